// pre_tc.cu -- tensor-core (tcgen05) pre forward for bf16 activations, and
// the library's device error word.
#include <cuda_runtime.h>
#include <stdint.h>

#include "launch.h"
#include "mhc_common.cuh"

namespace mhc {

// Latched by kernels whose bounded waits ran out; read and cleared by
// mhc_get_last_device_error().
__device__ unsigned g_device_error;

cudaError_t read_and_clear_device_error(unsigned* word, cudaStream_t s) {
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(word, g_device_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned));
}

bool pre_tc_supports(int64_t T, int64_t D) {
    (void)T;
    (void)D;
    return false;
}

cudaError_t launch_pre_tc(const void*, const float*, const float*, const float*, int64_t, int64_t,
                          int, float, void*, float*, float*, float*, float*, float*,
                          cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace mhc
