// pre_bwd_noalloc.cu -- mhc_pre_bwd for callers that cannot allocate device
// memory.
//
// mhc_pre_bwd asks its caller for scratch (per-token records and the dphi
// partials of each token block).  Some callers have no way to provide it: a
// custom-op or plugin interface that hands the op its tensors but no
// workspace, a runtime that plans all device memory ahead of time and forbids
// allocation once it runs, or a latency-bound loop where cudaMalloc's implicit
// device synchronisation is not acceptable.  This entry point takes its
// scratch from a fixed-size array in the library's own device memory instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it (MHC_PRE_BWD_NOALLOC_SCRATCH_BYTES) until the process
// exits.  In host code its name is only a host-side stand-in, never a device
// address: the device address is fetched with cudaGetSymbolAddress, with the
// device current, on the first call in each CUDA context, and passed to the
// kernels.  The cache is keyed by the context's unique id, so a context
// created later on the same device (after cudaDeviceReset, or a non-primary
// context) gets its own lookup.  A first call in a context made while its
// stream is being captured returns MHC_ERR_UNSUPPORTED instead of looking the
// address up.  All calls share the array and it keeps the last call's
// contents; every kernel here writes each scratch element before it reads it,
// so nothing needs clearing.  Calls that overlap on the GPU (for example on
// two streams of one device) race on the array.
#include <cuda.h>

#include <mutex>

#include "../../include/mhc.h"
#include "launch.h"

namespace mhc {

static __device__ __align__(256) unsigned char g_pre_bwd_scratch[MHC_PRE_BWD_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kLogits = 24;   // 2n + n^2 gate logits for n = 4
constexpr int kMaxContexts = 64;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

std::mutex g_setup_mutex;
struct Entry {
    unsigned long long ctx_id;
    void* ptr;
};
Entry g_cache[kMaxContexts];
int g_ncache = 0;

// Unique id of the calling thread's current context (0 if there is none or
// the driver entry points are unavailable).
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    if (get_current == nullptr || get_id == nullptr) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the scratch array in the current context, looked up on
// the first call in that context.  `status` is MHC_ERR_UNSUPPORTED when that
// first call comes while `stream` is capturing, MHC_ERR_CUDA when the context
// or the symbol cannot be resolved.
void* scratch_in_current_context(cudaStream_t stream, mhc_status* status) {
    unsigned long long id = current_context_id();
    if (id == 0) {
        // no context is current on this thread yet: make the current device's
        // primary context current (cudaSetDevice initialises it)
        int dev = -1;
        if (cudaGetDevice(&dev) == cudaSuccess && cudaSetDevice(dev) == cudaSuccess) id = current_context_id();
    }
    if (id == 0) {
        *status = MHC_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    for (int i = 0; i < g_ncache; ++i)
        if (g_cache[i].ctx_id == id) return g_cache[i].ptr;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        *status = MHC_ERR_CUDA;
        return nullptr;
    }
    if (cap != cudaStreamCaptureStatusNone) {
        *status = MHC_ERR_UNSUPPORTED;
        return nullptr;
    }
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_pre_bwd_scratch) != cudaSuccess || ptr == nullptr) {
        *status = MHC_ERR_CUDA;
        return nullptr;
    }
    if (g_ncache < kMaxContexts) g_cache[g_ncache++] = Entry{id, ptr};
    return ptr;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace mhc

extern "C" mhc_status mhc_pre_bwd_noalloc(mhc_dtype dt, const void* g_in, const float* dH_post,
                                          const float* dH_res, const void* x, const float* phi,
                                          const float* b, const float* alpha, const float* proj,
                                          const float* inv_rms, int64_t T, int n, int64_t D,
                                          int iters, void* dx, float* dphi, float* db,
                                          float* dalpha, cudaStream_t stream) {
    if (dt != MHC_F32 && dt != MHC_BF16) return MHC_ERR_INVALID_ARG;
    if (T < 0 || D <= 0) return MHC_ERR_INVALID_ARG;
    if (n != 4) return MHC_ERR_UNSUPPORTED;
    if (D % (dt == MHC_BF16 ? 8 : 4) != 0) return MHC_ERR_UNSUPPORTED;
    if (T > (int64_t(1) << 31) || D > (int64_t(1) << 24)) return MHC_ERR_UNSUPPORTED;
    if (iters < 1) return MHC_ERR_INVALID_ARG;
    if (iters > MHC_MAX_ITERS) return MHC_ERR_UNSUPPORTED;
    if (T == 0) {
        // the parameter gradients of an empty batch are zero
        const void* out[] = {dphi, db, dalpha};
        for (const void* p : out) {
            if (p == nullptr) return MHC_ERR_INVALID_ARG;
            if (!mhc::aligned16(p)) return MHC_ERR_MISALIGNED;
        }
        return mhc::zero_param_grads(D, dphi, db, dalpha, stream) == cudaSuccess ? MHC_OK : MHC_ERR_CUDA;
    }
    const void* ptrs[] = {g_in, dH_post, dH_res, x, phi, b, alpha, proj, inv_rms, dx, dphi, db, dalpha};
    for (const void* p : ptrs) {
        if (p == nullptr) return MHC_ERR_INVALID_ARG;
        if (!mhc::aligned16(p)) return MHC_ERR_MISALIGNED;
    }
    // Scratch plan: T per-token records, as many dphi token blocks as both the
    // usual plan and the fixed array allow (at least one), then the bf16 phi
    // blocks of the one-pass kernel.
    const size_t rec_bytes = static_cast<size_t>(T) * mhc::REC * sizeof(float);
    const size_t part_bytes = static_cast<size_t>(4 * D) * mhc::kLogits * sizeof(float);
    const size_t phi_bytes = mhc::pre_bwd_fused_phi_bytes(D);
    const size_t cap = MHC_PRE_BWD_NOALLOC_SCRATCH_BYTES;
    if (rec_bytes + part_bytes + phi_bytes > cap) return MHC_ERR_UNSUPPORTED;   // too large for the array
    int64_t nb = mhc::pre_bwd_plan(T, D).nb;
    const int64_t fit = static_cast<int64_t>((cap - rec_bytes - phi_bytes) / part_bytes);
    if (nb > fit) nb = fit;
    mhc_status st = MHC_OK;
    void* ws = mhc::scratch_in_current_context(stream, &st);
    if (ws == nullptr) return st;
    const cudaError_t e = mhc::launch_pre_bwd_blocks(dt == MHC_BF16, g_in, dH_post, dH_res, x, phi, b,
                                                     alpha, proj, inv_rms, T, D, iters, dx, dphi, db,
                                                     dalpha, ws, nb, stream);
    return e == cudaSuccess ? MHC_OK : MHC_ERR_CUDA;
}
