// launch.h -- host-side launchers shared between the ABI layer and the kernel
// translation units (internal to libmhc_gb300.so, C++ linkage).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mhc {

// Record per token written by the pre backward's per-token kernel (floats).
constexpr int REC = 64;
constexpr int REC_U = 0;        // [0, 24)  u = inv_rms * alpha_grp * dlogits
constexpr int REC_HPRE = 24;    // [24, 28) H_pre
constexpr int REC_COEF = 28;    // 28       coefficient of x in the RMSNorm backward
constexpr int REC_DL = 32;      // [32, 56) dlogits
constexpr int REC_DA = 56;      // [56, 59) per-token dalpha terms
constexpr int REC_DHPRE = 60;   // [60, 64) dH_pre (input of the per-token kernel), then
constexpr int REC_DSIG = 60;    //          s_i (1 - s_i) of the pre gates (its output)
constexpr int REC_S = 29;       // 29       inv_rms

// Sizes of the pre backward's dphi partial reduction.
struct PreBwdPlan {
    int64_t nb;          // token blocks (dphi partials)
    int64_t tb;          // tokens per block
    size_t rec_bytes;    // T * REC floats
    size_t part_bytes;   // nb * K * NG floats
    size_t phi_bytes;    // bf16 phi blocks of the one-pass kernel
    size_t total_bytes;
};
PreBwdPlan pre_bwd_plan(int64_t T, int64_t D);

// The gradients of phi [4D, 24], b [24] and alpha [3] of an empty batch: sums
// over no tokens, so zero.  Writes them with three memsets on `s`.
cudaError_t zero_param_grads(int64_t D, float* dphi, float* db, float* dalpha, cudaStream_t s);

// Forward (CUDA-core path: projection + gates, then the H_pre mix; no mix
// when x_in is null).
cudaError_t launch_pre_cc(bool bf16, const void* x, const float* phi, const float* b,
                          const float* alpha, int64_t T, int64_t D, int iters, float eps,
                          void* x_in, float* H_pre, float* H_post, float* H_res,
                          float* proj, float* inv_rms, cudaStream_t s);

// H_post and H_res from a saved projection (the side of the inference
// critical-path split).
cudaError_t launch_post_res_gates(const float* proj, const float* b, const float* alpha, int64_t T, int iters,
                                  float* H_post, float* H_res, cudaStream_t s);

cudaError_t launch_post(bool bf16, const void* x, const void* y, const float* H_post,
                        const float* H_res, int64_t T, int64_t D, void* x_next,
                        cudaStream_t s);

// The residual update with openPangu's stability changes (post_norm.cu).
bool post_norm_supports(bool bf16, int64_t D);
cudaError_t launch_post_norm(bool bf16, const void* x, const void* y, const float* H_post, const float* H_res,
                             int flags, float eps, int64_t T, int64_t D, void* x_next, float* inv_rms_y,
                             float* inv_rms_out, cudaStream_t s);
cudaError_t launch_post_norm_bwd(bool bf16, const void* g_next, const void* x, const void* y, const float* H_post,
                                 const float* H_res, int flags, float eps, const float* inv_rms_y,
                                 const float* inv_rms_out, int64_t T, int64_t D, void* dx, void* dy,
                                 float* dH_post, float* dH_res, cudaStream_t s);

cudaError_t launch_post_bwd(bool bf16, const void* g, const void* x, const void* y,
                            const float* H_post, const float* H_res, int64_t T, int64_t D,
                            void* dx, void* dy, float* dH_post, float* dH_res,
                            cudaStream_t s);

cudaError_t launch_pre_bwd(bool bf16, const void* g_in, const float* dH_post,
                           const float* dH_res, const void* x, const float* phi,
                           const float* b, const float* alpha, const float* proj,
                           const float* inv_rms, int64_t T, int64_t D, int iters, void* dx,
                           float* dphi, float* db, float* dalpha, void* ws,
                           cudaStream_t s);

cudaError_t launch_pre_bwd_blocks(bool bf16, const void* g_in, const float* dH_post,
                                  const float* dH_res, const void* x, const float* phi,
                                  const float* b, const float* alpha, const float* proj,
                                  const float* inv_rms, int64_t T, int64_t D, int iters, void* dx,
                                  float* dphi, float* db, float* dalpha, void* ws, int64_t nb,
                                  cudaStream_t s);

// One-pass cluster kernel of the pre backward (bf16; pre_bwd_fused.cu): the
// dH_pre dots, the rest of u and the RMSNorm coefficient, dx and the dphi
// partials (one per cluster, at most `max_parts`).  It expects records from
// the per-token kernel run without dH_pre and writes their pre-gate parts.
// It first packs phi as bf16 pair blocks into `phi2` (pre_bwd_fused_phi_bytes).
bool pre_bwd_fused_supports(int64_t T, int64_t D);
size_t pre_bwd_fused_phi_bytes(int64_t D);
// bf16 phi blocks of the one-pass kernel, packed into the workspace.
cudaError_t launch_pre_bwd_phi_pack(const float* phi, int64_t D, void* phi2, cudaStream_t s);
cudaError_t launch_pre_bwd_fused_main(const void* g_in, const void* x, const float* phi,
                                      const float* proj, const float* alpha, float* rec,
                                      int64_t T, int64_t D, int64_t max_parts, void* dx,
                                      float* part, void* phi2, int64_t* nparts, cudaStream_t s);

// Tensor-core main step of the pre backward (bf16; pre_bwd_tc.cu).
bool pre_bwd_tc_supports(int64_t T, int64_t D);
cudaError_t launch_pre_bwd_tc_main(const void* g_in, const void* x, const float* phi, const float* rec,
                                   int64_t T, int64_t D, int64_t nb, void* dx, float* part,
                                   cudaStream_t s);

}  // namespace mhc
