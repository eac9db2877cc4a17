// mhc_abi.cu -- the extern "C" entry points of libmhc_gb300.so.
//
// Host-side validation and dispatch only: every step of the layer runs in the
// kernels of kernels_fwd.cu, kernels_bwd.cu and pre_tc.cu.  Nothing here
// allocates memory or synchronises the host (mhc_get_last_device_error
// synchronises the given stream by contract).
#include <math.h>
#include <string.h>

#include "../../include/mhc.h"
#include "launch.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks shared by every entry point.  `ptrs` must all be non-null and
// 16-byte aligned when T > 0.
mhc_status check_common(mhc_dtype dt, int64_t T, int n, int64_t D, const void* const* ptrs,
                        int nptr) {
    if (dt != MHC_F32 && dt != MHC_BF16) return MHC_ERR_INVALID_ARG;
    if (T < 0 || D <= 0) return MHC_ERR_INVALID_ARG;
    if (n != 4) return MHC_ERR_UNSUPPORTED;
    const int64_t vec = dt == MHC_BF16 ? 8 : 4;
    if (D % vec != 0) return MHC_ERR_UNSUPPORTED;
    // keep every element index of x (T * n * D) far inside int64 and the
    // grid dimensions inside their limits
    if (T > (int64_t(1) << 31) || D > (int64_t(1) << 24)) return MHC_ERR_UNSUPPORTED;
    if (T == 0) return MHC_OK;
    for (int i = 0; i < nptr; ++i) {
        if (ptrs[i] == nullptr) return MHC_ERR_INVALID_ARG;
        if (!aligned16(ptrs[i])) return MHC_ERR_MISALIGNED;
    }
    return MHC_OK;
}

mhc_status check_iters(int iters) {
    if (iters < 1) return MHC_ERR_INVALID_ARG;
    if (iters > MHC_MAX_ITERS) return MHC_ERR_UNSUPPORTED;
    return MHC_OK;
}

mhc_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MHC_OK : MHC_ERR_CUDA; }

// The parameter gradients of an empty batch (T = 0): every other pointer may
// be null then, these three must be valid.
mhc_status empty_batch_param_grads(int64_t D, float* dphi, float* db, float* dalpha, cudaStream_t s) {
    if (dphi == nullptr || db == nullptr || dalpha == nullptr) return MHC_ERR_INVALID_ARG;
    if (!aligned16(dphi) || !aligned16(db) || !aligned16(dalpha)) return MHC_ERR_MISALIGNED;
    return from_cuda(mhc::zero_param_grads(D, dphi, db, dalpha, s));
}

}  // namespace

namespace mhc {
cudaError_t zero_param_grads(int64_t D, float* dphi, float* db, float* dalpha, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(dphi, 0, static_cast<size_t>(4 * D) * 24 * sizeof(float), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(db, 0, 24 * sizeof(float), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dalpha, 0, 3 * sizeof(float), s);
    return e;
}
}  // namespace mhc

namespace mhc {
// Defined in pre_tc.cu: the tensor-core pre forward (bf16).  Returns
// cudaErrorNotSupported when the shape is outside what it covers.
cudaError_t launch_pre_tc(const void* x, const float* phi, const float* b, const float* alpha,
                          int64_t T, int64_t D, int iters, float eps, void* x_in, float* H_pre,
                          float* H_post, float* H_res, float* proj, float* inv_rms,
                          cudaStream_t s);
bool pre_tc_supports(int64_t T, int64_t D);
cudaError_t read_and_clear_device_error(unsigned* word, cudaStream_t s);
cudaError_t set_force_timeout_pre(unsigned on);   // pre_tc.cu
cudaError_t set_force_timeout_bwd(unsigned on);   // pre_bwd_fused.cu
// Defined in post_pre_tc.cu: layer l's residual update fused with layer
// l + 1's pre forward (bf16).
bool post_pre_tc_supports(int64_t T, int64_t D);
size_t post_pre_tc_workspace_bytes(int64_t T);
cudaError_t launch_post_pre_tc(const void* x, const void* y, const float* H_post_l, const float* H_res_l,
                               const float* phi, const float* b, const float* alpha, int64_t T, int64_t D,
                               int iters, float eps, void* x_next, void* x_in, float* H_pre, float* H_post,
                               float* H_res, float* proj, float* inv_rms, void* workspace, cudaStream_t s);
}  // namespace mhc

extern "C" {

const char* mhc_status_string(mhc_status s) {
    switch (s) {
        case MHC_OK: return "MHC_OK";
        case MHC_ERR_INVALID_ARG: return "MHC_ERR_INVALID_ARG: null pointer, bad size, iters, eps or workspace";
        case MHC_ERR_UNSUPPORTED: return "MHC_ERR_UNSUPPORTED: n != 4, D not a multiple of the vector width, or iters too large";
        case MHC_ERR_MISALIGNED: return "MHC_ERR_MISALIGNED: a pointer is not 16-byte aligned";
        case MHC_ERR_CUDA: return "MHC_ERR_CUDA: a CUDA call or kernel launch failed";
        case MHC_ERR_TIMEOUT: return "MHC_ERR_TIMEOUT: a bounded device-side wait gave up";
    }
    return "MHC_ERR_UNKNOWN";
}

const char* mhc_version(void) { return "mhc_gb300 0.1.0 sm_103a"; }

mhc_status mhc_get_last_device_error(cudaStream_t stream) {
    unsigned word = 0;
    if (mhc::read_and_clear_device_error(&word, stream) != cudaSuccess) return MHC_ERR_CUDA;
    return word == 0 ? MHC_OK : MHC_ERR_TIMEOUT;
}

mhc_status mhc_test_force_timeout(int on) {
    const unsigned v = on ? 1u : 0u;
    if (mhc::set_force_timeout_pre(v) != cudaSuccess) return MHC_ERR_CUDA;
    return from_cuda(mhc::set_force_timeout_bwd(v));
}

mhc_status mhc_pre(mhc_dtype dt, const void* x, const float* phi, const float* b,
                   const float* alpha, int64_t T, int n, int64_t D, int iters, float eps,
                   void* x_in, float* H_pre, float* H_post, float* H_res, float* proj,
                   float* inv_rms, cudaStream_t stream) {
    const void* ptrs[] = {x, phi, b, alpha, x_in, H_pre, H_post, H_res, proj, inv_rms};
    mhc_status st = check_common(dt, T, n, D, ptrs, 10);
    if (st != MHC_OK) return st;
    if ((st = check_iters(iters)) != MHC_OK) return st;
    if (!(eps >= 0.0f) || !isfinite(eps)) return MHC_ERR_INVALID_ARG;
    if (T == 0) return MHC_OK;
    if (dt == MHC_BF16 && mhc::pre_tc_supports(T, D))
        return from_cuda(mhc::launch_pre_tc(x, phi, b, alpha, T, D, iters, eps, x_in, H_pre, H_post,
                                            H_res, proj, inv_rms, stream));
    return from_cuda(mhc::launch_pre_cc(dt == MHC_BF16, x, phi, b, alpha, T, D, iters, eps, x_in,
                                        H_pre, H_post, H_res, proj, inv_rms, stream));
}

mhc_status mhc_pre_gates(mhc_dtype dt, const void* x, const float* phi, const float* b,
                         const float* alpha, int64_t T, int n, int64_t D, int iters, float eps,
                         float* H_pre, float* H_post, float* H_res, float* proj, float* inv_rms,
                         cudaStream_t stream) {
    const void* ptrs[] = {x, phi, b, alpha, H_pre, H_post, H_res, proj, inv_rms};
    mhc_status st = check_common(dt, T, n, D, ptrs, 9);
    if (st != MHC_OK) return st;
    if ((st = check_iters(iters)) != MHC_OK) return st;
    if (!(eps >= 0.0f) || !isfinite(eps)) return MHC_ERR_INVALID_ARG;
    if (T == 0) return MHC_OK;
    // the forward kernels with no x_in buffer skip the mix
    if (dt == MHC_BF16 && mhc::pre_tc_supports(T, D))
        return from_cuda(mhc::launch_pre_tc(x, phi, b, alpha, T, D, iters, eps, nullptr, H_pre, H_post,
                                            H_res, proj, inv_rms, stream));
    return from_cuda(mhc::launch_pre_cc(dt == MHC_BF16, x, phi, b, alpha, T, D, iters, eps, nullptr,
                                        H_pre, H_post, H_res, proj, inv_rms, stream));
}

mhc_status mhc_pre_critical(mhc_dtype dt, const void* x, const float* phi, const float* b,
                            const float* alpha, int64_t T, int n, int64_t D, float eps, void* x_in,
                            float* H_pre, float* proj, float* inv_rms, cudaStream_t stream) {
    const void* ptrs[] = {x, phi, b, alpha, x_in, H_pre, proj, inv_rms};
    mhc_status st = check_common(dt, T, n, D, ptrs, 8);
    if (st != MHC_OK) return st;
    if (!(eps >= 0.0f) || !isfinite(eps)) return MHC_ERR_INVALID_ARG;
    if (T == 0) return MHC_OK;
    // the forward kernels with no H_post / H_res buffers skip Sinkhorn and
    // those gates (iters is then unused)
    if (dt == MHC_BF16 && mhc::pre_tc_supports(T, D))
        return from_cuda(mhc::launch_pre_tc(x, phi, b, alpha, T, D, 1, eps, x_in, H_pre, nullptr, nullptr, proj,
                                            inv_rms, stream));
    return from_cuda(mhc::launch_pre_cc(dt == MHC_BF16, x, phi, b, alpha, T, D, 1, eps, x_in, H_pre, nullptr,
                                        nullptr, proj, inv_rms, stream));
}

mhc_status mhc_post_res_gates(const float* proj, const float* b, const float* alpha, int64_t T, int n,
                              int iters, float* H_post, float* H_res, cudaStream_t stream) {
    if (T < 0) return MHC_ERR_INVALID_ARG;
    if (n != 4) return MHC_ERR_UNSUPPORTED;
    if (T > (int64_t(1) << 31)) return MHC_ERR_UNSUPPORTED;
    mhc_status st = check_iters(iters);
    if (st != MHC_OK) return st;
    if (T == 0) return MHC_OK;
    const void* ptrs[] = {proj, b, alpha, H_post, H_res};
    for (const void* p : ptrs) {
        if (p == nullptr) return MHC_ERR_INVALID_ARG;
        if (!aligned16(p)) return MHC_ERR_MISALIGNED;
    }
    return from_cuda(mhc::launch_post_res_gates(proj, b, alpha, T, iters, H_post, H_res, stream));
}

mhc_status mhc_post(mhc_dtype dt, const void* x, const void* y, const float* H_post,
                    const float* H_res, int64_t T, int n, int64_t D, void* x_next,
                    cudaStream_t stream) {
    const void* ptrs[] = {x, y, H_post, H_res, x_next};
    mhc_status st = check_common(dt, T, n, D, ptrs, 5);
    if (st != MHC_OK || T == 0) return st;
    return from_cuda(mhc::launch_post(dt == MHC_BF16, x, y, H_post, H_res, T, D, x_next, stream));
}

mhc_status mhc_post_norm(mhc_dtype dt, const void* x, const void* y, const float* H_post,
                         const float* H_res, int flags, float eps, int64_t T, int n, int64_t D,
                         void* x_next, float* inv_rms_y, float* inv_rms_out, cudaStream_t stream) {
    const void* ptrs[] = {x, y, H_post, H_res, x_next, inv_rms_y, inv_rms_out};
    mhc_status st = check_common(dt, T, n, D, ptrs, 7);
    if (st != MHC_OK) return st;
    if (flags < 0 || flags > (MHC_POST_SANDWICH_NORM | MHC_POST_BLOCK_NORM)) return MHC_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || !isfinite(eps)) return MHC_ERR_INVALID_ARG;
    if (!mhc::post_norm_supports(dt == MHC_BF16, D)) return MHC_ERR_UNSUPPORTED;
    if (T == 0) return MHC_OK;
    return from_cuda(mhc::launch_post_norm(dt == MHC_BF16, x, y, H_post, H_res, flags, eps, T, D, x_next,
                                           inv_rms_y, inv_rms_out, stream));
}

mhc_status mhc_post_norm_bwd(mhc_dtype dt, const void* g_next, const void* x, const void* y,
                             const float* H_post, const float* H_res, int flags, float eps,
                             const float* inv_rms_y, const float* inv_rms_out, int64_t T, int n,
                             int64_t D, void* dx, void* dy, float* dH_post, float* dH_res,
                             cudaStream_t stream) {
    const void* ptrs[] = {g_next, x, y, H_post, H_res, inv_rms_y, inv_rms_out, dx, dy, dH_post, dH_res};
    mhc_status st = check_common(dt, T, n, D, ptrs, 11);
    if (st != MHC_OK) return st;
    if (flags < 0 || flags > (MHC_POST_SANDWICH_NORM | MHC_POST_BLOCK_NORM)) return MHC_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || !isfinite(eps)) return MHC_ERR_INVALID_ARG;
    if (!mhc::post_norm_supports(dt == MHC_BF16, D)) return MHC_ERR_UNSUPPORTED;
    if (T == 0) return MHC_OK;
    return from_cuda(mhc::launch_post_norm_bwd(dt == MHC_BF16, g_next, x, y, H_post, H_res, flags, eps, inv_rms_y,
                                               inv_rms_out, T, D, dx, dy, dH_post, dH_res, stream));
}

mhc_status mhc_post_bwd(mhc_dtype dt, const void* g_next, const void* x, const void* y,
                        const float* H_post, const float* H_res, int64_t T, int n, int64_t D,
                        void* dx, void* dy, float* dH_post, float* dH_res, cudaStream_t stream) {
    const void* ptrs[] = {g_next, x, y, H_post, H_res, dx, dy, dH_post, dH_res};
    mhc_status st = check_common(dt, T, n, D, ptrs, 9);
    if (st != MHC_OK || T == 0) return st;
    return from_cuda(mhc::launch_post_bwd(dt == MHC_BF16, g_next, x, y, H_post, H_res, T, D, dx, dy,
                                          dH_post, dH_res, stream));
}

size_t mhc_post_pre_workspace_bytes(mhc_dtype dt, int64_t T, int n, int64_t D) {
    const void* none[] = {nullptr};
    if (T <= 0 || check_common(dt, T, n, D, none, 0) != MHC_OK) return 0;
    if (dt == MHC_BF16 && mhc::post_pre_tc_supports(T, D)) return mhc::post_pre_tc_workspace_bytes(T);
    return 0;
}

mhc_status mhc_post_pre(mhc_dtype dt, const void* x, const void* y, const float* H_post_l,
                        const float* H_res_l, const float* phi, const float* b, const float* alpha,
                        int64_t T, int n, int64_t D, int iters, float eps, void* x_next, void* x_in,
                        float* H_pre, float* H_post, float* H_res, float* proj, float* inv_rms,
                        void* workspace, size_t ws_bytes, cudaStream_t stream) {
    const void* ptrs[] = {x, y, H_post_l, H_res_l, phi, b, alpha, x_next, x_in,
                          H_pre, H_post, H_res, proj, inv_rms};
    mhc_status st = check_common(dt, T, n, D, ptrs, 14);
    if (st != MHC_OK) return st;
    if ((st = check_iters(iters)) != MHC_OK) return st;
    if (!(eps >= 0.0f) || !isfinite(eps)) return MHC_ERR_INVALID_ARG;
    if (T == 0) return MHC_OK;
    const size_t need = mhc_post_pre_workspace_bytes(dt, T, n, D);
    if (need > 0) {
        if (workspace == nullptr || ws_bytes < need) return MHC_ERR_INVALID_ARG;
        if (!aligned16(workspace)) return MHC_ERR_MISALIGNED;
        return from_cuda(mhc::launch_post_pre_tc(x, y, H_post_l, H_res_l, phi, b, alpha, T, D, iters, eps,
                                                 x_next, x_in, H_pre, H_post, H_res, proj, inv_rms, workspace,
                                                 stream));
    }
    // other shapes: the two steps one after the other, on the stored x_next
    st = from_cuda(mhc::launch_post(dt == MHC_BF16, x, y, H_post_l, H_res_l, T, D, x_next, stream));
    if (st != MHC_OK) return st;
    return mhc_pre(dt, x_next, phi, b, alpha, T, n, D, iters, eps, x_in, H_pre, H_post, H_res, proj,
                   inv_rms, stream);
}

int mhc_kernel_launches(const char* op, mhc_dtype dt, int64_t T, int n, int64_t D) {
    if (op == nullptr) return -1;
    const void* none[] = {nullptr};
    if (check_common(dt, T, n, D, none, 0) != MHC_OK) return -1;
    if (T == 0) return 0;
    if (strcmp(op, "mhc_pre") == 0)
        return dt == MHC_BF16 && mhc::pre_tc_supports(T, D) ? 1 : 2;
    if (strcmp(op, "mhc_post") == 0 || strcmp(op, "mhc_post_bwd") == 0) return 1;
    if (strcmp(op, "mhc_post_norm") == 0 || strcmp(op, "mhc_post_norm_bwd") == 0)
        return mhc::post_norm_supports(dt == MHC_BF16, D) ? 1 : -1;
    if (strcmp(op, "mhc_post_pre") == 0) {
        if (dt == MHC_BF16 && mhc::post_pre_tc_supports(T, D)) return 2;
        return 1 + (dt == MHC_BF16 && mhc::pre_tc_supports(T, D) ? 1 : 2);
    }
    if (strcmp(op, "mhc_pre_bwd") == 0) return 5;   // both paths: 5 launches
    if (strcmp(op, "mhc_pre_gates") == 0) return 1;   // no mix: one kernel on either path
    if (strcmp(op, "mhc_pre_critical") == 0) return dt == MHC_BF16 && mhc::pre_tc_supports(T, D) ? 1 : 2;
    if (strcmp(op, "mhc_post_res_gates") == 0) return 1;
    if (strcmp(op, "mhc_layer_bwd_recompute") == 0) return 1 + 1 + 5;
    return -1;
}

size_t mhc_pre_bwd_workspace_bytes(mhc_dtype dt, int64_t T, int n, int64_t D) {
    (void)dt;
    if (T <= 0 || n != 4 || D <= 0) return 0;
    return mhc::pre_bwd_plan(T, D).total_bytes;
}

mhc_status mhc_pre_bwd(mhc_dtype dt, const void* g_in, const float* dH_post, const float* dH_res,
                       const void* x, const float* phi, const float* b, const float* alpha,
                       const float* proj, const float* inv_rms, int64_t T, int n, int64_t D,
                       int iters, void* dx, float* dphi, float* db, float* dalpha,
                       void* workspace, size_t ws_bytes, cudaStream_t stream) {
    const void* ptrs[] = {g_in, dH_post, dH_res, x, phi, b, alpha, proj, inv_rms,
                          dx, dphi, db, dalpha, workspace};
    mhc_status st = check_common(dt, T, n, D, ptrs, 14);
    if (st != MHC_OK) return st;
    if ((st = check_iters(iters)) != MHC_OK) return st;
    if (T == 0) return empty_batch_param_grads(D, dphi, db, dalpha, stream);
    if (ws_bytes < mhc::pre_bwd_plan(T, D).total_bytes) return MHC_ERR_INVALID_ARG;
    return from_cuda(mhc::launch_pre_bwd(dt == MHC_BF16, g_in, dH_post, dH_res, x, phi, b, alpha,
                                         proj, inv_rms, T, D, iters, dx, dphi, db, dalpha,
                                         workspace, stream));
}

}  // extern "C"

namespace {

// Scratch of mhc_layer_bwd_recompute: the recomputed gates and saved state,
// the gate gradients, then mhc_pre_bwd's own scratch; 256-byte regions.
struct RecomputeLayout {
    size_t H_pre, H_post, H_res, proj, inv_rms, dH_post, dH_res, bwd, total;
};

RecomputeLayout recompute_layout(int64_t T, int64_t D) {
    auto r = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
    const size_t t = static_cast<size_t>(T);
    RecomputeLayout L;
    size_t o = 0;
    L.H_pre = o;   o += r(t * 16);
    L.H_post = o;  o += r(t * 16);
    L.H_res = o;   o += r(t * 64);
    L.proj = o;    o += r(t * 96);
    L.inv_rms = o; o += r(t * 4);
    L.dH_post = o; o += r(t * 16);
    L.dH_res = o;  o += r(t * 64);
    L.bwd = o;     o += mhc::pre_bwd_plan(T, D).total_bytes;
    L.total = o;
    return L;
}

}  // namespace

extern "C" {

size_t mhc_layer_bwd_recompute_workspace_bytes(mhc_dtype dt, int64_t T, int n, int64_t D) {
    const void* none[] = {nullptr};
    if (T <= 0 || check_common(dt, T, n, D, none, 0) != MHC_OK) return 0;
    return recompute_layout(T, D).total;
}

mhc_status mhc_layer_bwd_recompute(mhc_dtype dt, const void* g_in, const void* g_next, const void* x,
                                   const void* y, const float* phi, const float* b, const float* alpha,
                                   int64_t T, int n, int64_t D, int iters, float eps, void* dx, void* dy,
                                   float* dphi, float* db, float* dalpha, void* workspace, size_t ws_bytes,
                                   cudaStream_t stream) {
    const void* ptrs[] = {g_in, g_next, x, y, phi, b, alpha, dx, dy, dphi, db, dalpha, workspace};
    mhc_status st = check_common(dt, T, n, D, ptrs, 13);
    if (st != MHC_OK) return st;
    if ((st = check_iters(iters)) != MHC_OK) return st;
    if (!(eps >= 0.0f) || !isfinite(eps)) return MHC_ERR_INVALID_ARG;
    if (T == 0) return empty_batch_param_grads(D, dphi, db, dalpha, stream);
    const RecomputeLayout L = recompute_layout(T, D);
    if (ws_bytes < L.total) return MHC_ERR_INVALID_ARG;
    unsigned char* w = static_cast<unsigned char*>(workspace);
    float* H_pre = reinterpret_cast<float*>(w + L.H_pre);
    float* H_post = reinterpret_cast<float*>(w + L.H_post);
    float* H_res = reinterpret_cast<float*>(w + L.H_res);
    float* proj = reinterpret_cast<float*>(w + L.proj);
    float* inv_rms = reinterpret_cast<float*>(w + L.inv_rms);
    float* dH_post = reinterpret_cast<float*>(w + L.dH_post);
    float* dH_res = reinterpret_cast<float*>(w + L.dH_res);
    st = mhc_pre_gates(dt, x, phi, b, alpha, T, n, D, iters, eps, H_pre, H_post, H_res, proj, inv_rms, stream);
    if (st != MHC_OK) return st;
    st = mhc_post_bwd(dt, g_next, x, y, H_post, H_res, T, n, D, dx, dy, dH_post, dH_res, stream);
    if (st != MHC_OK) return st;
    return mhc_pre_bwd(dt, g_in, dH_post, dH_res, x, phi, b, alpha, proj, inv_rms, T, n, D, iters, dx, dphi,
                       db, dalpha, w + L.bwd, ws_bytes - L.bwd, stream);
}

}  // extern "C"
