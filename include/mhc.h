/*
 * mhc.h -- C ABI of the GB300 (sm_103a) mHC layer library (libmhc_gb300.so).
 *
 * The layer is the manifold-constrained hyper-connection of the "openPangu 2.0
 * -- architecture, training and Ascend systems" analysis notes, section 5.3:
 * for each token t with n residual streams x[t] in R^{n x D}, K = n*D,
 *
 *   x_bar  = RMSNorm(x[t])                 (flattened n*D row, unit weight)
 *   proj   = x_bar . phi                   (phi in R^{K x G}, G = 2n + n^2)
 *   logits = alpha_group * proj + b        (groups pre | post | res)
 *   H_pre  = sigmoid(logits[0:n])          in (0, 1)
 *   H_post = 2 sigmoid(logits[n:2n])       in (0, 2)
 *   H_res  = Sinkhorn(exp(reshape(logits[2n:], n, n)))   doubly stochastic
 *   x_in   = sum_i H_pre[i] x[t, i]                          (mhc_pre)
 *   x_next[i] = sum_j H_res[i, j] x[t, j] + H_post[i] y[t]   (mhc_post)
 *
 * The ranges of the gates and the doubly stochastic H_res (non-negative, rows
 * and columns summing to 1) are those of the Ascend mHC Triton operator
 * article (paragraph defining H^res / H^pre / H^post).  One Sinkhorn round
 * normalises the rows, then the columns; H_res[i][j] is logit 2n + i*n + j.
 *
 * Conventions shared by every entry point:
 *   - All pointers are device pointers owned by the caller.  The library
 *     allocates no memory; scratch space is passed in (mhc_pre_bwd).
 *   - Tensors are dense, row-major, with the shapes given per argument.
 *     Activations (x, y, x_in, x_next, g_in, g_next, dx, dy) have type `dt`;
 *     gates, phi, b, alpha, saved state and parameter gradients are float32.
 *   - Every pointer must be 16-byte aligned.  n must be 4.  D must be a
 *     multiple of 8 (bf16) or 4 (float32).  T = 0 launches no kernel; the
 *     backward entry points then write zero parameter gradients (below).
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) and
 *     never synchronise the host.  A bad argument returns an error before
 *     anything is launched; a failed launch returns MHC_ERR_CUDA.  Errors that
 *     only the device can see (a bounded wait that ran out) are latched in a
 *     device word and reported by mhc_get_last_device_error().
 *   - Results are deterministic: no floating-point atomics.
 */
#ifndef MHC_GB300_H
#define MHC_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MHC_OK = 0,
    MHC_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad iters/eps, short workspace */
    MHC_ERR_UNSUPPORTED = 2,  /* n != 4, D not a multiple of the vector width, iters > MHC_MAX_ITERS */
    MHC_ERR_MISALIGNED = 3,   /* a pointer is not 16-byte aligned */
    MHC_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
    MHC_ERR_TIMEOUT = 5       /* a bounded device-side wait gave up (see mhc_get_last_device_error) */
} mhc_status;

typedef enum { MHC_F32 = 0, MHC_BF16 = 1 } mhc_dtype;

/* Largest Sinkhorn round count the kernels accept (the backward keeps the
 * per-round normalisers of one token in registers / local memory). */
#define MHC_MAX_ITERS 64

/* Human-readable name of a status code (static string, never NULL). */
const char* mhc_status_string(mhc_status s);

/* Library version string, e.g. "mhc_gb300 0.1.0 sm_103a". */
const char* mhc_version(void);

/* Synchronises `stream`, then reads and clears the library's device error
 * word on the current device.  Returns MHC_OK if no kernel latched an error,
 * MHC_ERR_TIMEOUT if a bounded wait ran out, MHC_ERR_CUDA if the
 * synchronisation itself failed. */
mhc_status mhc_get_last_device_error(cudaStream_t stream);

/*
 * mhc_pre -- forward of the read side (steps RMSNorm, projection, gates,
 * Sinkhorn and the H_pre mix of section 5.3 of the openPangu 2.0 notes).
 *
 *   x       [T, n, D]  dt      the n-stream residual state
 *   phi     [n*D, G]   float   projection W_mHC (row k = i*D + d)
 *   b       [G]        float   logit bias
 *   alpha   [3]        float   logit scales of the pre, post and res groups
 *   iters              int     Sinkhorn rounds, 1 .. MHC_MAX_ITERS
 *   eps                float   RMSNorm epsilon (>= 0, inside the sqrt)
 * outputs (written):
 *   x_in    [T, D]     dt      sum_i H_pre[i] x[i]  (fp32 sum, one rounding)
 *   H_pre   [T, n]     float
 *   H_post  [T, n]     float
 *   H_res   [T, n, n]  float
 *   proj    [T, G]     float   x_bar . phi (saved for mhc_pre_bwd)
 *   inv_rms [T]        float   1/sqrt(mean(x^2) + eps) (saved for mhc_pre_bwd)
 */
mhc_status mhc_pre(mhc_dtype dt, const void* x, const float* phi,
                   const float* b, const float* alpha, int64_t T, int n,
                   int64_t D, int iters, float eps, void* x_in, float* H_pre,
                   float* H_post, float* H_res, float* proj, float* inv_rms,
                   cudaStream_t stream);

/*
 * mhc_post -- forward of the write side (residual update of section 5.3):
 *   x_next[t, i] = sum_j H_res[t, i, j] x[t, j] + H_post[t, i] y[t]
 *
 *   x [T, n, D] dt; y [T, D] dt; H_post [T, n] float; H_res [T, n, n] float
 *   x_next [T, n, D] dt (written; must not alias x or y)
 */
mhc_status mhc_post(mhc_dtype dt, const void* x, const void* y,
                    const float* H_post, const float* H_res, int64_t T, int n,
                    int64_t D, void* x_next, cudaStream_t stream);

/*
 * mhc_post_norm -- the residual update with openPangu's stability changes
 * (section 5.4 of the openPangu 2.0 notes), each selected by a bit of `flags`:
 *   MHC_POST_SANDWICH_NORM  y' = y r_y, r_y = 1/sqrt(mean_D(y^2) + eps): the
 *                           sublayer output normalised before the H_post
 *                           write-back ("sandwich normalisation");
 *   MHC_POST_BLOCK_NORM     x_next = z s, z = H_res x + H_post y',
 *                           s = 1/sqrt(mean_{n*D}(z^2) + eps): the updated
 *                           multi-stream state normalised ("block-level
 *                           post-normalisation"; the pages apply it after
 *                           the first layer and every fifth one).
 * Unit weights; eps inside the square root.  flags = 0 is mhc_post.
 *
 *   x [T, n, D] dt; y [T, D] dt; H_post [T, n], H_res [T, n, n] float
 * outputs (written): x_next [T, n, D] dt; inv_rms_y [T], inv_rms_out [T]
 *   float (r_y and s, 1 where the step is off; saved for the backward).
 * MHC_ERR_INVALID_ARG for flags outside 0..3; MHC_ERR_UNSUPPORTED when D is
 * above 8192 (bf16) or 4096 (float32).
 */
#define MHC_POST_SANDWICH_NORM 1
#define MHC_POST_BLOCK_NORM 2
mhc_status mhc_post_norm(mhc_dtype dt, const void* x, const void* y,
                         const float* H_post, const float* H_res, int flags,
                         float eps, int64_t T, int n, int64_t D, void* x_next,
                         float* inv_rms_y, float* inv_rms_out, cudaStream_t stream);

/*
 * mhc_post_norm_bwd -- gradients of <g_next, x_next> for mhc_post_norm with
 * the same flags, eps and the saved inv_rms_y, inv_rms_out:
 *   dx, dy written (not added); dH_post [T, n], dH_res [T, n, n] written.
 */
mhc_status mhc_post_norm_bwd(mhc_dtype dt, const void* g_next, const void* x,
                             const void* y, const float* H_post,
                             const float* H_res, int flags, float eps,
                             const float* inv_rms_y, const float* inv_rms_out,
                             int64_t T, int n, int64_t D, void* dx, void* dy,
                             float* dH_post, float* dH_res, cudaStream_t stream);

/*
 * mhc_post_pre -- mhc_post of layer l followed by mhc_pre of layer l + 1 on
 * the x_next it stores, in one pass over x and y where the shape allows (the
 * cross-layer fusion of the inference critical path, section 11.3 of the
 * openPangu 2.0 notes; each step as in section 5.3):
 *   x_next = mhc_post(x, y, H_post_l, H_res_l)                (stored in dt)
 *   (x_in, H_pre, H_post, H_res, proj, inv_rms) = mhc_pre(x_next, phi, b, alpha)
 *
 *   x [T, n, D] dt; y [T, D] dt; H_post_l [T, n], H_res_l [T, n, n] float
 *     (layer l's gates); phi, b, alpha, iters, eps: layer l + 1, as mhc_pre
 * outputs (written; none may alias an input):
 *   x_next [T, n, D] dt   bit-identical to mhc_post's
 *   x_in, H_pre, H_post, H_res, proj, inv_rms   as mhc_pre on the stored x_next
 *   workspace  device scratch of at least mhc_post_pre_workspace_bytes() bytes,
 *              16-byte aligned (NULL when that is 0); ws_bytes its size
 * bf16 shapes the fused kernel covers take two kernels that run at once: the
 * fused pass, and the x_in mix on the SMs the fused pass leaves free (it
 * reads each token tile once the fused pass has counted it done in the
 * workspace).  Every other shape runs mhc_post, then mhc_pre.  Errors as
 * mhc_pre; MHC_ERR_INVALID_ARG for a missing or short workspace.
 */
mhc_status mhc_post_pre(mhc_dtype dt, const void* x, const void* y,
                        const float* H_post_l, const float* H_res_l,
                        const float* phi, const float* b, const float* alpha,
                        int64_t T, int n, int64_t D, int iters, float eps,
                        void* x_next, void* x_in, float* H_pre, float* H_post,
                        float* H_res, float* proj, float* inv_rms,
                        void* workspace, size_t ws_bytes, cudaStream_t stream);

/* Bytes of scratch mhc_post_pre needs for these sizes (0: none). */
size_t mhc_post_pre_workspace_bytes(mhc_dtype dt, int64_t T, int n, int64_t D);

/*
 * mhc_post_bwd -- gradients of <g_next, x_next> for mhc_post:
 *   dx[t, j]      = sum_i H_res[t, i, j] g_next[t, i]     (written, not added)
 *   dy[t]         = sum_i H_post[t, i] g_next[t, i]
 *   dH_post[t, i] = <g_next[t, i], y[t]>
 *   dH_res[t,i,j] = <g_next[t, i], x[t, j]>
 *
 *   g_next, x, dx [T, n, D] dt; y, dy [T, D] dt;
 *   H_post, dH_post [T, n] float; H_res, dH_res [T, n, n] float
 */
mhc_status mhc_post_bwd(mhc_dtype dt, const void* g_next, const void* x,
                        const void* y, const float* H_post, const float* H_res,
                        int64_t T, int n, int64_t D, void* dx, void* dy,
                        float* dH_post, float* dH_res, cudaStream_t stream);

/*
 * mhc_test_force_timeout -- test hook of the failure path, off by default.
 * While on (nonzero), every launch of the bf16 forward kernels (the
 * tensor-core kernel and the small-batch cluster kernel of mhc_pre,
 * mhc_pre_gates and mhc_pre_critical) and of the pre backward's one-pass
 * cluster kernel (mhc_pre_bwd) makes thread 0 of each CTA wait on an mbarrier
 * that nothing arrives on; the wait gives up after about 100 us, the kernel
 * latches its device error word and returns before starting any copy or
 * tensor-memory allocation, leaving its outputs unwritten.  The next
 * mhc_get_last_device_error() then reports MHC_ERR_TIMEOUT, and the context
 * stays usable.  Synchronous for the backward (it writes a device flag); the
 * forward kernels take the setting as a launch parameter.  Applies to the
 * current device.  Not for production use.
 */
mhc_status mhc_test_force_timeout(int on);

/* Number of kernels the entry point `op` ("mhc_pre", "mhc_pre_gates",
 * "mhc_pre_critical", "mhc_post_res_gates",
 * "mhc_post", "mhc_post_norm", "mhc_post_norm_bwd", "mhc_post_pre",
 * "mhc_post_bwd", "mhc_pre_bwd" or "mhc_layer_bwd_recompute") launches for these sizes; -1 for an
 * unknown op or sizes the entry point would reject.  Useful when sizing CUDA
 * graphs or counting launches. */
int mhc_kernel_launches(const char* op, mhc_dtype dt, int64_t T, int n, int64_t D);

/* Bytes of scratch mhc_pre_bwd needs for these sizes (0 for T = 0). */
size_t mhc_pre_bwd_workspace_bytes(mhc_dtype dt, int64_t T, int n, int64_t D);

/*
 * mhc_pre_bwd -- backward of mhc_pre given the gradient of x_in and the
 * gradients of H_post and H_res (as produced by mhc_post_bwd).  The
 * Sinkhorn forward is recomputed from `proj`; its derivative is the exact
 * reverse mode of the unrolled `iters`-round map.
 *
 *   g_in    [T, D]     dt      dL/dx_in
 *   dH_post [T, n]     float   dL/dH_post
 *   dH_res  [T, n, n]  float   dL/dH_res
 *   x, phi, b, alpha, iters        as passed to mhc_pre
 *   proj, inv_rms      float   as written by mhc_pre
 * outputs:
 *   dx      [T, n, D]  dt      ACCUMULATED: dx += pre-side gradient (the
 *                              H_pre mix plus the projection / RMSNorm path),
 *                              so that after mhc_post_bwd it holds dL/dx
 *   dphi    [n*D, G]   float   written
 *   db      [G]        float   written
 *   dalpha  [3]        float   written
 *   workspace, ws_bytes        device scratch of at least
 *                              mhc_pre_bwd_workspace_bytes() bytes
 *
 * Data parallelism: dphi, db and dalpha are sums over this call's tokens, so
 * ranks that each hold a slice of the batch add them (one all-reduce) to get
 * the full-batch gradient; every other output is per token.  For T = 0 the
 * call writes zero parameter gradients (dphi, db and dalpha, the sums over no
 * tokens, with memsets on `stream`), so a rank with no tokens contributes
 * zero to that sum; the per-token pointers may then be null, dphi, db and
 * dalpha may not.
 */
mhc_status mhc_pre_bwd(mhc_dtype dt, const void* g_in, const float* dH_post,
                       const float* dH_res, const void* x, const float* phi,
                       const float* b, const float* alpha, const float* proj,
                       const float* inv_rms, int64_t T, int n, int64_t D,
                       int iters, void* dx, float* dphi, float* db,
                       float* dalpha, void* workspace, size_t ws_bytes,
                       cudaStream_t stream);

/* Size of the fixed device scratch array behind mhc_pre_bwd_noalloc. */
#define MHC_PRE_BWD_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * mhc_pre_bwd_noalloc -- mhc_pre_bwd for callers that cannot allocate device
 * memory.  (The pages have no counterpart: this is a packaging variant.)
 *
 * mhc_pre_bwd needs caller-provided scratch.  Some callers cannot provide
 * it: a custom-op or plugin interface that hands an op its tensors but no
 * workspace, a runtime that plans every device allocation up front and
 * forbids allocating once it runs, or a latency-bound loop that cannot afford
 * cudaMalloc's implicit device synchronisation.  This entry point takes its
 * scratch from a fixed array inside the library's device memory instead and
 * calls no allocating routine.
 *
 * Arguments and results are those of mhc_pre_bwd without the workspace.
 * Limits and behaviour:
 *   - The array holds MHC_PRE_BWD_NOALLOC_SCRATCH_BYTES (16 MiB) on every GPU
 *     that loads the library, until the process exits.  The call returns
 *     MHC_ERR_UNSUPPORTED when T * 256 bytes of per-token records, one
 *     4*D x 24 float32 partial of dphi and D * 256 bytes of bf16 phi blocks
 *     exceed it (for D = 5120: T <= 52,736).
 *   - The first call in each CUDA context looks up the array's device address
 *     in that context (cudaGetSymbolAddress) and keeps it for that context;
 *     a context created later (for example after cudaDeviceReset) gets a
 *     lookup of its own.  That first call must not come while `stream` is
 *     being captured: it then returns MHC_ERR_UNSUPPORTED and does nothing.
 *   - All calls share the array; calls that overlap on the GPU race on it.
 *     Every element is written before it is read, so no state carries over
 *     from one call to the next.
 *   - T = 0 writes zero parameter gradients, as mhc_pre_bwd.
 */
mhc_status mhc_pre_bwd_noalloc(mhc_dtype dt, const void* g_in, const float* dH_post,
                               const float* dH_res, const void* x, const float* phi,
                               const float* b, const float* alpha, const float* proj,
                               const float* inv_rms, int64_t T, int n, int64_t D, int iters,
                               void* dx, float* dphi, float* db, float* dalpha,
                               cudaStream_t stream);

/*
 * The inference critical-path split.  The openPangu 2.0 notes (section 11.3,
 * the inference system) put the previous layer's merge, the RMSNorm and H^pre
 * on the critical path that feeds the sublayer, and move H^post and H^res
 * (with Sinkhorn) to a low-priority side stream that overlaps the sublayer.
 * The two calls below are that split: mhc_pre_critical writes what the
 * sublayer needs (x_in) and the saved state; mhc_post_res_gates computes
 * H^post and H^res from the saved projection and may run on another stream,
 * ordered after mhc_pre_critical by an event.  Together they write the same
 * values as mhc_pre, bit for bit.
 */

/*
 * mhc_pre_critical -- mhc_pre without H_post, H_res and Sinkhorn: x_in,
 * H_pre, proj and inv_rms exactly as mhc_pre writes them (same kernels and
 * arithmetic).  Arguments, layouts, ownership and errors as mhc_pre; there is
 * no iters (no Sinkhorn runs).
 */
mhc_status mhc_pre_critical(mhc_dtype dt, const void* x, const float* phi, const float* b,
                            const float* alpha, int64_t T, int n, int64_t D, float eps, void* x_in,
                            float* H_pre, float* proj, float* inv_rms, cudaStream_t stream);

/*
 * mhc_post_res_gates -- H_post = 2 sigmoid(logits[n:2n]) and H_res =
 * Sinkhorn(exp(reshape(logits[2n:], n, n))), `iters` rounds, from the
 * projection proj [T, 2n+n^2] (float32, as mhc_pre / mhc_pre_critical wrote
 * it), with logits = alpha_group * proj + b as in mhc_pre.  Writes H_post
 * [T, n] and H_res [T, n, n] (float32), bit for bit the values mhc_pre
 * writes.  proj must be complete on `stream` (an event if it was written on
 * another one).  n must be 4; iters in [1, MHC_MAX_ITERS]; every pointer
 * 16-byte aligned; T = 0 is a no-op.
 */
mhc_status mhc_post_res_gates(const float* proj, const float* b, const float* alpha, int64_t T, int n,
                              int iters, float* H_post, float* H_res, cudaStream_t stream);

/*
 * Recompute-oriented backward.  The Ascend mHC Triton operator article
 * (paragraphs on the activation memory of mHC and on recompute inside a
 * layer and across layers) keeps, for each mHC layer, only the input of
 * hc_pre (the multi-stream state x) and the sublayer's output y, and
 * recomputes everything else during the backward.  The two calls below do
 * that: mhc_pre_gates recomputes the gates and the saved state from x, and
 * mhc_layer_bwd_recompute is the whole layer's backward from (x, y) and the
 * incoming gradients.  Across layers, x of layer l + 1 is restored from
 * layer l's (x, y) with mhc_post_pre (or mhc_pre_gates, then mhc_post).
 */

/*
 * mhc_pre_gates -- mhc_pre without the H_pre mix: the same kernel and the
 * same arithmetic, so H_pre, H_post, H_res, proj and inv_rms are bit for bit
 * those mhc_pre writes for the same inputs.  x_in is neither computed nor
 * written.  Arguments, layouts, ownership and errors as mhc_pre.
 */
mhc_status mhc_pre_gates(mhc_dtype dt, const void* x, const float* phi,
                         const float* b, const float* alpha, int64_t T, int n,
                         int64_t D, int iters, float eps, float* H_pre,
                         float* H_post, float* H_res, float* proj,
                         float* inv_rms, cudaStream_t stream);

/* Bytes of scratch mhc_layer_bwd_recompute needs (0 for T = 0): the
 * recomputed gates and saved state (196 B per token), dH_post and dH_res
 * (80 B per token), each region rounded up to 256 B, then
 * mhc_pre_bwd_workspace_bytes(). */
size_t mhc_layer_bwd_recompute_workspace_bytes(mhc_dtype dt, int64_t T, int n,
                                               int64_t D);

/*
 * mhc_layer_bwd_recompute -- the backward of one mHC layer (mhc_pre, the
 * sublayer's output y, mhc_post) from its inputs alone:
 *   mhc_pre_gates(x)   -> H_pre, H_post, H_res, proj, inv_rms   (scratch)
 *   mhc_post_bwd       -> dx (written), dy, dH_post, dH_res     (dH: scratch)
 *   mhc_pre_bwd        -> dx (accumulated), dphi, db, dalpha
 * on `stream`, in that order.  The results are bit for bit those of
 * mhc_post_bwd then mhc_pre_bwd given the state a mhc_pre call on the same x
 * saved.
 *
 *   g_in    [T, D]     dt      dL/dx_in
 *   g_next  [T, n, D]  dt      dL/dx_next
 *   x, phi, b, alpha, iters, eps   as passed to mhc_pre
 *   y       [T, D]     dt      the sublayer output, as passed to mhc_post
 * outputs (written):
 *   dx      [T, n, D]  dt      dL/dx (both paths)
 *   dy      [T, D]     dt      dL/dy
 *   dphi    [n*D, G]   float
 *   db      [G]        float
 *   dalpha  [3]        float
 *   workspace, ws_bytes        device scratch of at least
 *                              mhc_layer_bwd_recompute_workspace_bytes() bytes
 * Errors as mhc_pre_bwd; MHC_ERR_INVALID_ARG for a missing or short
 * workspace.  Data parallelism and T = 0 (zero dphi, db, dalpha) as
 * mhc_pre_bwd.
 */
mhc_status mhc_layer_bwd_recompute(mhc_dtype dt, const void* g_in, const void* g_next,
                                   const void* x, const void* y, const float* phi,
                                   const float* b, const float* alpha, int64_t T, int n,
                                   int64_t D, int iters, float eps, void* dx, void* dy,
                                   float* dphi, float* db, float* dalpha, void* workspace,
                                   size_t ws_bytes, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MHC_GB300_H */
