// post_norm.cu -- the residual update with openPangu's stability changes
// (section 5.4 of the "openPangu 2.0 -- architecture, training and Ascend
// systems" notes), forward and backward, each change optional:
//   sandwich norm: the sublayer output y is RMS-normalised over D before
//                  the H_post write-back, y' = y r_y, r_y = (mean(y^2)+eps)^-1/2;
//   block norm:    the updated state z = H_res x + H_post y' is
//                  RMS-normalised over its flattened n*D row,
//                  x_next = z s, s = (mean(z^2)+eps)^-1/2.
// Unit weights, eps inside the square root.
//
// One CTA per token (a token is 10 KB of y and 40 KB of x at D = 5120):
// the row statistics need the whole row before anything is written, so the
// block-normalised update is formed twice, once for sum z^2 and once to store
// it; the second reading of x hits L2 (the CTAs in flight hold a few tens of
// MB).  y, and in the backward the y-side gradient, stay in registers: a
// thread holds MP pieces of 16 bytes, so D <= NT * MP * (16 / element).
// The flags are template arguments, so a step that is off costs nothing.
#include <cuda_runtime.h>
#include <stdint.h>

#include "launch.h"
#include "mhc_common.cuh"

namespace mhc {
namespace {

// CTA shapes (threads, 16-byte pieces per thread and row, CTAs per SM), the
// fastest of those compared at T = 32768, D = 5120 before the backward's
// prefetch (forward 0.51-0.61 ms, backward 0.85-1.42 ms for flags 0-3;
// 512 threads x 2 pieces: 0.66-1.0 and 1.2-2.1 ms).  With the prefetch and
// one wave of CTAs the backward takes 0.77-1.24 ms.  Both cover D <= 8192
// (bf16) and 4096 (float32).
constexpr int FWD_NT = 128, FWD_MP = 8, FWD_MIN = 4;
constexpr int BWD_NT = 256, BWD_MP = 4, BWD_MIN = 2;
constexpr int MAX_PIECES = 1024;         // NT * MP of both
static_assert(FWD_NT * FWD_MP == MAX_PIECES && BWD_NT * BWD_MP == MAX_PIECES, "same width limit");
constexpr int SANDWICH = 1, BLOCK = 2;

// Sum over the CTA of NT threads (every thread gets the total).
template <int NT>
__device__ __forceinline__ float block_sum(float v, float* red) {
    v = warp_sum(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();                     // red is free (previous use done)
    if (l == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < NT / 32; ++i) t += red[i];
    return t;
}

// Several sums at once: v[0..N) over the CTA.
template <int NT, int N>
__device__ __forceinline__ void block_sums(float (&v)[N], float* red) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
#pragma unroll
    for (int k = 0; k < N; ++k) v[k] = warp_sum(v[k]);
    __syncthreads();
    if (l == 0) {
#pragma unroll
        for (int k = 0; k < N; ++k) red[k * (NT / 32) + w] = v[k];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < N; ++k) {
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < NT / 32; ++i) t += red[k * (NT / 32) + i];
        v[k] = t;
    }
}

struct Gates {
    float H[4][4], Hp[4];
};

__device__ __forceinline__ Gates load_gates(const float* H_post, const float* H_res, int64_t t) {
    Gates g;
    const float4 hp = reinterpret_cast<const float4*>(H_post)[t];
    const float4* hr4 = reinterpret_cast<const float4*>(H_res + t * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 r = hr4[i];
        g.H[i][0] = r.x; g.H[i][1] = r.y; g.H[i][2] = r.z; g.H[i][3] = r.w;
    }
    g.Hp[0] = hp.x; g.Hp[1] = hp.y; g.Hp[2] = hp.z; g.Hp[3] = hp.w;
    return g;
}

// z_i = sum_j H[i][j] x_j + H_post[i] y', mhc_post's order of operations.
__device__ __forceinline__ float post_elem(const Gates& g, int i, float x0, float x1, float x2, float x3, float yv) {
    return fmaf(g.Hp[i], yv, fmaf(g.H[i][3], x3, fmaf(g.H[i][2], x2, fmaf(g.H[i][1], x1, g.H[i][0] * x0))));
}

// Asks L2 for a contiguous range ahead of its use (a hint: no data reaches
// the SM, nothing waits for it).  Pieces of at most 32 KB, 16-byte multiples.
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
    const char* c = static_cast<const char*>(p);
    for (uint32_t off = 0; off < bytes; off += 32768u) {
        const uint32_t n = bytes - off < 32768u ? bytes - off : 32768u;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c + off), "r"(n) : "memory");
    }
}

template <typename TA, int flags, int PN_THREADS = FWD_NT, int MAXP = FWD_MP>
__global__ void __launch_bounds__(FWD_NT, FWD_MIN)
post_norm_kernel(const TA* __restrict__ x, const TA* __restrict__ y, const float* __restrict__ H_post,
                 const float* __restrict__ H_res, float eps, int64_t T, int64_t D,
                 TA* __restrict__ x_next, float* __restrict__ inv_rms_y, float* __restrict__ inv_rms_out) {
    constexpr int V = Vec<TA>::N;
    __shared__ float red[PN_THREADS / 32];
    const int tid = threadIdx.x;
    const int64_t QD = D / V;
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        const Gates g = load_gates(H_post, H_res, t);
        const TA* xt = x + t * 4 * D;
        // y' in registers
        float yv[MAXP][V];
        float ssq = 0.f;
#pragma unroll
        for (int k = 0; k < MAXP; ++k) {
            const int64_t q = tid + static_cast<int64_t>(k) * PN_THREADS;
            if (q < QD) {
                Vec<TA>::unpack(ld16_stream(y + t * D + q * V), yv[k]);
#pragma unroll
                for (int e = 0; e < V; ++e) ssq = fmaf(yv[k][e], yv[k][e], ssq);
            }
        }
        float ry = 1.0f;
        if constexpr ((flags & SANDWICH) != 0) {
            ry = 1.0f / sqrtf(block_sum<PN_THREADS>(ssq, red) / static_cast<float>(D) + eps);
#pragma unroll
            for (int k = 0; k < MAXP; ++k)
#pragma unroll
                for (int e = 0; e < V; ++e) yv[k][e] *= ry;
        }
        float s = 1.0f;
        if constexpr ((flags & BLOCK) != 0) {
            float zz = 0.f;
#pragma unroll
            for (int k = 0; k < MAXP; ++k) {
                const int64_t q = tid + static_cast<int64_t>(k) * PN_THREADS;
                if (q >= QD) continue;
                float f[4][V];
#pragma unroll
                for (int j = 0; j < 4; ++j) Vec<TA>::unpack(ld16(xt + j * D + q * V), f[j]);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        const float z = post_elem(g, i, f[0][e], f[1][e], f[2][e], f[3][e], yv[k][e]);
                        zz = fmaf(z, z, zz);
                    }
            }
            s = 1.0f / sqrtf(block_sum<PN_THREADS>(zz, red) / static_cast<float>(4 * D) + eps);
        }
#pragma unroll
        for (int k = 0; k < MAXP; ++k) {
            const int64_t q = tid + static_cast<int64_t>(k) * PN_THREADS;
            if (q >= QD) continue;
            float f[4][V];
#pragma unroll
            for (int j = 0; j < 4; ++j) Vec<TA>::unpack(ld16_stream(xt + j * D + q * V), f[j]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float o[V];
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const float z = post_elem(g, i, f[0][e], f[1][e], f[2][e], f[3][e], yv[k][e]);
                    o[e] = ((flags & BLOCK) != 0) ? z * s : z;
                }
                st16_stream(x_next + t * 4 * D + i * D + q * V, Vec<TA>::pack(o));
            }
        }
        if (tid == 0) {
            inv_rms_y[t] = ry;
            inv_rms_out[t] = s;
        }
    }
}

template <typename TA, int flags, int PN_THREADS = BWD_NT, int MAXP = BWD_MP>
__global__ void __launch_bounds__(BWD_NT, BWD_MIN)
post_norm_bwd_kernel(const TA* __restrict__ g_next, const TA* __restrict__ x, const TA* __restrict__ y,
                     const float* __restrict__ H_post, const float* __restrict__ H_res, float eps,
                     const float* __restrict__ inv_rms_y, const float* __restrict__ inv_rms_out, int64_t T,
                     int64_t D, TA* __restrict__ dx, TA* __restrict__ dy, float* __restrict__ dH_post,
                     float* __restrict__ dH_res) {
    constexpr int V = Vec<TA>::N;
    __shared__ float red[20 * (PN_THREADS / 32)];
    const int tid = threadIdx.x;
    const int64_t QD = D / V;
    (void)eps;
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        const Gates g = load_gates(H_post, H_res, t);
        const float ry = ((flags & SANDWICH) != 0) ? inv_rms_y[t] : 1.0f;
        const float s = ((flags & BLOCK) != 0) ? inv_rms_out[t] : 1.0f;
        const TA* xt = x + t * 4 * D;
        const TA* gt = g_next + t * 4 * D;
        // A token's loads come in dependent steps (the block-norm sum, then
        // the gradient pass), so have L2 fetch this CTA's next token while
        // this one works through them: 9% faster with both steps on, and
        // with neither.  (In the forward the same hint slowed the two-pass
        // block norm, so it has none.)
        if (tid == 0 && t + gridDim.x < T) {
            const int64_t tn = t + gridDim.x;
            bulk_prefetch_l2(x + tn * 4 * D, static_cast<uint32_t>(4 * D * sizeof(TA)));
            bulk_prefetch_l2(g_next + tn * 4 * D, static_cast<uint32_t>(4 * D * sizeof(TA)));
            bulk_prefetch_l2(y + tn * D, static_cast<uint32_t>(D * sizeof(TA)));
        }
        float yv[MAXP][V];   // y' = y r_y
#pragma unroll
        for (int k = 0; k < MAXP; ++k) {
            const int64_t q = tid + static_cast<int64_t>(k) * PN_THREADS;
            if (q < QD) {
                Vec<TA>::unpack(ld16_stream(y + t * D + q * V), yv[k]);
#pragma unroll
                for (int e = 0; e < V; ++e) yv[k][e] *= ry;
            }
        }
        // block norm: c = <g, u> over the row, u = z s the stored output before rounding
        float c = 0.f;
        if constexpr ((flags & BLOCK) != 0) {
            float gu = 0.f;
#pragma unroll
            for (int k = 0; k < MAXP; ++k) {
                const int64_t q = tid + static_cast<int64_t>(k) * PN_THREADS;
                if (q >= QD) continue;
                float f[4][V], gg[4][V];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    Vec<TA>::unpack(ld16(xt + j * D + q * V), f[j]);
                    Vec<TA>::unpack(ld16(gt + j * D + q * V), gg[j]);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int e = 0; e < V; ++e)
                        gu = fmaf(gg[i][e], post_elem(g, i, f[0][e], f[1][e], f[2][e], f[3][e], yv[k][e]) * s, gu);
            }
            c = block_sum<PN_THREADS>(gu, red) / static_cast<float>(4 * D);
        }
        float dyv[MAXP][V];  // gradient reaching y'
        float acc[20];       // dH_post[4], dH_res[16]
#pragma unroll
        for (int a = 0; a < 20; ++a) acc[a] = 0.f;
#pragma unroll
        for (int k = 0; k < MAXP; ++k) {
            const int64_t q = tid + static_cast<int64_t>(k) * PN_THREADS;
            if (q >= QD) continue;
            float f[4][V], dz[4][V];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                Vec<TA>::unpack(ld16_stream(xt + j * D + q * V), f[j]);
                Vec<TA>::unpack(ld16_stream(gt + j * D + q * V), dz[j]);
            }
            if constexpr ((flags & BLOCK) != 0) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        const float u = post_elem(g, i, f[0][e], f[1][e], f[2][e], f[3][e], yv[k][e]) * s;
                        dz[i][e] = s * fmaf(-u, c, dz[i][e]);
                    }
            }
            // mhc_post's backward with dz for the output gradient and y' for y
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float o[V];
#pragma unroll
                for (int e = 0; e < V; ++e)
                    o[e] = fmaf(g.H[3][j], dz[3][e], fmaf(g.H[2][j], dz[2][e], fmaf(g.H[1][j], dz[1][e], g.H[0][j] * dz[0][e])));
                st16_stream(dx + t * 4 * D + j * D + q * V, Vec<TA>::pack(o));
            }
#pragma unroll
            for (int e = 0; e < V; ++e) {
                dyv[k][e] = fmaf(g.Hp[3], dz[3][e], fmaf(g.Hp[2], dz[2][e], fmaf(g.Hp[1], dz[1][e], g.Hp[0] * dz[0][e])));
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[i] = fmaf(dz[i][e], yv[k][e], acc[i]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[4 + 4 * i + j] = fmaf(dz[i][e], f[j][e], acc[4 + 4 * i + j]);
                }
            }
        }
        // sandwich norm: dy = r_y (dy' - y' <dy', y'> / D)
        float c2 = 0.f;
        if constexpr ((flags & SANDWICH) != 0) {
            float dd = 0.f;
#pragma unroll
            for (int k = 0; k < MAXP; ++k) {
                const int64_t q = tid + static_cast<int64_t>(k) * PN_THREADS;
                if (q >= QD) continue;
#pragma unroll
                for (int e = 0; e < V; ++e) dd = fmaf(dyv[k][e], yv[k][e], dd);
            }
            c2 = block_sum<PN_THREADS>(dd, red) / static_cast<float>(D);
        }
#pragma unroll
        for (int k = 0; k < MAXP; ++k) {
            const int64_t q = tid + static_cast<int64_t>(k) * PN_THREADS;
            if (q >= QD) continue;
            float o[V];
#pragma unroll
            for (int e = 0; e < V; ++e) o[e] = ((flags & SANDWICH) != 0) ? ry * fmaf(-yv[k][e], c2, dyv[k][e]) : dyv[k][e];
            st16_stream(dy + t * D + q * V, Vec<TA>::pack(o));
        }
        block_sums<PN_THREADS>(acc, red);
        if (tid < 4) dH_post[t * 4 + tid] = acc[tid];
        else if (tid < 20) dH_res[t * 16 + tid - 4] = acc[tid];
    }
}

// CTAs per launch: `per_sm` for every SM, at most one per token.
int grid_for(int64_t T, int per_sm) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 148;
    const int64_t cap = static_cast<int64_t>(n) * per_sm;
    return static_cast<int>(T < cap ? T : cap);
}

bool post_norm_supports_impl(bool bf16, int64_t D) {
    const int64_t V = bf16 ? 8 : 4;
    return D % V == 0 && D / V <= MAX_PIECES;
}

template <typename TA, int F>
void fwd(const void* x, const void* y, const float* H_post, const float* H_res, float eps, int64_t T, int64_t D,
         void* x_next, float* inv_rms_y, float* inv_rms_out, cudaStream_t s) {
    post_norm_kernel<TA, F><<<grid_for(T, 16), FWD_NT, 0, s>>>(
        static_cast<const TA*>(x), static_cast<const TA*>(y), H_post, H_res, eps, T, D, static_cast<TA*>(x_next),
        inv_rms_y, inv_rms_out);
}

template <typename TA, int F>
void bwd(const void* g_next, const void* x, const void* y, const float* H_post, const float* H_res, float eps,
         const float* inv_rms_y, const float* inv_rms_out, int64_t T, int64_t D, void* dx, void* dy,
         float* dH_post, float* dH_res, cudaStream_t s) {
    // one wave of resident CTAs (two per SM), so that every token after a
    // CTA's first has been prefetched: 3% faster than 16 per SM with both steps
    post_norm_bwd_kernel<TA, F><<<grid_for(T, BWD_MIN), BWD_NT, 0, s>>>(
        static_cast<const TA*>(g_next), static_cast<const TA*>(x), static_cast<const TA*>(y), H_post, H_res, eps,
        inv_rms_y, inv_rms_out, T, D, static_cast<TA*>(dx), static_cast<TA*>(dy), dH_post, dH_res);
}

}  // namespace

bool post_norm_supports(bool bf16, int64_t D) { return post_norm_supports_impl(bf16, D); }

cudaError_t launch_post_norm(bool bf16, const void* x, const void* y, const float* H_post, const float* H_res,
                             int flags, float eps, int64_t T, int64_t D, void* x_next, float* inv_rms_y,
                             float* inv_rms_out, cudaStream_t s) {
#define MHC_PN_FWD(TA, F) fwd<TA, F>(x, y, H_post, H_res, eps, T, D, x_next, inv_rms_y, inv_rms_out, s)
    switch (flags + (bf16 ? 4 : 0)) {
        case 0: MHC_PN_FWD(float, 0); break;
        case 1: MHC_PN_FWD(float, 1); break;
        case 2: MHC_PN_FWD(float, 2); break;
        case 3: MHC_PN_FWD(float, 3); break;
        case 4: MHC_PN_FWD(__nv_bfloat16, 0); break;
        case 5: MHC_PN_FWD(__nv_bfloat16, 1); break;
        case 6: MHC_PN_FWD(__nv_bfloat16, 2); break;
        case 7: MHC_PN_FWD(__nv_bfloat16, 3); break;
        default: return cudaErrorInvalidValue;
    }
#undef MHC_PN_FWD
    return cudaGetLastError();
}

cudaError_t launch_post_norm_bwd(bool bf16, const void* g_next, const void* x, const void* y, const float* H_post,
                                 const float* H_res, int flags, float eps, const float* inv_rms_y,
                                 const float* inv_rms_out, int64_t T, int64_t D, void* dx, void* dy,
                                 float* dH_post, float* dH_res, cudaStream_t s) {
#define MHC_PN_BWD(TA, F) \
    bwd<TA, F>(g_next, x, y, H_post, H_res, eps, inv_rms_y, inv_rms_out, T, D, dx, dy, dH_post, dH_res, s)
    switch (flags + (bf16 ? 4 : 0)) {
        case 0: MHC_PN_BWD(float, 0); break;
        case 1: MHC_PN_BWD(float, 1); break;
        case 2: MHC_PN_BWD(float, 2); break;
        case 3: MHC_PN_BWD(float, 3); break;
        case 4: MHC_PN_BWD(__nv_bfloat16, 0); break;
        case 5: MHC_PN_BWD(__nv_bfloat16, 1); break;
        case 6: MHC_PN_BWD(__nv_bfloat16, 2); break;
        case 7: MHC_PN_BWD(__nv_bfloat16, 3); break;
        default: return cudaErrorInvalidValue;
    }
#undef MHC_PN_BWD
    return cudaGetLastError();
}

}  // namespace mhc
