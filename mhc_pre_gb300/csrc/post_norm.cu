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
#include "tc_ptx.cuh"

namespace mhc {

// This file's device error word (latched by bounded waits that ran out).
__device__ unsigned g_post_norm_error;

cudaError_t read_and_clear_post_norm_error(unsigned* word) {
    cudaError_t e = cudaMemcpyFromSymbol(word, g_post_norm_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_post_norm_error, &zero, sizeof(unsigned));
}

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


// ---- staged backward (bf16 rows that fit in shared memory) ---------------
// A token's x, g_next and y rows (18 D bytes) arrive in shared memory by
// bulk copies into one of two buffers, the next token's rows while this one
// is worked (one CTA per SM), so the block-norm pass and the gradient pass
// read them on chip instead of waiting on global loads in turn.  The
// per-element expressions are those of the kernel above, evaluated on column
// pairs with packed fp32 multiply-adds; the sums over the row are formed in
// another order (per stream and per column parity, then added).  Thread tid
// takes the 16-byte pieces tid, tid + NT, ...; nothing per piece is kept
// between the passes: y' is re-read from the buffer, and with the sandwich
// norm dy' (fp32) is parked over the piece's own g_next values of streams 0
// and 1, which the gradient pass has just consumed.
constexpr uint64_t STG_WAIT_NS = 1000000000ull;   // 1 s

// Two adjacent columns at once: packed fp32 multiply-adds (each lane rounds
// as fmaf / a plain product), so the results are those of the scalar
// expressions above.
__device__ __forceinline__ float2 bc2(float v) { return make_float2(v, v); }
__device__ __forceinline__ float2 bf16_pair(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ uint32_t bf16_pack_pair(float2 v) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
    return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t word_of(const uint4& u, int w) {
    return w == 0 ? u.x : w == 1 ? u.y : w == 2 ? u.z : u.w;
}
// post_elem on a column pair
__device__ __forceinline__ float2 post_elem2(const Gates& g, int i, float2 x0, float2 x1, float2 x2, float2 x3,
                                             float2 yv) {
    return __ffma2_rn(bc2(g.Hp[i]), yv,
                      __ffma2_rn(bc2(g.H[i][3]), x3,
                                 __ffma2_rn(bc2(g.H[i][2]), x2, __ffma2_rn(bc2(g.H[i][1]), x1, __fmul2_rn(bc2(g.H[i][0]), x0)))));
}

template <int NT, int flags>
__global__ void __launch_bounds__(NT, 1)
post_norm_bwd_staged_kernel(const __nv_bfloat16* __restrict__ g_next, const __nv_bfloat16* __restrict__ x,
                            const __nv_bfloat16* __restrict__ y, const float* __restrict__ H_post,
                            const float* __restrict__ H_res, const float* __restrict__ inv_rms_y,
                            const float* __restrict__ inv_rms_out, int64_t T, int64_t D,
                            __nv_bfloat16* __restrict__ dx, __nv_bfloat16* __restrict__ dy,
                            float* __restrict__ dH_post, float* __restrict__ dH_res) {
    using TA = __nv_bfloat16;
    constexpr int V = 8;
    extern __shared__ __align__(128) unsigned char stage[];   // 2 x [x 4D | g 4D | y D]
    __shared__ float red[20 * (NT / 32)];
    __shared__ __align__(8) uint64_t full[2];
    const int tid = threadIdx.x;
    const int64_t QD = D / V;
    const int64_t G = gridDim.x;
    const uint32_t buf_bytes = static_cast<uint32_t>(18 * D);
    const uint32_t sb = ptx::smem_u32(stage);
    const uint32_t bar0 = ptx::smem_u32(&full[0]);
    if (tid == 0) {
        for (int b = 0; b < 2; ++b) ptx::mbar_init(bar0 + 8u * b, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    // thread 0: token t's three rows into buffer b
    auto issue = [&](int b, int64_t t) {
        const uint32_t bar = bar0 + 8u * static_cast<uint32_t>(b);
        const uint32_t dst = sb + static_cast<uint32_t>(b) * buf_bytes;
        ptx::mbar_arrive_expect_tx(bar, buf_bytes);
        ptx::bulk_load(dst, x + t * 4 * D, static_cast<uint32_t>(8 * D), bar);
        ptx::bulk_load(dst + static_cast<uint32_t>(8 * D), g_next + t * 4 * D, static_cast<uint32_t>(8 * D), bar);
        ptx::bulk_load(dst + static_cast<uint32_t>(16 * D), y + t * D, static_cast<uint32_t>(2 * D), bar);
    };
    if (tid == 0) {
        for (int b = 0; b < 2; ++b)
            if (blockIdx.x + b * G < T) issue(b, blockIdx.x + b * G);
    }
    bool aborted = false;
    int k = 0;
    for (int64_t t = blockIdx.x; t < T; t += G, ++k) {
        const int b = k & 1;
        const uint32_t par = static_cast<uint32_t>(k >> 1) & 1u;
        const Gates g = load_gates(H_post, H_res, t);
        const float ry = ((flags & SANDWICH) != 0) ? inv_rms_y[t] : 1.0f;
        const float s = ((flags & BLOCK) != 0) ? inv_rms_out[t] : 1.0f;
        // bounded wait for the token's rows; every thread waits, and all
        // leave together if any gave up
        bool timed_out = false;
        {
            const uint32_t bar = bar0 + 8u * static_cast<uint32_t>(b);
            if (!ptx::mbar_try_wait(bar, par)) {
                const uint64_t t0 = ptx::globaltimer();
                while (!ptx::mbar_try_wait(bar, par)) {
                    if (ptx::globaltimer() - t0 > STG_WAIT_NS) {
                        timed_out = true;
                        break;
                    }
                }
            }
        }
        if (__syncthreads_or(timed_out)) {
            if (tid == 0) atomicOr(&g_post_norm_error, 1u);
            aborted = true;
            break;
        }
        TA* xs = reinterpret_cast<TA*>(stage + static_cast<size_t>(b) * buf_bytes);
        TA* gs = xs + 4 * D;
        const TA* ys = xs + 8 * D;
        // y' = y r_y of piece q
        auto load_y = [&](int64_t q, float (&yv)[V]) {
            Vec<TA>::unpack(*reinterpret_cast<const uint4*>(ys + q * V), yv);
#pragma unroll
            for (int e = 0; e < V; ++e) yv[e] *= ry;
        };
        // block norm: c = <g, u> over the row, u = z s the stored output before rounding
        float c = 0.f;
        if constexpr ((flags & BLOCK) != 0) {
            float2 gu2[4] = {};   // one partial sum per stream: four independent chains
#pragma unroll 2
            for (int64_t q = tid; q < QD; q += NT) {
                const uint4 yp = *reinterpret_cast<const uint4*>(ys + q * V);
                uint4 xp[4], gp[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    xp[j] = *reinterpret_cast<const uint4*>(xs + j * D + q * V);
                    gp[j] = *reinterpret_cast<const uint4*>(gs + j * D + q * V);
                }
#pragma unroll
                for (int w2 = 0; w2 < V / 2; ++w2) {
                    const float2 yv = __fmul2_rn(bf16_pair(word_of(yp, w2)), bc2(ry));
                    const float2 f0 = bf16_pair(word_of(xp[0], w2)), f1 = bf16_pair(word_of(xp[1], w2));
                    const float2 f2 = bf16_pair(word_of(xp[2], w2)), f3 = bf16_pair(word_of(xp[3], w2));
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        gu2[i] = __ffma2_rn(bf16_pair(word_of(gp[i], w2)),
                                            __fmul2_rn(post_elem2(g, i, f0, f1, f2, f3, yv), bc2(s)), gu2[i]);
                }
            }
            const float gu = ((gu2[0].x + gu2[0].y) + (gu2[1].x + gu2[1].y)) + ((gu2[2].x + gu2[2].y) + (gu2[3].x + gu2[3].y));
            c = block_sum<NT>(gu, red) / static_cast<float>(4 * D);
        }
        float2 acc2[20];   // dH_post[4], dH_res[16], even and odd columns apart
#pragma unroll
        for (int a = 0; a < 20; ++a) acc2[a] = make_float2(0.f, 0.f);
        float2 dd2 = make_float2(0.f, 0.f);  // <dy', y'> (sandwich norm)
#pragma unroll 2
        for (int64_t q = tid; q < QD; q += NT) {
            const uint4 yp = *reinterpret_cast<const uint4*>(ys + q * V);
            uint4 xp[4], gp[4];
            uint32_t op[4][V / 2];   // dx of the piece, bf16 pairs per stream
            float2 dyv[V / 2];       // gradient reaching y'
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                xp[j] = *reinterpret_cast<const uint4*>(xs + j * D + q * V);
                gp[j] = *reinterpret_cast<const uint4*>(gs + j * D + q * V);
            }
#pragma unroll
            for (int w2 = 0; w2 < V / 2; ++w2) {
                const float2 yv = __fmul2_rn(bf16_pair(word_of(yp, w2)), bc2(ry));
                float2 f[4], dz[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    f[j] = bf16_pair(word_of(xp[j], w2));
                    dz[j] = bf16_pair(word_of(gp[j], w2));
                }
                if constexpr ((flags & BLOCK) != 0) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 u = __fmul2_rn(post_elem2(g, i, f[0], f[1], f[2], f[3], yv), bc2(s));
                        dz[i] = __fmul2_rn(bc2(s), __ffma2_rn(make_float2(-u.x, -u.y), bc2(c), dz[i]));
                    }
                }
                // mhc_post's backward with dz for the output gradient and y' for y
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    op[j][w2] = bf16_pack_pair(__ffma2_rn(
                        bc2(g.H[3][j]), dz[3],
                        __ffma2_rn(bc2(g.H[2][j]), dz[2], __ffma2_rn(bc2(g.H[1][j]), dz[1], __fmul2_rn(bc2(g.H[0][j]), dz[0])))));
                dyv[w2] = __ffma2_rn(bc2(g.Hp[3]), dz[3],
                                     __ffma2_rn(bc2(g.Hp[2]), dz[2], __ffma2_rn(bc2(g.Hp[1]), dz[1], __fmul2_rn(bc2(g.Hp[0]), dz[0]))));
                dd2 = __ffma2_rn(dyv[w2], yv, dd2);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc2[i] = __ffma2_rn(dz[i], yv, acc2[i]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc2[4 + 4 * i + j] = __ffma2_rn(dz[i], f[j], acc2[4 + 4 * i + j]);
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                st16_stream(dx + t * 4 * D + j * D + q * V, make_uint4(op[j][0], op[j][1], op[j][2], op[j][3]));
            if constexpr ((flags & SANDWICH) != 0) {
                // park dy' over this piece's g_next values of streams 0 and 1
                *reinterpret_cast<float4*>(gs + q * V) = make_float4(dyv[0].x, dyv[0].y, dyv[1].x, dyv[1].y);
                *reinterpret_cast<float4*>(gs + D + q * V) = make_float4(dyv[2].x, dyv[2].y, dyv[3].x, dyv[3].y);
            } else {
                st16_stream(dy + t * D + q * V, make_uint4(bf16_pack_pair(dyv[0]), bf16_pack_pair(dyv[1]),
                                                           bf16_pack_pair(dyv[2]), bf16_pack_pair(dyv[3])));
            }
        }
        const float dd = dd2.x + dd2.y;
        float acc[20];
#pragma unroll
        for (int a = 0; a < 20; ++a) acc[a] = acc2[a].x + acc2[a].y;
        // sandwich norm: dy = r_y (dy' - y' <dy', y'> / D)
        if constexpr ((flags & SANDWICH) != 0) {
            const float c2 = block_sum<NT>(dd, red) / static_cast<float>(D);
#pragma unroll 1
            for (int64_t q = tid; q < QD; q += NT) {
                float yv[V], o[V];
                load_y(q, yv);
                const float4 p0 = *reinterpret_cast<const float4*>(gs + q * V);
                const float4 p1 = *reinterpret_cast<const float4*>(gs + D + q * V);
                const float dyv[V] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
                for (int e = 0; e < V; ++e) o[e] = ry * fmaf(-yv[e], c2, dyv[e]);
                st16_stream(dy + t * D + q * V, Vec<TA>::pack(o));
            }
        }
        // this thread is done with the buffer: the next bulk copy into it
        // (async proxy) is ordered after its accesses by the barriers below
        ptx::fence_proxy_async_smem();
        // dH_post and dH_res: the 20 sums over the CTA (block_sums' order),
        // thread a < 20 adding up and writing sum a
        {
            const int wp = tid >> 5, ln = tid & 31;
#pragma unroll
            for (int a = 0; a < 20; ++a) acc[a] = warp_sum(acc[a]);
            __syncthreads();   // red is free (previous use done)
            if (ln == 0) {
#pragma unroll
                for (int a = 0; a < 20; ++a) red[a * (NT / 32) + wp] = acc[a];
            }
            __syncthreads();   // every thread is done with the buffer
            if (tid == 0 && t + 2 * G < T) issue(b, t + 2 * G);
            if (tid < 20) {
                float tot = 0.f;
#pragma unroll
                for (int i = 0; i < NT / 32; ++i) tot += red[tid * (NT / 32) + i];
                if (tid < 4) dH_post[t * 4 + tid] = tot;
                else dH_res[t * 16 + tid - 4] = tot;
            }
        }
    }
    if (aborted) {
        // let copies already issued land before the shared memory goes away
        const uint64_t t0 = ptx::globaltimer();
        while (ptx::globaltimer() - t0 < 20000ull) {
        }
    }
}

// ---- staged forward (bf16 rows that fit in shared memory) ----------------
// A token's x and y rows (10 D bytes) arrive in shared memory by bulk copies
// into one of two buffers, the next token's while this one is worked, so the
// statistics passes (sum of y^2, sum of z^2) and the store pass read them on
// chip instead of the store pass re-reading x from L2.  Two CTAs per SM.
// The per-element expressions are those of the kernel above (with no step,
// x_next is mhc_post's bit for bit); the row sums run over this CTA shape.
template <int NT, int flags>
__global__ void __launch_bounds__(NT, 2)
post_norm_fwd_staged_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ y,
                            const float* __restrict__ H_post, const float* __restrict__ H_res, float eps, int64_t T,
                            int64_t D, __nv_bfloat16* __restrict__ x_next, float* __restrict__ inv_rms_y,
                            float* __restrict__ inv_rms_out) {
    using TA = __nv_bfloat16;
    constexpr int V = 8;
    extern __shared__ __align__(128) unsigned char stage[];   // 2 x [x 4D | y D]
    __shared__ float red[NT / 32];
    __shared__ __align__(8) uint64_t full[2];
    const int tid = threadIdx.x;
    const int64_t QD = D / V;
    const int64_t G = gridDim.x;
    const uint32_t buf_bytes = static_cast<uint32_t>(10 * D);
    const uint32_t sb = ptx::smem_u32(stage);
    const uint32_t bar0 = ptx::smem_u32(&full[0]);
    if (tid == 0) {
        ptx::mbar_init(bar0, 1);
        ptx::mbar_init(bar0 + 8, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    // thread 0: token t's two rows into buffer b
    auto issue = [&](int b, int64_t t) {
        const uint32_t bar = bar0 + 8u * static_cast<uint32_t>(b);
        const uint32_t dst = sb + static_cast<uint32_t>(b) * buf_bytes;
        ptx::mbar_arrive_expect_tx(bar, buf_bytes);
        ptx::bulk_load(dst, x + t * 4 * D, static_cast<uint32_t>(8 * D), bar);
        ptx::bulk_load(dst + static_cast<uint32_t>(8 * D), y + t * D, static_cast<uint32_t>(2 * D), bar);
    };
    if (tid == 0) {
        for (int b = 0; b < 2; ++b)
            if (blockIdx.x + b * G < T) issue(b, blockIdx.x + b * G);
    }
    bool aborted = false;
    int k = 0;
    for (int64_t t = blockIdx.x; t < T; t += G, ++k) {
        const int b = k & 1;
        const Gates g = load_gates(H_post, H_res, t);
        bool timed_out = false;
        {
            const uint32_t bar = bar0 + 8u * static_cast<uint32_t>(b), par = static_cast<uint32_t>(k >> 1) & 1u;
            if (!ptx::mbar_try_wait(bar, par)) {
                const uint64_t t0 = ptx::globaltimer();
                while (!ptx::mbar_try_wait(bar, par)) {
                    if (ptx::globaltimer() - t0 > STG_WAIT_NS) {
                        timed_out = true;
                        break;
                    }
                }
            }
        }
        if (__syncthreads_or(timed_out)) {
            if (tid == 0) atomicOr(&g_post_norm_error, 1u);
            aborted = true;
            break;
        }
        const TA* xs = reinterpret_cast<const TA*>(stage + static_cast<size_t>(b) * buf_bytes);
        const TA* ys = xs + 4 * D;
        float ry = 1.0f;
        if constexpr ((flags & SANDWICH) != 0) {
            float ssq = 0.f;
#pragma unroll 2
            for (int64_t q = tid; q < QD; q += NT) {
                float yv[V];
                Vec<TA>::unpack(*reinterpret_cast<const uint4*>(ys + q * V), yv);
#pragma unroll
                for (int e = 0; e < V; ++e) ssq = fmaf(yv[e], yv[e], ssq);
            }
            ry = 1.0f / sqrtf(block_sum<NT>(ssq, red) / static_cast<float>(D) + eps);
        }
        float s = 1.0f;
        if constexpr ((flags & BLOCK) != 0) {
            float zz = 0.f;
#pragma unroll 2
            for (int64_t q = tid; q < QD; q += NT) {
                float yv[V], f[4][V];
                Vec<TA>::unpack(*reinterpret_cast<const uint4*>(ys + q * V), yv);
#pragma unroll
                for (int e = 0; e < V; ++e) yv[e] *= ry;
#pragma unroll
                for (int j = 0; j < 4; ++j) Vec<TA>::unpack(*reinterpret_cast<const uint4*>(xs + j * D + q * V), f[j]);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int e = 0; e < V; ++e) {
                        const float z = post_elem(g, i, f[0][e], f[1][e], f[2][e], f[3][e], yv[e]);
                        zz = fmaf(z, z, zz);
                    }
            }
            s = 1.0f / sqrtf(block_sum<NT>(zz, red) / static_cast<float>(4 * D) + eps);
        }
#pragma unroll 2
        for (int64_t q = tid; q < QD; q += NT) {
            float yv[V], f[4][V];
            Vec<TA>::unpack(*reinterpret_cast<const uint4*>(ys + q * V), yv);
            if constexpr ((flags & SANDWICH) != 0) {
#pragma unroll
                for (int e = 0; e < V; ++e) yv[e] *= ry;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) Vec<TA>::unpack(*reinterpret_cast<const uint4*>(xs + j * D + q * V), f[j]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float o[V];
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const float z = post_elem(g, i, f[0][e], f[1][e], f[2][e], f[3][e], yv[e]);
                    o[e] = ((flags & BLOCK) != 0) ? z * s : z;
                }
                st16_stream(x_next + t * 4 * D + i * D + q * V, Vec<TA>::pack(o));
            }
        }
        // this thread is done with the buffer; the barrier orders every
        // thread's reads before the next bulk copy into it
        ptx::fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            if (t + 2 * G < T) issue(b, t + 2 * G);
            inv_rms_y[t] = ry;
            inv_rms_out[t] = s;
        }
    }
    if (aborted) {
        // let copies already issued land before the shared memory goes away
        const uint64_t t0 = ptx::globaltimer();
        while (ptx::globaltimer() - t0 < 20000ull) {
        }
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

// The staged forward: bf16 rows whose two buffers (20 D bytes) fit.
constexpr int STGF_NT = 256;
size_t staged_smem_limit();

bool staged_fwd_supports(bool bf16, int64_t D) {
    return bf16 && D % 8 == 0 && static_cast<size_t>(20 * D) <= staged_smem_limit();
}

template <int F>
cudaError_t fwd_staged(const void* x, const void* y, const float* H_post, const float* H_res, float eps, int64_t T,
                       int64_t D, void* x_next, float* inv_rms_y, float* inv_rms_out, cudaStream_t s) {
    auto k = post_norm_fwd_staged_kernel<STGF_NT, F>;
    const size_t smem = static_cast<size_t>(20 * D);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    using B = __nv_bfloat16;
    k<<<grid_for(T, 2), STGF_NT, smem, s>>>(static_cast<const B*>(x), static_cast<const B*>(y), H_post, H_res, eps,
                                            T, D, static_cast<B*>(x_next), inv_rms_y, inv_rms_out);
    return cudaGetLastError();
}

// Width of the staged backward (two buffers, one CTA per SM).  At T = 32768,
// D = 5120 (flags 0 / 1 / 2 / 3): 256 threads 0.70 / 0.76 / 1.00 / 1.13 ms;
// one buffer and two CTAs per SM 0.99 / 0.96 / 1.08 / 1.12; 320 threads (two
// pieces each) 0.72 / 0.83 / 1.13 / 1.27; the kernel above 1.24 ms with both
// flags.
constexpr int STG_NT = 256;

// Shared memory the staged backward may take per CTA on the current device
// (the opt-in limit less room for its static arrays), 0 if unknown.
size_t staged_smem_limit() {
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return 0;
    return optin > 4096 ? static_cast<size_t>(optin) - 4096 : 0;
}

bool staged_bwd_supports(bool bf16, int64_t D) {
    return bf16 && D % 8 == 0 && static_cast<size_t>(2 * 18 * D) <= staged_smem_limit();
}

template <int F>
cudaError_t bwd_staged(const void* g_next, const void* x, const void* y, const float* H_post, const float* H_res,
                       const float* inv_rms_y, const float* inv_rms_out, int64_t T, int64_t D, void* dx, void* dy,
                       float* dH_post, float* dH_res, cudaStream_t s) {
    auto k = post_norm_bwd_staged_kernel<STG_NT, F>;
    const size_t smem = static_cast<size_t>(2 * 18 * D);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    using B = __nv_bfloat16;
    k<<<grid_for(T, 1), STG_NT, smem, s>>>(
        static_cast<const B*>(g_next), static_cast<const B*>(x), static_cast<const B*>(y), H_post, H_res, inv_rms_y,
        inv_rms_out, T, D, static_cast<B*>(dx), static_cast<B*>(dy), dH_post, dH_res);
    return cudaGetLastError();
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
    if (staged_fwd_supports(bf16, D)) {
#define MHC_PN_STGF(F) fwd_staged<F>(x, y, H_post, H_res, eps, T, D, x_next, inv_rms_y, inv_rms_out, s)
        switch (flags) {
            case 0: return MHC_PN_STGF(0);
            case 1: return MHC_PN_STGF(1);
            case 2: return MHC_PN_STGF(2);
            case 3: return MHC_PN_STGF(3);
        }
#undef MHC_PN_STGF
        return cudaErrorInvalidValue;
    }
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
    if (staged_bwd_supports(bf16, D)) {
#define MHC_PN_STG_F(F) bwd_staged<F>(g_next, x, y, H_post, H_res, inv_rms_y, inv_rms_out, T, D, dx, dy, dH_post, dH_res, s)
        switch (flags) {
            case 0: return MHC_PN_STG_F(0);
            case 1: return MHC_PN_STG_F(1);
            case 2: return MHC_PN_STG_F(2);
            case 3: return MHC_PN_STG_F(3);
        }
#undef MHC_PN_STG_F
        return cudaErrorInvalidValue;
    }
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
