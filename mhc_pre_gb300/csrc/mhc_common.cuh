// mhc_common.cuh -- device helpers shared by the mHC kernels (sm_103a).
//
// Gate arithmetic follows section 5.3 of the "openPangu 2.0 -- architecture,
// training and Ascend systems" notes:
//   logits = alpha_group * proj + b, H_pre = sigmoid, H_post = 2 sigmoid,
//   H_res = Sinkhorn(exp(reshape(res logits, 4, 4))), one round = rows then
//   columns.
// The kernels start Sinkhorn from exp(L - rowmax): the row normalisation that
// follows cancels any per-row factor, so this equals exp(L) in value and in
// gradient while keeping exp() finite for peaked logits.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace mhc {

constexpr int NS = 4;                  // residual streams
constexpr int NG = 2 * NS + NS * NS;   // 24 gate logits
constexpr int MAX_ITERS = 64;

// ------------------------------------------------------------------------
// 16-byte activation vectors: 8 bf16 or 4 float, widened to float.
// ------------------------------------------------------------------------
template <typename TA> struct Vec;

template <> struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void unpack(const uint4& u, float (&f)[8]) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[8]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// x_in of one 16-byte piece (8 columns): sum_i h[i] x_i for the four
// streams' pieces, h.x x_0 first, then one fmaf per stream, rounded to bf16
// once.  Column pairs go through packed fp32 multiply-adds; each lane rounds
// as the scalar product and fmaf chain would.
__device__ __forceinline__ uint4 mix4_bf16(const uint4& x0, const uint4& x1, const uint4& x2, const uint4& x3,
                                           const float4& h) {
    const float2 hx = make_float2(h.x, h.x), hy = make_float2(h.y, h.y);
    const float2 hz = make_float2(h.z, h.z), hw = make_float2(h.w, h.w);
    const uint32_t a0[4] = {x0.x, x0.y, x0.z, x0.w}, a1[4] = {x1.x, x1.y, x1.z, x1.w};
    const uint32_t a2[4] = {x2.x, x2.y, x2.z, x2.w}, a3[4] = {x3.x, x3.y, x3.z, x3.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 f0 = make_float2(__uint_as_float(a0[q] << 16), __uint_as_float(a0[q] & 0xffff0000u));
        const float2 f1 = make_float2(__uint_as_float(a1[q] << 16), __uint_as_float(a1[q] & 0xffff0000u));
        const float2 f2 = make_float2(__uint_as_float(a2[q] << 16), __uint_as_float(a2[q] & 0xffff0000u));
        const float2 f3 = make_float2(__uint_as_float(a3[q] << 16), __uint_as_float(a3[q] & 0xffff0000u));
        const float2 v = __ffma2_rn(hw, f3, __ffma2_rn(hz, f2, __ffma2_rn(hy, f1, __fmul2_rn(hx, f0))));
        const __nv_bfloat162 b = __floats2bfloat162_rn(v.x, v.y);
        o[q] = *reinterpret_cast<const uint32_t*>(&b);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

template <> struct Vec<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void unpack(const uint4& u, float (&f)[4]) {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                          __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
};

// Plain cached 16-byte load (data that is read again soon).
__device__ __forceinline__ uint4 ld16(const void* p) {
    return *reinterpret_cast<const uint4*>(p);
}
// Streaming 16-byte load: read once, evict first.
__device__ __forceinline__ uint4 ld16_stream(const void* p) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
}
// Streaming 16-byte store.
__device__ __forceinline__ void st16_stream(void* p, const uint4& v) {
    __stcs(reinterpret_cast<uint4*>(p), v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------------------------------------
// Gates of one token.
// ------------------------------------------------------------------------
__device__ __forceinline__ int group_of(int g) { return g < NS ? 0 : (g < 2 * NS ? 1 : 2); }

// Hardware reciprocal approximation (rcp.approx.f32, within about one ulp);
// the Sinkhorn normalisers and gates tolerate it by orders of magnitude.
__device__ __forceinline__ float fast_rcp(float v) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ float sigmoid_f(float v) { return fast_rcp(1.0f + expf(-v)); }

// logits[g] = alpha[group(g)] * proj[g] + b[g]  (one fused multiply-add, so
// the backward reproduces the forward's logits bit for bit).
__device__ __forceinline__ void make_logits(const float (&proj)[NG], const float* alpha,
                                            const float* b, float (&lg)[NG]) {
    const float a0 = alpha[0], a1 = alpha[1], a2 = alpha[2];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        const float a = g < NS ? a0 : (g < 2 * NS ? a1 : a2);
        lg[g] = fmaf(a, proj[g], b[g]);
    }
}

// M = exp(L - rowmax), row-major 4x4.
__device__ __forceinline__ void sinkhorn_start(const float* L, float (&M)[16]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float m = fmaxf(fmaxf(L[4 * i], L[4 * i + 1]), fmaxf(L[4 * i + 2], L[4 * i + 3]));
#pragma unroll
        for (int j = 0; j < 4; ++j) M[4 * i + j] = expf(L[4 * i + j] - m);
    }
}

__device__ __forceinline__ void normalise_rows(float (&M)[16], float* sums) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float s = (M[4 * i] + M[4 * i + 1]) + (M[4 * i + 2] + M[4 * i + 3]);
        if (sums) sums[i] = s;
        const float r = fast_rcp(s);
#pragma unroll
        for (int j = 0; j < 4; ++j) M[4 * i + j] *= r;
    }
}

__device__ __forceinline__ void normalise_cols(float (&M)[16], float* sums) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float c = (M[j] + M[4 + j]) + (M[8 + j] + M[12 + j]);
        if (sums) sums[j] = c;
        const float r = fast_rcp(c);
#pragma unroll
        for (int i = 0; i < 4; ++i) M[4 * i + j] *= r;
    }
}

// H_res = `iters` rounds of (rows, columns) from exp(L - rowmax).
__device__ __forceinline__ void sinkhorn_fwd(const float* L, int iters, float (&M)[16]) {
    sinkhorn_start(L, M);
    for (int it = 0; it < iters; ++it) {
        normalise_rows(M, nullptr);
        normalise_cols(M, nullptr);
    }
}

// dL = d/dL <dH, Sinkhorn(L)> for the unrolled map (exact reverse mode).
// The forward keeps each round's row and column sums; walking back, the
// earlier iterate is rebuilt by multiplying those sums back in, and the VJP
// of Y = X / s is dX = (dY - sum(dY * Y)) / s along the normalised axis
// (the quotient formed as a product with the correctly rounded 1/s, one
// reciprocal per row or column instead of four divisions).
static __device__ __noinline__ void sinkhorn_vjp(const float* L, int iters, const float* dH,
                                          float* dL) {
    float rs[MAX_ITERS][4], cs[MAX_ITERS][4];
    float M[16];
    sinkhorn_start(L, M);
    for (int it = 0; it < iters; ++it) {
        normalise_rows(M, rs[it]);
        normalise_cols(M, cs[it]);
    }
    float g[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) g[e] = dH[e];
    for (int it = iters - 1; it >= 0; --it) {
        // column step: Y = M, divisor c_j
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float t = (g[j] * M[j] + g[4 + j] * M[4 + j]) + (g[8 + j] * M[8 + j] + g[12 + j] * M[12 + j]);
            const float c = cs[it][j];
            const float rc = __frcp_rn(c);   // one reciprocal for the column's four quotients
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                g[4 * i + j] = (g[4 * i + j] - t) * rc;
                M[4 * i + j] *= c;           // rebuild the row-normalised P
            }
        }
        // row step: Y = P, divisor s_i
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float t = (g[4 * i] * M[4 * i] + g[4 * i + 1] * M[4 * i + 1]) +
                            (g[4 * i + 2] * M[4 * i + 2] + g[4 * i + 3] * M[4 * i + 3]);
            const float s = rs[it][i];
            const float rs_i = __frcp_rn(s);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                g[4 * i + j] = (g[4 * i + j] - t) * rs_i;
                M[4 * i + j] *= s;           // rebuild the previous iterate
            }
        }
    }
    float M0[16];
    sinkhorn_start(L, M0);
#pragma unroll
    for (int e = 0; e < 16; ++e) dL[e] = g[e] * M0[e];
}

// H_pre alone (the inference critical path): the same expression as in
// token_gates.
__device__ __forceinline__ void token_pre_gates(const float (&proj)[NG], const float* alpha,
                                                const float* b, float (&hpre)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) hpre[i] = sigmoid_f(fmaf(alpha[0], proj[i], b[i]));
}

// H_post and H_res from the projection (the side of the critical-path
// split): the same expressions as in token_gates.
__device__ __forceinline__ void token_post_res_gates(const float (&proj)[NG], const float* alpha,
                                                     const float* b, int iters, float (&hpost)[4],
                                                     float (&hres)[16]) {
    float lg[NG];
    make_logits(proj, alpha, b, lg);
#pragma unroll
    for (int i = 0; i < 4; ++i) hpost[i] = 2.0f * sigmoid_f(lg[NS + i]);
    sinkhorn_fwd(lg + 2 * NS, iters, hres);
}

// All gates of one token from its projection.
__device__ __forceinline__ void token_gates(const float (&proj)[NG], const float* alpha,
                                            const float* b, int iters, float (&hpre)[4],
                                            float (&hpost)[4], float (&hres)[16]) {
    float lg[NG];
    make_logits(proj, alpha, b, lg);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        hpre[i] = sigmoid_f(lg[i]);
        hpost[i] = 2.0f * sigmoid_f(lg[NS + i]);
    }
    sinkhorn_fwd(lg + 2 * NS, iters, hres);
}

}  // namespace mhc
