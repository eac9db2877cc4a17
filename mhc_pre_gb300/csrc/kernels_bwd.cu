// kernels_bwd.cu -- backward kernels of the mHC layer (sm_103a).
//
// post backward (one warp per token):
//   dx[j] = sum_i H_res[i,j] g[i],  dy = sum_i H_post[i] g[i],
//   dH_post[i] = <g[i], y>,         dH_res[i,j] = <g[i], x[j]>
// pre backward, bf16 widths the cluster kernel tiles (pre_bwd_fused.cu):
//   1. token  (thread per token): gate derivatives, Sinkhorn VJP from the
//      recomputed forward, the post / residual parts of u = inv_rms *
//      alpha_grp * dlogits and their share of the RMSNorm coefficient of x,
//      written to a per-token record (none of it needs dH_pre)
//   2. one-pass cluster kernel: dH_pre, the pre-gate parts, dx, dphi partials
//   3. reduce : dphi over partials, db and dalpha over tokens (fixed order,
//      no atomics)
// otherwise (float32, other widths) five launches:
//   1. dots   (warp per token): dH_pre[i] = <g_in, x[i]>
//   2. token  as above, now with dH_pre
//   3. main   (K slice x token block, tensor cores for bf16 widths that are
//      a multiple of 256): dx += H_pre[i] g_in + phi u + coef x, and the
//      block's partial dphi = sum_t x_t u_t^T
//   4. reduce : as above
// Derivation (with s = inv_rms, v = alpha_grp * dlogits, proj = s * x.phi):
//   dx_norm = s * phi v - s^2 * x * (v . proj) / K,   dphi = sum_t s_t x_t v_t^T
// Layer definition: "openPangu 2.0 -- architecture, training and Ascend
// systems" notes, section 5.3; recompute instead of storing the Sinkhorn
// iterates follows the recompute paragraph of the Ascend mHC Triton operator
// article.
#include "launch.h"
#include "mhc_common.cuh"

namespace mhc {
namespace {

template <typename TA>
__global__ void __launch_bounds__(256)
post_bwd_kernel(const TA* __restrict__ g, const TA* __restrict__ x, const TA* __restrict__ y,
                const float* __restrict__ H_post, const float* __restrict__ H_res, int64_t T,
                int64_t D, TA* __restrict__ dx, TA* __restrict__ dy, float* __restrict__ dH_post,
                float* __restrict__ dH_res) {
    constexpr int V = Vec<TA>::N;
    const int lane = threadIdx.x & 31;
    const int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    const int64_t QD = D / V;
    const float4 hp = reinterpret_cast<const float4*>(H_post)[t];
    const float4* hr4 = reinterpret_cast<const float4*>(H_res + t * 16);
    const float4 r0 = hr4[0], r1 = hr4[1], r2 = hr4[2], r3 = hr4[3];
    const float H[4][4] = {{r0.x, r0.y, r0.z, r0.w}, {r1.x, r1.y, r1.z, r1.w},
                           {r2.x, r2.y, r2.z, r2.w}, {r3.x, r3.y, r3.z, r3.w}};
    const float Hp[4] = {hp.x, hp.y, hp.z, hp.w};
    float ap[4] = {0.f, 0.f, 0.f, 0.f};
    float ar[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) ar[e] = 0.f;

    const TA* gp = g + t * 4 * D;
    const TA* xp = x + t * 4 * D;
    const TA* yp = y + t * D;
    for (int64_t q = lane; q < QD; q += 32) {
        float fg[4][V], fx[4][V], fy[V];
#pragma unroll
        for (int i = 0; i < 4; ++i) Vec<TA>::unpack(ld16_stream(gp + i * D + q * V), fg[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) Vec<TA>::unpack(ld16_stream(xp + j * D + q * V), fx[j]);
        Vec<TA>::unpack(ld16_stream(yp + q * V), fy);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float o[V];
#pragma unroll
            for (int e = 0; e < V; ++e)
                o[e] = fmaf(H[3][j], fg[3][e], fmaf(H[2][j], fg[2][e], fmaf(H[1][j], fg[1][e], H[0][j] * fg[0][e])));
            st16_stream(dx + t * 4 * D + j * D + q * V, Vec<TA>::pack(o));
        }
        {
            float o[V];
#pragma unroll
            for (int e = 0; e < V; ++e)
                o[e] = fmaf(Hp[3], fg[3][e], fmaf(Hp[2], fg[2][e], fmaf(Hp[1], fg[1][e], Hp[0] * fg[0][e])));
            st16_stream(dy + t * D + q * V, Vec<TA>::pack(o));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int e = 0; e < V; ++e) {
                ap[i] = fmaf(fg[i][e], fy[e], ap[i]);
#pragma unroll
                for (int j = 0; j < 4; ++j) ar[4 * i + j] = fmaf(fg[i][e], fx[j][e], ar[4 * i + j]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) ap[i] = warp_sum(ap[i]);
#pragma unroll
    for (int e = 0; e < 16; ++e) ar[e] = warp_sum(ar[e]);
    if (lane == 0) {
        reinterpret_cast<float4*>(dH_post)[t] = make_float4(ap[0], ap[1], ap[2], ap[3]);
        float4* o = reinterpret_cast<float4*>(dH_res + t * 16);
#pragma unroll
        for (int v = 0; v < 4; ++v) o[v] = make_float4(ar[4 * v], ar[4 * v + 1], ar[4 * v + 2], ar[4 * v + 3]);
    }
}

// 1. dH_pre[i] = <g_in, x[i]>, one warp per token.
template <typename TA>
__global__ void __launch_bounds__(256)
pre_bwd_dots_kernel(const TA* __restrict__ g_in, const TA* __restrict__ x, int64_t T, int64_t D,
                    float* __restrict__ rec) {
    constexpr int V = Vec<TA>::N;
    const int lane = threadIdx.x & 31;
    const int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    const int64_t QD = D / V;
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    for (int64_t q = lane; q < QD; q += 32) {
        float fg[V];
        Vec<TA>::unpack(ld16(g_in + t * D + q * V), fg);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float fx[V];
            Vec<TA>::unpack(ld16(x + t * 4 * D + i * D + q * V), fx);
#pragma unroll
            for (int e = 0; e < V; ++e) a[i] = fmaf(fg[e], fx[e], a[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = warp_sum(a[i]);
    if (lane == 0)
        reinterpret_cast<float4*>(rec + t * REC + REC_DHPRE)[0] = make_float4(a[0], a[1], a[2], a[3]);
}

// 2. Per-token gate backward, one thread per token.
__global__ void __launch_bounds__(128)
pre_bwd_token_kernel(const float* __restrict__ dH_post, const float* __restrict__ dH_res,
                     const float* __restrict__ b, const float* __restrict__ alpha,
                     const float* __restrict__ proj, const float* __restrict__ inv_rms, int64_t T,
                     int64_t K, int iters, int have_dhpre, float* __restrict__ rec) {
    // a programmatically dependent kernel after this one may start now; it
    // waits for this kernel's completion before reading the records
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= T) return;
    float* r = rec + t * REC;
    float pj[NG];
#pragma unroll
    for (int v = 0; v < NG / 4; ++v) {
        const float4 p = reinterpret_cast<const float4*>(proj + t * NG)[v];
        pj[4 * v] = p.x; pj[4 * v + 1] = p.y; pj[4 * v + 2] = p.z; pj[4 * v + 3] = p.w;
    }
    float lg[NG];
    make_logits(pj, alpha, b, lg);
    // without dH_pre (the one-pass kernel computes it later) the pre gates'
    // terms are left at zero here and completed there
    const float4 dhp4 = have_dhpre ? reinterpret_cast<const float4*>(r + REC_DHPRE)[0]
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 dhq4 = reinterpret_cast<const float4*>(dH_post)[t];
    const float dhp[4] = {dhp4.x, dhp4.y, dhp4.z, dhp4.w};
    const float dhq[4] = {dhq4.x, dhq4.y, dhq4.z, dhq4.w};
    float dl[NG], hpre[4], dsig[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float sp = sigmoid_f(lg[i]);
        const float sq = sigmoid_f(lg[NS + i]);
        hpre[i] = sp;
        dsig[i] = sp * (1.0f - sp);
        dl[i] = dhp[i] * dsig[i];
        dl[NS + i] = dhq[i] * 2.0f * sq * (1.0f - sq);
    }
    float dhr[16];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const float4 d = reinterpret_cast<const float4*>(dH_res + t * 16)[v];
        dhr[4 * v] = d.x; dhr[4 * v + 1] = d.y; dhr[4 * v + 2] = d.z; dhr[4 * v + 3] = d.w;
    }
    sinkhorn_vjp(lg + 2 * NS, iters, dhr, dl + 2 * NS);

    const float s = inv_rms[t];
    const float a[3] = {alpha[0], alpha[1], alpha[2]};
    float vp = 0.f, da[3] = {0.f, 0.f, 0.f}, u[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        const int grp = group_of(g);
        const float v = a[grp] * dl[g];
        vp = fmaf(v, pj[g], vp);
        da[grp] = fmaf(dl[g], pj[g], da[grp]);
        u[g] = s * v;
    }
    // the record in 16-byte pieces (slots 30, 31 and 59 are unused)
    float4* r4 = reinterpret_cast<float4*>(r);
#pragma unroll
    for (int v = 0; v < NG / 4; ++v) {
        r4[(REC_U >> 2) + v] = make_float4(u[4 * v], u[4 * v + 1], u[4 * v + 2], u[4 * v + 3]);
        r4[(REC_DL >> 2) + v] = make_float4(dl[4 * v], dl[4 * v + 1], dl[4 * v + 2], dl[4 * v + 3]);
    }
    r4[REC_HPRE >> 2] = make_float4(hpre[0], hpre[1], hpre[2], hpre[3]);
    r4[REC_COEF >> 2] = make_float4(-s * s * vp / static_cast<float>(K), s, 0.f, 0.f);
    r4[REC_DSIG >> 2] = make_float4(dsig[0], dsig[1], dsig[2], dsig[3]);
    r4[REC_DA >> 2] = make_float4(da[0], da[1], da[2], 0.f);
}

// 3. dx += H_pre[i] g_in + phi u + coef x over a K slice, and the partial
//    dphi of a token block.  Each thread owns two consecutive k.
constexpr int MB_THREADS = 128;
constexpr int MB_KS = 2 * MB_THREADS;   // K elements per CTA

// Two consecutive activations of one token, kept in their storage form
// (one 32-bit word for bf16, two floats for float32) until they are used.
template <typename TA> struct Pair;
template <> struct Pair<__nv_bfloat16> {
    using Raw = uint32_t;
    __device__ __forceinline__ static Raw load(const __nv_bfloat16* p) {
        return *reinterpret_cast<const uint32_t*>(p);
    }
    __device__ __forceinline__ static float2 widen(Raw w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    __device__ __forceinline__ static void store(__nv_bfloat16* p, float2 v) {
        *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v.x, v.y);
    }
};
template <> struct Pair<float> {
    using Raw = float2;
    __device__ __forceinline__ static Raw load(const float* p) { return *reinterpret_cast<const float2*>(p); }
    __device__ __forceinline__ static float2 widen(Raw w) { return w; }
    __device__ __forceinline__ static void store(float* p, float2 v) { *reinterpret_cast<float2*>(p) = v; }
};

// cp.async of 4 or 8 bytes (zero fill when `valid` is false).
template <int BYTES>
__device__ __forceinline__ void cp_async_small(void* smem, const void* gmem, bool valid) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    const int n = valid ? BYTES : 0;
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;\n" ::"r"(s), "l"(gmem), "n"(BYTES), "r"(n)
                 : "memory");
}
__device__ __forceinline__ void cp_async_16(void* smem, const void* gmem, bool valid) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit_group() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// Packed fused multiply-add on two float32 lanes (fma.rn.f32x2).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(r)
        : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)),
          "l"(*reinterpret_cast<unsigned long long*>(&c)));
    return *reinterpret_cast<float2*>(&r);
}

// Shared-memory pipeline of the main kernel: each stage holds MB_TS tokens'
// records and, per thread, its two activations of x, g_in and dx.
constexpr int MB_TS = 12;
template <typename TA> struct MainCfg {
    static constexpr int STAGES = sizeof(TA) == 2 ? 3 : 2;
    static constexpr int RAW = 2 * static_cast<int>(sizeof(TA));          // bytes per thread per array
    static constexpr int REC_BYTES = MB_TS * 32 * 4;
    static constexpr int ARR_BYTES = MB_TS * MB_THREADS * RAW;
    static constexpr int STAGE_BYTES = REC_BYTES + 3 * ARR_BYTES;
    static constexpr int SMEM = STAGES * STAGE_BYTES;
};

template <typename TA>
__global__ void __launch_bounds__(MB_THREADS)
pre_bwd_main_kernel(const TA* __restrict__ g_in, const TA* __restrict__ x,
                    const float* __restrict__ phi, const float* __restrict__ rec, int64_t T,
                    int64_t D, int64_t tb, TA* __restrict__ dx, float* __restrict__ part) {
    using P = Pair<TA>;
    using Raw = typename P::Raw;
    using Cfg = MainCfg<TA>;
    constexpr int S = Cfg::STAGES;
    extern __shared__ __align__(16) unsigned char msm[];
    const int tid = threadIdx.x;
    const int64_t K = 4 * D;
    const int64_t k0 = static_cast<int64_t>(blockIdx.x) * MB_KS + 2 * tid;
    const bool active = k0 < K;
    const int si = active ? static_cast<int>(k0 / D) : 0;
    const int64_t d0 = active ? k0 - si * D : 0;
    const int64_t tbeg = static_cast<int64_t>(blockIdx.y) * tb;
    const int64_t tend = tbeg + tb < T ? tbeg + tb : T;
    const int ntok = tend > tbeg ? static_cast<int>(tend - tbeg) : 0;
    const int nst = (ntok + MB_TS - 1) / MB_TS;

    auto st_rec = [&](int b) { return reinterpret_cast<float*>(msm + b * Cfg::STAGE_BYTES); };
    auto st_arr = [&](int b, int a) {
        return reinterpret_cast<Raw*>(msm + b * Cfg::STAGE_BYTES + Cfg::REC_BYTES + a * Cfg::ARR_BYTES);
    };
    auto issue = [&](int st) {
        const int b = st % S;
        const int64_t c0 = tbeg + static_cast<int64_t>(st) * MB_TS;
        float* r = st_rec(b);
        for (int q = tid; q < MB_TS * 8; q += MB_THREADS) {
            const int tt = q >> 3, v = q & 7;
            const bool ok = c0 + tt < tend;
            cp_async_16(r + tt * 32 + v * 4, ok ? rec + (c0 + tt) * REC + v * 4 : rec, ok);
        }
        Raw* xa = st_arr(b, 0);
        Raw* ga = st_arr(b, 1);
        Raw* da = st_arr(b, 2);
#pragma unroll 4
        for (int tt = 0; tt < MB_TS; ++tt) {
            const int64_t t = c0 + tt;
            const bool ok = active && t < tend;
            cp_async_small<sizeof(Raw)>(xa + tt * MB_THREADS + tid, ok ? x + t * K + k0 : x, ok);
            cp_async_small<sizeof(Raw)>(ga + tt * MB_THREADS + tid, ok ? g_in + t * D + d0 : g_in, ok);
            cp_async_small<sizeof(Raw)>(da + tt * MB_THREADS + tid, ok ? dx + t * K + k0 : dx, ok);
        }
    };

    // phi rows k0, k0+1 and the dphi accumulators, paired per logit g
    float2 ph[NG], acc[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        ph[g] = active ? make_float2(phi[k0 * NG + g], phi[(k0 + 1) * NG + g]) : make_float2(0.f, 0.f);
        acc[g] = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int st = 0; st < S - 1; ++st) {
        if (st < nst) issue(st);
        cp_async_commit_group();
    }
    for (int st = 0; st < nst; ++st) {
        cp_async_wait_group<S - 2>();
        __syncthreads();   // stage st landed for every thread; stage st-1 is free
        if (st + S - 1 < nst) issue(st + S - 1);
        cp_async_commit_group();
        const int b = st % S;
        const float* r = st_rec(b);
        const Raw* xa = st_arr(b, 0);
        const Raw* ga = st_arr(b, 1);
        const Raw* da = st_arr(b, 2);
        const int64_t c0 = tbeg + static_cast<int64_t>(st) * MB_TS;
        const int nt = static_cast<int>(tend - c0 < MB_TS ? tend - c0 : MB_TS);
        if (active) {
            for (int tt = 0; tt < nt; ++tt) {
                const float2 xv = P::widen(xa[tt * MB_THREADS + tid]);
                const float2 gv = P::widen(ga[tt * MB_THREADS + tid]);
                const float2 dv = P::widen(da[tt * MB_THREADS + tid]);
                const float4* u4 = reinterpret_cast<const float4*>(r + tt * 32);
                float2 sa = make_float2(0.f, 0.f), sb = make_float2(0.f, 0.f);   // (phi u) for k0, k0+1
#pragma unroll
                for (int v = 0; v < NG / 4; ++v) {
                    const float4 u = u4[v];
                    const float uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int g = 4 * v + e;
                        const float2 u2 = make_float2(uu[e], uu[e]);
                        if (e & 1) sb = ffma2(ph[g], u2, sb);
                        else sa = ffma2(ph[g], u2, sa);
                        acc[g] = ffma2(xv, u2, acc[g]);
                    }
                }
                const float s0 = sa.x + sb.x, s1 = sa.y + sb.y;
                const float hpre = r[tt * 32 + REC_HPRE + si], coef = r[tt * 32 + REC_COEF];
                float2 o;
                o.x = dv.x + fmaf(hpre, gv.x, fmaf(coef, xv.x, s0));
                o.y = dv.y + fmaf(hpre, gv.y, fmaf(coef, xv.y, s1));
                P::store(dx + (c0 + tt) * K + k0, o);
            }
        }
    }
    cp_async_wait_group<0>();
    if (active) {
        float* p = part + (static_cast<int64_t>(blockIdx.y) * K + k0) * NG;
#pragma unroll
        for (int g = 0; g < NG; ++g) { p[g] = acc[g].x; p[NG + g] = acc[g].y; }
    }
}

template <typename TA>
void set_main_smem_once() {
    static bool done = false;   // the attribute is per function and context-wide
    if (!done) {
        cudaFuncSetAttribute(pre_bwd_main_kernel<TA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             MainCfg<TA>::SMEM);
        done = true;
    }
}

constexpr int BIAS_W = 28;          // bias partial: dlogits[24], da[3], one unused float

// 4a. dphi = sum over token blocks of the partials (fixed order).
__global__ void __launch_bounds__(256)
pre_bwd_reduce_phi_kernel(const float* __restrict__ part, int64_t nb, int64_t n4,
                          float* __restrict__ dphi, const float* __restrict__ bpart, int nbb,
                          float* __restrict__ db, float* __restrict__ dalpha) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        // the partials' loads go out four at a time (one round trip per four
        // blocks, not per block); the sum keeps block order
        const float4* pp = reinterpret_cast<const float4*>(part) + i;
        float4 s = pp[0];
        int64_t bb = 1;
        for (; bb + 4 <= nb; bb += 4) {
            const float4 v0 = pp[bb * n4], v1 = pp[(bb + 1) * n4], v2 = pp[(bb + 2) * n4], v3 = pp[(bb + 3) * n4];
            s.x += v0.x; s.y += v0.y; s.z += v0.z; s.w += v0.w;
            s.x += v1.x; s.y += v1.y; s.z += v1.z; s.w += v1.w;
            s.x += v2.x; s.y += v2.y; s.z += v2.z; s.w += v2.w;
            s.x += v3.x; s.y += v3.y; s.z += v3.z; s.w += v3.w;
        }
        for (; bb < nb; ++bb) {
            const float4 v = pp[bb * n4];
            s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
        }
        reinterpret_cast<float4*>(dphi)[i] = s;
    }
    // db and dalpha: the bias partials of every token block, in block order
    if (blockIdx.x == 0 && threadIdx.x < NG + 3) {
        float tot = 0.f;
        for (int b = 0; b < nbb; ++b) tot += bpart[b * BIAS_W + threadIdx.x];
        if (threadIdx.x < NG) db[threadIdx.x] = tot;
        else dalpha[threadIdx.x - NG] = tot;
    }
}

// 4b. db[g] = sum_t dlogits[t, g] and dalpha[c] = sum_t da[t, c], in two
//     deterministic steps.  Here, block b sums its contiguous token range:
//     a warp reads four tokens' 28 floats (dlogits[24], da[3], one unused)
//     at a time as float4 pieces, lanes 7k + v holding piece v of token k;
//     then a fixed-shape tree over the lanes and the warps.  The per-block
//     partials [nbb][28] are summed in order by block 0 of the dphi reduction.
__global__ void __launch_bounds__(256)
pre_bwd_bias_partial_kernel(const float* __restrict__ rec, int64_t T, float* __restrict__ bpart) {
    __shared__ float4 wsum[8][BIAS_W / 4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t per = (T + gridDim.x - 1) / gridDim.x;
    const int64_t t_begin = static_cast<int64_t>(blockIdx.x) * per;
    const int64_t t_end = t_begin + per < T ? t_begin + per : T;
    const int k = lane / 7, v = lane - 7 * (lane / 7);   // token slot, piece
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane < 28) {
        // loads of four token rows per round trip; the sum keeps token order
#pragma unroll 4
        for (int64_t t = t_begin + warp * 4 + k; t < t_end; t += 32) {
            const float4 a = reinterpret_cast<const float4*>(rec + t * REC + REC_DL)[v];
            acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
        }
    }
    // lanes v, v + 7, v + 14, v + 21 hold piece v of the four token slots
#pragma unroll
    for (int j = 1; j < 4; ++j) {
        const float x = __shfl_sync(0xffffffffu, acc.x, (lane + 7 * j) & 31);
        const float y = __shfl_sync(0xffffffffu, acc.y, (lane + 7 * j) & 31);
        const float z = __shfl_sync(0xffffffffu, acc.z, (lane + 7 * j) & 31);
        const float w = __shfl_sync(0xffffffffu, acc.w, (lane + 7 * j) & 31);
        if (lane < 7) { acc.x += x; acc.y += y; acc.z += z; acc.w += w; }
    }
    if (lane < 7) wsum[warp][lane] = acc;
    __syncthreads();
    if (threadIdx.x < BIAS_W / 4) {
        float4 tot = wsum[0][threadIdx.x];
#pragma unroll
        for (int w2 = 1; w2 < 8; ++w2) {
            const float4 a = wsum[w2][threadIdx.x];
            tot.x += a.x; tot.y += a.y; tot.z += a.z; tot.w += a.w;
        }
        reinterpret_cast<float4*>(bpart + static_cast<int64_t>(blockIdx.x) * BIAS_W)[threadIdx.x] = tot;
    }
}

}  // namespace

PreBwdPlan pre_bwd_plan(int64_t T, int64_t D) {
    PreBwdPlan p{};
    const int64_t K = 4 * D;
    int64_t nb = (T + 255) / 256;
    if (nb > 16) nb = 16;
    if (nb < 1) nb = 1;
    p.nb = nb;
    p.tb = (T + nb - 1) / nb;
    p.rec_bytes = static_cast<size_t>(T) * REC * sizeof(float);
    p.part_bytes = static_cast<size_t>(nb) * K * NG * sizeof(float);
    p.phi_bytes = pre_bwd_fused_phi_bytes(D);
    p.total_bytes = T > 0 ? p.rec_bytes + p.part_bytes + p.phi_bytes : 0;
    return p;
}

cudaError_t launch_post_bwd(bool bf16, const void* g, const void* x, const void* y,
                            const float* H_post, const float* H_res, int64_t T, int64_t D,
                            void* dx, void* dy, float* dH_post, float* dH_res, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>((T * 32 + 255) / 256));
    if (bf16)
        post_bwd_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(g), static_cast<const __nv_bfloat16*>(x),
            static_cast<const __nv_bfloat16*>(y), H_post, H_res, T, D, static_cast<__nv_bfloat16*>(dx),
            static_cast<__nv_bfloat16*>(dy), dH_post, dH_res);
    else
        post_bwd_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(g), static_cast<const float*>(x),
                                                    static_cast<const float*>(y), H_post, H_res, T, D,
                                                    static_cast<float*>(dx), static_cast<float*>(dy),
                                                    dH_post, dH_res);
    return cudaGetLastError();
}

// The pre backward with room for at most nb dphi partials (scratch = T * REC
// floats of records, nb * K * NG floats of partials, then D * 256 bytes of
// bf16 phi blocks): launch_pre_bwd passes the plan's nb, the entry point with
// a fixed scratch array its own.
cudaError_t launch_pre_bwd_blocks(bool bf16, const void* g_in, const float* dH_post,
                                  const float* dH_res, const void* x, const float* phi,
                                  const float* b, const float* alpha, const float* proj,
                                  const float* inv_rms, int64_t T, int64_t D, int iters, void* dx,
                                  float* dphi, float* db, float* dalpha, void* ws, int64_t nb,
                                  cudaStream_t s) {
    const int64_t K = 4 * D;
    const int64_t tb = (T + nb - 1) / nb;
    float* rec = static_cast<float*>(ws);
    float* part = reinterpret_cast<float*>(static_cast<char*>(ws) + static_cast<size_t>(T) * REC * sizeof(float));
    const dim3 gw(static_cast<unsigned>((T * 32 + 255) / 256));
    const dim3 gt(static_cast<unsigned>((T + 127) / 128));
    const dim3 gm(static_cast<unsigned>((K + MB_KS - 1) / MB_KS), static_cast<unsigned>(nb));
    int64_t nparts = nb;
    if (bf16 && pre_bwd_fused_supports(T, D)) {
        // one pass: phi packed for the cluster kernel, the per-token gate
        // backward (it does not need dH_pre), then the cluster kernel finds
        // dH_pre and does the rest; it starts while the per-token kernel
        // finishes and waits for its records only where it reads them
        void* phi2 = static_cast<char*>(ws) + static_cast<size_t>(T) * REC * sizeof(float) +
                     static_cast<size_t>(nb) * K * NG * sizeof(float);
        const cudaError_t ep = launch_pre_bwd_phi_pack(phi, D, phi2, s);
        if (ep != cudaSuccess) return ep;
        pre_bwd_token_kernel<<<gt, 128, 0, s>>>(dH_post, dH_res, b, alpha, proj, inv_rms, T, K, iters, 0, rec);
        const cudaError_t e = launch_pre_bwd_fused_main(g_in, x, phi, proj, alpha, rec, T, D, nb, dx, part,
                                                        phi2, &nparts, s);
        if (e != cudaSuccess) return e;
    } else if (bf16) {
        pre_bwd_dots_kernel<__nv_bfloat16><<<gw, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(g_in),
                                                              static_cast<const __nv_bfloat16*>(x), T, D, rec);
        pre_bwd_token_kernel<<<gt, 128, 0, s>>>(dH_post, dH_res, b, alpha, proj, inv_rms, T, K, iters, 1, rec);
        if (pre_bwd_tc_supports(T, D)) {
            const cudaError_t e = launch_pre_bwd_tc_main(g_in, x, phi, rec, T, D, nb, dx, part, s);
            if (e != cudaSuccess) return e;
        } else {
            set_main_smem_once<__nv_bfloat16>();
            pre_bwd_main_kernel<__nv_bfloat16><<<gm, MB_THREADS, MainCfg<__nv_bfloat16>::SMEM, s>>>(
                static_cast<const __nv_bfloat16*>(g_in), static_cast<const __nv_bfloat16*>(x), phi, rec, T, D,
                tb, static_cast<__nv_bfloat16*>(dx), part);
        }
    } else {
        pre_bwd_dots_kernel<float><<<gw, 256, 0, s>>>(static_cast<const float*>(g_in),
                                                      static_cast<const float*>(x), T, D, rec);
        pre_bwd_token_kernel<<<gt, 128, 0, s>>>(dH_post, dH_res, b, alpha, proj, inv_rms, T, K, iters, 1, rec);
        set_main_smem_once<float>();
        pre_bwd_main_kernel<float><<<gm, MB_THREADS, MainCfg<float>::SMEM, s>>>(static_cast<const float*>(g_in),
                                                             static_cast<const float*>(x), phi, rec, T, D,
                                                             tb, static_cast<float*>(dx), part);
    }
    const int64_t n4 = K * NG / 4;
    const dim3 gr(static_cast<unsigned>((n4 + 255) / 256 < 4096 ? (n4 + 255) / 256 : 4096));
    // the bias partials go where the bf16 phi blocks were (dead once the
    // main kernel is done; the region is reserved on every path)
    float* bpart = reinterpret_cast<float*>(static_cast<char*>(ws) + static_cast<size_t>(T) * REC * sizeof(float) +
                                            static_cast<size_t>(nb) * K * NG * sizeof(float));
    int64_t nbb = (T + 255) / 256;
    const int64_t fit = static_cast<int64_t>(pre_bwd_fused_phi_bytes(D) / (BIAS_W * sizeof(float)));
    if (nbb > 128) nbb = 128;
    if (nbb > fit) nbb = fit;
    if (nbb < 1) nbb = 1;
    pre_bwd_bias_partial_kernel<<<static_cast<unsigned>(nbb), 256, 0, s>>>(rec, T, bpart);
    pre_bwd_reduce_phi_kernel<<<gr, 256, 0, s>>>(part, nparts, n4, dphi, bpart, static_cast<int>(nbb), db, dalpha);
    return cudaGetLastError();
}

cudaError_t launch_pre_bwd(bool bf16, const void* g_in, const float* dH_post,
                           const float* dH_res, const void* x, const float* phi, const float* b,
                           const float* alpha, const float* proj, const float* inv_rms, int64_t T,
                           int64_t D, int iters, void* dx, float* dphi, float* db, float* dalpha,
                           void* ws, cudaStream_t s) {
    return launch_pre_bwd_blocks(bf16, g_in, dH_post, dH_res, x, phi, b, alpha, proj, inv_rms, T, D, iters,
                                 dx, dphi, db, dalpha, ws, pre_bwd_plan(T, D).nb, s);
}

}  // namespace mhc
