// pre_small.cu -- the pre forward of the mHC layer for decode-sized batches
// (bf16, at most 56 tokens: one cluster per eight).
//
// What it computes is the same per-token map as the tensor-core kernel
// (section 5.3 of the "openPangu 2.0 -- architecture, training and Ascend
// systems" notes): inv_rms over the flattened 4*D row, proj = x_bar . phi
// (24 logits), the gates (Sinkhorn for H_res only when H_res is asked for),
// and x_in = sum_i H_pre[i] x[i] when x_in is asked for.
//
// At a few tokens the work is reading phi (4*D x 24 floats, 1.97 MB at
// D = 5120) and a chain of latencies; the tensor-core kernel's ring of
// 64-token boxes and its eight MMAs per stage only add to that chain.  Here
// one cluster of 16 CTAs (one per SM) per eight tokens splits K (each cluster
// reads all of phi; the later ones from L2):
//   * CTA c brings its K-slice of phi (fp32, contiguous) into shared memory
//     with one bulk copy, and the tokens' matching slices of x with plain
//     loads by every thread meanwhile;
//   * each warp takes 1/16 of the slice's rows; lane (token, group of six
//     logits, row phase) accumulates in fp32, and for one logit group the
//     token's squares;
//   * the warps' partials are added in a fixed order, and each token's
//     CTA partial goes (distributed shared memory, then a cluster barrier) to
//     the CTA that owns the token, which adds the 16 partials in CTA order,
//     forms inv_rms, proj and H_pre and broadcasts H_pre to the cluster;
//   * after a second cluster barrier every CTA mixes its share of the
//     columns (warps 1..15) while warp 0 of each owner runs the other gates
//     and Sinkhorn.
// Every sum runs in a fixed order, so results do not depend on timing, and
// mhc_pre, mhc_pre_gates and mhc_pre_critical agree bit for bit.  The one
// wait, on phi's bulk copy, is bounded (about a second); on expiry the kernel
// latches its device error word and skips its work, still passing both
// cluster barriers (the call's outputs are then not valid).
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "launch.h"
#include "mhc_common.cuh"
#include "tc_ptx.cuh"

namespace mhc {

// This file's device error word (latched when the bounded wait runs out).
__device__ unsigned g_small_error;

cudaError_t read_and_clear_small_error(unsigned* word) {
    cudaError_t e = cudaMemcpyFromSymbol(word, g_small_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_small_error, &zero, sizeof(unsigned));
}

namespace sm {

constexpr int CS = 16;                 // CTAs of the cluster
constexpr int NT = 512;                // 16 warps
constexpr int NW = NT / 32;
constexpr int TMAX = 8;                // tokens per cluster
constexpr int TCAP = 56;               // tokens per launch (one cluster per TMAX)
constexpr int PF = 28;                 // partial record: 24 logits, sum of x^2, pad (floats)
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;   // 1 s

struct Params {
    const __nv_bfloat16* x;
    const float* phi;
    const float* b;
    const float* alpha;
    int T, D, iters;
    float eps;
    unsigned force_timeout;            // test hook
    __nv_bfloat16* x_in;
    float* H_pre;
    float* H_post;
    float* H_res;
    float* proj;
    float* inv_rms;
};

// Byte offsets in the dynamic shared memory of a width D (KS = D / 4 rows
// of phi and x per CTA).
struct Layout {
    uint32_t phi, xs, xrow, wpart, recv, hpre, gate, bar, total;
    __host__ __device__ static Layout make(int D) {
        Layout L;
        const uint32_t ks = static_cast<uint32_t>(D / 4);
        L.phi = 0;                                     // [KS][24] fp32
        L.xs = ks * NG * 4;                            // [TMAX][KS] bf16, rows padded by 16 B
        L.xrow = ks * 2 + 16;
        L.wpart = L.xs + TMAX * L.xrow;                // [NW][TMAX][PF]
        L.recv = L.wpart + NW * TMAX * PF * 4;         // [CS][PF]: the partials of this CTA's token
        L.hpre = L.recv + CS * PF * 4;                 // [TMAX][4]
        L.gate = L.hpre + TMAX * 16;                   // alpha[3], b[24]
        L.bar = L.gate + 32 * 4;
        L.total = L.bar + 16;
        return L;
    }
};

template <int RP>
__global__ void __launch_bounds__(NT, 1) pre_small_kernel(const Params batch) {
    extern __shared__ __align__(128) unsigned char smem[];
    // cluster j takes tokens [TMAX j, TMAX j + T) of the batch
    const int j0 = static_cast<int>(ptx::cluster_id_x()) * TMAX;
    Params p = batch;
    p.x += static_cast<int64_t>(j0) * 4 * p.D;
    if (p.x_in != nullptr) p.x_in += static_cast<int64_t>(j0) * p.D;
    p.H_pre += j0 * 4;
    if (p.H_post != nullptr) p.H_post += j0 * 4;
    if (p.H_res != nullptr) p.H_res += j0 * 16;
    p.proj += j0 * NG;
    p.inv_rms += j0;
    const int D = p.D, T = min(TMAX, batch.T - j0);
    const int KS = D / 4;
    const int64_t K = 4ll * D;
    const Layout L = Layout::make(D);
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bar = sbase + L.bar;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t c = ptx::cluster_ctarank();
    constexpr unsigned FULL = 0xffffffffu;

    if (p.force_timeout != 0u) {
        // test hook: one bounded wait that runs out, before any copy or
        // cluster exchange; every CTA of the launch leaves here
        if (tid == 0 && ptx::forced_wait_runs_out(bar, 100000ull)) atomicOr(&g_small_error, 1u);
        __syncthreads();
        return;
    }

    // ---- the CTA's K-slice of phi and of every token's x row ---------------
    float* gate_par = reinterpret_cast<float*>(smem + L.gate);
    if (tid < 3) gate_par[tid] = p.alpha[tid];
    if (tid >= 32 && tid < 32 + NG) gate_par[3 + tid - 32] = p.b[tid - 32];
    if (tid == 0) {
        ptx::mbar_init(bar, 1);
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(KS) * NG * 4);
        ptx::bulk_load(sbase + L.phi, p.phi + static_cast<int64_t>(c) * KS * NG, static_cast<uint32_t>(KS) * NG * 4, bar);
    }
    // the tokens' x slices with plain 16-byte loads by every thread, while
    // phi's copy is in flight
    {
        const int pieces = KS / 8;                     // 16-byte pieces of a token's slice
        for (int item = tid; item < T * pieces; item += NT) {
            const int t = item / pieces, q = item % pieces;
            *reinterpret_cast<uint4*>(smem + L.xs + t * L.xrow + q * 16) =
                ld16(p.x + t * K + static_cast<int64_t>(c) * KS + q * 8);
        }
    }
    __syncthreads();
    bool landed = ptx::mbar_try_wait(bar, 0);
    if (!landed) {
        const uint64_t t0 = ptx::globaltimer();
        while (!(landed = ptx::mbar_try_wait(bar, 0))) {
            if (ptx::globaltimer() - t0 > WAIT_LIMIT_NS) break;
        }
    }
    const bool ok = __syncthreads_and(landed) != 0;
    if (!ok && tid == 0) atomicOr(&g_small_error, 1u);

    // ---- partial dot products: warp w takes rows [w RW, (w + 1) RW) --------
    // Lane (t, lg, rp) = (lane / 4RP, lane / RP % 4, lane % RP) accumulates
    // logits 6 lg .. 6 lg + 5 of token t over the rows whose index within each
    // group of eight is rp mod RP (and, for lg = 0, their squares); the RP
    // lanes of one (t, lg) are added at the end.  With RP = 8 / (tokens a
    // warp covers) every lane works at any batch, and the warp's instruction
    // count does not grow with the number of tokens.
    const float* phs = reinterpret_cast<const float*>(smem + L.phi);
    float* wpart = reinterpret_cast<float*>(smem + L.wpart);
    if (ok) {
        const int RW = KS / NW;                        // a multiple of 8
        const int t = lane / (4 * RP), lg = (lane / RP) & 3, rp = lane % RP;
        float acc[6], sq = 0.f;
        {
            // logit pairs through packed fp32 multiply-adds (each lane rounds
            // as fmaf: the same chain per logit as one at a time)
            float2 a01 = make_float2(0.f, 0.f), a23 = a01, a45 = a01;
            if (t < T) {
                const __nv_bfloat16* xr = reinterpret_cast<const __nv_bfloat16*>(smem + L.xs + t * L.xrow);
                for (int k0 = warp * RW; k0 < (warp + 1) * RW; k0 += 8) {
#pragma unroll
                    for (int i = 0; i < 8 / RP; ++i) {
                        const int k = k0 + rp + RP * i;
                        const float xv = __bfloat162float(xr[k]);
                        const float2 xv2 = make_float2(xv, xv);
                        const float2* ph2 = reinterpret_cast<const float2*>(phs + k * NG + 6 * lg);
                        a01 = __ffma2_rn(xv2, ph2[0], a01);
                        a23 = __ffma2_rn(xv2, ph2[1], a23);
                        a45 = __ffma2_rn(xv2, ph2[2], a45);
                        if (lg == 0) sq = fmaf(xv, xv, sq);
                    }
                }
            }
            acc[0] = a01.x; acc[1] = a01.y; acc[2] = a23.x; acc[3] = a23.y; acc[4] = a45.x; acc[5] = a45.y;
        }
#pragma unroll
        for (int m = 1; m < RP; m <<= 1) {
#pragma unroll
            for (int j = 0; j < 6; ++j) acc[j] += __shfl_xor_sync(FULL, acc[j], m);
            sq += __shfl_xor_sync(FULL, sq, m);
        }
        if (t < T && rp == 0) {
            float* wp = wpart + (warp * TMAX + t) * PF;
#pragma unroll
            for (int j = 0; j < 6; ++j) wp[6 * lg + j] = acc[j];
            if (lg == 0) wp[NG] = sq;
        }
    }
    __syncthreads();
    // the CTA's partial record of token t (warps added in order) to the CTA
    // that owns token t
    if (ok && tid < T * (NG + 1)) {
        const int t = tid / (NG + 1), g = tid % (NG + 1);
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) v += wpart[(w * TMAX + t) * PF + g];
        const uint32_t dst = ptx::mapa(sbase + L.recv + (c * PF + g) * 4, static_cast<uint32_t>(t));
        asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dst), "f"(v) : "memory");
    }
    ptx::cluster_sync();

    // ---- the owner of token t = c: sums, inv_rms, proj, H_pre -------------
    const int t_own = static_cast<int>(c);
    float pj[NG], inv = 0.f;
    if (t_own < T && warp == 0) {
        const float* recv = reinterpret_cast<const float*>(smem + L.recv);
        float v = 0.f;
        if (lane <= NG)
            for (int s = 0; s < CS; ++s) v += recv[s * PF + lane];
        const float sq = __shfl_sync(FULL, v, NG);
        inv = 1.0f / sqrtf(sq / static_cast<float>(K) + p.eps);
#pragma unroll
        for (int g = 0; g < NG; ++g) pj[g] = __shfl_sync(FULL, v, g) * inv;
        float hp[4];
        token_pre_gates(pj, gate_par, gate_par + 3, hp);
        // H_pre to every CTA of the cluster (lane s writes CTA s's copy)
        if (lane < CS) {
            const uint32_t dst = ptx::mapa(sbase + L.hpre + t_own * 16, static_cast<uint32_t>(lane));
            ptx::st_cluster_v4(dst, hp[0], hp[1], hp[2], hp[3]);
        }
        if (lane == 0 && ok) {
            reinterpret_cast<float4*>(p.H_pre)[t_own] = make_float4(hp[0], hp[1], hp[2], hp[3]);
            p.inv_rms[t_own] = inv;
#pragma unroll
            for (int v4 = 0; v4 < NG / 4; ++v4)
                reinterpret_cast<float4*>(p.proj + static_cast<int64_t>(t_own) * NG)[v4] =
                    make_float4(pj[4 * v4], pj[4 * v4 + 1], pj[4 * v4 + 2], pj[4 * v4 + 3]);
        }
    }
    ptx::cluster_sync();   // H_pre of every token is in every CTA; no remote access after this

    // ---- mix: CTA c takes the 16-byte column pieces c, c + 16, ... ---------
    if (ok && p.x_in != nullptr) {
        const float4* hb = reinterpret_cast<const float4*>(smem + L.hpre);
        const int qpt = D / 8;                         // pieces per stream row
        const int per = (qpt - static_cast<int>(c) + CS - 1) / CS;
        // warps 1.. only: warp 0 of a token's owner runs Sinkhorn meanwhile
        for (int item = tid - 32; item < T * per; item += NT - 32) {
            if (item < 0) break;
            const int t = item / per, qq = static_cast<int>(c) + (item % per) * CS;
            const __nv_bfloat16* src = p.x + t * K + qq * 8;
            uint4 xv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) xv[i] = ld16(src + static_cast<int64_t>(i) * D);
            const float4 h = hb[t];
            st16_stream(p.x_in + static_cast<int64_t>(t) * D + qq * 8, mix4_bf16(xv[0], xv[1], xv[2], xv[3], h));
        }
    }
    // ---- the owner: the other gates (off the mix's path) -------------------
    if (ok && t_own < T && warp == 0 && p.H_res != nullptr) {
        float hp[4], hq[4], hr[16];
        token_gates(pj, gate_par, gate_par + 3, p.iters, hp, hq, hr);
        if (lane == 0) reinterpret_cast<float4*>(p.H_post)[t_own] = make_float4(hq[0], hq[1], hq[2], hq[3]);
        if (lane >= 1 && lane <= 4) {
            const int r = lane - 1;
            float4 o = make_float4(hr[0], hr[1], hr[2], hr[3]);
#pragma unroll
            for (int v4 = 1; v4 < 4; ++v4)
                if (r == v4) o = make_float4(hr[4 * v4], hr[4 * v4 + 1], hr[4 * v4 + 2], hr[4 * v4 + 3]);
            reinterpret_cast<float4*>(p.H_res + static_cast<int64_t>(t_own) * 16)[r] = o;
        }
    }
    if (!ok) {
        // let a copy still in flight land before the shared memory goes away
        const uint64_t t0 = ptx::globaltimer();
        while (ptx::globaltimer() - t0 < 20000ull) {
        }
    }
}

}  // namespace sm

// Clusters of the small-batch kernel that can be resident at once at width D,
// per device.  The clusters of a launch are independent (each reads all of
// phi); the path is taken only when they all fit at once, so that a batch
// costs one cluster's latency.
int small_clusters_resident(int64_t D) {
    static std::mutex mu;
    static int cached_dev[8] = {-1, -1, -1, -1, -1, -1, -1, -1};
    static int64_t cached_D[8];
    static int cached_n[8];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < 8; ++i)
        if (cached_dev[i] == dev && cached_D[i] == D) return cached_n[i];
    const size_t smem = sm::Layout::make(static_cast<int>(D)).total;
    auto k = sm::pre_small_kernel<1>;
    int n = 0;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) == cudaSuccess &&
        cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(sm::CS * 16);
        cfg.blockDim = dim3(sm::NT);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = sm::CS;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) n = 0;
    }
    for (int i = 0; i < 8; ++i)
        if (cached_dev[i] < 0) {
            cached_dev[i] = dev;
            cached_D[i] = D;
            cached_n[i] = n;
            break;
        }
    return n;
}

bool pre_small_supports(int64_t T, int64_t D) {
    if (T < 1 || T > sm::TCAP || D <= 0 || D % 512 != 0) return false;
    int dev = 0, optin = 0, cl = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&cl, cudaDevAttrClusterLaunch, dev) != cudaSuccess || cl == 0)
        return false;
    if (sm::Layout::make(static_cast<int>(D)).total > static_cast<uint32_t>(optin)) return false;
    return small_clusters_resident(D) >= static_cast<int>((T + sm::TMAX - 1) / sm::TMAX);
}

cudaError_t launch_pre_small(const void* x, const float* phi, const float* b, const float* alpha, int64_t T,
                             int64_t D, int iters, float eps, void* x_in, float* H_pre, float* H_post,
                             float* H_res, float* proj, float* inv_rms, unsigned force_timeout, cudaStream_t s) {
    const size_t smem = sm::Layout::make(static_cast<int>(D)).total;
    // row phases per (token, logit group): all 32 lanes of a warp busy
    void (*k)(sm::Params) = T <= 1 ? sm::pre_small_kernel<8>
                          : T <= 2 ? sm::pre_small_kernel<4>
                          : T <= 4 ? sm::pre_small_kernel<2>
                                   : sm::pre_small_kernel<1>;   // clusters of eight tokens
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    sm::Params prm;
    prm.x = static_cast<const __nv_bfloat16*>(x);
    prm.phi = phi;
    prm.b = b;
    prm.alpha = alpha;
    prm.T = static_cast<int>(T);
    prm.D = static_cast<int>(D);
    prm.iters = iters;
    prm.eps = eps;
    prm.force_timeout = force_timeout;
    prm.x_in = static_cast<__nv_bfloat16*>(x_in);
    prm.H_pre = H_pre;
    prm.H_post = H_post;
    prm.H_res = H_res;
    prm.proj = proj;
    prm.inv_rms = inv_rms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sm::CS * ((T + sm::TMAX - 1) / sm::TMAX)));
    cfg.blockDim = dim3(sm::NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = sm::CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, prm);
}

}  // namespace mhc
