// pre_tc.cu -- fused tensor-core pre forward of the mHC layer (bf16, n = 4),
// and the library's device error word.
//
// What it computes, per token (section 5.3 of the "openPangu 2.0 --
// architecture, training and Ascend systems" notes): inv_rms over the
// flattened 4*D row, proj = x_bar . phi (24 logits), gates and Sinkhorn, and
// x_in = sum_i H_pre[i] x[i].
//
// Design (GB300, one CTA per SM, persistent):
//   * A cluster of C CTAs owns a tile of 128 tokens at a time.  CTA c owns the
//     D-slice [c*D/C, (c+1)*D/C) of every stream, i.e. a K-slice of 4*D/C
//     columns of the projection, whose phi rows stay resident in shared
//     memory as bf16 hi + lo halves (phi = hi + lo to 2^-17 relative).
//   * A TMA producer warp streams the tile's x slice (128 tokens x 64
//     columns per stage, 128-byte swizzle) through a ring of stages; one
//     thread issues tcgen05.mma (M = 128 tokens, N = 48 = 24 hi + 24 lo
//     columns, K = 16) accumulating in TMEM (two accumulators, so the next
//     tile's MMAs overlap this tile's epilogue); four warps sum x^2 per token
//     from the same stages.
//   * Eight epilogue warps read the partial logits from TMEM, publish them in
//     shared memory, and each CTA reduces 128/C tokens over the cluster's C
//     partials through distributed shared memory, computes the gates and
//     Sinkhorn, writes them out and pushes H_pre back to every CTA.  Each
//     CTA then mixes its own D-slice: x is read from HBM once (TMA, kept in
//     L2 with an evict-last hint) and read a second time from L2 for the mix.
//   * Every wait is bounded (about one second); on expiry the kernel latches
//     the device error word, lets the other roles drain and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "launch.h"
#include "mhc_common.cuh"
#include "tc_ptx.cuh"

namespace mhc {

// Latched by kernels whose bounded waits ran out; read and cleared by
// mhc_get_last_device_error().
__device__ unsigned g_device_error;

cudaError_t read_and_clear_bwd_tc_error(unsigned* word);      // pre_bwd_tc.cu
cudaError_t read_and_clear_bwd_fused_error(unsigned* word);   // pre_bwd_fused.cu

cudaError_t read_and_clear_device_error(unsigned* word, cudaStream_t s) {
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(word, g_device_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    unsigned other = 0;
    e = read_and_clear_bwd_tc_error(&other);
    if (e != cudaSuccess) return e;
    *word |= other;
    other = 0;
    e = read_and_clear_bwd_fused_error(&other);
    *word |= other;
    return e;
}

namespace tc {

constexpr int TILE_M = 128;                       // tokens per tile (MMA M)
constexpr int KW = 64;                            // K columns per stage (128 B rows)
constexpr int STAGES = 5;
constexpr int NB = 48;                            // MMA N: 24 hi + 24 lo
constexpr int STAGE_BYTES = TILE_M * KW * 2;      // 16 KB
constexpr int PHI_CHUNK_BYTES = NB * KW * 2;      // 6 KB
constexpr int MAX_NCH = 20;                       // K-slice <= 1280 columns
constexpr int NTHREADS = 512;                     // 16 warps
constexpr int SS_WARP0 = 2, NSS = 2;              // x^2 warps (two token rows per lane)
constexpr int GATE_WARP0 = 4, NGATE = 4;          // TMEM readers, cluster reduction, gates
constexpr int MIX_WARP0 = 8, NMIX = 8;            // x_in = sum_i H_pre[i] x[i]
constexpr int REC = 25;                           // partial record: 24 logits + sum x^2
constexpr int TMEM_COLS = 128;                    // two 64-column accumulators
constexpr uint32_t IDESC = ptx::idesc_bf16_f32(TILE_M, NB);
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;  // 1 s

enum : int {
    BAR_FULL = 0,
    BAR_EMPTY = BAR_FULL + STAGES,
    BAR_ACC_FULL = BAR_EMPTY + STAGES,
    BAR_ACC_EMPTY = BAR_ACC_FULL + 2,
    BAR_SS_FULL = BAR_ACC_EMPTY + 2,
    BAR_SS_EMPTY = BAR_SS_FULL + 2,
    BAR_PEER = BAR_SS_EMPTY + 2,
    BAR_HPRE = BAR_PEER + 1,
    BAR_MIX_DONE = BAR_HPRE + 2,
    NBARS = BAR_MIX_DONE + 2
};

// Byte offsets inside the (1024-aligned) dynamic shared memory.
struct Layout {
    uint32_t phi, stages, xbuf, hpre, ssbuf, bars, misc, total;
    __host__ __device__ static Layout make(int nch) {
        Layout L;
        L.phi = 0;
        L.stages = static_cast<uint32_t>(nch) * PHI_CHUNK_BYTES;   // multiple of 1024
        L.xbuf = L.stages + STAGES * STAGE_BYTES;
        L.hpre = L.xbuf + TILE_M * REC * 4;
        L.ssbuf = L.hpre + 2 * TILE_M * 16;
        L.bars = L.ssbuf + 2 * TILE_M * 4;
        L.misc = L.bars + NBARS * 8;
        L.total = L.misc + 64 + 32 * 4;   // tmem slot, abort flag, alpha, b
        return L;
    }
};

struct Params {
    const __nv_bfloat16* x;
    const float* phi;
    const float* b;
    const float* alpha;
    int64_t T;
    int D, Dc, nch, iters;
    float eps;
    int ntiles;
    __nv_bfloat16* x_in;
    float* H_pre;
    float* H_post;
    float* H_res;
    float* proj;
    float* inv_rms;
};

// Bounded wait on an mbarrier phase.  Returns false (and latches the error
// word) once about a second has passed, or at once if another role of this
// CTA already gave up.
template <bool CLUSTER>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (CLUSTER ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (CLUSTER ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (*abort_flag) return false;
            if (ptx::globaltimer() - t0 > WAIT_LIMIT_NS) {
                atomicOr(&g_device_error, 1u);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

template <int C>
__global__ void __launch_bounds__(NTHREADS, 1)
pre_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const Params p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const Layout L = Layout::make(p.nch);
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bars = sbase + L.bars;
    auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 16);
    float* gate_par = reinterpret_cast<float*>(smem + L.misc + 64);   // alpha[3], b[24]
    float* xbuf = reinterpret_cast<float*>(smem + L.xbuf);
    float* ssbuf = reinterpret_cast<float*>(smem + L.ssbuf);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t c = ptx::cluster_ctarank();
    const int cid = static_cast<int>(ptx::cluster_id_x());
    const int ncl = static_cast<int>(ptx::nclusters_x());
    const int D = p.D, Dc = p.Dc, nch = p.nch;
    const int cpd = Dc / KW;                       // chunks per stream
    const int64_t K = 4ll * D;
    constexpr int TPC = TILE_M / C;                // tokens each CTA reduces

    // ---- set-up: barriers, TMEM, gate parameters, resident phi slice ------
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar(BAR_FULL + s), 1);
            ptx::mbar_init(bar(BAR_EMPTY + s), 1 + NSS * 32);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(bar(BAR_ACC_FULL + i), 1);
            ptx::mbar_init(bar(BAR_ACC_EMPTY + i), 128);
            ptx::mbar_init(bar(BAR_SS_FULL + i), NSS * 32);
            ptx::mbar_init(bar(BAR_SS_EMPTY + i), 128);
            ptx::mbar_init(bar(BAR_HPRE + i), C);
            ptx::mbar_init(bar(BAR_MIX_DONE + i), NMIX * 32);
        }
        ptx::mbar_init(bar(BAR_PEER), C);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) ptx::prefetch_tmap(&tmap_x);
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (tid < 3) gate_par[tid] = p.alpha[tid];
    if (tid >= 32 && tid < 32 + NG) gate_par[3 + tid - 32] = p.b[tid - 32];
    // phi slice -> bf16 hi / lo rows in the swizzled K-major layout of the
    // MMA's B operand: chunk ch, row n (< 24: hi of logit n, else lo of
    // logit n - 24), 16-byte piece q of the row at (q ^ (n & 7)).
    for (int item = tid; item < nch * 8 * NG; item += NTHREADS) {
        const int g = item % NG;
        const int q = (item / NG) % 8;
        const int ch = item / (NG * 8);
        const int i = ch / cpd, sub = ch % cpd;
        const int64_t k0 = static_cast<int64_t>(i) * D + static_cast<int64_t>(c) * Dc + sub * KW + q * 8;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float v0 = p.phi[(k0 + 2 * e) * NG + g];
            const float v1 = p.phi[(k0 + 2 * e + 1) * NG + g];
            const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
            const float2 hf = __bfloat1622float2(h);
            const __nv_bfloat162 l = __floats2bfloat162_rn(v0 - hf.x, v1 - hf.y);
            hi[e] = *reinterpret_cast<const uint32_t*>(&h);
            lo[e] = *reinterpret_cast<const uint32_t*>(&l);
        }
        unsigned char* chunk = smem + L.phi + ch * PHI_CHUNK_BYTES;
        const int nh = g, nl = NG + g;
        *reinterpret_cast<uint4*>(chunk + nh * 128 + ((q ^ (nh & 7)) * 16)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(chunk + nl * 128 + ((q ^ (nl & 7)) * 16)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    ptx::cluster_sync();   // peers' barriers are initialised before any remote arrive
    const uint32_t tmem_base = *tmem_slot;

    constexpr unsigned FULL = 0xffffffffu;
    if (warp == 0) {
        // ------------------------------------------------ TMA producer ----
        // The whole warp walks the loop; lane 0 waits and issues.
        const uint64_t pol = ptx::policy_evict_last();
        int stage = 0;
        uint32_t round = 0;
        for (int j = cid; j < p.ntiles; j += ncl) {
            const int t0 = j * TILE_M;
            for (int ch = 0; ch < nch; ++ch) {
                const int i = ch / cpd, sub = ch % cpd;
                const int xk = i * D + static_cast<int>(c) * Dc + sub * KW;
                bool ok = true;
                if (lane == 0) ok = wait_bar<false>(bar(BAR_EMPTY + stage), (round & 1) ^ 1, abort_flag);
                if (!__shfl_sync(FULL, ok, 0)) goto done;
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(bar(BAR_FULL + stage), STAGE_BYTES);
                    ptx::tma_load_2d(sbase + L.stages + stage * STAGE_BYTES, &tmap_x, xk, t0,
                                     bar(BAR_FULL + stage), pol);
                }
                __syncwarp();
                if (++stage == STAGES) { stage = 0; ++round; }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer -----
        int stage = 0;
        uint32_t round = 0;
        int it = 0;
        for (int j = cid; j < p.ntiles; j += ncl, ++it) {
            const int tb = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            bool ok = true;
            if (lane == 0) ok = wait_bar<false>(bar(BAR_ACC_EMPTY + tb), (use & 1) ^ 1, abort_flag);
            if (!__shfl_sync(FULL, ok, 0)) goto done;
            ptx::tc_fence_after();
            const uint32_t d_tmem = tmem_base + tb * 64;
            for (int ch = 0; ch < nch; ++ch) {
                if (lane == 0) ok = wait_bar<false>(bar(BAR_FULL + stage), round & 1, abort_flag);
                if (!__shfl_sync(FULL, ok, 0)) goto done;
                ptx::tc_fence_after();
                if (lane == 0) {
                    const uint32_t a0 = sbase + L.stages + stage * STAGE_BYTES;
                    const uint32_t b0 = sbase + L.phi + ch * PHI_CHUNK_BYTES;
#pragma unroll
                    for (int kk = 0; kk < KW / 16; ++kk)
                        ptx::tc_mma_f16(d_tmem, ptx::sw128_kmajor_desc(a0 + kk * 32),
                                        ptx::sw128_kmajor_desc(b0 + kk * 32), IDESC, (ch | kk) != 0);
                    ptx::tc_commit(bar(BAR_EMPTY + stage));
                }
                __syncwarp();
                if (++stage == STAGES) { stage = 0; ++round; }
            }
            if (lane == 0) ptx::tc_commit(bar(BAR_ACC_FULL + tb));
            __syncwarp();
        }
    } else if (warp < GATE_WARP0) {
        // ------------------------------------------ sum of squares --------
        const int r0 = (warp - SS_WARP0) * 32 + lane;   // token rows r0 and r0 + 64
        int stage = 0;
        uint32_t round = 0;
        int it = 0;
        for (int j = cid; j < p.ntiles; j += ncl, ++it) {
            const int tb = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            float ss[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
            for (int ch = 0; ch < nch; ++ch) {
                if (!__all_sync(FULL, wait_bar<false>(bar(BAR_FULL + stage), round & 1, abort_flag))) goto done;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int r = r0 + 64 * h;
                    const unsigned char* rowp = smem + L.stages + stage * STAGE_BYTES + r * 128;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint4 v = *reinterpret_cast<const uint4*>(rowp + ((k ^ (r & 7)) * 16));
                        float f[8];
                        Vec<__nv_bfloat16>::unpack(v, f);
#pragma unroll
                        for (int e2 = 0; e2 < 8; e2 += 2) {
                            ss[h][0] = fmaf(f[e2], f[e2], ss[h][0]);
                            ss[h][1] = fmaf(f[e2 + 1], f[e2 + 1], ss[h][1]);
                        }
                    }
                }
                ptx::mbar_arrive(bar(BAR_EMPTY + stage));
                if (++stage == STAGES) { stage = 0; ++round; }
            }
            if (!__all_sync(FULL, wait_bar<false>(bar(BAR_SS_EMPTY + tb), (use & 1) ^ 1, abort_flag))) goto done;
            ssbuf[tb * TILE_M + r0] = ss[0][0] + ss[0][1];
            ssbuf[tb * TILE_M + r0 + 64] = ss[1][0] + ss[1][1];
            ptx::mbar_arrive(bar(BAR_SS_FULL + tb));
        }
    } else if (warp < MIX_WARP0) {
        // ------------------------------------------------- gates ----------
        // TMEM -> partial logits; publish; reduce this CTA's tokens over the
        // cluster; gates and Sinkhorn; push H_pre to every CTA.
        const int row = (warp & 3) * 32 + lane;        // TMEM lane quarter = warp % 4
        const uint32_t xbuf_a = sbase + L.xbuf;
        const int half = lane >> 4, hl = lane & 15;    // two tokens per warp, 16 lanes each
        int it = 0;
        bool aborted = false;
        for (int j = cid; j < p.ntiles; j += ncl, ++it) {
            const int tb = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            const int64_t t0 = static_cast<int64_t>(j) * TILE_M;
            float z[NG];
            float ssv = 0.f;
            bool ok = !aborted && wait_bar<false>(bar(BAR_ACC_FULL + tb), use & 1, abort_flag);
            ok = __all_sync(FULL, ok);
            if (ok) {
                ptx::tc_fence_after();
                uint32_t v[3][16];
                const uint32_t ta = tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) + tb * 64;
                ptx::tmem_ld16(ta, v[0]);
                ptx::tmem_ld16(ta + 16, v[1]);
                ptx::tmem_ld16(ta + 32, v[2]);
                ptx::tmem_wait_ld();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(BAR_ACC_EMPTY + tb));
#pragma unroll
                for (int g = 0; g < NG; ++g) {
                    const int h = g, l = NG + g;
                    z[g] = __uint_as_float(v[h >> 4][h & 15]) + __uint_as_float(v[l >> 4][l & 15]);
                }
            }
            ok = __all_sync(FULL, ok && wait_bar<false>(bar(BAR_SS_FULL + tb), use & 1, abort_flag));
            if (ok) {
                ssv = ssbuf[tb * TILE_M + row];
                ptx::mbar_arrive(bar(BAR_SS_EMPTY + tb));
            }
            // xbuf is reused: every CTA must have pulled the previous tile's
            // partials (they push its H_pre only after pulling), and the
            // H_pre buffer this tile fills must be free (mix of tile it-2).
            if (it >= 1) {
                const int pt = it - 1;
                ok = __all_sync(FULL, ok && wait_bar<true>(bar(BAR_HPRE + (pt & 1)), (pt >> 1) & 1, abort_flag));
            }
            ok = __all_sync(FULL, ok && wait_bar<false>(bar(BAR_MIX_DONE + tb), (use & 1) ^ 1, abort_flag));
            if (ok) {
                float* rec = xbuf + row * REC;
#pragma unroll
                for (int g = 0; g < NG; ++g) rec[g] = z[g];
                rec[NG] = ssv;
            }
            if (!ok) aborted = true;
            ptx::fence_acq_rel_cluster();
            ptx::named_bar_sync(1, NGATE * 32);
            if (warp == GATE_WARP0 && lane < C && !aborted) ptx::mbar_arrive_remote(ptx::mapa(bar(BAR_PEER), lane));
            if (!__all_sync(FULL, !aborted && wait_bar<true>(bar(BAR_PEER), it & 1, abort_flag))) aborted = true;
            if (!aborted) {
                for (int tt0 = (warp - GATE_WARP0) * 2; tt0 < TPC; tt0 += NGATE * 2) {
                    const int tt = tt0 + half;
                    const bool real = tt < TPC;
                    const int r = static_cast<int>(c) * TPC + (real ? tt : 0);
                    float va = 0.f, vb = 0.f;
                    if (real) {
                        const uint32_t a = xbuf_a + static_cast<uint32_t>((r * REC + hl) * 4);
#pragma unroll
                        for (int s = 0; s < C; ++s) va += ptx::ld_cluster_f32(ptx::mapa(a, s));
                        if (hl + 16 < REC) {
#pragma unroll
                            for (int s = 0; s < C; ++s) vb += ptx::ld_cluster_f32(ptx::mapa(a + 64, s));
                        }
                    }
                    float pj[NG];
#pragma unroll
                    for (int g = 0; g < NG; ++g) pj[g] = __shfl_sync(FULL, g < 16 ? va : vb, g & 15, 16);
                    const float sq = __shfl_sync(FULL, vb, NG - 16, 16);
                    const float inv = 1.0f / sqrtf(sq / static_cast<float>(K) + p.eps);
#pragma unroll
                    for (int g = 0; g < NG; ++g) pj[g] *= inv;
                    float hp[4], hq[4], hr[16];
                    token_gates(pj, gate_par, gate_par + 3, p.iters, hp, hq, hr);
                    const int64_t t = t0 + r;
                    if (real && t < p.T) {
                        if (hl < 6)
                            reinterpret_cast<float4*>(p.proj + t * NG)[hl] =
                                make_float4(pj[4 * hl], pj[4 * hl + 1], pj[4 * hl + 2], pj[4 * hl + 3]);
                        else if (hl == 6) p.inv_rms[t] = inv;
                        else if (hl == 7) reinterpret_cast<float4*>(p.H_pre)[t] = make_float4(hp[0], hp[1], hp[2], hp[3]);
                        else if (hl == 8) reinterpret_cast<float4*>(p.H_post)[t] = make_float4(hq[0], hq[1], hq[2], hq[3]);
                        else if (hl < 13) {
                            const int v = hl - 9;
                            reinterpret_cast<float4*>(p.H_res + t * 16)[v] =
                                make_float4(hr[4 * v], hr[4 * v + 1], hr[4 * v + 2], hr[4 * v + 3]);
                        }
                    }
                    if (real && hl < C) {
                        const uint32_t dst = sbase + L.hpre + static_cast<uint32_t>((tb * TILE_M + r) * 16);
                        ptx::st_cluster_v4(ptx::mapa(dst, hl), hp[0], hp[1], hp[2], hp[3]);
                        ptx::fence_acq_rel_cluster();
                    }
                }
            }
            ptx::named_bar_sync(1, NGATE * 32);
            if (warp == GATE_WARP0 && lane < C && !aborted) ptx::mbar_arrive_remote(ptx::mapa(bar(BAR_HPRE + tb), lane));
            if (ptx::named_bar_or(2, NGATE * 32, aborted)) break;
        }
    } else {
        // --------------------------------------------------- mix ----------
        // x_in = sum_i H_pre[i] x[i] over this CTA's D-slice; x read again
        // (from L2 when the tile's first read is recent enough).
        const int mtid = tid - MIX_WARP0 * 32;          // 0..255
        int it = 0;
        for (int j = cid; j < p.ntiles; j += ncl, ++it) {
            const int tb = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            const int64_t t0 = static_cast<int64_t>(j) * TILE_M;
            if (!__all_sync(FULL, wait_bar<true>(bar(BAR_HPRE + tb), use & 1, abort_flag))) break;
            const float4* hb = reinterpret_cast<const float4*>(smem + L.hpre) + tb * TILE_M;
            const int qpt = Dc / 8;
            const int items = TILE_M * qpt;
            for (int base = 0; base < items; base += NMIX * 32 * 4) {
                uint4 xv[4][4];
                int64_t tok[4];
                int qq[4], rr[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int idx = base + m * NMIX * 32 + mtid;
                    rr[m] = idx / qpt;
                    qq[m] = idx - rr[m] * qpt;
                    tok[m] = (idx < items) ? t0 + rr[m] : p.T;
                    if (tok[m] < p.T) {
                        const __nv_bfloat16* src = p.x + tok[m] * K + static_cast<int64_t>(c) * Dc + qq[m] * 8;
#pragma unroll
                        for (int i = 0; i < 4; ++i) xv[m][i] = ld16_stream(src + static_cast<int64_t>(i) * D);
                    }
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    if (tok[m] < p.T) {
                        const float4 h = hb[rr[m]];
                        float f0[8], f1[8], f2[8], f3[8], o[8];
                        Vec<__nv_bfloat16>::unpack(xv[m][0], f0);
                        Vec<__nv_bfloat16>::unpack(xv[m][1], f1);
                        Vec<__nv_bfloat16>::unpack(xv[m][2], f2);
                        Vec<__nv_bfloat16>::unpack(xv[m][3], f3);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            o[q] = fmaf(h.w, f3[q], fmaf(h.z, f2[q], fmaf(h.y, f1[q], h.x * f0[q])));
                        st16_stream(p.x_in + tok[m] * D + static_cast<int64_t>(c) * Dc + qq[m] * 8,
                                    Vec<__nv_bfloat16>::pack(o));
                    }
                }
            }
            ptx::mbar_arrive(bar(BAR_MIX_DONE + tb));
        }
    }
done:
    __syncthreads();
    if (*abort_flag) {
        // let copies already issued land before the shared memory goes away
        const uint64_t t0 = ptx::globaltimer();
        while (ptx::globaltimer() - t0 < 20000ull) {
        }
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, TMEM_COLS);
    }
    ptx::cluster_sync();
}

// ------------------------------------------------------------------ host ---

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// Cluster size for a width D: phi slice of 4*D/C columns resident (<= 1280)
// and a D-slice that is a whole number of 64-column stages.
int cluster_for(int64_t D) {
    for (int C : {16, 8, 4, 2}) {
        if (D % (KW * C) != 0) continue;
        if (4 * D / C > MAX_NCH * KW) continue;
        return C;
    }
    return 0;
}

size_t smem_bytes(int nch) { return Layout::make(nch).total + 1024; }

template <int C>
int max_clusters(size_t smem) {
    // per device ordinal, computed once
    static int cache[64];
    static std::once_flag once[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::call_once(once[dev], [&] {
        int n = 0;
        auto k = pre_tc_kernel<C>;
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem_bytes(MAX_NCH))) != cudaSuccess ||
            (C > 8 && cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)) {
            cache[dev] = 0;
            return;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(C * 64);
        cfg.blockDim = dim3(NTHREADS);
        cfg.dynamicSmemBytes = smem_bytes(MAX_NCH);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) n = 0;
        cache[dev] = n;
    });
    (void)smem;
    return cache[dev];
}

int max_clusters_for(int C, size_t smem) {
    switch (C) {
        case 16: return max_clusters<16>(smem);
        case 8: return max_clusters<8>(smem);
        case 4: return max_clusters<4>(smem);
        case 2: return max_clusters<2>(smem);
    }
    return 0;
}

template <int C>
cudaError_t launch(const CUtensorMap& tm, const Params& prm, int nclusters, size_t smem, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nclusters * C));
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, pre_tc_kernel<C>, tm, prm);
}

}  // namespace tc

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() { return tc::encode_fn(); }

bool pre_tc_supports(int64_t T, int64_t D) {
    if (T < tc::TILE_M || D > (int64_t(1) << 20)) return false;
    if (4 * D * T >= (int64_t(1) << 46)) return false;
    const int C = tc::cluster_for(D);
    if (C == 0 || tc::encode_fn() == nullptr) return false;
    const int nch = static_cast<int>(4 * D / C / tc::KW);
    return tc::max_clusters_for(C, tc::smem_bytes(nch)) > 0;
}

cudaError_t launch_pre_tc(const void* x, const float* phi, const float* b, const float* alpha,
                          int64_t T, int64_t D, int iters, float eps, void* x_in, float* H_pre,
                          float* H_post, float* H_res, float* proj, float* inv_rms,
                          cudaStream_t s) {
    const int C = tc::cluster_for(D);
    auto encode = tc::encode_fn();
    if (C == 0 || encode == nullptr) return cudaErrorNotSupported;
    const int64_t K = 4 * D;
    CUtensorMap tm;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K * 2)};
    const cuuint32_t box[2] = {tc::KW, tc::TILE_M};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    tc::Params prm;
    prm.x = static_cast<const __nv_bfloat16*>(x);
    prm.phi = phi;
    prm.b = b;
    prm.alpha = alpha;
    prm.T = T;
    prm.D = static_cast<int>(D);
    prm.Dc = static_cast<int>(D / C);
    prm.nch = static_cast<int>(K / C / tc::KW);
    prm.iters = iters;
    prm.eps = eps;
    prm.ntiles = static_cast<int>((T + tc::TILE_M - 1) / tc::TILE_M);
    prm.x_in = static_cast<__nv_bfloat16*>(x_in);
    prm.H_pre = H_pre;
    prm.H_post = H_post;
    prm.H_res = H_res;
    prm.proj = proj;
    prm.inv_rms = inv_rms;
    const size_t smem = tc::smem_bytes(prm.nch);
    int ncl = tc::max_clusters_for(C, smem);
    if (ncl <= 0) return cudaErrorNotSupported;
    if (ncl > prm.ntiles) ncl = prm.ntiles;
    switch (C) {
        case 16: return tc::launch<16>(tm, prm, ncl, smem, s);
        case 8: return tc::launch<8>(tm, prm, ncl, smem, s);
        case 4: return tc::launch<4>(tm, prm, ncl, smem, s);
        case 2: return tc::launch<2>(tm, prm, ncl, smem, s);
    }
    return cudaErrorNotSupported;
}

}  // namespace mhc
