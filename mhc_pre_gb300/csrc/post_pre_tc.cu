// post_pre_tc.cu -- the residual update of layer l fused with the pre step of
// layer l + 1 (bf16, n = 4), on tensor cores.
//
// What it computes, per token (section 5.3 of the "openPangu 2.0 --
// architecture, training and Ascend systems" notes, two consecutive layers;
// the fusion follows the inference critical-path split of section 11.3):
//   x_next[i] = sum_j H_res[i][j] x[j] + H_post[i] y          (layer l, stored bf16)
//   then, on the stored x_next, everything mhc_pre computes for layer l + 1:
//   inv_rms, proj = x_bar . phi, the gates, Sinkhorn, and
//   x_in = sum_i H_pre'[i] x_next[i].
// One pass over x and y: x_next is formed in shared memory, stored once, and
// projected from there, so the separate pre step's read of x_next (2 K bytes
// per token) disappears.
//
// Design (GB300, one CTA per SM, persistent; the cluster layout, resident
// phi, MMA, gate and Sinkhorn roles are those of pre_tc.cu):
//   * A stage is one 32-column chunk of a 64-token tile: the x box of all four
//     streams (16 KB) and the y box (4 KB), brought by TMA into one of four
//     20 KB slots (phi takes 120 KB of shared memory).  Rows are 64 bytes, in
//     the 64-byte swizzle; the MMA reads them with K = 32 per stage.
//   * Eight post warps turn the x box into x_next in place, with the same
//     multiply-add order as mhc_post (so the two agree bit for bit), and one
//     of them stores it with a TMA store; the slot is free once the store
//     and the MMA thread have read it.
//   * The MMA thread projects the slot's two stream pairs against phi and
//     forms the Gram products, into the same accumulators as pre_tc.
//   * x_in = sum_i H_pre'[i] x_next[i] is a second kernel on the SMs the
//     clusters leave idle (40 of 152 with clusters of 16), launched behind this
//     one (programmatic dependent launch) so that both run at once.  Each CTA
//     of a cluster counts a tile done twice in a per-tile word of the
//     workspace, with release semantics: once its Sinkhorn warp has written
//     the tile's H_pre', once its x_next stores have completed (a TMA store's
//     writes are visible to plain loads only then).  The mix kernel reads a
//     tile (x_next from L2) once its count is complete; it never holds this
//     kernel up, so it is correct whenever it gets to run.
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

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// This file's device error word (latched by bounded waits that ran out).
__device__ unsigned g_post_pre_error;

cudaError_t read_and_clear_post_pre_error(unsigned* word) {
    cudaError_t e = cudaMemcpyFromSymbol(word, g_post_pre_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_post_pre_error, &zero, sizeof(unsigned));
}

namespace pp {

constexpr int TILE_M = 64;                        // tokens per tile
constexpr int KW = 32;                            // columns per chunk (64 B rows)
constexpr int STAGES = 4;
constexpr int NB = 48;                            // MMA N per stream: 24 hi + 24 lo
constexpr int ROW = KW * 2;                       // 64 B
constexpr int SUB_BYTES = TILE_M * ROW;           // one stream of a chunk: 4 KB
constexpr int PAIR_BYTES = 2 * SUB_BYTES;         // a stream pair: 8 KB, one MMA's A
constexpr int X_BYTES = 4 * SUB_BYTES;            // x box of a stage: 16 KB
constexpr int SLOT_BYTES = X_BYTES + SUB_BYTES;   // [x box | y box]: 20 KB
constexpr int PHI_CHUNK_BYTES = NB * ROW;         // 3 KB
constexpr int MAX_NCH = 40;                       // K-slice <= 1280 columns
constexpr int GATE_WARP0 = 2, NGATE = 4;          // TMEM readers, cluster reduction
constexpr int SK_WARP = 6;                        // Sinkhorn, other gates, outputs
// Eight post warps: the post arithmetic sits on every slot's turnover (four
// warps: 0.92 ms at T = 32768, D = 5120; eight: 0.82; two: 1.17).
constexpr int POST_WARP0 = 7, NPOST = 8;          // x_next in the slot
constexpr int POST_TPT = NPOST / 2;               // post threads per token
constexpr int POST_PPT = 4 / POST_TPT;            // 16-byte pieces per post thread and row
static_assert(NPOST == 2 || NPOST == 4 || NPOST == 8, "post threads split a token row evenly");
constexpr int NTHREADS = (POST_WARP0 + NPOST) * 32;
constexpr int SKF = 28;                           // hand-off record: proj[24], inv_rms (floats)
constexpr int REC = 25;                           // partial record: 24 logits + sum x^2
constexpr int RB = 28;                            // its stride in floats
constexpr uint32_t REC_TX = REC * 4;
constexpr int TMEM_COLS = 512;
constexpr uint32_t GRAM_COL = 256;                // projection at 0 / 128, Gram at 256 / 384
constexpr uint32_t IDESC = ptx::idesc_bf16_f32(2 * TILE_M, 2 * NB);
constexpr uint32_t IDESC_GRAM = ptx::idesc_bf16_f32(2 * TILE_M, 2 * TILE_M);
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;

enum : int {
    BAR_FULL = 0,                   // [2] the slot's boxes landed
    BAR_XREADY = BAR_FULL + STAGES,  // [2] x_next formed in the slot
    BAR_EMPTY = BAR_XREADY + STAGES, // [2] MMA and the x_next store are done with the slot
    BAR_ACC_FULL = BAR_EMPTY + STAGES,
    BAR_ACC_EMPTY = BAR_ACC_FULL + 2,
    BAR_RECV = BAR_ACC_EMPTY + 2,
    BAR_RFREE = BAR_RECV + 1,
    BAR_SKFULL = BAR_RFREE + 1,
    BAR_SKEMPTY = BAR_SKFULL + 2,
    NBARS = BAR_SKEMPTY + 2
};

struct Layout {
    uint32_t phi, stages, recv, sk, bars, misc, total;
    __host__ __device__ static Layout make(int nch, int tpc) {
        Layout L;
        L.phi = 0;
        L.stages = (static_cast<uint32_t>(nch) * PHI_CHUNK_BYTES + 1023u) & ~1023u;
        L.recv = L.stages + STAGES * SLOT_BYTES;      // [C senders][TILE_M / C tokens][2 halves][RB]
        L.sk = L.recv + 2 * TILE_M * RB * 4;          // [2][tpc][SKF]
        L.bars = L.sk + 2 * tpc * SKF * 4;
        L.misc = L.bars + NBARS * 8;
        L.total = L.misc + 64 + 32 * 4;               // tmem slot, abort flag, alpha, b
        return L;
    }
};

struct Params {
    const __nv_bfloat16* x;
    const __nv_bfloat16* y;
    const float* H_post_l;   // layer l's gates [T, 4], [T, 16]
    const float* H_res_l;
    const float* phi;        // layer l + 1
    const float* b;
    const float* alpha;
    int64_t T;
    int D, Dc, nch, iters;
    float eps;
    int ntiles;
    unsigned* tile_done;     // [ntiles] completion counts (zeroed before the launch)
    float* H_pre;
    float* H_post;
    float* H_res;
    float* proj;
    float* inv_rms;
};

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

template <bool CLUSTER>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (CLUSTER ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (CLUSTER ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (*abort_flag) return false;
            if (ptx::globaltimer() - t0 > WAIT_LIMIT_NS) {
                atomicOr(&g_post_pre_error, 1u);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

template <int C>
__global__ void __launch_bounds__(NTHREADS, 1)
post_pre_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_y,
                   const __grid_constant__ CUtensorMap tmap_xn, const Params p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    constexpr int TPC = TILE_M / C;                // tokens each CTA reduces
    const Layout L = Layout::make(p.nch, TPC);
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bars = sbase + L.bars;
    auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 16);
    float* gate_par = reinterpret_cast<float*>(smem + L.misc + 64);   // alpha[3], b[24]
    const float* recv = reinterpret_cast<const float*>(smem + L.recv);

    ptx::griddep_launch_dependents();   // the mix kernel may start on the idle SMs
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t c = ptx::cluster_ctarank();
    const int cid = static_cast<int>(ptx::cluster_id_x());
    const int ncl = static_cast<int>(ptx::nclusters_x());
    const int D = p.D, Dc = p.Dc, nch = p.nch;
    const int cpd = Dc / KW;                       // chunks per stream = stages per tile
    const int64_t K = 4ll * D;
    const int ntl = p.ntiles > cid ? (p.ntiles - cid + ncl - 1) / ncl : 0;   // tiles of this cluster

    // ---- set-up: barriers, TMEM, gate parameters, resident phi slice ------
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar(BAR_FULL + s), 1);
            ptx::mbar_init(bar(BAR_XREADY + s), 1);
            ptx::mbar_init(bar(BAR_EMPTY + s), 2);   // the MMA's commit and the x_next store
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(bar(BAR_ACC_FULL + i), 1);
            ptx::mbar_init(bar(BAR_ACC_EMPTY + i), 128);
            ptx::mbar_init(bar(BAR_SKFULL + i), 1);
            ptx::mbar_init(bar(BAR_SKEMPTY + i), 1);
        }
        ptx::mbar_init(bar(BAR_RECV), 1);
        ptx::mbar_init(bar(BAR_RFREE), C);
        // receive barriers are armed one use ahead, before any peer can send
        if (ntl > 0) ptx::mbar_arrive_expect_tx(bar(BAR_RECV), 2 * TILE_M * REC_TX);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmap_x);
        ptx::prefetch_tmap(&tmap_y);
        ptx::prefetch_tmap(&tmap_xn);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (tid < 3) gate_par[tid] = p.alpha[tid];
    if (tid >= 32 && tid < 32 + NG) gate_par[3 + tid - 32] = p.b[tid - 32];
    // phi slice -> bf16 hi / lo rows in the 64-byte-swizzled K-major layout
    // of the MMA's B operand: chunk ch = (pair, chunk of the slice, stream in
    // the pair), row n (< 24: hi of logit n, else lo), 16-byte piece q of the
    // row at q ^ ((n >> 1) & 3).  Item (ch, q, g) is 8 consecutive K rows of
    // logit g.  A thread issues the loads of all its items before it converts
    // any, so that the set-up waits for one round trip to memory, not one per
    // item.
    {
        constexpr int PHI_ITEMS = (MAX_NCH * 4 * NG + NTHREADS - 1) / NTHREADS;
        const int nitems = nch * 4 * NG;
        float v[PHI_ITEMS][8];
#pragma unroll
        for (int m = 0; m < PHI_ITEMS; ++m) {
            const int item = tid + m * NTHREADS;
            if (item < nitems) {
                const int g = item % NG;
                const int q = (item / NG) % 4;
                const int ch = item / (NG * 4);
                const int pr = ch / (2 * cpd), rem = ch % (2 * cpd);
                const int sub = rem >> 1, i = 2 * pr + (rem & 1);
                const int64_t k0 = static_cast<int64_t>(i) * D + static_cast<int64_t>(sub * C + c) * KW + q * 8;
#pragma unroll
                for (int e = 0; e < 8; ++e) v[m][e] = p.phi[(k0 + e) * NG + g];
            }
        }
#pragma unroll
        for (int m = 0; m < PHI_ITEMS; ++m) {
            const int item = tid + m * NTHREADS;
            if (item < nitems) {
                const int g = item % NG;
                const int q = (item / NG) % 4;
                const int ch = item / (NG * 4);
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(v[m][2 * e], v[m][2 * e + 1]);
                    const float2 hf = __bfloat1622float2(h);
                    const __nv_bfloat162 l = __floats2bfloat162_rn(v[m][2 * e] - hf.x, v[m][2 * e + 1] - hf.y);
                    hi[e] = *reinterpret_cast<const uint32_t*>(&h);
                    lo[e] = *reinterpret_cast<const uint32_t*>(&l);
                }
                unsigned char* chunk = smem + L.phi + ch * PHI_CHUNK_BYTES;
                const int nh = g, nl = NG + g;
                *reinterpret_cast<uint4*>(chunk + nh * ROW + ((q ^ ((nh >> 1) & 3)) * 16)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(chunk + nl * ROW + ((q ^ ((nl >> 1) & 3)) * 16)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
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
        const uint64_t pol = ptx::policy_evict_normal();   // x and y are read again by the mix
        int stage = 0;
        uint32_t round = 0;
        for (int j = cid; j < p.ntiles; j += ncl) {
            const int t0 = j * TILE_M;
            for (int sub = 0; sub < cpd; ++sub) {
                const int xd = (sub * C + static_cast<int>(c)) * KW;   // chunks interleaved over the cluster
                bool ok = true;
                if (lane == 0) ok = wait_bar<false>(bar(BAR_EMPTY + stage), (round & 1) ^ 1, abort_flag);
                if (!__shfl_sync(FULL, ok, 0)) goto done;
                if (lane == 0) {
                    const uint32_t dst = sbase + L.stages + stage * SLOT_BYTES;
                    ptx::mbar_arrive_expect_tx(bar(BAR_FULL + stage), SLOT_BYTES);
                    ptx::tma_load_3d(dst, &tmap_x, xd, t0, 0, bar(BAR_FULL + stage), pol);
                    ptx::tma_load_2d(dst + X_BYTES, &tmap_y, xd, t0, bar(BAR_FULL + stage), pol);
                }
                __syncwarp();
                if (++stage == STAGES) { stage = 0; ++round; }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer -----
        const uint64_t desc_stage0 = ptx::sw64_kmajor_desc(sbase + L.stages);
        const uint64_t desc_phi0 = ptx::sw64_kmajor_desc(sbase + L.phi);
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
            const uint32_t d_tmem = tmem_base + tb * 128;
            for (int sub = 0; sub < cpd; ++sub) {
                if (lane == 0) ok = wait_bar<false>(bar(BAR_XREADY + stage), round & 1, abort_flag);
                if (!__shfl_sync(FULL, ok, 0)) goto done;
                ptx::tc_fence_after();
                if (lane == 0) {
#pragma unroll
                    for (int pr = 0; pr < 2; ++pr) {
                        // A: the pair's 128 rows of x_next; B: the pair's phi chunks
                        const uint64_t da = ptx::desc_add(desc_stage0, stage * SLOT_BYTES + pr * PAIR_BYTES);
                        const uint64_t db = ptx::desc_add(desc_phi0, (pr * cpd + sub) * 2 * PHI_CHUNK_BYTES);
#pragma unroll
                        for (int kk = 0; kk < KW / 16; ++kk) {
                            const uint64_t dak = ptx::desc_add(da, kk * 32);
                            const uint32_t acc = (sub | pr | kk) != 0;
                            ptx::tc_mma_f16(d_tmem, dak, ptx::desc_add(db, kk * 32), IDESC, acc);
                            ptx::tc_mma_f16(d_tmem + GRAM_COL, dak, dak, IDESC_GRAM, acc);
                        }
                    }
                    ptx::tc_commit(bar(BAR_EMPTY + stage));
                }
                __syncwarp();
                if (++stage == STAGES) { stage = 0; ++round; }
            }
            if (lane == 0) ptx::tc_commit(bar(BAR_ACC_FULL + tb));
            __syncwarp();
        }
    } else if (warp < SK_WARP) {
        // ------------------------------------------------- gates ----------
        // As in pre_tc.cu: TMEM -> partial records pushed to each token's
        // reducer; the reducers sum them and hand the projection to the
        // Sinkhorn warp.
        const int row = (warp & 3) * 32 + lane;        // TMEM lane quarter = warp % 4
        const int tok = row & (TILE_M - 1), hs = row / TILE_M;   // hs is the same across a warp
        const int half = lane >> 4, hl = lane & 15;    // two tokens per warp, 16 lanes each
        const uint32_t rk = static_cast<uint32_t>(tok / TPC);   // reducer of this token
        const uint32_t rec_dst = ptx::mapa(
            sbase + L.recv + static_cast<uint32_t>((((c * TPC) + tok % TPC) * 2 + hs) * RB * 4), rk);
        const uint32_t recv_bar = ptx::mapa(bar(BAR_RECV), rk);
        int it = 0;
        for (int j = cid; j < p.ntiles; j += ncl, ++it) {
            const int tb = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            float z[NG];
            float ssv = 0.f;
            bool ok = __all_sync(FULL, wait_bar<false>(bar(BAR_ACC_FULL + tb), use & 1, abort_flag));
            if (ok) {
                ptx::tc_fence_after();
                uint32_t v[3][16], gd[2][16];
                const uint32_t lanes = static_cast<uint32_t>((warp & 3) * 32) << 16;
                const uint32_t ta = tmem_base + lanes + tb * 128 + hs * NB;
                ptx::tmem_ld16(ta, v[0]);
                ptx::tmem_ld16(ta + 16, v[1]);
                ptx::tmem_ld16(ta + 32, v[2]);
                // Gram columns 32 (warp % 4) .. +31: lane l holds row 32 (warp % 4) + l,
                // whose diagonal entry is column l of these loads
                const uint32_t tg = tmem_base + lanes + GRAM_COL + tb * 128 + (warp & 3) * 32;
                ptx::tmem_ld16(tg, gd[0]);
                ptx::tmem_ld16(tg + 16, gd[1]);
                ptx::tmem_wait_ld();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(BAR_ACC_EMPTY + tb));
#pragma unroll
                for (int g = 0; g < NG; ++g) {
                    const int h = g, l = NG + g;
                    z[g] = __uint_as_float(v[h >> 4][h & 15]) + __uint_as_float(v[l >> 4][l & 15]);
                }
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    if (hl == k) ssv = __uint_as_float(half ? gd[1][k] : gd[0][k]);
            }
            // the reducers have read the previous tile's records
            if (it >= 1) ok = ok && __all_sync(FULL, wait_bar<true>(bar(BAR_RFREE), (it - 1) & 1, abort_flag));
            if (ok) {
#pragma unroll
                for (int v4 = 0; v4 < NG / 4; ++v4)
                    ptx::st_async_v4(rec_dst + 16 * v4, z[4 * v4], z[4 * v4 + 1], z[4 * v4 + 2], z[4 * v4 + 3],
                                     recv_bar);
                ptx::st_async_b32(rec_dst + 4 * NG, ssv, recv_bar);
            }
            // the Sinkhorn warp is done with this parity's hand-off (tile it-2)
            if (it >= 2) ok = ok && __all_sync(FULL, wait_bar<false>(bar(BAR_SKEMPTY + tb), (use - 1) & 1, abort_flag));
            ok = ok && __all_sync(FULL, wait_bar<true>(bar(BAR_RECV), it & 1, abort_flag));
            if (ok) {
                for (int tt0 = (warp - GATE_WARP0) * 2; tt0 < TPC; tt0 += NGATE * 2) {
                    const int tt = tt0 + half;
                    const bool real = tt < TPC;
                    float va = 0.f, vb = 0.f;
                    if (real) {
#pragma unroll
                        for (int s = 0; s < C; ++s) {
#pragma unroll
                            for (int h2 = 0; h2 < 2; ++h2) {
                                const float* rec = recv + ((s * TPC + tt) * 2 + h2) * RB;
                                va += rec[hl];
                                if (hl + 16 < REC) vb += rec[hl + 16];
                            }
                        }
                    }
                    float pj[NG];
#pragma unroll
                    for (int g = 0; g < NG; ++g) pj[g] = __shfl_sync(FULL, g < 16 ? va : vb, g & 15, 16);
                    const float sq = __shfl_sync(FULL, vb, NG - 16, 16);
                    const float inv = 1.0f / sqrtf(sq / static_cast<float>(K) + p.eps);
#pragma unroll
                    for (int g = 0; g < NG; ++g) pj[g] *= inv;
                    if (real && hl < SKF / 4) {
                        // hand-off record: proj[24], inv_rms
                        float4 o = make_float4(inv, 0.f, 0.f, 0.f);
#pragma unroll
                        for (int v = 0; v < NG / 4; ++v)
                            if (hl == v) o = make_float4(pj[4 * v], pj[4 * v + 1], pj[4 * v + 2], pj[4 * v + 3]);
                        reinterpret_cast<float4*>(smem + L.sk)[(tb * TPC + tt) * (SKF / 4) + hl] = o;
                    }
                }
            }
            // every gate warp is done with the records: arm the barrier for the
            // next tile's, then tell every sender the buffer is free
            ptx::fence_proxy_async_smem();
            if (ptx::named_bar_or(1, NGATE * 32, !ok)) break;
            if (warp == GATE_WARP0) {
                if (lane == 0) ptx::mbar_arrive(bar(BAR_SKFULL + tb));
                if (lane == 0 && it + 1 < ntl) ptx::mbar_arrive_expect_tx(bar(BAR_RECV), 2 * TILE_M * REC_TX);
                __syncwarp();
                // a credit: the records read above already feed the sums
                if (lane < C) ptx::mbar_arrive_remote_relaxed(ptx::mapa(bar(BAR_RFREE), static_cast<uint32_t>(lane)));
            }
        }
    } else if (warp == SK_WARP) {
        // ----------------------------------------- Sinkhorn and outputs ---
        // Layer l + 1's other gates and every per-token output (as pre_tc.cu).
        const int l8 = lane & 7;
        int it = 0;
        for (int j = cid; j < p.ntiles; j += ncl, ++it) {
            const int tb = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            if (!__all_sync(FULL, wait_bar<false>(bar(BAR_SKFULL + tb), use & 1, abort_flag))) break;
            const int64_t t0 = static_cast<int64_t>(j) * TILE_M;
            for (int tt0 = 0; tt0 < TPC; tt0 += 4) {
                const int tt = tt0 + (lane >> 3);
                const bool real = tt < TPC;
                float pj[NG], inv = 0.f;
#pragma unroll
                for (int g = 0; g < NG; ++g) pj[g] = 0.f;
                if (real) {
                    const float4* rec = reinterpret_cast<const float4*>(smem + L.sk) + (tb * TPC + tt) * (SKF / 4);
#pragma unroll
                    for (int v = 0; v < NG / 4; ++v) {
                        const float4 a = rec[v];
                        pj[4 * v] = a.x; pj[4 * v + 1] = a.y; pj[4 * v + 2] = a.z; pj[4 * v + 3] = a.w;
                    }
                    inv = rec[NG / 4].x;
                }
                float hp[4], hq[4], hr[16];
                token_gates(pj, gate_par, gate_par + 3, p.iters, hp, hq, hr);
                const int64_t t = t0 + static_cast<int>(c) * TPC + tt;
                if (real && t < p.T) {
#pragma unroll
                    for (int rep = 0; rep < 2; ++rep) {
                        const int k = l8 + 8 * rep;
                        float4 o = make_float4(hp[0], hp[1], hp[2], hp[3]);
#pragma unroll
                        for (int v = 0; v < NG / 4; ++v)
                            if (k == v) o = make_float4(pj[4 * v], pj[4 * v + 1], pj[4 * v + 2], pj[4 * v + 3]);
                        if (k == 8) o = make_float4(hq[0], hq[1], hq[2], hq[3]);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            if (k == 9 + v) o = make_float4(hr[4 * v], hr[4 * v + 1], hr[4 * v + 2], hr[4 * v + 3]);
                        if (k < 6) reinterpret_cast<float4*>(p.proj + t * NG)[k] = o;
                        else if (k == 6) p.inv_rms[t] = inv;
                        else if (k == 7) reinterpret_cast<float4*>(p.H_pre)[t] = o;
                        else if (k == 8) reinterpret_cast<float4*>(p.H_post)[t] = o;
                        else if (k < 13) reinterpret_cast<float4*>(p.H_res + t * 16)[k - 9] = o;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(bar(BAR_SKEMPTY + tb));
                // this CTA's H_pre' of the tile is written
                __threadfence();
                red_release_add(p.tile_done + j, 1u);
            }
        }
    } else {
        // --------------------------------------------------- post ---------
        // x_next = H_res x + H_post y, in place in the slot: POST_TPT threads
        // per token, each with POST_PPT of the row's four 16-byte pieces (8
        // columns) in each of the 4 streams and y.  A token row of every
        // stream and of y has the same 64-byte swizzle (rows are 64 apart), so
        // one offset serves all five.  The leader stores the stage.
        const int pt = tid - POST_WARP0 * 32;
        const int t = pt / POST_TPT, q0 = (pt % POST_TPT) * POST_PPT;
        const bool leader = pt == 0;
        int stage = 0, it = 0;
        uint32_t round = 0;
        for (int j = cid; j < p.ntiles; j += ncl, ++it) {
            const int t0 = j * TILE_M;
            const int64_t tgl = static_cast<int64_t>(t0) + t;
            float H[4][4], Hp[4];
            {
                float4 r[4] = {}, hq = {};
                if (tgl < p.T) {
                    const float4* hr4 = reinterpret_cast<const float4*>(p.H_res_l + tgl * 16);
                    r[0] = hr4[0]; r[1] = hr4[1]; r[2] = hr4[2]; r[3] = hr4[3];
                    hq = reinterpret_cast<const float4*>(p.H_post_l)[tgl];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    H[i][0] = r[i].x; H[i][1] = r[i].y; H[i][2] = r[i].z; H[i][3] = r[i].w;
                }
                Hp[0] = hq.x; Hp[1] = hq.y; Hp[2] = hq.z; Hp[3] = hq.w;
            }
            for (int sub = 0; sub < cpd; ++sub) {
                const bool ok = __all_sync(FULL, wait_bar<false>(bar(BAR_FULL + stage), round & 1, abort_flag));
                if (ok) {
                    unsigned char* slot = smem + L.stages + stage * SLOT_BYTES;
#pragma unroll
                    for (int q = q0; q < q0 + POST_PPT; ++q) {
                        const uint32_t off = static_cast<uint32_t>(t * ROW + ((q ^ ((t >> 1) & 3)) << 4));
                        float f[4][8], fy[8];
#pragma unroll
                        for (int s = 0; s < 4; ++s)
                            Vec<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4*>(slot + s * SUB_BYTES + off), f[s]);
                        Vec<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4*>(slot + X_BYTES + off), fy);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            // mhc_post's order, H[i][0] x0 + ... + H_post y, as
                            // pairs of lanes (each lane one IEEE fma)
                            float o[8];
#pragma unroll
                            for (int el = 0; el < 8; el += 2) {
                                float2 a = __fmul2_rn(make_float2(H[i][0], H[i][0]), make_float2(f[0][el], f[0][el + 1]));
                                a = __ffma2_rn(make_float2(H[i][1], H[i][1]), make_float2(f[1][el], f[1][el + 1]), a);
                                a = __ffma2_rn(make_float2(H[i][2], H[i][2]), make_float2(f[2][el], f[2][el + 1]), a);
                                a = __ffma2_rn(make_float2(H[i][3], H[i][3]), make_float2(f[3][el], f[3][el + 1]), a);
                                a = __ffma2_rn(make_float2(Hp[i], Hp[i]), make_float2(fy[el], fy[el + 1]), a);
                                o[el] = a.x;
                                o[el + 1] = a.y;
                            }
                            *reinterpret_cast<uint4*>(slot + i * SUB_BYTES + off) = Vec<__nv_bfloat16>::pack(o);
                        }
                    }
                    // the MMA and the TMA store read the slot through the async proxy
                    ptx::fence_proxy_async_smem();
                }
                if (ptx::named_bar_or(2, NPOST * 32, !ok)) goto done;
                if (leader) {
                    // x_next of the stage to global memory; the slot is free for
                    // the producer once the MMAs (their commit) and this store
                    // have read it
                    ptx::tma_store_3d(&tmap_xn, (sub * C + static_cast<int>(c)) * KW, t0, 0,
                                      sbase + L.stages + stage * SLOT_BYTES);
                    ptx::bulk_commit();
                    ptx::mbar_arrive(bar(BAR_XREADY + stage));
                    ptx::bulk_wait_read<0>();
                    ptx::mbar_arrive(bar(BAR_EMPTY + stage));
                    if (sub == 0 && it > 0) {
                        // every store of the previous tile has completed: the mix
                        // kernel may read that x_next back with plain loads
                        ptx::bulk_wait<1>();
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                        red_release_add(p.tile_done + (j - ncl), 1u);
                    }
                }
                if (++stage == STAGES) { stage = 0; ++round; }
            }
        }
        if (leader && it > 0) {
            ptx::bulk_wait<0>();
            asm volatile("fence.proxy.async.global;" ::: "memory");
            red_release_add(p.tile_done + (cid + (it - 1) * ncl), 1u);
        }
    }
done:
    // x_next stores read shared memory and must land before the kernel ends
    if (warp == POST_WARP0 && lane == 0) ptx::bulk_wait<0>();
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

// ------------------------------------------------------------------ mix ----
// x_in = sum_i H_pre'[i] x_next[i] (mhc_pre's sum), on the SMs the cluster
// kernel leaves idle.  Eight CTAs share a tile, MIX_TOK tokens each, and the
// groups of eight take tiles in turn, so a few tiles are in flight, each read
// back from L2 soon after the cluster kernel stored it.  One CTA per SM: its
// dynamic shared memory keeps a second one (and a cluster CTA) off the SM.
constexpr int MIX_THREADS = 512;
constexpr int MIX_GROUP = 8;                      // CTAs per tile
constexpr int MIX_TOK = TILE_M / MIX_GROUP;       // tokens per CTA and tile
constexpr int MIX_UNROLL = 5;
constexpr size_t MIX_SMEM = 116 * 1024;

__global__ void __launch_bounds__(MIX_THREADS, 1)
post_pre_mix_kernel(const __nv_bfloat16* __restrict__ x_next, const float* H_pre, __nv_bfloat16* __restrict__ x_in,
                    const unsigned* tile_done, unsigned need, int64_t T, int D, int ntiles) {
    __shared__ float4 hp[MIX_TOK];
    __shared__ int stop;
    const int tid = threadIdx.x;
    const int ngroups = static_cast<int>(gridDim.x) / MIX_GROUP;
    const int group = static_cast<int>(blockIdx.x) / MIX_GROUP, part = static_cast<int>(blockIdx.x) % MIX_GROUP;
    const int64_t K = 4ll * D;
    const int qpt = D / 8;                         // 16-byte pieces per stream row
    if (tid == 0) stop = 0;
    __syncthreads();
    for (int j = group; group < ngroups && j < ntiles; j += ngroups) {
        const int64_t t0 = static_cast<int64_t>(j) * TILE_M + part * MIX_TOK;
        const int nt = T - t0 < MIX_TOK ? static_cast<int>(T - t0) : MIX_TOK;
        if (nt <= 0) continue;
        if (tid == 0) {
            // every CTA of the tile's cluster has written its H_pre' and
            // completed its x_next stores (acquire pairs with their release)
            const uint64_t w0 = ptx::globaltimer();
            while (ld_acquire(tile_done + j) < need) {
                if (ptx::globaltimer() - w0 > WAIT_LIMIT_NS) {
                    atomicOr(&g_post_pre_error, 2u);
                    stop = 1;
                    break;
                }
                __nanosleep(128);
            }
        }
        __syncthreads();
        if (stop) break;
        if (tid < nt) hp[tid] = __ldcg(reinterpret_cast<const float4*>(H_pre) + t0 + tid);
        __syncthreads();
        const int items = nt * qpt;
        // item idx = (row r, piece q), idx = r qpt + q; a thread's item moves by
        // MIX_THREADS a step, so r, q and the item's offsets into x_next and
        // x_in advance with a carry (no division or multiply per item)
        const int dr = MIX_THREADS / qpt, dq = MIX_THREADS - dr * qpt;
        int r_at = tid / qpt, q_at = tid - r_at * qpt;
        int64_t xo_at = (t0 + r_at) * K + q_at * 8, io_at = (t0 + r_at) * D + q_at * 8;
        const int64_t xstep = dr * K + dq * 8, xcarry = K - qpt * 8;
        const int64_t istep = static_cast<int64_t>(dr) * D + dq * 8, icarry = static_cast<int64_t>(D) - qpt * 8;
        for (int base = 0; base < items; base += MIX_THREADS * MIX_UNROLL) {
            uint4 xv[MIX_UNROLL][4];
            int64_t io[MIX_UNROLL];
            int rr[MIX_UNROLL];
#pragma unroll
            for (int m = 0; m < MIX_UNROLL; ++m) {
                rr[m] = r_at < nt ? r_at : -1;
                io[m] = io_at;
                const int64_t xo = xo_at;
                q_at += dq;
                r_at += dr;
                xo_at += xstep;
                io_at += istep;
                if (q_at >= qpt) {
                    q_at -= qpt;
                    ++r_at;
                    xo_at += xcarry;
                    io_at += icarry;
                }
                if (rr[m] >= 0) {
                    const uint4* src = reinterpret_cast<const uint4*>(x_next + xo);
#pragma unroll
                    for (int i = 0; i < 4; ++i) xv[m][i] = __ldcg(src + static_cast<int64_t>(i) * (D / 8));
                }
            }
#pragma unroll
            for (int m = 0; m < MIX_UNROLL; ++m) {
                if (rr[m] >= 0)
                    st16_stream(x_in + io[m], mix4_bf16(xv[m][0], xv[m][1], xv[m][2], xv[m][3], hp[rr[m]]));
            }
        }
        __syncthreads();   // hp is refilled for the next tile
    }
    // complete only after the cluster kernel (its other outputs) has
    if (tid == 0) ptx::griddep_wait();
}

// ------------------------------------------------------------------ host ---

// Cluster size for a width D: phi slice of 4*D/C columns resident (<= 1280)
// and a D-slice of whole 32-column chunks.
int cluster_for(int64_t D) {
    for (int C : {16, 8, 4, 2}) {
        if (D % (KW * C) != 0) continue;
        if (4 * D / C > MAX_NCH * KW) continue;
        return C;
    }
    return 0;
}

size_t smem_bytes(int nch, int C) { return Layout::make(nch, TILE_M / C).total + 1024; }

template <int C>
int max_clusters() {
    static int cache[64];
    static std::once_flag once[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::call_once(once[dev], [&] {
        int n = 0;
        auto k = post_pre_tc_kernel<C>;
        const size_t smem = smem_bytes(MAX_NCH, C);
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
                cudaSuccess ||
            (C > 8 && cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)) {
            cache[dev] = 0;
            return;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(C * 64);
        cfg.blockDim = dim3(NTHREADS);
        cfg.dynamicSmemBytes = smem;
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
    return cache[dev];
}

int max_clusters_for(int C) {
    switch (C) {
        case 16: return max_clusters<16>();
        case 8: return max_clusters<8>();
        case 4: return max_clusters<4>();
        case 2: return max_clusters<2>();
    }
    return 0;
}

template <int C>
cudaError_t launch(const CUtensorMap& tx, const CUtensorMap& ty, const CUtensorMap& txn, const Params& prm,
                   int nclusters, size_t smem, cudaStream_t s) {
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
    return cudaLaunchKernelEx(&cfg, post_pre_tc_kernel<C>, tx, ty, txn, prm);
}

// (d, token, stream) view of a [T, 4, D] bf16 tensor; boxes of 32 columns x
// 64 tokens x 4 streams, laid out in shared memory as [stream][token][32].
bool encode_x4(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* tm, const void* base, int64_t T,
               int64_t D) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T), 4};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(8 * D), static_cast<cuuint64_t>(2 * D)};
    const cuuint32_t box[3] = {KW, TILE_M, 4};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [T, D] bf16 in boxes of 32 columns x 64 tokens.
bool encode_y(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* tm, const void* base, int64_t T, int64_t D) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(2 * D)};
    const cuuint32_t box[2] = {KW, TILE_M};
    const cuuint32_t estr[2] = {1, 1};
    return encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace pp

size_t post_pre_tc_workspace_bytes(int64_t T) {
    const int64_t ntiles = (T + pp::TILE_M - 1) / pp::TILE_M;
    return static_cast<size_t>((ntiles * 4 + 255) / 256 * 256);
}

bool post_pre_tc_supports(int64_t T, int64_t D) {
    if (T < 1 || D > (int64_t(1) << 20) || T >= (int64_t(1) << 31)) return false;
    if (4 * D * T >= (int64_t(1) << 46)) return false;
    const int C = pp::cluster_for(D);
    return C != 0 && tensor_map_encoder() != nullptr && pp::max_clusters_for(C) > 0;
}

cudaError_t launch_post_pre_tc(const void* x, const void* y, const float* H_post_l, const float* H_res_l,
                               const float* phi, const float* b, const float* alpha, int64_t T, int64_t D,
                               int iters, float eps, void* x_next, void* x_in, float* H_pre, float* H_post,
                               float* H_res, float* proj, float* inv_rms, void* workspace, cudaStream_t s) {
    const int C = pp::cluster_for(D);
    auto encode = tensor_map_encoder();
    if (C == 0 || encode == nullptr) return cudaErrorNotSupported;
    CUtensorMap tx, ty, txn;
    if (!pp::encode_x4(encode, &tx, x, T, D) || !pp::encode_y(encode, &ty, y, T, D) ||
        !pp::encode_x4(encode, &txn, x_next, T, D))
        return cudaErrorInvalidValue;
    pp::Params prm;
    prm.x = static_cast<const __nv_bfloat16*>(x);
    prm.y = static_cast<const __nv_bfloat16*>(y);
    prm.H_post_l = H_post_l;
    prm.H_res_l = H_res_l;
    prm.phi = phi;
    prm.b = b;
    prm.alpha = alpha;
    prm.T = T;
    prm.D = static_cast<int>(D);
    prm.Dc = static_cast<int>(D / C);
    prm.nch = static_cast<int>(4 * D / C / pp::KW);
    prm.iters = iters;
    prm.eps = eps;
    prm.ntiles = static_cast<int>((T + pp::TILE_M - 1) / pp::TILE_M);
    prm.tile_done = static_cast<unsigned*>(workspace);
    prm.H_pre = H_pre;
    prm.H_post = H_post;
    prm.H_res = H_res;
    prm.proj = proj;
    prm.inv_rms = inv_rms;
    const size_t smem = pp::smem_bytes(prm.nch, C);
    int ncl = pp::max_clusters_for(C);
    if (ncl <= 0) return cudaErrorNotSupported;
    if (ncl > prm.ntiles) ncl = prm.ntiles;
    cudaError_t e = cudaMemsetAsync(workspace, 0, static_cast<size_t>(prm.ntiles) * 4, s);
    if (e != cudaSuccess) return e;
    switch (C) {
        case 16: e = pp::launch<16>(tx, ty, txn, prm, ncl, smem, s); break;
        case 8: e = pp::launch<8>(tx, ty, txn, prm, ncl, smem, s); break;
        case 4: e = pp::launch<4>(tx, ty, txn, prm, ncl, smem, s); break;
        case 2: e = pp::launch<2>(tx, ty, txn, prm, ncl, smem, s); break;
        default: e = cudaErrorNotSupported;
    }
    if (e != cudaSuccess) return e;
    // the mix kernel: on the SMs the clusters leave free, in groups of eight
    // CTAs (all SMs when none is free: it then runs after the cluster kernel)
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(pp::post_pre_mix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(pp::MIX_SMEM));
    });
    if (attr_err != cudaSuccess) return attr_err;
    int free_sm = nsm - ncl * C;
    if (free_sm < pp::MIX_GROUP) free_sm = nsm;
    int ngroups = free_sm / pp::MIX_GROUP;
    if (ngroups > prm.ntiles) ngroups = prm.ntiles;
    if (ngroups < 1) ngroups = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ngroups * pp::MIX_GROUP));
    cfg.blockDim = dim3(pp::MIX_THREADS);
    cfg.dynamicSmemBytes = pp::MIX_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, pp::post_pre_mix_kernel, static_cast<const __nv_bfloat16*>(x_next),
                              static_cast<const float*>(H_pre), static_cast<__nv_bfloat16*>(x_in),
                              static_cast<const unsigned*>(workspace), static_cast<unsigned>(2 * C), T,
                              static_cast<int>(D), prm.ntiles);
}

}  // namespace mhc
