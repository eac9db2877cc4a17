// pre_bwd_fused.cu -- one-pass tensor-core pre backward of the mHC layer
// (bf16, n = 4) on thread-block clusters.
//
// What it computes, per token t (the layer of section 5.3 of the "openPangu
// 2.0 -- architecture, training and Ascend systems" notes, differentiated;
// the gates are recomputed from the saved projection as in the recompute
// paragraph of the Ascend mHC Triton operator article):
//   dH_pre[i] = <g_in, x[i]>,   dl_pre[i] = dH_pre[i] s_i (1 - s_i)
//   u_pre[i]  = inv_rms alpha_pre dl_pre[i]
//   coef      = coef_rest - inv_rms (u_pre . proj_pre) / K
//   dx[t, k] += H_pre[i(k)] g_in[t, d(k)] + (phi u_t)[k] + coef x[t, k]
//   dphi_part[k, g] = sum_t x[t, k] u[t, g]
// The other 20 entries of u, coef_rest (the post and residual gates'
// share of the RMSNorm coefficient) and the Sinkhorn backward come from the
// per-token kernel that runs first: none of them depends on dH_pre.
//
// Design (GB300, one CTA per SM, persistent):
//   * A cluster of C CTAs owns a tile of 64 tokens at a time; CTA r owns the
//     64-column chunks r, r + C, r + 2C, ... of every stream (nck of them),
//     so that the cluster reads 64 C contiguous columns of a row at a time.
//   * First pass (dot warps): TMA brings, per chunk and stream pair, a 16 KB
//     x box (64 tokens x 64 columns x 2 streams) and the 8 KB g_in box into
//     a ring of its own; four warps sum g_in * x[i] per token.  The C
//     partial dot products of each token are exchanged through distributed
//     shared memory and two warps finish u and coef for the tile.
//   * Second pass (MMA and epilogue): a second ring brings, per chunk and
//     stream pair, the same x box again (now from L2), the pair's phi block
//     (bf16, packed once per launch in the workspace) and the g_in box.  One
//     thread issues tcgen05.mma:
//       D1 = U' . PHI2^T  (M = 128 = 64 tokens x 2 streams, N = 64, K = 64):
//         U' holds u in the first 32 K-columns of rows 0..63 and in the last
//         32 of rows 64..127, PHI2 holds phi of stream 2p in its first 32
//         K-columns and of stream 2p+1 in its last 32, so the two halves of
//         D1 are (phi u) of the two streams;
//       D2 += X^T . U     (M = 128 = 2 streams x 64 columns, read MN-major
//         from the box, N = 32 (24 logits), K = 64 tokens): the dphi partial
//         of the CTA's columns, resident in TMEM for the whole kernel.
//     Four epilogue warps per stream pair (one token and stream per thread,
//     as the TMEM lane layout gives) form the increment H_pre g_in + D1 +
//     coef x in bf16 over the x rows it came from, and one thread adds that
//     box to dx with a TMA reduction (the add happens in L2), so dx is never
//     staged on chip.
//   * With phi streamed, shared memory holds two rings deep enough for the
//     two passes to run side by side; the producer serves both without
//     blocking and issues a tile's second-pass boxes only after its first
//     pass ones, so that they come from L2.
//   * u enters both products in bf16, far inside the tolerance of the bf16
//     dx and of the dphi sums.
//   * Every wait is bounded (about one second); on expiry the kernel latches
//     its device error word and returns.
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
__device__ unsigned g_bwd_fused_error;
// Test hook (mhc_test_force_timeout): nonzero makes pre_bwd_fused_kernel run
// one bounded wait that nothing completes, then return.
__device__ unsigned g_force_timeout_bwd;

cudaError_t set_force_timeout_bwd(unsigned on) {
    return cudaMemcpyToSymbol(g_force_timeout_bwd, &on, sizeof(unsigned));
}

cudaError_t read_and_clear_bwd_fused_error(unsigned* word) {
    cudaError_t e = cudaMemcpyFromSymbol(word, g_bwd_fused_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_bwd_fused_error, &zero, sizeof(unsigned));
}

namespace bwdfu {

constexpr int TT = 64;                      // tokens per tile
constexpr int KC = 64;                      // columns per chunk
constexpr int MAX_NCK = 5;                  // chunks per stream per CTA
constexpr int SUB = TT * 128;               // one stream of a box: 64 tokens x 128 B = 8 KB
constexpr int PBOX = 2 * SUB;               // x box of a stream pair: 16 KB
constexpr int GBOX = SUB;                   // g_in box: 8 KB
constexpr int PHIB = KC * 128;              // phi block of a pair: 64 columns x [phi 2p | phi 2p+1]
constexpr int ASLOTS = 3;                   // first pass: [x pair box | g_in box]
constexpr int A_SLOT = PBOX + GBOX;         // 24 KB
constexpr int BSLOTS = 4;                   // second pass: [x pair box | phi block | g_in box]
constexpr int B_SLOT = PBOX + PHIB + GBOX;  // 32 KB
constexpr int NTHREADS = 512;               // 16 warps
constexpr int DOT_WARP0 = 2, NDOT = 4;      // first-pass dot products
constexpr int PREP_WARP0 = 6, NPREP = 2;    // cluster reduction, u and coef
constexpr int EPI_WARP0 = 8, NEPI = 8;      // dx epilogue (4 warps per stream pair), then dphi
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t D1_COL = 0;              // one 64-column buffer per stream pair
constexpr uint32_t D2_COL = 128;            // (chunk, pair) -> 32 columns
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;
constexpr int LEAD = 15;                    // ring-A positions the first pass may run ahead of ring B

// Rings.  Every consumer of a ring visits each of its positions in order
// (an mbarrier parity wait is only sound one phase behind):
//   A: the four dot warps;
//   B: the MMA thread (a commit: its products are done) and the leader of
//      the position's stream pair (its dx reduction has read the box).  Pair
//      p's positions fall in slots p and p + 2 only, so each pair also sees
//      every phase of its own slots.
constexpr uint32_t AEMPTY_COUNT = NDOT;
static_assert(LEAD >= 2 * MAX_NCK, "the first pass must be able to finish the tile ring B waits on");
constexpr uint32_t BEMPTY_COUNT = 2;
static_assert(BSLOTS % 2 == 0, "each stream pair owns every other slot of ring B");

enum : int {
    BAR_AFULL = 0,
    BAR_AEMPTY = BAR_AFULL + ASLOTS,
    BAR_BFULL = BAR_AEMPTY + ASLOTS,
    BAR_BEMPTY = BAR_BFULL + BSLOTS,
    BAR_UFULL = BAR_BEMPTY + BSLOTS,
    BAR_UEMPTY = BAR_UFULL + 1,
    BAR_D1FULL = BAR_UEMPTY + 1,
    BAR_D1EMPTY = BAR_D1FULL + 2,
    BAR_D2DONE = BAR_D1EMPTY + 2,
    BAR_PFULL = BAR_D2DONE + 1,             // partial dots of a tile parity, from every peer
    BAR_PEMPTY = BAR_PFULL + 2,             // every peer has read them
    NBARS = BAR_PEMPTY + 2
};

struct Layout {
    static constexpr uint32_t AR = 0;
    static constexpr uint32_t BR = AR + ASLOTS * A_SLOT;
    static constexpr uint32_t UA = BR + BSLOTS * B_SLOT;       // 128 rows x 128 B
    static constexpr uint32_t U2 = UA + 128 * 128;             // 32 rows x 128 B
    static constexpr uint32_t SC = U2 + 32 * 128;              // per token: H_pre[4], coef
    static constexpr uint32_t PART = SC + TT * 32;             // [2][TT] float4
    static constexpr uint32_t BARS = PART + 2 * TT * 16;
    static constexpr uint32_t MISC = BARS + NBARS * 8;
    static constexpr uint32_t TOTAL = MISC + 64;
};
constexpr size_t SMEM_BYTES = Layout::TOTAL + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
static_assert(Layout::BR % 1024 == 0 && Layout::UA % 1024 == 0 && Layout::U2 % 1024 == 0, "alignment");
static_assert(A_SLOT % 1024 == 0 && B_SLOT % 1024 == 0, "alignment");

struct Params {
    const float* proj;     // [T, 24]
    const float* alpha;    // [3]
    float* rec;            // [T, REC]
    float* part;           // [clusters, K, 24]
    int64_t T;
    int D;
    int nck;               // chunks per stream per CTA
    int ntiles;
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         bool cluster_scope = false) {
    auto test = [&] {
        return cluster_scope ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
    };
    if (test()) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (test()) return true;
        if ((it & 63) == 0) {
            if (*abort_flag) return false;
            if (ptx::globaltimer() - t0 > WAIT_LIMIT_NS) {
                atomicOr(&g_bwd_fused_error, 1u);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// PHI2 in global memory, rows of 64 bf16 (128 B, swizzled by TMA on load):
// block (pair p, chunk q) holds, in row r, phi[(2p) D + 64q + r, 0..31] then
// phi[(2p + 1) D + 64q + r, 0..31], logits 24..31 zero.
__global__ void __launch_bounds__(256)
pre_bwd_phi_pack_kernel(const float* __restrict__ phi, int64_t D, __nv_bfloat16* __restrict__ phi2) {
    const int64_t nq = D / KC;
    const int64_t items = 2 * nq * KC * 8;          // (pair, chunk, row, 16-byte piece)
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; it < items;
         it += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int piece = static_cast<int>(it & 7);
        const int64_t row = it >> 3;                // (p * nq + q) * 64 + r
        const int r = static_cast<int>(row % KC);
        const int64_t pq = row / KC;
        const int p = static_cast<int>(pq / nq);
        const int64_t q = pq % nq;
        const int a = piece >> 2, g0 = (piece & 3) * 8;
        const int64_t k = (2 * p + a) * D + q * KC + r;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int g = g0 + 2 * e;
            w[e] = pack_bf16x2(g < NG ? phi[k * NG + g] : 0.f, g + 1 < NG ? phi[k * NG + g + 1] : 0.f);
        }
        reinterpret_cast<uint4*>(phi2)[it] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

__global__ void __launch_bounds__(NTHREADS, 1)
pre_bwd_fused_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dx,
                     const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_phi,
                     const Params p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    auto bar = [&](int i) { return sbase + Layout::BARS + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Layout::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Layout::MISC + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (g_force_timeout_bwd != 0u) {
        // test hook: one bounded wait that runs out, before anything async
        // starts; the kernel still waits for the per-token kernel it may
        // have started beside (programmatic dependent launch) before leaving
        if (tid == 0 && ptx::forced_wait_runs_out(ptx::smem_u32(smem), 100000ull))
            atomicOr(&g_bwd_fused_error, 1u);
        __syncthreads();
        ptx::griddep_wait();
        return;
    }
    constexpr unsigned FULL = 0xffffffffu;
    const uint32_t C = ptx::cluster_nctarank();
    const uint32_t rank = ptx::cluster_ctarank();
    const int cl = static_cast<int>(ptx::cluster_id_x());
    const int ncl = static_cast<int>(ptx::nclusters_x());
    const int nck = p.nck;
    const int D = p.D;
    const int nq = D / KC;                         // 64-column chunks per stream
    const int64_t K = 4 * static_cast<int64_t>(D);
    const int ntl = p.ntiles > cl ? (p.ntiles - cl + ncl - 1) / ncl : 0;
    auto tile_t0 = [&](int jl) { return static_cast<int64_t>(cl + jl * ncl) * TT; };
    auto chunk_col = [&](int c) { return (c * static_cast<int>(C) + static_cast<int>(rank)) * KC; };

    // ---- set-up ----------------------------------------------------------
    if (tid == 0) {
        for (int s = 0; s < ASLOTS; ++s) {
            ptx::mbar_init(bar(BAR_AFULL + s), 1);
            ptx::mbar_init(bar(BAR_AEMPTY + s), AEMPTY_COUNT);
        }
        for (int s = 0; s < BSLOTS; ++s) {
            ptx::mbar_init(bar(BAR_BFULL + s), 1);
            ptx::mbar_init(bar(BAR_BEMPTY + s), BEMPTY_COUNT);
        }
        ptx::mbar_init(bar(BAR_UFULL), NPREP * 32);
        ptx::mbar_init(bar(BAR_UEMPTY), 1 + NEPI);
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar(BAR_D1FULL + b), 1);
            ptx::mbar_init(bar(BAR_D1EMPTY + b), 4);
            ptx::mbar_init(bar(BAR_PFULL + b), C);
            ptx::mbar_init(bar(BAR_PEMPTY + b), C);
        }
        ptx::mbar_init(bar(BAR_D2DONE), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tm_x);
        ptx::prefetch_tmap(&tm_dx);
        ptx::prefetch_tmap(&tm_g);
        ptx::prefetch_tmap(&tm_phi);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    // U' and U start zero; the preparation warps only ever write their u parts.
    for (int i = tid; i < (128 * 128 + 32 * 128) / 16; i += NTHREADS)
        reinterpret_cast<uint4*>(smem + Layout::UA)[i] = make_uint4(0u, 0u, 0u, 0u);
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    ptx::cluster_sync();   // peers' barriers are initialised before any remote arrive

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ----
        // Positions of both rings run over (tile, chunk, stream pair).  Lane 0
        // polls the two rings without blocking; a ring-B box is issued only
        // after the ring-A box of the same position (so that it comes from
        // L2), and ring A stays at most LEAD positions ahead of ring B, so
        // that the x and g_in it brings in (24 KB a position and CTA, about
        // 40 MB over 112 CTAs) are still in L2 for the second pass.  At
        // T = 32768, D = 5120 a lead of 15 positions (a tile and a half) took
        // 0.900 ms with DRAM reads 1.03x those of a 10-position lead; 10 took
        // 1.087 ms, 12 0.990, 20-30 0.901-0.910, and up to two whole tiles
        // ahead 0.906-0.912 with reads 1.08x.  LEAD >= 2 * MAX_NCK, so the
        // first pass of the tile that ring B waits on can always finish.
        // First pass: normal priority.  An evict-last hint would keep the
        // boxes for the second pass no better (it comes one tile later) and
        // the lines keep that priority after the kernel ends: the next
        // kernel then finds L2 full of them (the forward ran 20% slower).
        const uint64_t keep = ptx::policy_evict_normal();
        const uint64_t drop = ptx::policy_evict_first();   // second pass: last use
        const int npos = ntl * nck * 2;
        int na = 0, nb = 0;
        uint64_t idle_since = ptx::globaltimer();
        while (na < npos || nb < npos) {
            int moved = 0;
            if (lane == 0) {
                if (na < npos && na - nb <= LEAD) {
                    const int slot = na % ASLOTS;
                    if (ptx::mbar_test_wait(bar(BAR_AEMPTY + slot), ((na / ASLOTS) & 1) ^ 1)) {
                        const int jl = na / (2 * nck), c = (na >> 1) % nck, pr = na & 1;
                        const int64_t t0 = tile_t0(jl);
                        const uint32_t dst = sbase + Layout::AR + slot * A_SLOT;
                        const uint32_t fb = bar(BAR_AFULL + slot);
                        ptx::mbar_arrive_expect_tx(fb, A_SLOT);
                        ptx::tma_load_3d(dst, &tm_x, chunk_col(c), static_cast<int>(t0), 2 * pr, fb, keep);
                        ptx::tma_load_2d(dst + PBOX, &tm_g, chunk_col(c), static_cast<int>(t0), fb, keep);
                        ++na;
                        moved = 1;
                    }
                }
                if (nb < na) {
                    const int slot = nb % BSLOTS;
                    if (ptx::mbar_test_wait(bar(BAR_BEMPTY + slot), ((nb / BSLOTS) & 1) ^ 1)) {
                        const int jl = nb / (2 * nck), c = (nb >> 1) % nck, pr = nb & 1;
                        const int64_t t0 = tile_t0(jl);
                        const uint32_t dst = sbase + Layout::BR + slot * B_SLOT;
                        const uint32_t fb = bar(BAR_BFULL + slot);
                        ptx::mbar_arrive_expect_tx(fb, B_SLOT);
                        ptx::tma_load_3d(dst, &tm_x, chunk_col(c), static_cast<int>(t0), 2 * pr, fb, drop);
                        ptx::tma_load_2d(dst + PBOX, &tm_phi, 0, (pr * nq + c * static_cast<int>(C) +
                                                                   static_cast<int>(rank)) * KC, fb, keep);
                        ptx::tma_load_2d(dst + PBOX + PHIB, &tm_g, chunk_col(c), static_cast<int>(t0), fb, drop);
                        ++nb;
                        moved = 1;
                    }
                }
                if (moved) {
                    idle_since = ptx::globaltimer();
                } else if (*abort_flag) {
                    moved = -1;
                } else if (ptx::globaltimer() - idle_since > WAIT_LIMIT_NS) {
                    atomicOr(&g_bwd_fused_error, 1u);
                    *abort_flag = 1;
                    moved = -1;
                }
            }
            moved = __shfl_sync(FULL, moved, 0);
            na = __shfl_sync(FULL, na, 0);
            nb = __shfl_sync(FULL, nb, 0);
            if (moved < 0) goto done;
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer -----
        constexpr uint32_t IDESC1 = ptx::idesc_bf16_f32(128, KC);               // D1: both K-major
        constexpr uint32_t IDESC2 = ptx::idesc_bf16_f32(128, 32) | (1u << 15);  // D2: A (x^T) MN-major
        // descriptors built once; the loop only moves their start address
        const uint64_t desc_xmn = ptx::sw128_mnmajor_desc(sbase + Layout::BR, SUB, 1024);
        const uint64_t desc_phi = ptx::sw128_kmajor_desc(sbase + Layout::BR + PBOX);
        const uint64_t desc_u2 = ptx::sw128_kmajor_desc(sbase + Layout::U2);
        const uint64_t desc_ua = ptx::sw128_kmajor_desc(sbase + Layout::UA);
        int s = 0;
        for (int ju = 0; ju < ntl; ++ju) {
            bool ok = true;
            if (lane == 0) ok = wait_bar(bar(BAR_UFULL), ju & 1, abort_flag);
            if (!__shfl_sync(FULL, ok, 0)) goto done;
            for (int c = 0; c < nck; ++c, ++s) {
                for (int pp = 0; pp < 2; ++pp) {
                    const int n = (ju * nck + c) * 2 + pp;
                    const int slot = n % BSLOTS;
                    if (lane == 0)
                        ok = wait_bar(bar(BAR_BFULL + slot), (n / BSLOTS) & 1, abort_flag) &&
                             wait_bar(bar(BAR_D1EMPTY + pp), (s & 1) ^ 1, abort_flag);
                    if (!__shfl_sync(FULL, ok, 0)) goto done;
                    ptx::tc_fence_after();
                    if (lane == 0) {
                        // D2 first: the commit of D1FULL then also tells the pair's
                        // epilogue that the MMA no longer reads the x box, which it
                        // overwrites with the dx increment
                        const uint64_t dx2 = ptx::desc_add(desc_xmn, slot * B_SLOT);
#pragma unroll
                        for (int kk = 0; kk < TT / 16; ++kk)
                            ptx::tc_mma_f16(tmem + D2_COL + (c * 2 + pp) * 32, ptx::desc_add(dx2, kk * 2048),
                                            ptx::desc_add(desc_u2, kk * 32), IDESC2, (ju | kk) != 0);
                        const uint64_t dphi = ptx::desc_add(desc_phi, slot * B_SLOT);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            ptx::tc_mma_f16(tmem + D1_COL + pp * KC, ptx::desc_add(desc_ua, kk * 32),
                                            ptx::desc_add(dphi, kk * 32), IDESC1, kk != 0);
                        ptx::tc_commit(bar(BAR_D1FULL + pp));
                        ptx::tc_commit(bar(BAR_BEMPTY + slot));
                    }
                    __syncwarp();
                }
            }
            if (lane == 0) ptx::tc_commit(bar(BAR_UEMPTY));
            __syncwarp();
        }
        if (lane == 0) ptx::tc_commit(bar(BAR_D2DONE));
        __syncwarp();
    } else if (warp < PREP_WARP0) {
        // -------------------------------------- first pass: dot products --
        const int q = tid - DOT_WARP0 * 32;            // 0..127
        const int t = q >> 1, h = q & 1;               // token, half of each chunk
        int n = 0;                                     // ring-A position
        for (int jd = 0; jd < ntl; ++jd) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            bool ok = true;
            for (int c = 0; c < nck && ok; ++c) {
#pragma unroll
                for (int pr = 0; pr < 2; ++pr, ++n) {
                    const int slot = n % ASLOTS;
                    ok = ok && __all_sync(FULL, wait_bar(bar(BAR_AFULL + slot), (n / ASLOTS) & 1, abort_flag));
                    if (!ok) break;
                    const unsigned char* xb = smem + Layout::AR + slot * A_SLOT;
                    const unsigned char* gb = xb + PBOX;
#pragma unroll
                    for (int cq = 0; cq < 4; ++cq) {
                        const uint32_t off = static_cast<uint32_t>(t * 128 + (((h * 4 + cq) ^ (t & 7)) << 4));
                        float fg[8];
                        Vec<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4*>(gb + off), fg);
#pragma unroll
                        for (int s2 = 0; s2 < 2; ++s2) {
                            float fx[8];
                            Vec<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4*>(xb + s2 * SUB + off), fx);
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[2 * pr + s2] = fmaf(fg[e], fx[e], acc[2 * pr + s2]);
                        }
                    }
                    // the slot's next bytes come through the async proxy (TMA)
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(bar(BAR_AEMPTY + slot));
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] += __shfl_xor_sync(FULL, acc[i], 1);
            const int ps = jd & 1;
            if (ok) ok = __all_sync(FULL, wait_bar(bar(BAR_PEMPTY + ps), ((jd >> 1) & 1) ^ 1, abort_flag, true));
            if (ok && h == 0)
                reinterpret_cast<float4*>(smem + Layout::PART + ps * TT * 16)[t] =
                    make_float4(acc[0], acc[1], acc[2], acc[3]);
            if (ptx::named_bar_or(1, NDOT * 32, !ok)) goto done;
            if (warp == DOT_WARP0 && lane < static_cast<int>(C)) {
                ptx::fence_acq_rel_cluster();
                ptx::mbar_arrive_remote(ptx::mapa(bar(BAR_PFULL + ps), static_cast<uint32_t>(lane)));
            }
        }
    } else if (warp < EPI_WARP0) {
        // ------------------------------ cluster reduction, u and coef -----
        const int t = tid - PREP_WARP0 * 32;           // 0..63: token of the tile
        // the per-token kernel before this one (which may still be running:
        // programmatic dependent launch) wrote the records read below
        ptx::griddep_wait();
        const float apre = p.alpha[0];
        const float invK = 1.0f / static_cast<float>(K);
        for (int jl = 0; jl < ntl; ++jl) {
            const int64_t tg = tile_t0(jl) + t;
            const bool valid = tg < p.T;
            float u[32], hp[4] = {0.f, 0.f, 0.f, 0.f}, ds[4] = {0.f, 0.f, 0.f, 0.f};
            float pj[4] = {0.f, 0.f, 0.f, 0.f}, coef_rest = 0.f, s = 0.f;
#pragma unroll
            for (int g = 0; g < 32; ++g) u[g] = 0.f;
            if (valid) {
                const float* rr = p.rec + tg * REC;
#pragma unroll
                for (int v = 1; v < 6; ++v) {
                    const float4 a = reinterpret_cast<const float4*>(rr + REC_U)[v];
                    u[4 * v] = a.x; u[4 * v + 1] = a.y; u[4 * v + 2] = a.z; u[4 * v + 3] = a.w;
                }
                const float4 a = reinterpret_cast<const float4*>(rr + REC_HPRE)[0];
                hp[0] = a.x; hp[1] = a.y; hp[2] = a.z; hp[3] = a.w;
                const float4 cs = reinterpret_cast<const float4*>(rr + REC_COEF)[0];
                coef_rest = cs.x;
                s = cs.y;
                const float4 dd = reinterpret_cast<const float4*>(rr + REC_DSIG)[0];
                ds[0] = dd.x; ds[1] = dd.y; ds[2] = dd.z; ds[3] = dd.w;
                const float4 pq = reinterpret_cast<const float4*>(p.proj + tg * NG)[0];
                pj[0] = pq.x; pj[1] = pq.y; pj[2] = pq.z; pj[3] = pq.w;
            }
            const int ps = jl & 1;
            bool ok = __all_sync(FULL, wait_bar(bar(BAR_PFULL + ps), (jl >> 1) & 1, abort_flag, true));
            float dh[4] = {0.f, 0.f, 0.f, 0.f};
            if (ok) {
                const uint32_t src = sbase + Layout::PART + ps * TT * 16 + t * 16;
#pragma unroll 4
                for (uint32_t pr = 0; pr < C; ++pr) {
                    const float4 v = ptx::ld_cluster_v4(ptx::mapa(src, pr));
                    dh[0] += v.x; dh[1] += v.y; dh[2] += v.z; dh[3] += v.w;
                }
            }
            if (ptx::named_bar_or(2, NPREP * 32, !ok)) goto done;
            if (t < static_cast<int>(C)) {
                // a credit: the partials read above already feed dh
                ptx::mbar_arrive_remote_relaxed(ptx::mapa(bar(BAR_PEMPTY + ps), static_cast<uint32_t>(t)));
            }
            float dl[4], cadd = 0.f, da0 = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dl[i] = dh[i] * ds[i];
                u[i] = s * apre * dl[i];
                cadd = fmaf(u[i], pj[i], cadd);
                da0 = fmaf(dl[i], pj[i], da0);
            }
            const float coef = coef_rest - s * cadd * invK;
            if (valid && rank == 0) {
                reinterpret_cast<float4*>(p.rec + tg * REC + REC_DL)[0] = make_float4(dl[0], dl[1], dl[2], dl[3]);
                p.rec[tg * REC + REC_DA] = da0;
            }
            if (!__all_sync(FULL, wait_bar(bar(BAR_UEMPTY), (jl & 1) ^ 1, abort_flag))) goto done;
            // U' rows t and 64 + t; U column t (rows g < 24); per-token scalars
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                const uint4 w = make_uint4(pack_bf16x2(u[8 * qq], u[8 * qq + 1]), pack_bf16x2(u[8 * qq + 2], u[8 * qq + 3]),
                                           pack_bf16x2(u[8 * qq + 4], u[8 * qq + 5]),
                                           pack_bf16x2(u[8 * qq + 6], u[8 * qq + 7]));
                *reinterpret_cast<uint4*>(smem + Layout::UA + ptx::sw128_off(t, qq * 8)) = w;
                *reinterpret_cast<uint4*>(smem + Layout::UA + ptx::sw128_off(64 + t, 32 + qq * 8)) = w;
            }
#pragma unroll
            for (int g = 0; g < NG; ++g)
                *reinterpret_cast<__nv_bfloat16*>(smem + Layout::U2 + ptx::sw128_off(g, t)) = __float2bfloat16_rn(u[g]);
            float* sc = reinterpret_cast<float*>(smem + Layout::SC) + t * 8;
            reinterpret_cast<float4*>(sc)[0] = make_float4(hp[0], hp[1], hp[2], hp[3]);
            sc[4] = coef;
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(bar(BAR_UFULL));
        }
    } else {
        // ------------------------------------------------- epilogue -------
        const int e = tid - EPI_WARP0 * 32;            // 0..255
        const int pp = e >> 7;                         // stream pair
        const int q = e & 127;                         // TMEM lane = row of D1 / D2
        const int t = q & 63;                          // token of the tile
        const int si = 2 * pp + (q >> 6);              // stream
        const int wq = warp & 3;                       // TMEM lane quarter of this warp
        const bool leader = q == 0;                    // issues the pair's dx reductions
        int s = 0;
        bool aborted = false;
        for (int ju = 0; ju < ntl && !aborted; ++ju) {
            const int t0 = static_cast<int>(tile_t0(ju));
            // every thread of the pair passes the same named barriers, so a
            // failed wait is carried in `ok` and acted on at the barrier
            bool ok = __all_sync(FULL, wait_bar(bar(BAR_UFULL), ju & 1, abort_flag));
            float hpre = 0.f, cf = 0.f;
            if (ok) {
                const float* sc = reinterpret_cast<const float*>(smem + Layout::SC) + t * 8;
                hpre = sc[si];
                cf = sc[4];
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(BAR_UEMPTY));
            }
            for (int c = 0; c < nck; ++c, ++s) {
                const int n = (ju * nck + c) * 2 + pp;
                const int slot = n % BSLOTS;
                ok = ok && __all_sync(FULL, wait_bar(bar(BAR_D1FULL + pp), s & 1, abort_flag)) &&
                     __all_sync(FULL, wait_bar(bar(BAR_BFULL + slot), (n / BSLOTS) & 1, abort_flag));
                unsigned char* box = smem + Layout::BR + slot * B_SLOT;
                unsigned char* xb = box + (q >> 6) * SUB;
                if (ok) {
                    ptx::tc_fence_after();
                    uint32_t v[4][16];
                    const uint32_t ta = tmem + (static_cast<uint32_t>(wq * 32) << 16) + D1_COL + pp * KC;
#pragma unroll
                    for (int h16 = 0; h16 < 4; ++h16) ptx::tmem_ld16(ta + h16 * 16, v[h16]);
                    ptx::tmem_wait_ld();
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(bar(BAR_D1EMPTY + pp));
                    const unsigned char* gb = box + PBOX + PHIB;
                    // dx increment of this token and stream, written over the
                    // x row it was computed from (same swizzled place); column
                    // pairs through packed fp32 multiply-adds, each lane rounded
                    // as fmaf
                    const float2 hp2 = make_float2(hpre, hpre), cf2 = make_float2(cf, cf);
#pragma unroll
                    for (int cq = 0; cq < 8; ++cq) {
                        const uint32_t off = static_cast<uint32_t>(t * 128 + ((cq ^ (t & 7)) << 4));
                        const uint4 xw = *reinterpret_cast<const uint4*>(xb + off);
                        const uint4 gw = *reinterpret_cast<const uint4*>(gb + off);
                        const uint32_t xa[4] = {xw.x, xw.y, xw.z, xw.w}, ga[4] = {gw.x, gw.y, gw.z, gw.w};
                        uint32_t ow[4];
#pragma unroll
                        for (int w2 = 0; w2 < 4; ++w2) {
                            const int col = cq * 8 + 2 * w2;
                            const float2 fx = make_float2(__uint_as_float(xa[w2] << 16), __uint_as_float(xa[w2] & 0xffff0000u));
                            const float2 fg = make_float2(__uint_as_float(ga[w2] << 16), __uint_as_float(ga[w2] & 0xffff0000u));
                            const float2 d1 = make_float2(__uint_as_float(v[col >> 4][col & 15]),
                                                          __uint_as_float(v[(col + 1) >> 4][(col + 1) & 15]));
                            const float2 o2 = __ffma2_rn(hp2, fg, __ffma2_rn(cf2, fx, d1));
                            const __nv_bfloat162 ob = __floats2bfloat162_rn(o2.x, o2.y);
                            ow[w2] = *reinterpret_cast<const uint32_t*>(&ob);
                        }
                        *reinterpret_cast<uint4*>(xb + off) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                    }
                    ptx::fence_proxy_async_smem();
                }
                if (ptx::named_bar_or(3 + pp, 128, !ok)) {
                    aborted = true;
                    break;
                }
                if (leader) {
                    // dx[t0.., 2pp..2pp+1, chunk] += the pair's box; the slot is
                    // free once the reduction has read it
                    ptx::tma_reduce_add_3d(&tm_dx, chunk_col(c), t0, 2 * pp, sbase + Layout::BR + slot * B_SLOT);
                    ptx::bulk_commit();
                    ptx::bulk_wait_read<0>();
                    ptx::mbar_arrive(bar(BAR_BEMPTY + slot));
                }
            }
        }
        if (leader) ptx::bulk_wait<0>();   // the reductions are complete before the kernel ends
        // dphi partial of this cluster: D2 row q of (chunk c, pair pp) is
        // column k = si * D + 64 (c C + rank) + t.
        if (!aborted && __all_sync(FULL, wait_bar(bar(BAR_D2DONE), 0, abort_flag))) {
            ptx::tc_fence_after();
            float* out = p.part + static_cast<int64_t>(cl) * K * NG;
            for (int c = 0; c < nck; ++c) {
                uint32_t w0[16], w1[16];
                const uint32_t ta = tmem + (static_cast<uint32_t>(wq * 32) << 16) + D2_COL + (c * 2 + pp) * 32;
                ptx::tmem_ld16(ta, w0);
                ptx::tmem_ld16(ta + 16, w1);
                ptx::tmem_wait_ld();
                float4* o4 = reinterpret_cast<float4*>(out + (static_cast<int64_t>(si) * D + chunk_col(c) + t) * NG);
                const bool any = ntl > 0;
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                    o4[v4] = any ? make_float4(__uint_as_float(w0[4 * v4]), __uint_as_float(w0[4 * v4 + 1]),
                                               __uint_as_float(w0[4 * v4 + 2]), __uint_as_float(w0[4 * v4 + 3]))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int v4 = 0; v4 < 2; ++v4)
                    o4[4 + v4] = any ? make_float4(__uint_as_float(w1[4 * v4]), __uint_as_float(w1[4 * v4 + 1]),
                                                   __uint_as_float(w1[4 * v4 + 2]), __uint_as_float(w1[4 * v4 + 3]))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
            }
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
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
    ptx::cluster_sync();   // no CTA leaves while a peer may still touch its shared memory
}

// Smallest cluster whose per-CTA share is a whole number of 64-column chunks
// per stream, at most MAX_NCK of them (dphi accumulators in TMEM).
int cluster_for(int64_t D) {
    if (D <= 0 || D % KC != 0) return 0;
    const int64_t nc = D / KC;
    for (int C : {1, 2, 4, 8, 16})
        if (nc % C == 0 && nc / C <= MAX_NCK) return C;
    return 0;
}

bool set_attributes_once() {
    static int ok = -1;
    static std::once_flag once;
    std::call_once(once, [] {
        ok = cudaFuncSetAttribute(pre_bwd_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(SMEM_BYTES)) == cudaSuccess &&
             cudaFuncSetAttribute(pre_bwd_fused_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                 cudaSuccess;
    });
    return ok == 1;
}

cudaLaunchConfig_t config(int C, int nclusters, cudaStream_t s, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nclusters * C));
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// Clusters of size C that fit on the device at once (per device, cached).
int max_clusters(int C) {
    static int cache[64][5];
    static std::once_flag once[64][5];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int ci = 0;
    while ((1 << ci) < C) ++ci;
    if (ci > 4 || (1 << ci) != C) return 0;
    std::call_once(once[dev][ci], [&] {
        int n = 0;
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg = config(C, 152 / C > 0 ? 152 / C : 1, nullptr, attr);
        if (!set_attributes_once() || cudaOccupancyMaxActiveClusters(&n, pre_bwd_fused_kernel, &cfg) != cudaSuccess)
            n = 0;
        cache[dev][ci] = n;
    });
    return cache[dev][ci];
}

// dims (d, t, stream) of a [T, 4, D] tensor: box = 64 columns x 64 tokens x
// 2 streams, laid out in shared memory as [stream][token][64 columns]
bool encode_x(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* tm, const void* base, int64_t T, int64_t D) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T), 4};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(8 * D), static_cast<cuuint64_t>(2 * D)};
    const cuuint32_t box[3] = {KC, TT, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A [rows, inner] bf16 matrix read in boxes of 64 x 64.
bool encode_2d(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* tm, const void* base, int64_t inner,
               int64_t rows) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(2 * inner)};
    const cuuint32_t box[2] = {KC, TT};
    const cuuint32_t estr[2] = {1, 1};
    return encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace bwdfu

bool pre_bwd_fused_supports(int64_t T, int64_t D) {
    if (T < 1 || T >= (int64_t(1) << 31) || 4 * D * T >= (int64_t(1) << 46)) return false;
    const int C = bwdfu::cluster_for(D);
    return C > 0 && tensor_map_encoder() != nullptr && bwdfu::max_clusters(C) > 0;
}

size_t pre_bwd_fused_phi_bytes(int64_t D) { return static_cast<size_t>(D) * 256; }

cudaError_t launch_pre_bwd_fused_main(const void* g_in, const void* x, const float* phi,
                                      const float* proj, const float* alpha, float* rec,
                                      int64_t T, int64_t D, int64_t max_parts, void* dx,
                                      float* part, void* phi2, int64_t* nparts, cudaStream_t s) {
    auto encode = tensor_map_encoder();
    const int C = bwdfu::cluster_for(D);
    if (encode == nullptr || C == 0 || !bwdfu::set_attributes_once()) return cudaErrorNotSupported;
    CUtensorMap tx, tdx, tg, tphi;
    if (!bwdfu::encode_x(encode, &tx, x, T, D) || !bwdfu::encode_x(encode, &tdx, dx, T, D) ||
        !bwdfu::encode_2d(encode, &tg, g_in, D, T) || !bwdfu::encode_2d(encode, &tphi, phi2, bwdfu::KC, 2 * D))
        return cudaErrorInvalidValue;
    (void)phi;
    (void)phi2;
    bwdfu::Params prm;
    prm.proj = proj;
    prm.alpha = alpha;
    prm.rec = rec;
    prm.part = part;
    prm.T = T;
    prm.D = static_cast<int>(D);
    prm.nck = static_cast<int>(D / bwdfu::KC / C);
    prm.ntiles = static_cast<int>((T + bwdfu::TT - 1) / bwdfu::TT);
    int64_t ncl = bwdfu::max_clusters(C);
    if (ncl > prm.ntiles) ncl = prm.ntiles;
    if (ncl > max_parts) ncl = max_parts;
    if (ncl <= 0) return cudaErrorNotSupported;
    *nparts = ncl;
    // Programmatic dependent launch: the kernel may start while the
    // per-token kernel before it finishes; only the reduction warps need that
    // kernel's records, and they wait for it (griddepcontrol.wait).
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = bwdfu::config(C, static_cast<int>(ncl), s, attr);
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, bwdfu::pre_bwd_fused_kernel, tx, tdx, tg, tphi, prm);
}

cudaError_t launch_pre_bwd_phi_pack(const float* phi, int64_t D, void* phi2, cudaStream_t s) {
    // phi as bf16 pair blocks for the second pass (read from L2 by TMA)
    const int64_t pack_items = 2 * (D / bwdfu::KC) * bwdfu::KC * 8;
    const int64_t pack_blocks = (pack_items + 255) / 256;
    bwdfu::pre_bwd_phi_pack_kernel<<<static_cast<unsigned>(pack_blocks < 1024 ? pack_blocks : 1024), 256, 0, s>>>(
        phi, D, static_cast<__nv_bfloat16*>(phi2));
    return cudaGetLastError();
}

}  // namespace mhc
