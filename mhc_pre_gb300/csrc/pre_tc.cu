// pre_tc.cu -- fused tensor-core pre forward of the mHC layer (bf16, n = 4),
// and the library's device error word.
//
// What it computes, per token (section 5.3 of the "openPangu 2.0 --
// architecture, training and Ascend systems" notes): inv_rms over the
// flattened 4*D row, proj = x_bar . phi (24 logits), gates and Sinkhorn, and
// x_in = sum_i H_pre[i] x[i].  With no x_in buffer the mix warps only keep
// the hand-off protocol and the kernel computes the gates and saved state
// alone (the recompute of the Ascend mHC operator article's backward).
//
// Design (GB300, one CTA per SM, persistent):
//   * A cluster of C CTAs owns a tile of 64 tokens at a time (small tiles keep
//     the time between the two reads of x short enough for L2 to serve the
//     second).  For the projection, CTA c owns the 64-column chunks c, c + C,
//     c + 2C, ... of every stream (4*D/C columns), whose phi rows stay
//     resident in shared memory as bf16 hi + lo halves (phi = hi + lo to
//     2^-17 relative).  Interleaving the chunks makes the cluster read 64*C
//     contiguous columns of each token row at a time, which DRAM serves far
//     better than C scattered 128-byte pieces.  For the mix, CTA c owns the
//     contiguous columns [c*D/C, (c+1)*D/C).
//   * A TMA producer warp streams the tile's x slice through a ring of 16 KB
//     stages (64 tokens x 64 columns of two streams, 128-byte swizzle); one
//     thread issues tcgen05.mma with the stage's 128 rows (two streams of 64
//     tokens) as A: against the two streams' phi chunks side by side (N = 96
//     = 2 x (24 hi + 24 lo)), each row keeping the half of its own stream,
//     and against the stage itself (N = 128), whose diagonal is each row's
//     sum of x^2.  Few, large MMAs matter: a tcgen05.mma issues every few
//     tens of cycles at best.  Accumulators live in TMEM, two of each, so
//     the next tile's MMAs overlap this tile's epilogue.
//   * Four gate warps read each token's two partial records (one per
//     stream of a pair) from TMEM and push them, with the partial sum of
//     squares, into the shared memory of the CTA that reduces that token
//     (st.async completing on the receiver's mbarrier: no fences).  Each CTA reduces 64/C tokens over the C
//     partials, computes H_pre first and pushes it to every CTA of the
//     cluster the same way, and only then runs the other gates and Sinkhorn
//     and writes them out.  Credit barriers (records read, H_pre used) let
//     consecutive tiles overlap without a cluster-wide rendezvous.
//   * Eight mix warps form x_in = sum_i H_pre[i] x[i] over the CTA's D-slice:
//     x is read from HBM once (TMA, normal L2 priority) and a second time,
//     soon after, for the mix, from L2.
//   * Every wait is bounded (about one second); on expiry the kernel latches
//     the device error word, lets the other roles drain and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "launch.h"
#include "mhc_common.cuh"
#include "tc_ptx.cuh"

namespace mhc {

// Latched by kernels whose bounded waits ran out; read and cleared by
// mhc_get_last_device_error().
__device__ unsigned g_device_error;
// Test hook (mhc_test_force_timeout): nonzero makes pre_tc_kernel run one
// bounded wait that nothing completes, then return.  Passed to the kernel as
// a launch parameter (no global read at the kernel's start).
static std::atomic<unsigned> g_force_timeout_pre{0u};

cudaError_t set_force_timeout_pre(unsigned on) {
    g_force_timeout_pre.store(on);
    return cudaSuccess;
}

cudaError_t read_and_clear_bwd_tc_error(unsigned* word);      // pre_bwd_tc.cu
cudaError_t read_and_clear_bwd_fused_error(unsigned* word);   // pre_bwd_fused.cu
cudaError_t read_and_clear_post_pre_error(unsigned* word);    // post_pre_tc.cu
cudaError_t read_and_clear_post_norm_error(unsigned* word);   // post_norm.cu
cudaError_t read_and_clear_small_error(unsigned* word);       // pre_small.cu
bool pre_small_supports(int64_t T, int64_t D);                 // pre_small.cu
cudaError_t launch_pre_small(const void* x, const float* phi, const float* b, const float* alpha, int64_t T,
                             int64_t D, int iters, float eps, void* x_in, float* H_pre, float* H_post,
                             float* H_res, float* proj, float* inv_rms, unsigned force_timeout, cudaStream_t s);

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
    if (e != cudaSuccess) return e;
    *word |= other;
    other = 0;
    e = read_and_clear_post_pre_error(&other);
    if (e != cudaSuccess) return e;
    *word |= other;
    other = 0;
    e = read_and_clear_post_norm_error(&other);
    if (e != cudaSuccess) return e;
    *word |= other;
    other = 0;
    e = read_and_clear_small_error(&other);
    *word |= other;
    return e;
}

namespace tc {

constexpr int TILE_M = 64;                        // tokens per tile (MMA M)
constexpr int KW = 64;                            // K columns per chunk (128 B rows)
constexpr int STAGES = 5;
constexpr int NB = 48;                            // MMA N: 24 hi + 24 lo
constexpr int SUB_BYTES = TILE_M * KW * 2;        // one stream of a stage: 8 KB
constexpr int STAGE_BYTES = 2 * SUB_BYTES;        // a stage holds a stream pair: 16 KB
constexpr int PHI_CHUNK_BYTES = NB * KW * 2;      // 6 KB
constexpr int MAX_NCH = 20;                       // K-slice <= 1280 columns
constexpr int NTHREADS = 512;                     // 16 warps
constexpr int GATE_WARP0 = 2, NGATE = 4;          // TMEM readers, cluster reduction, H_pre
constexpr int SK_WARP0 = 6, NSK = 2;             // Sinkhorn, other gates, outputs (one per tile parity)
constexpr int MIX_WARP0 = 8, NMIX = 8;            // x_in = sum_i H_pre[i] x[i]
static_assert(GATE_WARP0 + NGATE == SK_WARP0 && SK_WARP0 + NSK == MIX_WARP0 && MIX_WARP0 + NMIX == NTHREADS / 32,
              "warp roles: producer, MMA, gates, Sinkhorn, mix");
// Token pieces a mix thread loads before it computes (4 streams x 16 B each).
// Two keep the mix ahead of the tiles; four put so many L2 reads in flight
// that the TMA stream's boxes land later and the whole kernel slows by 4%.
constexpr int MIX_UNROLL = 2;
constexpr int SKF = 28;                           // hand-off record: proj[24], inv_rms (floats)
constexpr int NHP = 4;                            // H_pre buffers: tiles between reducers and mixes
constexpr int REC = 25;                           // partial record: 24 logits + sum x^2
constexpr int RB = 28;                            // its stride in floats (16-byte aligned)
constexpr uint32_t REC_TX = REC * 4;              // bytes of one record pushed to its reducer
constexpr int TMEM_COLS = 512;                    // two (projection, Gram) accumulator pairs
constexpr uint32_t GRAM_COL = 256;                // projection at 0 / 128, Gram at 256 / 384
// One MMA covers a whole stage: its two 64-token stream boxes are the 128
// rows of A.  B for the projection is the two streams' phi chunks one after
// the other (N = 96), so rows of the first stream keep columns 0..47 and
// rows of the second columns 48..95; the Gram product is the stage times
// its own transpose (N = 128), whose diagonal holds the sums of squares.
constexpr uint32_t IDESC = ptx::idesc_bf16_f32(2 * TILE_M, 2 * NB);
constexpr uint32_t IDESC_GRAM = ptx::idesc_bf16_f32(2 * TILE_M, 2 * TILE_M);
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;  // 1 s

enum : int {
    BAR_FULL = 0,
    BAR_EMPTY = BAR_FULL + STAGES,
    BAR_ACC_FULL = BAR_EMPTY + STAGES,
    BAR_ACC_EMPTY = BAR_ACC_FULL + 2,
    BAR_RECV = BAR_ACC_EMPTY + 2,    // this CTA's tokens: every peer's partial record arrived
    BAR_RFREE = BAR_RECV + 1,       // every reducer of the cluster has read the last tile's records
    BAR_HPRE = BAR_RFREE + 1,       // [NHP] H_pre of tile it (buffer it % NHP) arrived from the reducers
    BAR_HFREE = BAR_HPRE + NHP,     // [NHP] every CTA's mix has finished with that buffer
    BAR_SKFULL = BAR_HFREE + NHP,   // [2] reduced tokens handed to the Sinkhorn warp
    BAR_SKEMPTY = BAR_SKFULL + 2,   // [2] the Sinkhorn warp is done with them
    NBARS = BAR_SKEMPTY + 2
};

// Byte offsets inside the (1024-aligned) dynamic shared memory.
struct Layout {
    uint32_t phi, stages, recv, hpre, sk, bars, misc, total;
    __host__ __device__ static Layout make(int nch, int tpc) {
        Layout L;
        L.phi = 0;
        L.stages = static_cast<uint32_t>(nch) * PHI_CHUNK_BYTES;   // multiple of 1024
        L.recv = L.stages + STAGES * STAGE_BYTES;    // [C senders][TILE_M / C tokens][2 halves][RB]
        L.hpre = L.recv + 2 * TILE_M * RB * 4;
        L.sk = L.hpre + NHP * TILE_M * 16;            // [2][tpc][SKF]
        L.bars = L.sk + 2 * tpc * SKF * 4;
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
    unsigned force_timeout;   // test hook
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
    constexpr int TPC = TILE_M / C;                // tokens each CTA reduces
    const Layout L = Layout::make(p.nch, TPC);
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bars = sbase + L.bars;
    auto bar = [&](int i) { return bars + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 16);
    float* gate_par = reinterpret_cast<float*>(smem + L.misc + 64);   // alpha[3], b[24]
    const float* recv = reinterpret_cast<const float*>(smem + L.recv);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (p.force_timeout != 0u) {
        // test hook: one bounded wait that runs out, before anything async
        // starts; every CTA of the launch takes this path and none touches a
        // peer, so leaving here is safe
        if (tid == 0 && ptx::forced_wait_runs_out(ptx::smem_u32(smem), 100000ull)) atomicOr(&g_device_error, 1u);
        __syncthreads();
        return;
    }
    const uint32_t c = ptx::cluster_ctarank();
    const int cid = static_cast<int>(ptx::cluster_id_x());
    const int ncl = static_cast<int>(ptx::nclusters_x());
    const int D = p.D, Dc = p.Dc, nch = p.nch;
    const int cpd = Dc / KW;                       // chunks per stream
    const int64_t K = 4ll * D;
    const int ntl = p.ntiles > cid ? (p.ntiles - cid + ncl - 1) / ncl : 0;   // tiles of this cluster

    // ---- set-up: barriers, TMEM, gate parameters, resident phi slice ------
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar(BAR_FULL + s), 1);
            ptx::mbar_init(bar(BAR_EMPTY + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(bar(BAR_ACC_FULL + i), 1);
            ptx::mbar_init(bar(BAR_ACC_EMPTY + i), 128);
            ptx::mbar_init(bar(BAR_SKFULL + i), 1);
            ptx::mbar_init(bar(BAR_SKEMPTY + i), 1);
        }
        ptx::mbar_init(bar(BAR_RECV), 1);
        ptx::mbar_init(bar(BAR_RFREE), C);
        // receive barriers are armed one use ahead, before any peer can send:
        // records of the first tile, H_pre of the first two
        if (ntl > 0) ptx::mbar_arrive_expect_tx(bar(BAR_RECV), 2 * TILE_M * REC_TX);
        for (int i = 0; i < NHP; ++i) {
            ptx::mbar_init(bar(BAR_HPRE + i), 1);
            ptx::mbar_init(bar(BAR_HFREE + i), C);
            if (i < ntl) ptx::mbar_arrive_expect_tx(bar(BAR_HPRE + i), TILE_M * 16);
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
        // The first ring loads go out now, so that they are in flight while
        // phi is staged (a fresh slot needs no wait); the producer loop below
        // skips them.
        ptx::prefetch_tmap(&tmap_x);
        const uint64_t pol = ptx::policy_evict_normal();
        const int first = ntl * (nch / 2) < STAGES ? ntl * (nch / 2) : STAGES;
        for (int n = 0; n < first; ++n) {
            const int j = cid + (n / (nch / 2)) * ncl, st = n % (nch / 2);
            const int pr = st / cpd, sub = st % cpd;
            ptx::mbar_arrive_expect_tx(bar(BAR_FULL + n), STAGE_BYTES);
            ptx::tma_load_3d(sbase + L.stages + n * STAGE_BYTES, &tmap_x, (sub * C + static_cast<int>(c)) * KW,
                             j * TILE_M, 2 * pr, bar(BAR_FULL + n), pol);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (tid < 3) gate_par[tid] = p.alpha[tid];
    if (tid >= 32 && tid < 32 + NG) gate_par[3 + tid - 32] = p.b[tid - 32];
    // phi slice -> bf16 hi / lo rows in the swizzled K-major layout of the
    // MMA's B operand: chunk ch, row n (< 24: hi of logit n, else lo of
    // logit n - 24), 16-byte piece q of the row at (q ^ (n & 7)).  Item
    // (ch, q, g) is 8 consecutive K rows of logit g.  A thread issues the
    // loads of all its items before it converts any, so that the set-up
    // waits for one round trip to memory, not one per item.
    {
        constexpr int PHI_ITEMS = (MAX_NCH * 8 * NG + NTHREADS - 1) / NTHREADS;
        const int nitems = nch * 8 * NG;
        float v[PHI_ITEMS][8];
#pragma unroll
        for (int m = 0; m < PHI_ITEMS; ++m) {
            const int item = tid + m * NTHREADS;
            if (item < nitems) {
                const int g = item % NG;
                const int q = (item / NG) % 8;
                const int ch = item / (NG * 8);
                // chunk order: stream pair, chunk of the slice, stream in the
                // pair, so that the two phi chunks one stage needs are one
                // 96-row B operand
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
                const int q = (item / NG) % 8;
                const int ch = item / (NG * 8);
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
                *reinterpret_cast<uint4*>(chunk + nh * 128 + ((q ^ (nh & 7)) * 16)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(chunk + nl * 128 + ((q ^ (nl & 7)) * 16)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
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
        // The whole warp walks the loop; lane 0 waits and issues.
        const uint64_t pol = ptx::policy_evict_normal();
        const int first = ntl * (nch / 2) < STAGES ? ntl * (nch / 2) : STAGES;   // issued at set-up
        int stage = 0, n = 0;
        uint32_t round = 0;
        for (int j = cid; j < p.ntiles; j += ncl) {
            const int t0 = j * TILE_M;
            for (int st = 0; st < nch / 2; ++st, ++n) {
                if (n < first) {
                    if (++stage == STAGES) { stage = 0; ++round; }
                    continue;
                }
                const int pr = st / cpd, sub = st % cpd;       // stream pair, chunk of the slice
                const int xd = (sub * C + static_cast<int>(c)) * KW;   // chunks interleaved over the cluster
                bool ok = true;
                if (lane == 0) ok = wait_bar<false>(bar(BAR_EMPTY + stage), (round & 1) ^ 1, abort_flag);
                if (!__shfl_sync(FULL, ok, 0)) goto done;
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(bar(BAR_FULL + stage), STAGE_BYTES);
                    ptx::tma_load_3d(sbase + L.stages + stage * STAGE_BYTES, &tmap_x, xd, t0, 2 * pr,
                                     bar(BAR_FULL + stage), pol);
                }
                __syncwarp();
                if (++stage == STAGES) { stage = 0; ++round; }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer -----
        const uint64_t desc_stage0 = ptx::sw128_kmajor_desc(sbase + L.stages);
        const uint64_t desc_phi0 = ptx::sw128_kmajor_desc(sbase + L.phi);
        if (p.x_in == nullptr) {
            // No mix (the gates alone): lane 0 walks the loop by itself, every
            // instruction in it being a single thread's, and the other lanes
            // wait at the kernel's final barrier.  Its MMAs then issue sooner:
            // the gates-only forward 0.388 -> 0.331 ms at T = 32768.  With the
            // mix the warp-wide loop below is kept: there its slower issue is
            // what keeps the projection from running ahead of the mix's L2
            // re-reads (this loop: 0.439 -> 0.555 ms, and 0.52-0.54 ms with two
            // or three H_pre buffers).
            if (lane == 0) {
                int stage = 0;
                uint32_t round = 0;
                int it = 0;
                for (int j = cid; j < p.ntiles; j += ncl, ++it) {
                    const int tb = it & 1;
                    const uint32_t use = static_cast<uint32_t>(it >> 1);
                    if (!wait_bar<false>(bar(BAR_ACC_EMPTY + tb), (use & 1) ^ 1, abort_flag)) goto done;
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + tb * 128;
                    for (int st = 0; st < nch / 2; ++st) {
                        if (!wait_bar<false>(bar(BAR_FULL + stage), round & 1, abort_flag)) goto done;
                        ptx::tc_fence_after();
                        const uint64_t da = ptx::desc_add(desc_stage0, stage * STAGE_BYTES);
                        const uint64_t db = ptx::desc_add(desc_phi0, st * 2 * PHI_CHUNK_BYTES);
#pragma unroll
                        for (int kk = 0; kk < KW / 16; ++kk) {
                            const uint64_t dak = ptx::desc_add(da, kk * 32);
                            const uint32_t acc = (st | kk) != 0;
                            ptx::tc_mma_f16(d_tmem, dak, ptx::desc_add(db, kk * 32), IDESC, acc);
                            ptx::tc_mma_f16(d_tmem + GRAM_COL, dak, dak, IDESC_GRAM, acc);
                        }
                        ptx::tc_commit(bar(BAR_EMPTY + stage));
                        if (++stage == STAGES) { stage = 0; ++round; }
                    }
                    ptx::tc_commit(bar(BAR_ACC_FULL + tb));
                }
            }
            goto done;
        }
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
            for (int st = 0; st < nch / 2; ++st) {
                if (lane == 0) ok = wait_bar<false>(bar(BAR_FULL + stage), round & 1, abort_flag);
                if (!__shfl_sync(FULL, ok, 0)) goto done;
                ptx::tc_fence_after();
                if (lane == 0) {
                    const uint64_t da = ptx::desc_add(desc_stage0, stage * STAGE_BYTES);
                    const uint64_t db = ptx::desc_add(desc_phi0, st * 2 * PHI_CHUNK_BYTES);
#pragma unroll
                    for (int kk = 0; kk < KW / 16; ++kk) {
                        const uint64_t dak = ptx::desc_add(da, kk * 32);
                        const uint32_t acc = (st | kk) != 0;
                        ptx::tc_mma_f16(d_tmem, dak, ptx::desc_add(db, kk * 32), IDESC, acc);
                        ptx::tc_mma_f16(d_tmem + GRAM_COL, dak, dak, IDESC_GRAM, acc);
                    }
                    ptx::tc_commit(bar(BAR_EMPTY + stage));
                }
                __syncwarp();
                if (++stage == STAGES) { stage = 0; ++round; }
            }
            if (lane == 0) ptx::tc_commit(bar(BAR_ACC_FULL + tb));
            __syncwarp();
        }
    } else if (warp < SK_WARP0) {
        // ------------------------------------------------- gates ----------
        // (1) TMEM -> this CTA's partial logits and sum of squares for every
        //     token row, pushed (st.async) to the CTA that reduces the token;
        // (2) this CTA's TPC tokens: sum the partials, H_pre (pushed to every
        //     CTA, it is all the mix waits for), and hand the projection to
        //     the Sinkhorn warp for the other gates and the outputs.
        // M = 128 accumulators: lane = row; rows 0..63 are the first stream of
        // each stage (streams 0, 2), rows 64..127 the second (1, 3).  Each
        // row is half of a token's partial record; both halves are pushed.
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
            // H_pre buffer it % NHP is free at every CTA (mix of tile it - NHP done)
            const int hs = it % NHP;
            if (it >= NHP)
                ok = ok && __all_sync(FULL, wait_bar<true>(bar(BAR_HFREE + hs), ((it / NHP) - 1) & 1, abort_flag));
            // the Sinkhorn warp is done with this parity's hand-off (tile it-2)
            if (it >= 2) ok = ok && __all_sync(FULL, wait_bar<false>(bar(BAR_SKEMPTY + tb), (use - 1) & 1, abort_flag));
            ok = ok && __all_sync(FULL, wait_bar<true>(bar(BAR_RECV), it & 1, abort_flag));
            if (ok) {
                for (int tt0 = (warp - GATE_WARP0) * 2; tt0 < TPC; tt0 += NGATE * 2) {
                    const int tt = tt0 + half;
                    const bool real = tt < TPC;
                    const int r = static_cast<int>(c) * TPC + (real ? tt : 0);
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
                    // the pre gates (same expression as in token_gates)
                    float hp[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) hp[i] = sigmoid_f(fmaf(gate_par[0], pj[i], gate_par[3 + i]));
                    if (real && hl < C)
                        ptx::st_async_v4(ptx::mapa(sbase + L.hpre + static_cast<uint32_t>((hs * TILE_M + r) * 16),
                                                   static_cast<uint32_t>(hl)),
                                         hp[0], hp[1], hp[2], hp[3],
                                         ptx::mapa(bar(BAR_HPRE + hs), static_cast<uint32_t>(hl)));
                    if (real && hl < SKF / 4) {
                        // hand-off record: proj[24], inv_rms (picked with constant
                        // indices so that pj stays in registers)
                        float4 o = make_float4(inv, 0.f, 0.f, 0.f);
#pragma unroll
                        for (int v = 0; v < NG / 4; ++v)
                            if (hl == v) o = make_float4(pj[4 * v], pj[4 * v + 1], pj[4 * v + 2], pj[4 * v + 3]);
                        reinterpret_cast<float4*>(smem + L.sk)[(tb * TPC + tt) * (SKF / 4) + hl] = o;
                    }
                }
            }
            // every gate warp is done with the records: arm the barrier for the
            // next tile's, then tell every sender the buffer is free (peers
            // refill it with st.async)
            ptx::fence_proxy_async_smem();
            if (ptx::named_bar_or(1, NGATE * 32, !ok)) break;
            if (warp == GATE_WARP0) {
                if (lane == 0) ptx::mbar_arrive(bar(BAR_SKFULL + tb));
                if (lane == 0 && it + 1 < ntl) ptx::mbar_arrive_expect_tx(bar(BAR_RECV), 2 * TILE_M * REC_TX);
                __syncwarp();
                // a credit: every record value read above already feeds this
                // warp's sums, so a relaxed arrive suffices (a cluster-scope
                // release would wait about a microsecond for the SM's
                // outstanding memory operations)
                if (lane < C) ptx::mbar_arrive_remote_relaxed(ptx::mapa(bar(BAR_RFREE), static_cast<uint32_t>(lane)));
            }
        }
    } else if (warp < MIX_WARP0) {
        // ----------------------------------------- Sinkhorn and outputs ---
        // The other gates of this CTA's reduced tokens (H_post, Sinkhorn for
        // H_res) and every per-token output, off the mix's critical path.
        // One warp per tile parity, so that a tile's Sinkhorn may take up to
        // two tile periods (it grows with the round count).  Eight lanes per
        // token; lane l8 writes outputs l8 and l8 + 8 of the 13 float4-sized
        // pieces: proj[0..5], inv_rms, H_pre, H_post, H_res[0..3].
        const int l8 = lane & 7;
        int it = 0;
        for (int j = cid; j < p.ntiles; j += ncl, ++it) {
            const int tb = it & 1;
            if (tb != warp - SK_WARP0) continue;
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
                float hp[4], hq[4] = {0.f, 0.f, 0.f, 0.f}, hr[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) hr[e] = 0.f;
                const bool side = p.H_res != nullptr;   // null: the critical path, no Sinkhorn
                if (side) token_gates(pj, gate_par, gate_par + 3, p.iters, hp, hq, hr);
                else token_pre_gates(pj, gate_par, gate_par + 3, hp);
                const int64_t t = t0 + static_cast<int>(c) * TPC + tt;
                if (real && t < p.T) {
#pragma unroll
                    for (int rep = 0; rep < 2; ++rep) {
                        const int k = l8 + 8 * rep;
                        if (!side && k >= 8) continue;
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
            if (lane == 0) ptx::mbar_arrive(bar(BAR_SKEMPTY + tb));
        }
    } else {
        // --------------------------------------------------- mix ----------
        // x_in = sum_i H_pre[i] x[i] over this CTA's D-slice; x read again
        // (from L2 when the tile's first read is recent enough).
        const int mtid = tid - MIX_WARP0 * 32;          // 0..255
        int it = 0;
        for (int j = cid; j < p.ntiles; j += ncl, ++it) {
            const int64_t t0 = static_cast<int64_t>(j) * TILE_M;
            const int hs = it % NHP;
            const bool ok = __all_sync(FULL, wait_bar<true>(bar(BAR_HPRE + hs), (it / NHP) & 1, abort_flag));
            const float4* hb = reinterpret_cast<const float4*>(smem + L.hpre) + hs * TILE_M;
            const int qpt = Dc / 8;
            // no x_in buffer: the gates alone (recompute of the saved state)
            const int items = (ok && p.x_in != nullptr) ? TILE_M * qpt : 0;
            // item idx = (row r, piece q) with idx = r qpt + q; each step moves a
            // thread's item by NMIX * 32, so r, q and the item's offsets into x
            // and x_in advance by fixed amounts with a carry (no division or
            // multiply per item)
            const int dr = (NMIX * 32) / qpt, dq = (NMIX * 32) - dr * qpt;
            const int rlim = p.T - t0 < TILE_M ? static_cast<int>(p.T - t0) : TILE_M;   // rows in the batch
            int r_at = mtid / qpt, q_at = mtid - r_at * qpt;
            int64_t xo_at = (t0 + r_at) * K + static_cast<int64_t>(c) * Dc + q_at * 8;
            int64_t io_at = (t0 + r_at) * D + static_cast<int64_t>(c) * Dc + q_at * 8;
            const int64_t xstep = dr * K + dq * 8, xcarry = K - qpt * 8;
            const int64_t istep = static_cast<int64_t>(dr) * D + dq * 8, icarry = D - qpt * 8;
            for (int base = 0; base < items; base += NMIX * 32 * MIX_UNROLL) {
                uint4 xv[MIX_UNROLL][4];
                int64_t io[MIX_UNROLL];
                int rr[MIX_UNROLL];
#pragma unroll
                for (int m = 0; m < MIX_UNROLL; ++m) {
                    rr[m] = r_at < rlim ? r_at : -1;
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
                        const __nv_bfloat16* src = p.x + xo;
#pragma unroll
                        for (int i = 0; i < 4; ++i) xv[m][i] = ld16_stream(src + static_cast<int64_t>(i) * D);
                    }
                }
#pragma unroll
                for (int m = 0; m < MIX_UNROLL; ++m) {
                    if (rr[m] >= 0)
                        st16_stream(p.x_in + io[m], mix4_bf16(xv[m][0], xv[m][1], xv[m][2], xv[m][3], hb[rr[m]]));
                }
            }
            // every mix thread is done with this tile's H_pre buffer: arm it
            // for tile it + NHP, then free it at every reducer (which refills
            // it with st.async)
            ptx::fence_proxy_async_smem();
            if (ptx::named_bar_or(3, NMIX * 32, !ok)) break;
            if (warp == MIX_WARP0) {
                if (lane == 0 && it + NHP < ntl) ptx::mbar_arrive_expect_tx(bar(BAR_HPRE + hs), TILE_M * 16);
                __syncwarp();
                // a credit: the H_pre values read from the buffer were used by
                // every mix thread before the named barrier above
                if (lane < C) ptx::mbar_arrive_remote_relaxed(ptx::mapa(bar(BAR_HFREE + hs), static_cast<uint32_t>(lane)));
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

size_t smem_bytes(int nch, int C) { return Layout::make(nch, TILE_M / C).total + 1024; }

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
                                 static_cast<int>(smem_bytes(MAX_NCH, C))) != cudaSuccess ||
            (C > 8 && cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)) {
            cache[dev] = 0;
            return;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(C * 64);
        cfg.blockDim = dim3(NTHREADS);
        cfg.dynamicSmemBytes = smem_bytes(MAX_NCH, C);
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
    // T < 64 is one partial tile: TMA fills the rows past T with zeros
    if (T < 1 || D > (int64_t(1) << 20)) return false;
    if (4 * D * T >= (int64_t(1) << 46)) return false;
    const int C = tc::cluster_for(D);
    if (C == 0 || tc::encode_fn() == nullptr) return false;
    const int nch = static_cast<int>(4 * D / C / tc::KW);
    return tc::max_clusters_for(C, tc::smem_bytes(nch, C)) > 0;
}

cudaError_t launch_pre_tc(const void* x, const float* phi, const float* b, const float* alpha,
                          int64_t T, int64_t D, int iters, float eps, void* x_in, float* H_pre,
                          float* H_post, float* H_res, float* proj, float* inv_rms,
                          cudaStream_t s) {
    // a few tokens: the cluster split-K kernel without the tensor-core ring
    if (pre_small_supports(T, D))
        return launch_pre_small(x, phi, b, alpha, T, D, iters, eps, x_in, H_pre, H_post, H_res, proj, inv_rms,
                                g_force_timeout_pre.load(), s);
    const int C = tc::cluster_for(D);
    auto encode = tc::encode_fn();
    if (C == 0 || encode == nullptr) return cudaErrorNotSupported;
    const int64_t K = 4 * D;
    // x as (d, token, stream): a box is 64 columns x 64 tokens x 2 streams,
    // laid out in shared memory as [stream][token][64 columns]
    CUtensorMap tm;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T), 4};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K * 2), static_cast<cuuint64_t>(D * 2)};
    const cuuint32_t box[3] = {tc::KW, tc::TILE_M, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, estr,
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
    prm.force_timeout = g_force_timeout_pre.load();
    prm.x_in = static_cast<__nv_bfloat16*>(x_in);
    prm.H_pre = H_pre;
    prm.H_post = H_post;
    prm.H_res = H_res;
    prm.proj = proj;
    prm.inv_rms = inv_rms;
    const size_t smem = tc::smem_bytes(prm.nch, C);
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
