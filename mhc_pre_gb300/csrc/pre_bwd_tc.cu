// pre_bwd_tc.cu -- tensor-core main step of the pre backward (bf16, n = 4).
//
// Given the per-token records of the pre backward (u = inv_rms * alpha_grp *
// dlogits, H_pre, the RMSNorm coefficient of x), this kernel does, for a
// K-slice of 256 columns and a block of tokens:
//   dx[t, k] += H_pre[t, i(k)] g_in[t, d(k)] + (phi u_t)[k] + coef_t x[t, k]
//   dphi_part[k, g] = sum_t x[t, k] u[t, g]
// Both contractions run on tcgen05 with fp32 accumulators in TMEM, for tiles
// of 128 tokens and chunks of 64 columns:
//   * D1[t, k] = U[t, 0:32] . A_phi[k, 0:32]^T  (M = 128 tokens, N = 64,
//     K = 32: the 24 logits padded by zero columns of A_phi; bf16 u and phi --
//     a small part of dx, far inside the bf16 dx tolerance);
//   * D2T[n, k] += U2T[n, t] . X[t, k]          (M = 128 rows of which 48 are
//     the hi and lo bf16 halves of u, N = 64 columns, K = 128 tokens).
// U2T (48 rows x 128 tokens) is one shared-memory block read K-major by the
// second MMA and MN-major (tokens contiguous) as the A operand of the first;
// X comes straight from the TMA stage, read MN-major.  x, dx and g_in arrive
// by TMA; each epilogue thread owns one token (its TMEM lane), reads its row
// of the three tiles with 16-byte swizzled loads and writes dx with 16-byte
// global stores.
//
// Derivation: openPangu 2.0 notes, section 5.3 (layer definition); recompute
// of the gates from the saved projection as in the Ascend mHC Triton operator
// article's recompute paragraph.
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
__device__ unsigned g_bwd_tc_error;

cudaError_t read_and_clear_bwd_tc_error(unsigned* word) {
    cudaError_t e = cudaMemcpyFromSymbol(word, g_bwd_tc_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_bwd_tc_error, &zero, sizeof(unsigned));
}

namespace bwdtc {

constexpr int KSLICE = 256;                 // K columns per CTA (inside one stream)
constexpr int KC = 64;                      // columns per chunk (MMA N)
constexpr int NCH = KSLICE / KC;            // 4 chunks
constexpr int TT = 128;                     // tokens per tile (MMA M)
constexpr int STAGES = 3;
constexpr int ARR_BYTES = TT * 128;         // one [128 tokens x 64 columns] bf16 box, 16 KB
constexpr int STAGE_BYTES = 3 * ARR_BYTES;  // x, dx, g_in
constexpr int APHI_CHUNK = KC * 128;        // 64 rows x 128 B
constexpr int U2_ATOM = 48 * 128;           // 48 rows x 64 tokens
constexpr int SC_OFF = 12288;               // per token H_pre[4], coef, pad (after U2T)
constexpr int UBUF_BYTES = 16384;           // U2T + scalars (+ the MMA's reads past row 48)
constexpr int NTHREADS = 384;               // 12 warps
constexpr int PREP_WARP0 = 2, NPREP = 2;
constexpr int EPI_WARP0 = 4, NEPI = 8;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t D1_COL = 0;              // two 64-column buffers
constexpr uint32_t D2_COL = 128;            // NCH x 64 columns
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;

enum : int {
    BAR_FULL = 0,
    BAR_EMPTY = BAR_FULL + STAGES,
    BAR_UFULL = BAR_EMPTY + STAGES,
    BAR_UEMPTY = BAR_UFULL + 2,
    BAR_D1FULL = BAR_UEMPTY + 2,
    BAR_D1EMPTY = BAR_D1FULL + 2,
    BAR_D2DONE = BAR_D1EMPTY + 2,
    NBARS = BAR_D2DONE + 1
};

// U buffers come first so that the first MMA's reads of rows 48..127 of the
// second U2T atom (whose results are never used) stay inside shared memory.
struct Layout {
    static constexpr uint32_t UBUF = 0;
    static constexpr uint32_t APHI = UBUF + 2 * UBUF_BYTES;
    static constexpr uint32_t STAGE = APHI + NCH * APHI_CHUNK;
    static constexpr uint32_t BARS = STAGE + STAGES * STAGE_BYTES;
    static constexpr uint32_t MISC = BARS + NBARS * 8;
    static constexpr uint32_t TOTAL = MISC + 32;
};
constexpr size_t SMEM_BYTES = Layout::TOTAL + 1024;

struct Params {
    const float* phi;
    const float* rec;
    __nv_bfloat16* dx;
    float* part;
    int64_t T;
    int64_t D;
    int64_t tb;            // tokens per block, a multiple of TT
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (*abort_flag) return false;
            if (ptx::globaltimer() - t0 > WAIT_LIMIT_NS) {
                atomicOr(&g_bwd_tc_error, 1u);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

using ptx::sw128_mnmajor_desc;
using ptx::sw128_off;

__global__ void __launch_bounds__(NTHREADS, 1)
pre_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dx,
                  const __grid_constant__ CUtensorMap tm_g, const Params p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    auto bar = [&](int i) { return sbase + Layout::BARS + 8u * static_cast<uint32_t>(i); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Layout::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Layout::MISC + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr unsigned FULL = 0xffffffffu;
    const int64_t D = p.D;
    const int64_t kbase = static_cast<int64_t>(blockIdx.x) * KSLICE;
    const int si = static_cast<int>(kbase / D);
    const int64_t dbase = kbase - si * D;
    const int64_t K = 4 * D;
    const int64_t tbeg = static_cast<int64_t>(blockIdx.y) * p.tb;
    const int64_t tend = tbeg + p.tb < p.T ? tbeg + p.tb : p.T;
    const int ntiles = tend > tbeg ? static_cast<int>((tend - tbeg + TT - 1) / TT) : 0;

    // ---- set-up ----------------------------------------------------------
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar(BAR_FULL + s), 1);
            ptx::mbar_init(bar(BAR_EMPTY + s), 1 + NEPI * 32);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar(BAR_UFULL + b), NPREP * 32);
            ptx::mbar_init(bar(BAR_UEMPTY + b), 1 + NEPI * 32);
            ptx::mbar_init(bar(BAR_D1FULL + b), 1);
            ptx::mbar_init(bar(BAR_D1EMPTY + b), NEPI * 32);
        }
        ptx::mbar_init(bar(BAR_D2DONE), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tm_x);
        ptx::prefetch_tmap(&tm_dx);
        ptx::prefetch_tmap(&tm_g);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    // A_phi: row k of the slice (chunk k / 64), columns g < 24 = bf16(phi[k, g]),
    // columns 24..31 zero (the MMAs read K = 0..31 only).
    for (int item = tid; item < KSLICE * 4; item += NTHREADS) {
        const int kl = item >> 2, q = item & 3;
        const int ch = kl / KC, r = kl % KC;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int g0 = q * 8 + 2 * e;
            const float v0 = g0 < NG ? p.phi[(kbase + kl) * NG + g0] : 0.f;
            const float v1 = g0 + 1 < NG ? p.phi[(kbase + kl) * NG + g0 + 1] : 0.f;
            const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
            w[e] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(smem + Layout::APHI + ch * APHI_CHUNK + sw128_off(r, q * 8)) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ----
        // normal priority: evict-last lines outlive the kernel and crowd the
        // next kernel's working set out of L2
        const uint64_t pol = ptx::policy_evict_normal();
        int stage = 0;
        uint32_t round = 0;
        for (int j = 0; j < ntiles; ++j) {
            const int t0 = static_cast<int>(tbeg + static_cast<int64_t>(j) * TT);
            for (int c = 0; c < NCH; ++c) {
                bool ok = true;
                if (lane == 0) ok = wait_bar(bar(BAR_EMPTY + stage), (round & 1) ^ 1, abort_flag);
                if (!__shfl_sync(FULL, ok, 0)) goto done;
                if (lane == 0) {
                    const uint32_t st = sbase + Layout::STAGE + stage * STAGE_BYTES;
                    const uint32_t fb = bar(BAR_FULL + stage);
                    ptx::mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    ptx::tma_load_2d(st, &tm_x, static_cast<int>(kbase + c * KC), t0, fb, pol);
                    ptx::tma_load_2d(st + ARR_BYTES, &tm_dx, static_cast<int>(kbase + c * KC), t0, fb, pol);
                    ptx::tma_load_2d(st + 2 * ARR_BYTES, &tm_g, static_cast<int>(dbase + c * KC), t0, fb, pol);
                }
                __syncwarp();
                if (++stage == STAGES) { stage = 0; ++round; }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer -----
        constexpr uint32_t IDESC1 = ptx::idesc_bf16_f32(TT, KC) | (1u << 15);    // A (U) MN-major
        constexpr uint32_t IDESC2 = ptx::idesc_bf16_f32(128, KC) | (1u << 16);   // B (X) MN-major
        // descriptors built once; the loop only moves their start address
        const uint64_t desc_aphi0 = ptx::sw128_kmajor_desc(sbase + Layout::APHI);
        const uint64_t desc_x0 = sw128_mnmajor_desc(sbase + Layout::STAGE, ARR_BYTES, 1024);
        const uint64_t desc_u2mn0 = sw128_mnmajor_desc(sbase + Layout::UBUF, U2_ATOM, 1024);
        const uint64_t desc_u2k0 = ptx::sw128_kmajor_desc(sbase + Layout::UBUF);
        int stage = 0;
        uint32_t round = 0;
        int q = 0;
        for (int j = 0; j < ntiles; ++j) {
            const int ub = j & 1;
            bool ok = true;
            if (lane == 0) ok = wait_bar(bar(BAR_UFULL + ub), (j >> 1) & 1, abort_flag);
            if (!__shfl_sync(FULL, ok, 0)) goto done;
            for (int c = 0; c < NCH; ++c, ++q) {
                const int db = q & 1;
                if (lane == 0) ok = wait_bar(bar(BAR_D1EMPTY + db), ((q >> 1) & 1) ^ 1, abort_flag);
                if (!__shfl_sync(FULL, ok, 0)) goto done;
                if (lane == 0) ok = wait_bar(bar(BAR_FULL + stage), round & 1, abort_flag);
                if (!__shfl_sync(FULL, ok, 0)) goto done;
                ptx::tc_fence_after();
                if (lane == 0) {
                    const uint64_t aphi = ptx::desc_add(desc_aphi0, c * APHI_CHUNK);
                    const uint64_t xs = ptx::desc_add(desc_x0, stage * STAGE_BYTES);
                    const uint32_t u2o = ub * UBUF_BYTES;
                    // D1 = U . A_phi^T: A = U2T read MN-major (tokens contiguous,
                    // 64-token atoms U2_ATOM apart), K = 32 logit rows
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
                        ptx::tc_mma_f16(tmem + D1_COL + db * KC, ptx::desc_add(desc_u2mn0, u2o + kk * 2048),
                                        ptx::desc_add(aphi, kk * 32), IDESC1, kk != 0);
                    // D2T += U2T . X: A = U2T K-major (rows 0..47 real), B = x tile
                    // MN-major, K = 128 tokens
#pragma unroll
                    for (int kk = 0; kk < TT / 16; ++kk)
                        ptx::tc_mma_f16(tmem + D2_COL + c * KC,
                                        ptx::desc_add(desc_u2k0, u2o + (kk >> 2) * U2_ATOM + (kk & 3) * 32),
                                        ptx::desc_add(xs, kk * 2048), IDESC2, (j | kk) != 0);
                    ptx::tc_commit(bar(BAR_D1FULL + db));
                    ptx::tc_commit(bar(BAR_EMPTY + stage));
                    if (c == NCH - 1) ptx::tc_commit(bar(BAR_UEMPTY + ub));
                }
                __syncwarp();
                if (++stage == STAGES) { stage = 0; ++round; }
            }
        }
        if (lane == 0) ptx::tc_commit(bar(BAR_D2DONE));
        __syncwarp();
    } else if (warp < EPI_WARP0) {
        // --------------------------------------------- U preparation ------
        const int pt = tid - PREP_WARP0 * 32;          // tokens pt and pt + 64
        for (int j = 0; j < ntiles; ++j) {
            const int ub = j & 1;
            if (!__all_sync(FULL, wait_bar(bar(BAR_UEMPTY + ub), ((j >> 1) & 1) ^ 1, abort_flag))) goto done;
            unsigned char* ubuf = smem + Layout::UBUF + ub * UBUF_BYTES;
            float* sc = reinterpret_cast<float*>(ubuf + SC_OFF);
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                const int tl = pt + 64 * h;
                const int64_t t = tbeg + static_cast<int64_t>(j) * TT + tl;
                float u[NG], hp[4], cf = 0.f;
                if (t < tend) {
                    const float4* r4 = reinterpret_cast<const float4*>(p.rec + t * REC);
#pragma unroll
                    for (int v = 0; v < 6; ++v) {
                        const float4 a = r4[v];
                        u[4 * v] = a.x; u[4 * v + 1] = a.y; u[4 * v + 2] = a.z; u[4 * v + 3] = a.w;
                    }
                    const float4 hh = r4[6];
                    hp[0] = hh.x; hp[1] = hh.y; hp[2] = hh.z; hp[3] = hh.w;
                    cf = p.rec[t * REC + REC_COEF];
                } else {
#pragma unroll
                    for (int g = 0; g < NG; ++g) u[g] = 0.f;
                    hp[0] = hp[1] = hp[2] = hp[3] = 0.f;
                }
                // U2T column tl: rows g < 24 hi(u[g]), rows 24 + g lo(u[g])
                unsigned char* at = ubuf + (tl >> 6) * U2_ATOM;
                const int tc = tl & 63;
#pragma unroll
                for (int g = 0; g < NG; ++g) {
                    const __nv_bfloat16 hi = __float2bfloat16_rn(u[g]);
                    const __nv_bfloat16 lo = __float2bfloat16_rn(u[g] - __bfloat162float(hi));
                    *reinterpret_cast<__nv_bfloat16*>(at + sw128_off(g, tc)) = hi;
                    *reinterpret_cast<__nv_bfloat16*>(at + sw128_off(NG + g, tc)) = lo;
                }
                reinterpret_cast<float4*>(sc)[2 * tl] = make_float4(hp[0], hp[1], hp[2], hp[3]);
                sc[8 * tl + 4] = cf;
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(bar(BAR_UFULL + ub));
        }
    } else {
        // ------------------------------------------------- epilogue -------
        // One token per thread (TMEM lane); warps 4-7 take columns 0..31 of
        // each 64-column chunk, warps 8-11 columns 32..63.
        const int qd = warp & 3;
        const int half = (warp - EPI_WARP0) >> 2;
        const int tl = qd * 32 + lane;                 // token row of the tile
        int stage = 0;
        uint32_t round = 0;
        int q = 0;
        bool aborted = false;
        for (int j = 0; j < ntiles && !aborted; ++j) {
            const int ub = j & 1;
            const int64_t t = tbeg + static_cast<int64_t>(j) * TT + tl;
            if (!__all_sync(FULL, wait_bar(bar(BAR_UFULL + ub), (j >> 1) & 1, abort_flag))) { aborted = true; break; }
            const float* sc = reinterpret_cast<const float*>(smem + Layout::UBUF + ub * UBUF_BYTES + SC_OFF);
            const float hpre = sc[8 * tl + si], cf = sc[8 * tl + 4];
            for (int c = 0; c < NCH; ++c, ++q) {
                const int db = q & 1;
                if (!__all_sync(FULL, wait_bar(bar(BAR_D1FULL + db), (q >> 1) & 1, abort_flag)) ||
                    !__all_sync(FULL, wait_bar(bar(BAR_FULL + stage), round & 1, abort_flag))) {
                    aborted = true;
                    break;
                }
                ptx::tc_fence_after();
                uint32_t v[2][16];
                const uint32_t ta = tmem + (static_cast<uint32_t>(qd * 32) << 16) + D1_COL + db * KC + half * 32;
                ptx::tmem_ld16(ta, v[0]);
                ptx::tmem_ld16(ta + 16, v[1]);
                ptx::tmem_wait_ld();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(BAR_D1EMPTY + db));
                const unsigned char* st = smem + Layout::STAGE + stage * STAGE_BYTES;
                uint4 xs4[4], ds4[4], gs4[4];
#pragma unroll
                for (int cq = 0; cq < 4; ++cq) {
                    const uint32_t off = static_cast<uint32_t>(tl * 128 + (((half * 4 + cq) ^ (tl & 7)) << 4));
                    xs4[cq] = *reinterpret_cast<const uint4*>(st + off);
                    ds4[cq] = *reinterpret_cast<const uint4*>(st + ARR_BYTES + off);
                    gs4[cq] = *reinterpret_cast<const uint4*>(st + 2 * ARR_BYTES + off);
                }
                // the stage's next bytes come through the async proxy (TMA)
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive(bar(BAR_EMPTY + stage));
                if (t < tend) {
                    __nv_bfloat16* dst = p.dx + t * K + kbase + c * KC + half * 32;
#pragma unroll
                    for (int cq = 0; cq < 4; ++cq) {
                        float fx[8], fd[8], fg[8], o[8];
                        Vec<__nv_bfloat16>::unpack(xs4[cq], fx);
                        Vec<__nv_bfloat16>::unpack(ds4[cq], fd);
                        Vec<__nv_bfloat16>::unpack(gs4[cq], fg);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int col = cq * 8 + e;
                            o[e] = fd[e] + fmaf(hpre, fg[e], fmaf(cf, fx[e], __uint_as_float(v[col >> 4][col & 15])));
                        }
                        *reinterpret_cast<uint4*>(dst + cq * 8) = Vec<__nv_bfloat16>::pack(o);
                    }
                }
                if (++stage == STAGES) { stage = 0; ++round; }
            }
            if (aborted) break;
            ptx::mbar_arrive(bar(BAR_UEMPTY + ub));
        }
        // dphi partial of this block from D2T (rows g: hi, rows 24 + g: lo).
        // Rows 0..47 sit in lane quarters 0 and 1; they go through shared
        // memory (the stage buffers are free once every MMA is done) so that
        // each thread can then sum one column k.
        bool ok = !aborted && ntiles > 0 && __all_sync(FULL, wait_bar(bar(BAR_D2DONE), 0, abort_flag));
        float* d2s = reinterpret_cast<float*>(smem + Layout::STAGE);      // [NCH][48][KC]
        ptx::named_bar_sync(2, NEPI * 32);   // every epilogue thread is done with the stages
        if (ok && qd < 2) {
            ptx::tc_fence_after();
            const int row = qd * 32 + lane;
            for (int c = half * 2; c < half * 2 + 2; ++c) {
#pragma unroll
                for (int h16 = 0; h16 < KC / 16; ++h16) {
                    uint32_t v[16];
                    ptx::tmem_ld16(tmem + (static_cast<uint32_t>(qd * 32) << 16) + D2_COL + c * KC + h16 * 16, v);
                    ptx::tmem_wait_ld();
                    if (row < 48) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) d2s[(c * 48 + row) * KC + h16 * 16 + e] = __uint_as_float(v[e]);
                    }
                }
            }
        }
        const bool any_bad = ptx::named_bar_or(1, NEPI * 32, !ok && ntiles > 0);
        const int et = tid - EPI_WARP0 * 32;            // 0..255: one column of the slice
        float* out = p.part + (static_cast<int64_t>(blockIdx.y) * K + kbase + et) * NG;
        if (ntiles == 0) {
#pragma unroll
            for (int g = 0; g < NG; ++g) out[g] = 0.f;
        } else if (!any_bad) {
            const int c = et / KC, k = et % KC;
#pragma unroll
            for (int g = 0; g < NG; ++g)
                out[g] = d2s[(c * 48 + g) * KC + k] + d2s[(c * 48 + NG + g) * KC + k];
        }
    }
done:
    __syncthreads();
    if (*abort_flag) {
        const uint64_t t0 = ptx::globaltimer();
        while (ptx::globaltimer() - t0 < 20000ull) {
        }
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

bool set_smem_once() {
    static int ok = -1;
    static std::once_flag once;
    std::call_once(once, [] {
        ok = cudaFuncSetAttribute(pre_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(SMEM_BYTES)) == cudaSuccess;
    });
    return ok == 1;
}

bool encode_2d(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* tm, const void* base, int64_t inner,
               int64_t rows) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner * 2)};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(TT)};
    const cuuint32_t estr[2] = {1, 1};
    return encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace bwdtc

bool pre_bwd_tc_supports(int64_t T, int64_t D) {
    return T >= bwdtc::TT && D % bwdtc::KSLICE == 0 && 4 * D * T < (int64_t(1) << 46) &&
           tensor_map_encoder() != nullptr;
}

cudaError_t launch_pre_bwd_tc_main(const void* g_in, const void* x, const float* phi, const float* rec,
                                   int64_t T, int64_t D, int64_t nb, void* dx, float* part,
                                   cudaStream_t s) {
    auto encode = tensor_map_encoder();
    if (encode == nullptr || !bwdtc::set_smem_once()) return cudaErrorNotSupported;
    const int64_t K = 4 * D;
    CUtensorMap tx, tdx, tg;
    if (!bwdtc::encode_2d(encode, &tx, x, K, T) || !bwdtc::encode_2d(encode, &tdx, dx, K, T) ||
        !bwdtc::encode_2d(encode, &tg, g_in, D, T))
        return cudaErrorInvalidValue;
    bwdtc::Params prm;
    prm.phi = phi;
    prm.rec = rec;
    prm.dx = static_cast<__nv_bfloat16*>(dx);
    prm.part = part;
    prm.T = T;
    prm.D = D;
    // token blocks are whole tiles, so no tile's dx write-back touches a
    // token of another block; blocks past the end write zero partials
    const int64_t per = (T + nb - 1) / nb;
    prm.tb = (per + bwdtc::TT - 1) / bwdtc::TT * bwdtc::TT;
    const dim3 grid(static_cast<unsigned>(K / bwdtc::KSLICE), static_cast<unsigned>(nb));
    bwdtc::pre_bwd_tc_kernel<<<grid, bwdtc::NTHREADS, bwdtc::SMEM_BYTES, s>>>(tx, tdx, tg, prm);
    return cudaGetLastError();
}

}  // namespace mhc
