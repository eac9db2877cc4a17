// kernels_fwd.cu -- CUDA-core forward kernels of the mHC layer (sm_103a).
//
//   pre_proj_gates_kernel : RMS statistic + x . phi projection + gates/Sinkhorn
//                           for a tile of 64 tokens (fp32 FMA on CUDA cores).
//   pre_mix_kernel        : x_in = sum_i H_pre[i] x[i]            (streaming)
//   post_kernel           : x_next[i] = sum_j H_res[i,j] x[j] + H_post[i] y
//
// Layer definition: "openPangu 2.0 -- architecture, training and Ascend
// systems" notes, section 5.3.  The float32 workload always runs here; bf16
// shapes the tensor-core pre kernel does not cover run here too.
#include "launch.h"
#include "mhc_common.cuh"

namespace mhc {
namespace {

constexpr int PT_TOK = 64;       // tokens per CTA (two per lane)
constexpr int PT_KC = 64;        // K elements per pipeline stage
constexpr int PT_THREADS = 128;  // four warps split each stage's K range

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    const int n = valid ? 16 : 0;  // 0 source bytes = zero fill
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

template <typename TA>
struct ProjSmem {
    static constexpr int V = 16 / sizeof(TA);            // elements per 16 B
    static constexpr int PITCH = PT_KC + V;              // padded token row
    static constexpr int X_BYTES = 2 * PT_TOK * PITCH * (int)sizeof(TA);
    static constexpr int P_BYTES = 2 * PT_KC * NG * 4;
    static constexpr int RED_BYTES = 4 * PT_TOK * (NG + 1) * 4;
    static constexpr int BYTES = (X_BYTES + P_BYTES) > RED_BYTES ? (X_BYTES + P_BYTES) : RED_BYTES;
};

template <typename TA>
__global__ void __launch_bounds__(PT_THREADS)
pre_proj_gates_kernel(const TA* __restrict__ x, const float* __restrict__ phi,
                      const float* __restrict__ b, const float* __restrict__ alpha, int64_t T,
                      int64_t D, int iters, float eps, float* __restrict__ H_pre,
                      float* __restrict__ H_post, float* __restrict__ H_res,
                      float* __restrict__ proj_out, float* __restrict__ inv_rms_out) {
    using S = ProjSmem<TA>;
    constexpr int V = S::V;
    constexpr int PITCH = S::PITCH;
    __shared__ __align__(16) unsigned char smem[S::BYTES];
    TA* xs = reinterpret_cast<TA*>(smem);                                  // [2][PT_TOK][PITCH]
    float* ps = reinterpret_cast<float*>(smem + S::X_BYTES);              // [2][PT_KC][NG]
    float* red = reinterpret_cast<float*>(smem);                          // [4][PT_TOK][NG+1]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t K = 4 * D;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * PT_TOK;
    const int nchunks = static_cast<int>((K + PT_KC - 1) / PT_KC);

    auto load_stage = [&](int c, int buf) {
        const int64_t k0 = static_cast<int64_t>(c) * PT_KC;
        constexpr int CPR = PT_KC / V;  // 16-byte pieces per token row
        for (int q = tid; q < PT_TOK * CPR; q += PT_THREADS) {
            const int r = q / CPR, cc = q % CPR;
            const int64_t t = t0 + r, k = k0 + cc * V;
            const bool ok = (t < T) && (k < K);
            cp_async16(xs + (buf * PT_TOK + r) * PITCH + cc * V, ok ? x + t * K + k : x, ok);
        }
        for (int q = tid; q < PT_KC * (NG / 4); q += PT_THREADS) {
            const int r = q / (NG / 4), cc = q % (NG / 4);
            const int64_t k = k0 + r;
            const bool ok = k < K;
            cp_async16(ps + (buf * PT_KC + r) * NG + cc * 4, ok ? phi + k * NG + cc * 4 : phi, ok);
        }
        cp_async_commit();
    };

    float acc_a[NG], acc_b[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) acc_a[g] = acc_b[g] = 0.f;
    float ss_a = 0.f, ss_b = 0.f;

    load_stage(0, 0);
    for (int c = 0; c < nchunks; ++c) {
        const int buf = c & 1;
        if (c + 1 < nchunks) {
            load_stage(c + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        // warp w owns K elements [16w, 16w+16) of this stage; lane owns
        // tokens `lane` and `lane + 32` of the tile.
        float fa[16], fb[16];
        {
            const TA* ra = xs + (buf * PT_TOK + lane) * PITCH + warp * 16;
            const TA* rb = xs + (buf * PT_TOK + lane + 32) * PITCH + warp * 16;
#pragma unroll
            for (int v = 0; v < 16 / V; ++v) {
                float tmp[V];
                Vec<TA>::unpack(*reinterpret_cast<const uint4*>(ra + v * V), tmp);
#pragma unroll
                for (int e = 0; e < V; ++e) fa[v * V + e] = tmp[e];
                Vec<TA>::unpack(*reinterpret_cast<const uint4*>(rb + v * V), tmp);
#pragma unroll
                for (int e = 0; e < V; ++e) fb[v * V + e] = tmp[e];
            }
        }
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            const float4* prow = reinterpret_cast<const float4*>(ps + (buf * PT_KC + warp * 16 + kk) * NG);
            float ph[NG];
#pragma unroll
            for (int v = 0; v < NG / 4; ++v) {
                const float4 p = prow[v];
                ph[4 * v] = p.x; ph[4 * v + 1] = p.y; ph[4 * v + 2] = p.z; ph[4 * v + 3] = p.w;
            }
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                acc_a[g] = fmaf(fa[kk], ph[g], acc_a[g]);
                acc_b[g] = fmaf(fb[kk], ph[g], acc_b[g]);
            }
            ss_a = fmaf(fa[kk], fa[kk], ss_a);
            ss_b = fmaf(fb[kk], fb[kk], ss_b);
        }
        __syncthreads();
    }

    // cross-warp reduction of the four K quarters (staging buffers reused)
    {
        float* ra = red + (warp * PT_TOK + lane) * (NG + 1);
        float* rb = red + (warp * PT_TOK + lane + 32) * (NG + 1);
#pragma unroll
        for (int g = 0; g < NG; ++g) { ra[g] = acc_a[g]; rb[g] = acc_b[g]; }
        ra[NG] = ss_a;
        rb[NG] = ss_b;
    }
    __syncthreads();
    if (tid < PT_TOK) {
        const int64_t t = t0 + tid;
        if (t < T) {
            float z[NG + 1];
#pragma unroll
            for (int g = 0; g <= NG; ++g) {
                z[g] = (red[(0 * PT_TOK + tid) * (NG + 1) + g] + red[(1 * PT_TOK + tid) * (NG + 1) + g]) +
                       (red[(2 * PT_TOK + tid) * (NG + 1) + g] + red[(3 * PT_TOK + tid) * (NG + 1) + g]);
            }
            const float inv = 1.0f / sqrtf(z[NG] / static_cast<float>(K) + eps);
            float proj[NG];
#pragma unroll
            for (int g = 0; g < NG; ++g) proj[g] = z[g] * inv;
            float4* po = reinterpret_cast<float4*>(proj_out + t * NG);
#pragma unroll
            for (int v = 0; v < NG / 4; ++v)
                po[v] = make_float4(proj[4 * v], proj[4 * v + 1], proj[4 * v + 2], proj[4 * v + 3]);
            inv_rms_out[t] = inv;
            if (H_res == nullptr) {
                // the critical path: H_pre only, no Sinkhorn
                float hp[4];
                token_pre_gates(proj, alpha, b, hp);
                reinterpret_cast<float4*>(H_pre)[t] = make_float4(hp[0], hp[1], hp[2], hp[3]);
            } else {
                float hp[4], hq[4], hr[16];
                token_gates(proj, alpha, b, iters, hp, hq, hr);
                reinterpret_cast<float4*>(H_pre)[t] = make_float4(hp[0], hp[1], hp[2], hp[3]);
                reinterpret_cast<float4*>(H_post)[t] = make_float4(hq[0], hq[1], hq[2], hq[3]);
                float4* hro = reinterpret_cast<float4*>(H_res + t * 16);
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    hro[v] = make_float4(hr[4 * v], hr[4 * v + 1], hr[4 * v + 2], hr[4 * v + 3]);
            }
        }
    }
}

template <typename TA>
__global__ void __launch_bounds__(256)
pre_mix_kernel(const TA* __restrict__ x, const float* __restrict__ H_pre, int64_t T, int64_t D,
               TA* __restrict__ x_in) {
    constexpr int V = Vec<TA>::N;
    const int64_t QD = D / V;
    const int64_t total = T * QD;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = idx / QD, q = idx - t * QD;
        const float4 h = reinterpret_cast<const float4*>(H_pre)[t];
        const TA* xp = x + t * 4 * D + q * V;
        float f0[V], f1[V], f2[V], f3[V], o[V];
        Vec<TA>::unpack(ld16_stream(xp), f0);
        Vec<TA>::unpack(ld16_stream(xp + D), f1);
        Vec<TA>::unpack(ld16_stream(xp + 2 * D), f2);
        Vec<TA>::unpack(ld16_stream(xp + 3 * D), f3);
#pragma unroll
        for (int e = 0; e < V; ++e) o[e] = fmaf(h.w, f3[e], fmaf(h.z, f2[e], fmaf(h.y, f1[e], h.x * f0[e])));
        st16_stream(x_in + t * D + q * V, Vec<TA>::pack(o));
    }
}

template <typename TA>
__global__ void __launch_bounds__(256)
post_kernel(const TA* __restrict__ x, const TA* __restrict__ y, const float* __restrict__ H_post,
            const float* __restrict__ H_res, int64_t T, int64_t D, TA* __restrict__ x_next) {
    constexpr int V = Vec<TA>::N;
    const int64_t QD = D / V;
    const int64_t total = T * QD;
    for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
         idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = idx / QD, q = idx - t * QD;
        const float4 hp = reinterpret_cast<const float4*>(H_post)[t];
        const float4* hr4 = reinterpret_cast<const float4*>(H_res + t * 16);
        const float4 r0 = hr4[0], r1 = hr4[1], r2 = hr4[2], r3 = hr4[3];
        const float H[4][4] = {{r0.x, r0.y, r0.z, r0.w}, {r1.x, r1.y, r1.z, r1.w},
                               {r2.x, r2.y, r2.z, r2.w}, {r3.x, r3.y, r3.z, r3.w}};
        const float Hp[4] = {hp.x, hp.y, hp.z, hp.w};
        const TA* xp = x + t * 4 * D + q * V;
        float f[4][V], fy[V];
#pragma unroll
        for (int j = 0; j < 4; ++j) Vec<TA>::unpack(ld16_stream(xp + j * D), f[j]);
        Vec<TA>::unpack(ld16_stream(y + t * D + q * V), fy);
        TA* op = x_next + t * 4 * D + q * V;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float o[V];
#pragma unroll
            for (int e = 0; e < V; ++e)
                o[e] = fmaf(Hp[i], fy[e],
                            fmaf(H[i][3], f[3][e], fmaf(H[i][2], f[2][e], fmaf(H[i][1], f[1][e], H[i][0] * f[0][e]))));
            st16_stream(op + i * D, Vec<TA>::pack(o));
        }
    }
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

int64_t stream_grid(int64_t total, int threads) {
    const int64_t need = (total + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
    return need < cap ? need : cap;
}

}  // namespace

cudaError_t launch_pre_cc(bool bf16, const void* x, const float* phi, const float* b,
                          const float* alpha, int64_t T, int64_t D, int iters, float eps,
                          void* x_in, float* H_pre, float* H_post, float* H_res, float* proj,
                          float* inv_rms, cudaStream_t s) {
    const dim3 g1(static_cast<unsigned>((T + PT_TOK - 1) / PT_TOK));
    const int vec = bf16 ? 8 : 4;
    const dim3 g2(static_cast<unsigned>(stream_grid(T * (D / vec), 256)));
    if (bf16) {
        pre_proj_gates_kernel<__nv_bfloat16><<<g1, PT_THREADS, 0, s>>>(
            static_cast<const __nv_bfloat16*>(x), phi, b, alpha, T, D, iters, eps, H_pre, H_post,
            H_res, proj, inv_rms);
        if (x_in != nullptr)
            pre_mix_kernel<__nv_bfloat16><<<g2, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), H_pre, T,
                                                             D, static_cast<__nv_bfloat16*>(x_in));
    } else {
        pre_proj_gates_kernel<float><<<g1, PT_THREADS, 0, s>>>(static_cast<const float*>(x), phi, b, alpha,
                                                               T, D, iters, eps, H_pre, H_post, H_res,
                                                               proj, inv_rms);
        if (x_in != nullptr)
            pre_mix_kernel<float><<<g2, 256, 0, s>>>(static_cast<const float*>(x), H_pre, T, D,
                                                     static_cast<float*>(x_in));
    }
    return cudaGetLastError();
}

// H_post and H_res of each token from its saved projection (thread per
// token): the side of the inference critical-path split.
__global__ void __launch_bounds__(128)
post_res_gates_kernel(const float* __restrict__ proj, const float* __restrict__ b,
                      const float* __restrict__ alpha, int64_t T, int iters, float* __restrict__ H_post,
                      float* __restrict__ H_res) {
    __shared__ float par[3 + NG];
    if (threadIdx.x < 3) par[threadIdx.x] = alpha[threadIdx.x];
    if (threadIdx.x < NG) par[3 + threadIdx.x] = b[threadIdx.x];
    __syncthreads();
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= T) return;
    float pj[NG];
#pragma unroll
    for (int v = 0; v < NG / 4; ++v) {
        const float4 a = reinterpret_cast<const float4*>(proj + t * NG)[v];
        pj[4 * v] = a.x; pj[4 * v + 1] = a.y; pj[4 * v + 2] = a.z; pj[4 * v + 3] = a.w;
    }
    float hq[4], hr[16];
    token_post_res_gates(pj, par, par + 3, iters, hq, hr);
    reinterpret_cast<float4*>(H_post)[t] = make_float4(hq[0], hq[1], hq[2], hq[3]);
    float4* hro = reinterpret_cast<float4*>(H_res + t * 16);
#pragma unroll
    for (int v = 0; v < 4; ++v) hro[v] = make_float4(hr[4 * v], hr[4 * v + 1], hr[4 * v + 2], hr[4 * v + 3]);
}

cudaError_t launch_post_res_gates(const float* proj, const float* b, const float* alpha, int64_t T, int iters,
                                  float* H_post, float* H_res, cudaStream_t s) {
    post_res_gates_kernel<<<static_cast<unsigned>((T + 127) / 128), 128, 0, s>>>(proj, b, alpha, T, iters,
                                                                               H_post, H_res);
    return cudaGetLastError();
}

cudaError_t launch_post(bool bf16, const void* x, const void* y, const float* H_post,
                        const float* H_res, int64_t T, int64_t D, void* x_next, cudaStream_t s) {
    const int vec = bf16 ? 8 : 4;
    const dim3 g(static_cast<unsigned>(stream_grid(T * (D / vec), 256)));
    if (bf16)
        post_kernel<__nv_bfloat16><<<g, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x),
                                                     static_cast<const __nv_bfloat16*>(y), H_post, H_res,
                                                     T, D, static_cast<__nv_bfloat16*>(x_next));
    else
        post_kernel<float><<<g, 256, 0, s>>>(static_cast<const float*>(x), static_cast<const float*>(y),
                                             H_post, H_res, T, D, static_cast<float*>(x_next));
    return cudaGetLastError();
}

}  // namespace mhc
