// Contribution decomposition of a GR read (analysis tool), CUDA cores, fp32 arithmetic.
//
// "【论文解读】 Qwen3.8 Flash Next", §二.6: GR never mixes branches, so the state a block reads
// is the initial state plus the writes of the blocks before it, and the read's output splits
// exactly into per-writer terms (eq auv). For reader v (state R, parameters γ, W_d, W_u) and
// writers u (outputs y^(u), write strengths s^(u)), per token:
//   coef_i[c]      = G_i[c] γ_i[c] / rms(R_i)          (the read's gate, gain and norm)
//   a_{u→v,i}[c]   = ¼ coef_i[c] s_i^(u) y^(u)[c],     a_{u→v} = Σ_i a_{u→v,i}
//   ‖a_{u→v}‖, ‖a_{u→v,i}‖ over the D channels,       π_uv = ‖a_{u→v}‖ / Σ_u' ‖a_{u'→v}‖
//   a_{0→v}[c]     = ¼ Σ_i coef_i[c] R0_i[c]          (the initial state's share)
//
// One kernel, persistent, TB tokens per CTA at a time (TB = 2 below rank 64, two CTAs per SM):
//   1. the read's gates, recomputed as the backward does (squared sums, z = ¼ W_d vec R̂,
//      h = SiLU(z), G = σ(W_u h)), into coef [TB][4D] fp32 in shared memory (the state rows are
//      read twice, the second time from L2, so that a row of D = 12288 still fits);
//   2. the writers in groups of kGroup: every thread owns 8-channel slots of one token, loads
//      the writers' 8 channels with 16-byte loads, and accumulates per writer Σ_c A² with
//      A = Σ_i s_i coef_i y, and Σ_c (coef_i y)² per branch (‖a_{u→v,i}‖ = |s_i|/4 of its root);
//      a warp reduce-scatter and a shared-memory sum over the token's warps finish the sums;
//   3. π from the norms this CTA wrote, and ‖a_{0→v}‖ when the initial state is given.
#include <math.h>

#include "gr_internal.h"
#include "gr_ptx.cuh"

namespace gr {
namespace {

constexpr int kGroup = 6;            // writers per group: 5 sums each, 30 of a warp's 32 lanes
constexpr int kSums = 5;             // Σ A², then Σ (coef_i y)² for the four branches

// σ(a) = 1/(1 + e^-a) with the fast exponential and division: a few ulp, far inside the fp32
// bounds of these paths; 0 and 1 at the ends (1/inf = 0).
__device__ __forceinline__ float sigm(float a) { return __fdividef(1.0f, 1.0f + __expf(-a)); }

// 256 threads; two CTAs per SM below rank 64 (each thread then has 128 registers), so that one
// CTA's gate recompute overlaps the other's writer pass.
template <int RM>
__host__ __device__ constexpr int dec_threads() { return 256; }

// Block sums of M per-thread values (NW warps); totals land in out[0..M).
template <int M, int NW>
__device__ __forceinline__ void block_sum(const float (&v)[M], float* red, float* out) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int k = 0; k < M; ++k) {
        float a = v[k];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0) red[warp * M + k] = a;
    }
    __syncthreads();
    for (int k = threadIdx.x; k < M; k += NW * 32) {
        float a = 0.f;
        for (int w = 0; w < NW; ++w) a += red[w * M + k];
        out[k] = a;
    }
    __syncthreads();
}

// Warp reduce-scatter of 32 values per lane: afterwards v[0] of lane j holds the warp's sum of
// value j (31 shuffles instead of 5 per value).
__device__ __forceinline__ void warp_reduce_scatter32(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int half = 16; half >= 1; half >>= 1) {
        const bool up = (lane & half) != 0;   // this lane keeps the upper half of the range
#pragma unroll
        for (int k = 0; k < half; ++k) {
            const float send = up ? v[k] : v[k + half];
            const float keep = up ? v[k + half] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, half);
        }
    }
}

__device__ __forceinline__ uint32_t word(const uint4& q, int j) {
    return j == 0 ? q.x : j == 1 ? q.y : j == 2 ? q.z : q.w;
}
__device__ __forceinline__ float comp(const float4& q, int j) {
    return j == 0 ? q.x : j == 1 ? q.y : j == 2 ? q.z : q.w;
}

// 8 consecutive channels of a row, kept in their stored form until used (4 registers for bf16);
// get(k) with a compile-time k gives channel k as fp32.
template <typename T> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
    uint4 q;
    __device__ __forceinline__ void load(const __nv_bfloat16* p) {
        q = __ldcs(reinterpret_cast<const uint4*>(p));   // streamed once
    }
    __device__ __forceinline__ void zero() { q = make_uint4(0u, 0u, 0u, 0u); }
    __device__ __forceinline__ float get(int k) const {
        const uint32_t w = word(q, k >> 1);
        return (k & 1) ? __uint_as_float(w & 0xffff0000u) : __uint_as_float(w << 16);
    }
};
template <> struct Raw8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float* p) {
        a = __ldcs(reinterpret_cast<const float4*>(p));
        b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    }
    __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ __forceinline__ float get(int k) const { return k < 4 ? comp(a, k) : comp(b, k - 4); }
};

// FULL: r == RM, so that every rank test is a compile-time constant.
template <typename T, int RM, int TB, bool FULL>
__global__ void __launch_bounds__(dec_threads<RM>(), RM > 32 ? 1 : 2)
decompose_kernel(int64_t N, int D, int r_arg, float eps, const T* __restrict__ R,
                 const float* __restrict__ gamma, const float* __restrict__ Wd,
                 const float* __restrict__ Wu, int U, const T* __restrict__ Y,
                 const float* __restrict__ S, const T* __restrict__ R0,
                 float* __restrict__ norm, float* __restrict__ bnorm, float* __restrict__ pi,
                 float* __restrict__ a0_norm) {
    constexpr int NT = dec_threads<RM>();
    constexpr int NW = NT / 32;
    constexpr int TPT = NT / TB;            // threads per token in the writer pass
    const int r = FULL ? RM : r_arg;
    constexpr int WPT = TPT / 32;           // warps per token
    extern __shared__ float smem[];
    const int K = kBranches * D;
    float* coef = smem;                                            // [TB][4D]
    float* red = coef + size_t(TB) * K;                            // [NW][max(32, TB·RM)]
    constexpr int RED = (TB * RM > 32 ? TB * RM : 32);
    float* tot = red + NW * RED;                                   // [TB·RM]
    float* hs = tot + TB * RM;                                     // [TB][RM]
    float* inv = hs + TB * RM;                                     // [TB][4]
    float* sS = inv + TB * kBranches;                              // [TB][kGroup][4]
    float* tsum = sS + TB * kGroup * kBranches;                    // [TB] Σ_u ‖a_{u→v}‖
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tt = tid / TPT, l = tid % TPT;
    const int nslot = D / 8;
    const int64_t ntiles = (N + TB - 1) / TB;

    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t t0 = tile * TB;
        const int nt = int(N - t0 < TB ? N - t0 : TB);
        __syncthreads();   // the previous tile is done with the shared arrays
        // 1a. squared sums (the state rows are read again in 1b, from L2)
        {
            float sq[TB * kBranches];
#pragma unroll
            for (int k = 0; k < TB * kBranches; ++k) sq[k] = 0.f;
#pragma unroll
            for (int t2 = 0; t2 < TB; ++t2)
#pragma unroll
                for (int i = 0; i < kBranches; ++i)
                    for (int c = tid; c < D; c += NT) {
                        const float f = t2 < nt ? to_f32(R[(t0 + t2) * K + i * D + c]) : 0.f;
                        sq[t2 * kBranches + i] = fmaf(f, f, sq[t2 * kBranches + i]);
                    }
            block_sum<TB * kBranches, NW>(sq, red, tot);
            if (tid < TB * kBranches) inv[tid] = rsqrtf(tot[tid] / float(D) + eps);
            if (tid < TB) tsum[tid] = 0.f;
            __syncthreads();
        }
        // 1b. z = ¼ W_d vec R̂, h = SiLU(z)
        {
            float az[TB * RM];
#pragma unroll
            for (int k = 0; k < TB * RM; ++k) az[k] = 0.f;
#pragma unroll 2
            for (int e = tid; e < K; e += NT) {
                const int i = e / D;
                const float ge = gamma[e];
                float wd[RM];
#pragma unroll
                for (int k = 0; k < RM; ++k) wd[k] = k < r ? Wd[size_t(k) * K + e] : 0.f;
#pragma unroll
                for (int t2 = 0; t2 < TB; ++t2) {
                    const float rv = t2 < nt ? to_f32(R[(t0 + t2) * K + e]) : 0.f;
                    const float rh = ge * rv * inv[t2 * kBranches + i];
#pragma unroll
                    for (int k = 0; k < RM; ++k)
                        az[t2 * RM + k] = fmaf(wd[k], rh, az[t2 * RM + k]);
                }
            }
            block_sum<TB * RM, NW>(az, red, tot);
            for (int q = tid; q < TB * RM; q += NT) {
                const float z = (q % RM) < r ? 0.25f * tot[q] : 0.f;
                hs[q] = z * sigm(z);
            }
            __syncthreads();
        }
        // 1c. coef = σ(W_u h) γ / rms (a row of W_u is r consecutive floats: 16-byte loads
        //     when r is a multiple of 4)
        const bool wu_vec = (r & 3) == 0;
#pragma unroll 2
        for (int e = tid; e < K; e += NT) {
            const int i = e / D;
            const float ge = gamma[e];
            float wu[RM];
            if (wu_vec) {
                const float4* row = reinterpret_cast<const float4*>(Wu + size_t(e) * r);
#pragma unroll
                for (int k = 0; k < RM; k += 4) {
                    const float4 q = k < r ? row[k / 4] : make_float4(0.f, 0.f, 0.f, 0.f);
                    wu[k] = q.x; wu[k + 1] = q.y; wu[k + 2] = q.z; wu[k + 3] = q.w;
                }
            } else {
#pragma unroll
                for (int k = 0; k < RM; ++k) wu[k] = k < r ? Wu[size_t(e) * r + k] : 0.f;
            }
#pragma unroll
            for (int t2 = 0; t2 < TB; ++t2) {
                float g = 0.f;
#pragma unroll
                for (int k = 0; k < RM; ++k) g = fmaf(wu[k], hs[t2 * RM + k], g);
                coef[t2 * K + e] = sigm(g) * ge * inv[t2 * kBranches + i];
            }
        }
        __syncthreads();
        // 2. the writers, kGroup at a time
        for (int u0 = 0; u0 < U; u0 += kGroup) {
            const int gn = U - u0 < kGroup ? U - u0 : kGroup;
            for (int q = tid; q < TB * kGroup * kBranches; q += NT) {
                const int t2 = q / (kGroup * kBranches), g = (q / kBranches) % kGroup;
                const int i = q % kBranches;
                sS[q] = (t2 < nt && g < gn)
                            ? S[(size_t(u0 + g) * N + t0 + t2) * kBranches + i] : 0.f;
            }
            __syncthreads();
            float v[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = 0.f;
            if (tt < nt) {
                for (int sl = l; sl < nslot; sl += TPT) {
                    Raw8<T> y[kGroup];
#pragma unroll
                    for (int g = 0; g < kGroup; ++g) {
                        if (g < gn)
                            y[g].load(Y + (size_t(u0 + g) * N + t0 + tt) * D + sl * 8);
                        else
                            y[g].zero();
                    }
                    float cf[kBranches][8];
#pragma unroll
                    for (int i = 0; i < kBranches; ++i) {
                        const float4* cp =
                            reinterpret_cast<const float4*>(coef + tt * K + i * D + sl * 8);
                        const float4 a = cp[0], b = cp[1];
                        cf[i][0] = a.x; cf[i][1] = a.y; cf[i][2] = a.z; cf[i][3] = a.w;
                        cf[i][4] = b.x; cf[i][5] = b.y; cf[i][6] = b.z; cf[i][7] = b.w;
                    }
#pragma unroll
                    for (int g = 0; g < kGroup; ++g) {
                        const float4 s4 =
                            *reinterpret_cast<const float4*>(sS + (tt * kGroup + g) * kBranches);
                        const float sv[kBranches] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            float A = 0.f;
#pragma unroll
                            for (int i = 0; i < kBranches; ++i) {
                                const float p = cf[i][k] * y[g].get(k);
                                A = fmaf(sv[i], p, A);
                                v[g * kSums + 1 + i] = fmaf(p, p, v[g * kSums + 1 + i]);
                            }
                            v[g * kSums] = fmaf(A, A, v[g * kSums]);
                        }
                    }
                }
            }
            warp_reduce_scatter32(v);
            if (lane < kGroup * kSums) red[warp * 32 + lane] = v[0];
            __syncthreads();
            for (int q = tid; q < TB * kGroup; q += NT) {
                const int t2 = q / kGroup, g = q % kGroup;
                if (t2 < nt && g < gn) {
                    float acc[kSums] = {0.f, 0.f, 0.f, 0.f, 0.f};
                    for (int w = t2 * WPT; w < (t2 + 1) * WPT; ++w)
#pragma unroll
                        for (int m = 0; m < kSums; ++m) acc[m] += red[w * 32 + g * kSums + m];
                    const size_t o = size_t(t0 + t2) * U + u0 + g;
                    const float nv = 0.25f * sqrtf(acc[0]);
                    norm[o] = nv;
                    if (bnorm) {
                        const float* sv = sS + (t2 * kGroup + g) * kBranches;
#pragma unroll
                        for (int i = 0; i < kBranches; ++i)
                            bnorm[o * kBranches + i] = 0.25f * fabsf(sv[i]) * sqrtf(acc[1 + i]);
                    }
                    atomicAdd(&tsum[t2], nv);
                }
            }
            __syncthreads();
        }
        // 3. π from the norms written above, and the initial state's share
        if (pi)
            for (int64_t q = tid; q < int64_t(nt) * U; q += NT) {
                const int t2 = int(q / U);
                const size_t o = size_t(t0) * U + size_t(q);
                const float ts = tsum[t2];
                pi[o] = ts > 0.f ? norm[o] / ts : 0.f;
            }
        if (R0) {
            float v[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = 0.f;
            if (tt < nt)
                for (int sl = l; sl < nslot; sl += TPT) {
                    Raw8<T> x0[kBranches];
#pragma unroll
                    for (int i = 0; i < kBranches; ++i)
                        x0[i].load(R0 + (t0 + tt) * K + i * D + sl * 8);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        float A = 0.f;
#pragma unroll
                        for (int i = 0; i < kBranches; ++i)
                            A = fmaf(coef[tt * K + i * D + sl * 8 + k], x0[i].get(k), A);
                        v[0] = fmaf(A, A, v[0]);
                    }
                }
            warp_reduce_scatter32(v);
            if (lane == 0) red[warp * 32] = v[0];
            __syncthreads();
            if (tid < nt) {
                float a = 0.f;
                for (int w = tid * WPT; w < (tid + 1) * WPT; ++w) a += red[w * 32];
                a0_norm[t0 + tid] = 0.25f * sqrtf(a);
            }
        }
    }
}

template <typename T, int RM, int TB, bool FULL>
cudaError_t launch_t(int64_t N, int D, int r, float eps, const void* R, const float* gamma,
                     const float* Wd, const float* Wu, int U, const void* Y, const float* S,
                     const void* R0, float* norm, float* bnorm, float* pi, float* a0_norm,
                     cudaStream_t st) {
    constexpr int NT = dec_threads<RM>();
    constexpr int RED = (TB * RM > 32 ? TB * RM : 32);
    const size_t K = size_t(kBranches) * D;
    const size_t smem = (size_t(TB) * K + size_t(NT / 32) * RED + 2 * TB * RM +
                         TB * kBranches + TB * kGroup * kBranches + TB) * 4;
    auto kern = decompose_kernel<T, RM, TB, FULL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int64_t ntiles = (N + TB - 1) / TB;
    const int64_t cap = int64_t(sm_count()) * per_sm;
    kern<<<unsigned(ntiles < cap ? ntiles : cap), NT, smem, st>>>(
        N, D, r, eps, static_cast<const T*>(R), gamma, Wd, Wu, U, static_cast<const T*>(Y), S,
        static_cast<const T*>(R0), norm, bnorm, pi, a0_norm);
    return cudaGetLastError();
}

// Tokens per CTA: 2 below rank 64 when two tokens' fp32 coefficients fit in about 100 KB of
// shared memory (two CTAs per SM), else 1.
template <typename T, int RM>
cudaError_t launch_rm(int64_t N, int D, int r, float eps, const void* R, const float* gamma,
                      const float* Wd, const float* Wu, int U, const void* Y, const float* S,
                      const void* R0, float* norm, float* bnorm, float* pi, float* a0_norm,
                      cudaStream_t st) {
    const size_t row = size_t(kBranches) * D * 4;
    const int tb_reg = RM <= 32 ? 2 : 1;
    const int tb_smem = row * 2 <= 100 * 1024 ? 2 : 1;
    const int tb = tb_reg < tb_smem ? tb_reg : tb_smem;
    if (tb >= 2 && RM <= 32)
        return r == RM ? launch_t<T, RM, (RM <= 32 ? 2 : 1), true>(
                             N, D, r, eps, R, gamma, Wd, Wu, U, Y, S, R0, norm, bnorm, pi,
                             a0_norm, st)
                       : launch_t<T, RM, (RM <= 32 ? 2 : 1), false>(
                             N, D, r, eps, R, gamma, Wd, Wu, U, Y, S, R0, norm, bnorm, pi,
                             a0_norm, st);
    return r == RM ? launch_t<T, RM, 1, true>(N, D, r, eps, R, gamma, Wd, Wu, U, Y, S, R0, norm,
                                              bnorm, pi, a0_norm, st)
                   : launch_t<T, RM, 1, false>(N, D, r, eps, R, gamma, Wd, Wu, U, Y, S, R0, norm,
                                               bnorm, pi, a0_norm, st);
}

template <typename T>
cudaError_t launch_dt(int64_t N, int D, int r, float eps, const void* R, const float* gamma,
                      const float* Wd, const float* Wu, int U, const void* Y, const float* S,
                      const void* R0, float* norm, float* bnorm, float* pi, float* a0_norm,
                      cudaStream_t st) {
    if (r <= 16)
        return launch_rm<T, 16>(N, D, r, eps, R, gamma, Wd, Wu, U, Y, S, R0, norm, bnorm, pi,
                                a0_norm, st);
    if (r <= 32)
        return launch_rm<T, 32>(N, D, r, eps, R, gamma, Wd, Wu, U, Y, S, R0, norm, bnorm, pi,
                                a0_norm, st);
    return launch_rm<T, 64>(N, D, r, eps, R, gamma, Wd, Wu, U, Y, S, R0, norm, bnorm, pi,
                            a0_norm, st);
}

}  // namespace

cudaError_t launch_decompose(int64_t N, int D, int r, float eps, int dtype, const void* R,
                             const float* gamma, const float* Wd, const float* Wu, int U,
                             const void* Y, const float* S, const void* R0, float* norm,
                             float* bnorm, float* pi, float* a0_norm, cudaStream_t st) {
    if (N == 0 || (U == 0 && !R0)) return cudaSuccess;
    if (dtype == GR_BF16)
        return launch_dt<__nv_bfloat16>(N, D, r, eps, R, gamma, Wd, Wu, U, Y, S, R0, norm,
                                        bnorm, pi, a0_norm, st);
    return launch_dt<float>(N, D, r, eps, R, gamma, Wd, Wu, U, Y, S, R0, norm, bnorm, pi,
                            a0_norm, st);
}

}  // namespace gr
