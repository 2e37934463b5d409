// Backward of the GR read and write (training), CUDA cores, fp32 arithmetic.
//
// The gradients of "【论文解读】 Qwen3.8 Flash Next", §二.4 (eq rms, eq gate, eq use_gate, eq s,
// eq write) by the chain rule. Per token t, with R̂_i = γ_i R_i inv_i, z = W_d vec R̂ / n_r,
// h = SiLU(z), G = σ(W_u h), u = W_w vec R̂ / n_r, s = 2σ(u), given dL/dx and dL/ds:
//   dG = dx ⊙ R̂ / n_r,  dR̂ = dx ⊙ G / n_r + (W_dᵀ dz + W_wᵀ du) / n_r,  dg = dG ⊙ G(1 − G)
//   dh = W_uᵀ dg,  dz = dh ⊙ SiLU'(z),  du = ds ⊙ 2σ(u)(1 − σ(u))
//   dR_i = inv_i γ_i ⊙ dR̂_i − inv_i³ R_i (Σ_c γ_i dR̂_i R_i) / D
//   dW_u = Σ_t dg ⊗ h,  dW_d = Σ_t dz ⊗ vec R̂ / n_r,  dW_w = Σ_t du ⊗ vec R̂ / n_r,
//   dγ = Σ_t dR̂ ⊙ R inv.
//
// Two kernels. The per-token kernel (persistent, TB tokens per CTA at a time with their state
// rows in shared memory in the state's type, so that each weight element loaded serves TB
// tokens) recomputes the read's intermediates, writes dR, and leaves the per-token factors of
// the parameter gradients in the caller's workspace: dg, vec R̂ and dR̂ ⊙ R inv ([N][4D] each)
// and [h | dz/n_r | du/n_r | 1] ([N][2r+5]). The reduction kernel then forms each parameter
// gradient as a sum over tokens of (small factor) × (long factor), a CTA per 256 columns and
// 128 tokens, fp32 atomics into the zeroed outputs. W_u is transposed into the workspace first.
#include <math.h>

#include "gr_internal.h"

namespace gr {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// σ(a) = 1/(1 + e^-a) with the fast exponential and division: a few ulp, far inside the fp32
// bounds of these paths; 0 and 1 at the ends (1/inf = 0).
__device__ __forceinline__ float sigm(float a) { return __fdividef(1.0f, 1.0f + __expf(-a)); }

// Sums of the first m of M per-thread values over the block; the totals land in out[0..m).
template <int M>
__device__ __forceinline__ void block_sum(const float (&v)[M], int m, float* red, float* out) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int k = 0; k < M; ++k) {
        if (k < m) {   // uniform over the block
            float a = v[k];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
            if (lane == 0) red[warp * M + k] = a;
        }
    }
    __syncthreads();
    for (int k = threadIdx.x; k < m; k += kThreads) {
        float a = 0.f;
        for (int w = 0; w < kWarps; ++w) a += red[w * M + k];
        out[k] = a;
    }
    __syncthreads();
}

// Sums of M per-thread values over a block of NW warps; the totals land in out[0..M).
template <int M, int NW>
__device__ __forceinline__ void block_sum_w(const float (&v)[M], float* red, float* out) {
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

// Threads of the per-token kernel: 512, or 256 at rank 64 (whose accumulators need more than
// the 128 registers a thread of a 512-thread block can have).
template <int RM>
__host__ __device__ constexpr int bwd_threads() { return RM > 32 ? 256 : 512; }

// RM: the largest rank of the instantiation (16, 32 or 64); TB: tokens per CTA at a time. Every
// weight element a thread loads serves the TB tokens (the weights stream from L2 once per TB
// tokens); the TB state rows sit in shared memory in the state's own type.
// FULL: r == RM, so that every rank test below is a compile-time constant (the common case of a
// rank that is itself 16, 32 or 64).
template <typename T, int RM, int TB, bool FULL>
__global__ void __launch_bounds__(bwd_threads<RM>())
read_backward_kernel(int64_t N, int D, int r_arg, float eps, const T* __restrict__ R,
                     const float* __restrict__ gamma, const float* __restrict__ Wd,
                     const float* __restrict__ WuT, const float* __restrict__ Ww,
                     const float* __restrict__ dx, const float* __restrict__ ds,
                     float* __restrict__ dR, float* __restrict__ DG, float* __restrict__ V,
                     float* __restrict__ P, float* __restrict__ S) {
    // WuT is W_u transposed, [r][4D]: for each k the block's threads read consecutive channels
    constexpr int M = RM + kBranches;
    constexpr int kBwdThreads = bwd_threads<RM>();
    constexpr int kBwdWarps = kBwdThreads / 32;
    const int r = FULL ? RM : r_arg;
    extern __shared__ float smem[];
    const int K = kBranches * D;
    const int ss = 2 * r + kBranches + 1;                   // row stride of S
    T* Rs = reinterpret_cast<T*>(smem);                     // [TB][4D] the state rows
    float* fl = smem + (size_t(TB) * K * sizeof(T) + 15) / 16 * 4;
    float* red = fl;                                        // [warps][TB·M]
    float* tot = red + kBwdWarps * TB * M;                  // [TB·M]
    float* q = tot + TB * M;                                // [TB][M] z|u, then dz|du
    float* hs = q + TB * M;                                 // [TB][RM] h
    float* inv = hs + TB * RM;                              // [TB][4]
    const int tid = threadIdx.x;
    const int64_t ntiles = (N + TB - 1) / TB;

    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t t0 = tile * TB;
        const int nt = int(N - t0 < TB ? N - t0 : TB);
        __syncthreads();   // the previous tile is done with the shared arrays
        float sq[TB * kBranches];
#pragma unroll
        for (int k = 0; k < TB * kBranches; ++k) sq[k] = 0.f;
#pragma unroll
        for (int tt = 0; tt < TB; ++tt)
#pragma unroll
            for (int i = 0; i < kBranches; ++i)
                for (int c = tid; c < D; c += kBwdThreads) {
                    const T v = tt < nt ? R[(t0 + tt) * K + i * D + c] : from_f32<T>(0.f);
                    Rs[tt * K + i * D + c] = v;
                    const float f = to_f32(v);
                    sq[tt * kBranches + i] = fmaf(f, f, sq[tt * kBranches + i]);
                }
        block_sum_w<TB * kBranches, kBwdWarps>(sq, red, tot);
        if (tid < TB * kBranches) inv[tid] = rsqrtf(tot[tid] / float(D) + eps);
        __syncthreads();
        // z = W_d vec R̂ / 4 (slots 0..r-1) and u = W_w vec R̂ / 4 (slots RM..RM+3) per token
        {
            float az[TB * M];
#pragma unroll
            for (int k = 0; k < TB * M; ++k) az[k] = 0.f;
#pragma unroll
            for (int i = 0; i < kBranches; ++i)
                for (int c = tid; c < D; c += kBwdThreads) {
                    const int e = i * D + c;
                    const float ge = gamma[e];
                    float wd[RM], ww[kBranches];
#pragma unroll
                    for (int k = 0; k < RM; ++k) wd[k] = k < r ? Wd[size_t(k) * K + e] : 0.f;
#pragma unroll
                    for (int j = 0; j < kBranches; ++j) ww[j] = Ww[size_t(j) * K + e];
#pragma unroll
                    for (int tt = 0; tt < TB; ++tt) {
                        const float rh = ge * to_f32(Rs[tt * K + e]) * inv[tt * kBranches + i];
#pragma unroll
                        for (int k = 0; k < RM; ++k)
                            az[tt * M + k] = fmaf(wd[k], rh, az[tt * M + k]);
#pragma unroll
                        for (int j = 0; j < kBranches; ++j)
                            az[tt * M + RM + j] = fmaf(ww[j], rh, az[tt * M + RM + j]);
                    }
                }
            block_sum_w<TB * M, kBwdWarps>(az, red, q);
        }
        for (int e2 = tid; e2 < TB * RM; e2 += kBwdThreads) {
            const int tt = e2 / RM, k = e2 - tt * RM;
            const float z = k < r ? 0.25f * q[tt * M + k] : 0.f;
            hs[e2] = z * sigm(z);
        }
        __syncthreads();
        // dg (streamed out) and the partial sums of dh = W_uᵀ dg
        {
            float adh[TB * RM];
#pragma unroll
            for (int k = 0; k < TB * RM; ++k) adh[k] = 0.f;
#pragma unroll
            for (int i = 0; i < kBranches; ++i)
                for (int c = tid; c < D; c += kBwdThreads) {
                    const int e = i * D + c;
                    const float ge = gamma[e];
                    float wu[RM];
#pragma unroll
                    for (int k = 0; k < RM; ++k) wu[k] = k < r ? WuT[size_t(k) * K + e] : 0.f;
#pragma unroll
                    for (int tt = 0; tt < TB; ++tt) {
                        float g = 0.f;
#pragma unroll
                        for (int k = 0; k < RM; ++k) g = fmaf(wu[k], hs[tt * RM + k], g);
                        const float G = sigm(g);
                        const float rh = ge * to_f32(Rs[tt * K + e]) * inv[tt * kBranches + i];
                        const float dxc = tt < nt ? dx[(t0 + tt) * D + c] : 0.f;
                        const float dg = 0.25f * dxc * rh * G * (1.0f - G);
                        if (tt < nt) __stcs(&DG[(t0 + tt) * K + e], dg);   // keep weights in L2
#pragma unroll
                        for (int k = 0; k < RM; ++k)
                            adh[tt * RM + k] = fmaf(wu[k], dg, adh[tt * RM + k]);
                    }
                }
            block_sum_w<TB * RM, kBwdWarps>(adh, red, tot);
        }
        // dz = dh ⊙ SiLU'(z), du = ds ⊙ 2σ'(u) into q (without the 1/4); the token's row of S
        // is [h | dz/4 | du/4 | 1]
        for (int e2 = tid; e2 < TB * M; e2 += kBwdThreads) {
            const int tt = e2 / M, k = e2 - tt * M;
            if (tt >= nt) continue;
            float* Srow = S + (t0 + tt) * ss;
            if (k < r) {
                const float z = 0.25f * q[e2];
                const float sg = sigm(z);
                Srow[k] = z * sg;
                q[e2] = tot[tt * RM + k] * sg * (1.0f + z * (1.0f - sg));
                Srow[r + k] = 0.25f * q[e2];
            } else if (k >= RM) {
                const int j = k - RM;
                const float sg = sigm(0.25f * q[e2]);
                q[e2] = ds[(t0 + tt) * kBranches + j] * 2.0f * sg * (1.0f - sg);
                Srow[2 * r + j] = 0.25f * q[e2];
                if (j == 0) Srow[2 * r + kBranches] = 1.0f;
            }
        }
        __syncthreads();
        // dR̂, the token's factors for dγ and the weight gradients, and γ ⊙ dR̂ into dR
        {
            float apr[TB * kBranches];
#pragma unroll
            for (int k = 0; k < TB * kBranches; ++k) apr[k] = 0.f;
#pragma unroll
            for (int i = 0; i < kBranches; ++i)
                for (int c = tid; c < D; c += kBwdThreads) {
                    const int e = i * D + c;
                    const float ge = gamma[e];
                    float wu[RM], wd[RM], ww[kBranches];
#pragma unroll
                    for (int k = 0; k < RM; ++k) {
                        wu[k] = k < r ? WuT[size_t(k) * K + e] : 0.f;
                        wd[k] = k < r ? Wd[size_t(k) * K + e] : 0.f;
                    }
#pragma unroll
                    for (int j = 0; j < kBranches; ++j) ww[j] = Ww[size_t(j) * K + e];
#pragma unroll
                    for (int tt = 0; tt < TB; ++tt) {
                        float g = 0.f, back = 0.f;   // W_u h and (W_dᵀ dz + W_wᵀ du) at e
#pragma unroll
                        for (int k = 0; k < RM; ++k) {
                            g = fmaf(wu[k], hs[tt * RM + k], g);
                            back = fmaf(wd[k], q[tt * M + k], back);
                        }
#pragma unroll
                        for (int j = 0; j < kBranches; ++j)
                            back = fmaf(ww[j], q[tt * M + RM + j], back);
                        const float G = sigm(g);
                        const float dxc = tt < nt ? dx[(t0 + tt) * D + c] : 0.f;
                        const float dRh = 0.25f * (dxc * G + back);
                        const float rv = to_f32(Rs[tt * K + e]);
                        const float ri = rv * inv[tt * kBranches + i];
                        const float a = dRh * ge;
                        if (tt < nt) {
                            __stcs(&V[(t0 + tt) * K + e], ge * ri);
                            __stcs(&P[(t0 + tt) * K + e], dRh * ri);
                            dR[(t0 + tt) * K + e] = a;
                        }
                        apr[tt * kBranches + i] = fmaf(a, rv, apr[tt * kBranches + i]);
                    }
                }
            block_sum_w<TB * kBranches, kBwdWarps>(apr, red, tot);
        }
#pragma unroll
        for (int tt = 0; tt < TB; ++tt) {
            if (tt >= nt) break;
#pragma unroll
            for (int i = 0; i < kBranches; ++i) {
                const float iv = inv[tt * kBranches + i];
                const float i3 = iv * iv * iv * tot[tt * kBranches + i] / float(D);
                for (int c = tid; c < D; c += kBwdThreads) {
                    const size_t e = size_t(t0 + tt) * K + i * D + c;
                    __stcs(&dR[e], iv * dR[e] - i3 * to_f32(Rs[tt * K + i * D + c]));
                }
            }
        }
    }
}

// out rows m < M: Σ over this CTA's tokens of S[t][soff + m] · B[t][j], added atomically to
// out0[m·K + j] (m < m0) or out1[(m − m0)·K + j]; or, transposed (one output), to
// out0[j·M + m]. One column j per thread, 32 tokens' small factors staged in shared memory.
template <int MM, int CW>
__global__ void __launch_bounds__(kThreads)
token_sum_kernel(int64_t N, int K, int M, const float* __restrict__ S, int s_stride, int soff,
                 const float* __restrict__ B, float* __restrict__ out0, float* __restrict__ out1,
                 int m0, bool transposed, int64_t tokens_per_cta) {
    // CW consecutive columns a thread (16- or 8-byte loads of the long factor), so that each
    // shared-memory read of a small factor serves CW columns; rows padded to a multiple of 4
    constexpr int MP = (MM + 3) / 4 * 4;
    __shared__ __align__(16) float sS[32][MP];
    const int j0 = (blockIdx.x * kThreads + threadIdx.x) * CW;
    const int64_t ta = int64_t(blockIdx.y) * tokens_per_cta;
    const int64_t tb = ta + tokens_per_cta < N ? ta + tokens_per_cta : N;
    float acc[MM][CW];
#pragma unroll
    for (int m = 0; m < MM; ++m)
#pragma unroll
        for (int c = 0; c < CW; ++c) acc[m][c] = 0.f;
    for (int64_t t0 = ta; t0 < tb; t0 += 32) {
        const int nt = int(tb - t0 < 32 ? tb - t0 : 32);
        for (int e = threadIdx.x; e < 32 * MP; e += kThreads) {
            const int tt = e / MP, m = e - tt * MP;
            sS[tt][m] = (tt < nt && m < M) ? S[(t0 + tt) * s_stride + soff + m] : 0.f;
        }
        __syncthreads();
        if (j0 < K) {
#pragma unroll 4
            for (int tt = 0; tt < nt; ++tt) {
                float b[CW];
                const float* bp = B + (t0 + tt) * K + j0;
                if (CW == 4) {
                    const float4 v = *reinterpret_cast<const float4*>(bp);
                    b[0] = v.x; b[CW > 1 ? 1 : 0] = v.y; b[CW > 2 ? 2 : 0] = v.z;
                    b[CW > 3 ? 3 : 0] = v.w;
                } else if (CW == 2) {
                    const float2 v = *reinterpret_cast<const float2*>(bp);
                    b[0] = v.x; b[CW > 1 ? 1 : 0] = v.y;
                } else {
                    b[0] = *bp;
                }
#pragma unroll
                for (int m4 = 0; m4 < MP; m4 += 4) {
                    const float4 s4 = *reinterpret_cast<const float4*>(&sS[tt][m4]);
                    const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (m4 + q < MM)
#pragma unroll
                            for (int c = 0; c < CW; ++c)
                                acc[m4 + q][c] = fmaf(sv[q], b[c], acc[m4 + q][c]);
                }
            }
        }
        __syncthreads();
    }
    if (j0 < K) {
#pragma unroll
        for (int m = 0; m < MM; ++m) {
            if (m < M) {
#pragma unroll
                for (int c = 0; c < CW; ++c) {
                    const int j = j0 + c;
                    if (transposed) atomicAdd(&out0[size_t(j) * M + m], acc[m][c]);
                    else if (m < m0) atomicAdd(&out0[size_t(m) * K + j], acc[m][c]);
                    else atomicAdd(&out1[size_t(m - m0) * K + j], acc[m][c]);
                }
            }
        }
    }
}

// W_u [K][r] -> its transpose [r][K].
__global__ void transpose_kernel(int K, int r, const float* __restrict__ Wu,
                                 float* __restrict__ WuT) {
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < int64_t(K) * r;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int k = int(e / K), j = int(e - int64_t(k) * K);
        WuT[e] = Wu[size_t(j) * r + k];
    }
}

// Backward of eq write: dy = Σ_i s_i dR'_i, ds_i = Σ_c dR'_i[c] y[c], dR = dR'.
template <typename T>
__global__ void __launch_bounds__(kThreads)
write_backward_kernel(int64_t N, int D, const float* __restrict__ dRp, const T* __restrict__ y,
                      const float* __restrict__ s, float* __restrict__ dR,
                      float* __restrict__ dy, float* __restrict__ ds) {
    __shared__ float red[kWarps * kBranches];
    __shared__ float tot[kBranches];
    const int K = kBranches * D;
    for (int64_t t = blockIdx.x; t < N; t += gridDim.x) {
        float sv[kBranches], a[kBranches] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < kBranches; ++i) sv[i] = s[t * kBranches + i];
        for (int c = threadIdx.x; c < D; c += kThreads) {
            const float yc = to_f32(y[t * D + c]);
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < kBranches; ++i) {
                const float g = dRp[t * K + i * D + c];
                acc = fmaf(sv[i], g, acc);
                a[i] = fmaf(g, yc, a[i]);
                if (dR != dRp) dR[t * K + i * D + c] = g;
            }
            dy[t * D + c] = acc;
        }
        block_sum<kBranches>(a, kBranches, red, tot);
        if (threadIdx.x < kBranches) ds[t * kBranches + threadIdx.x] = tot[threadIdx.x];
    }
}

int grid_tokens(int64_t N) {
    const int64_t cap = int64_t(sm_count()) * 4;
    return int(N < cap ? N : cap);
}

template <typename T, int RM, int TB, bool FULL>
cudaError_t launch_rb_t(int64_t N, int D, int r, float eps, const void* R, const float* gamma,
                        const float* Wd, const float* WuT, const float* Ww, const float* dx,
                        const float* ds, float* dR, float* DG, float* V, float* P, float* S,
                        cudaStream_t st) {
    constexpr int M = RM + kBranches;
    constexpr int kBwdThreads = bwd_threads<RM>();
    const size_t K = size_t(kBranches) * D;
    const size_t smem =
        (size_t(TB) * K * sizeof(T) + 15) / 16 * 16 +
        (size_t(kBwdThreads / 32) * TB * M + 2 * TB * M + TB * RM + TB * kBranches) * 4;
    auto kern = read_backward_kernel<T, RM, TB, FULL>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0;   // a persistent grid: as many CTAs as stay resident
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kBwdThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int64_t ntiles = (N + TB - 1) / TB;
    const int64_t cap = int64_t(sm_count()) * per_sm;
    kern<<<unsigned(ntiles < cap ? ntiles : cap), kBwdThreads, smem, st>>>(
        N, D, r, eps, static_cast<const T*>(R), gamma, Wd, WuT, Ww, dx, ds, dR, DG, V, P, S);
    return cudaGetLastError();
}

// The full-rank instantiation when r == RM, else the general one.
template <typename T, int RM, int TB>
cudaError_t launch_rb_tb(int64_t N, int D, int r, float eps, const void* R, const float* gamma,
                         const float* Wd, const float* WuT, const float* Ww, const float* dx,
                         const float* ds, float* dR, float* DG, float* V, float* P, float* S,
                         cudaStream_t st) {
    if (r == RM)
        return launch_rb_t<T, RM, TB, true>(N, D, r, eps, R, gamma, Wd, WuT, Ww, dx, ds, dR, DG,
                                            V, P, S, st);
    return launch_rb_t<T, RM, TB, false>(N, D, r, eps, R, gamma, Wd, WuT, Ww, dx, ds, dR, DG, V,
                                         P, S, st);
}

// The most tokens per CTA that the registers (TB·(RM+4) accumulators) and shared memory
// (TB state rows, up to about 200 KB) allow: 4, 2 or 1.
template <typename T, int RM>
cudaError_t launch_rb(int64_t N, int D, int r, float eps, const void* R, const float* gamma,
                      const float* Wd, const float* WuT, const float* Ww, const float* dx,
                      const float* ds, float* dR, float* DG, float* V, float* P, float* S,
                      cudaStream_t st) {
    const size_t row = size_t(kBranches) * D * sizeof(T);
    const int tb_reg = RM <= 16 ? 4 : RM <= 32 ? 2 : 1;
    const int tb_smem = row * 4 <= 200 * 1024 ? 4 : row * 2 <= 200 * 1024 ? 2 : 1;
    const int tb = tb_reg < tb_smem ? tb_reg : tb_smem;
    if (tb >= 4 && RM <= 16)
        return launch_rb_tb<T, RM, (RM <= 16 ? 4 : 1)>(N, D, r, eps, R, gamma, Wd, WuT, Ww, dx,
                                                       ds, dR, DG, V, P, S, st);
    if (tb >= 2 && RM <= 32)
        return launch_rb_tb<T, RM, (RM <= 32 ? 2 : 1)>(N, D, r, eps, R, gamma, Wd, WuT, Ww, dx,
                                                       ds, dR, DG, V, P, S, st);
    return launch_rb_tb<T, RM, 1>(N, D, r, eps, R, gamma, Wd, WuT, Ww, dx, ds, dR, DG, V, P, S,
                                  st);
}

template <int MM>
cudaError_t launch_sum(int64_t N, int K, int M, const float* S, int s_stride, int soff,
                       const float* B, float* out0, float* out1, int m0, bool transposed,
                       cudaStream_t st) {
    // 128 tokens per CTA: thousands of CTAs keep enough loads of the long factor in flight
    // (a few CTAs walking thousands of tokens each were latency-bound); the cost is one atomic
    // per output element and CTA row. Columns per thread: 4 up to 20 small factors, 2 up to
    // 40, else 1 (the accumulators are MM × CW registers).
    constexpr int CW = MM <= 20 ? 4 : MM <= 40 ? 2 : 1;
    const int gx = (K + kThreads * CW - 1) / (kThreads * CW);
    const int64_t per = 128;
    const int gy = int((N + per - 1) / per);
    token_sum_kernel<MM, CW><<<dim3(gx, gy), kThreads, 0, st>>>(
        N, K, M, S, s_stride, soff, B, out0, out1, m0, transposed, per);
    return cudaGetLastError();
}

}  // namespace

size_t read_backward_workspace(int64_t N, int D, int r) {
    const size_t K = size_t(kBranches) * D;
    return 3 * align256(size_t(N) * K * 4) + align256(size_t(N) * (2 * r + kBranches + 1) * 4) +
           align256(size_t(r) * K * 4);
}

cudaError_t launch_read_backward(int64_t N, int D, int r, float eps, int dtype, const void* R,
                                 const float* gamma, const float* Wd, const float* Wu,
                                 const float* Ww, const float* dx, const float* ds, float* dR,
                                 float* dgamma, float* dWd, float* dWu, float* dWw,
                                 void* workspace, cudaStream_t st) {
    const size_t K = size_t(kBranches) * D;
    char* ws = static_cast<char*>(workspace);
    float* DG = reinterpret_cast<float*>(ws);
    float* V = reinterpret_cast<float*>(ws + align256(size_t(N) * K * 4));
    float* P = reinterpret_cast<float*>(ws + 2 * align256(size_t(N) * K * 4));
    float* S = reinterpret_cast<float*>(ws + 3 * align256(size_t(N) * K * 4));
    float* WuT = reinterpret_cast<float*>(ws + 3 * align256(size_t(N) * K * 4) +
                                          align256(size_t(N) * (2 * r + kBranches + 1) * 4));
    const int ss = 2 * r + kBranches + 1;
    cudaError_t e;
    if ((e = cudaMemsetAsync(dgamma, 0, K * 4, st)) != cudaSuccess ||
        (e = cudaMemsetAsync(dWd, 0, size_t(r) * K * 4, st)) != cudaSuccess ||
        (e = cudaMemsetAsync(dWu, 0, size_t(r) * K * 4, st)) != cudaSuccess ||
        (e = cudaMemsetAsync(dWw, 0, size_t(kBranches) * K * 4, st)) != cudaSuccess)
        return e;
    if (N == 0) return cudaSuccess;
    transpose_kernel<<<sm_count() * 4, kThreads, 0, st>>>(int(K), r, Wu, WuT);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const bool bf = dtype == GR_BF16;
    if (r <= 16)
        e = bf ? launch_rb<__nv_bfloat16, 16>(N, D, r, eps, R, gamma, Wd, WuT, Ww, dx, ds, dR,
                                              DG, V, P, S, st)
               : launch_rb<float, 16>(N, D, r, eps, R, gamma, Wd, WuT, Ww, dx, ds, dR, DG, V, P,
                                      S, st);
    else if (r <= 32)
        e = bf ? launch_rb<__nv_bfloat16, 32>(N, D, r, eps, R, gamma, Wd, WuT, Ww, dx, ds, dR,
                                              DG, V, P, S, st)
               : launch_rb<float, 32>(N, D, r, eps, R, gamma, Wd, WuT, Ww, dx, ds, dR, DG, V, P,
                                      S, st);
    else
        e = bf ? launch_rb<__nv_bfloat16, 64>(N, D, r, eps, R, gamma, Wd, WuT, Ww, dx, ds, dR,
                                              DG, V, P, S, st)
               : launch_rb<float, 64>(N, D, r, eps, R, gamma, Wd, WuT, Ww, dx, ds, dR, DG, V, P,
                                      S, st);
    if (e != cudaSuccess) return e;
    const int Kk = int(K);
    // dW_u[j][k] = Σ_t dg[t][j] h[t][k]
    if (r <= 16) e = launch_sum<16>(N, Kk, r, S, ss, 0, DG, dWu, nullptr, r, true, st);
    else if (r <= 32) e = launch_sum<32>(N, Kk, r, S, ss, 0, DG, dWu, nullptr, r, true, st);
    else e = launch_sum<64>(N, Kk, r, S, ss, 0, DG, dWu, nullptr, r, true, st);
    if (e != cudaSuccess) return e;
    // dW_d[k][j] and dW_w[i][j] = Σ_t (dz/4, du/4)[t] vec R̂[t][j]
    const int m = r + kBranches;
    if (m <= 20) e = launch_sum<20>(N, Kk, m, S, ss, r, V, dWd, dWw, r, false, st);
    else if (m <= 36) e = launch_sum<36>(N, Kk, m, S, ss, r, V, dWd, dWw, r, false, st);
    else e = launch_sum<68>(N, Kk, m, S, ss, r, V, dWd, dWw, r, false, st);
    if (e != cudaSuccess) return e;
    // dγ[j] = Σ_t dR̂[t][j] R[t][j] inv[t]
    return launch_sum<1>(N, Kk, 1, S, ss, 2 * r + kBranches, P, dgamma, nullptr, 1, false, st);
}

cudaError_t launch_write_backward(int64_t N, int D, int dtype, const float* dRp, const void* y,
                                  const float* s, float* dR, float* dy, float* ds,
                                  cudaStream_t st) {
    if (N == 0) return cudaSuccess;
    if (dtype == GR_BF16)
        write_backward_kernel<__nv_bfloat16><<<grid_tokens(N), kThreads, 0, st>>>(
            N, D, dRp, static_cast<const __nv_bfloat16*>(y), s, dR, dy, ds);
    else
        write_backward_kernel<float><<<grid_tokens(N), kThreads, 0, st>>>(
            N, D, dRp, static_cast<const float*>(y), s, dR, dy, ds);
    return cudaGetLastError();
}

}  // namespace gr
