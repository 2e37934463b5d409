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
// Two kernels. The per-token kernel (one CTA per token, the token's state row in shared memory
// as fp32) recomputes the read's intermediates, writes dR, and leaves the per-token factors of
// the parameter gradients in the caller's workspace: dg, vec R̂ and dR̂ ⊙ R inv ([N][4D] each)
// and [h | dz/n_r | du/n_r | 1] ([N][2r+5]). The reduction kernel then forms each parameter
// gradient as a sum over tokens of (small factor) × (long factor), a CTA per 256 columns and a
// slice of the tokens, fp32 atomics into the zeroed outputs.
#include <math.h>

#include "gr_internal.h"

namespace gr {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float sigm(float a) { return 1.0f / (1.0f + expf(-a)); }

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

// RM: the largest rank of the instantiation (16, 32 or 64).
template <typename T, int RM>
__global__ void __launch_bounds__(kThreads)
read_backward_kernel(int64_t N, int D, int r, float eps, const T* __restrict__ R,
                     const float* __restrict__ gamma, const float* __restrict__ Wd,
                     const float* __restrict__ Wu, const float* __restrict__ Ww,
                     const float* __restrict__ dx, const float* __restrict__ ds,
                     float* __restrict__ dR, float* __restrict__ DG, float* __restrict__ V,
                     float* __restrict__ P, float* __restrict__ S) {
    constexpr int M = RM + kBranches;
    extern __shared__ float smem[];
    const int K = kBranches * D;
    const int ss = 2 * r + kBranches + 1;     // row stride of S
    float* Rs = smem;                         // [4D] the state row
    float* red = Rs + K;                      // [kWarps][M]
    float* tot = red + kWarps * M;            // [M]
    float* q = tot + M;                       // [M] z at 0..r-1, u at RM..RM+3; then dz, du
    float* inv = q + M;                       // [4]
    const int tid = threadIdx.x;

    for (int64_t t = blockIdx.x; t < N; t += gridDim.x) {
        __syncthreads();   // the previous token is done with the shared arrays
        const T* Rt = R + t * K;
        float sq[kBranches] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < kBranches; ++i)
            for (int c = tid; c < D; c += kThreads) {
                const float v = to_f32(Rt[i * D + c]);
                Rs[i * D + c] = v;
                sq[i] = fmaf(v, v, sq[i]);
            }
        block_sum<kBranches>(sq, kBranches, red, tot);
        if (tid < kBranches) inv[tid] = rsqrtf(tot[tid] / float(D) + eps);
        __syncthreads();
        // z = W_d vec R̂ / 4 and u = W_w vec R̂ / 4 (indices 0..r-1 and RM..RM+3; the slots
        // between stay zero, so that every index is a compile-time constant)
        float az[M];
#pragma unroll
        for (int k = 0; k < M; ++k) az[k] = 0.f;
#pragma unroll
        for (int i = 0; i < kBranches; ++i)
            for (int c = tid; c < D; c += kThreads) {
                const int e = i * D + c;
                const float rh = gamma[e] * Rs[e] * inv[i];
#pragma unroll
                for (int k = 0; k < RM; ++k)
                    if (k < r) az[k] = fmaf(Wd[size_t(k) * K + e], rh, az[k]);
#pragma unroll
                for (int j = 0; j < kBranches; ++j)
                    az[RM + j] = fmaf(Ww[size_t(j) * K + e], rh, az[RM + j]);
            }
        block_sum<M>(az, M, red, q);
        // q = [z, u] (scaled below); h = SiLU(z)
        float h[RM];
#pragma unroll
        for (int k = 0; k < RM; ++k) {
            const float z = k < r ? 0.25f * q[k] : 0.f;
            h[k] = z * sigm(z);
        }
        // dg and the partial sums of dh = W_uᵀ dg
        float adh[RM];
#pragma unroll
        for (int k = 0; k < RM; ++k) adh[k] = 0.f;
#pragma unroll
        for (int i = 0; i < kBranches; ++i)
            for (int c = tid; c < D; c += kThreads) {
                const int e = i * D + c;
                const float* wu = Wu + size_t(e) * r;
                float g = 0.f;
#pragma unroll
                for (int k = 0; k < RM; ++k)
                    if (k < r) g = fmaf(wu[k], h[k], g);
                const float G = sigm(g);
                const float rh = gamma[e] * Rs[e] * inv[i];
                const float dG = 0.25f * dx[t * D + c] * rh;
                const float dg = dG * G * (1.0f - G);
                DG[t * K + e] = dg;
#pragma unroll
                for (int k = 0; k < RM; ++k)
                    if (k < r) adh[k] = fmaf(wu[k], dg, adh[k]);
            }
        __syncthreads();   // every thread has read q before it is overwritten
        block_sum<RM>(adh, r, red, tot);
        // dz = dh ⊙ SiLU'(z), du = ds ⊙ 2σ'(u); q becomes [dz, .., du] (without the 1/4), and
        // the token's row of S is [h | dz/4 | du/4 | 1]
        if (tid < r) {
            const float z = 0.25f * q[tid];
            const float sg = sigm(z);
            S[t * ss + tid] = z * sg;
            q[tid] = tot[tid] * sg * (1.0f + z * (1.0f - sg));
            S[t * ss + r + tid] = 0.25f * q[tid];
        } else if (tid >= RM && tid < RM + kBranches) {
            const int j = tid - RM;
            const float sg = sigm(0.25f * q[tid]);
            q[tid] = ds[t * kBranches + j] * 2.0f * sg * (1.0f - sg);
            S[t * ss + 2 * r + j] = 0.25f * q[tid];
        }
        if (tid == 0) S[t * ss + 2 * r + kBranches] = 1.0f;
        __syncthreads();
        // dR̂, the token's factors for dγ and the weight gradients, and γ ⊙ dR̂ into dR
        float apr[kBranches] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < kBranches; ++i)
            for (int c = tid; c < D; c += kThreads) {
                const int e = i * D + c;
                const float* wu = Wu + size_t(e) * r;
                float g = 0.f;
#pragma unroll
                for (int k = 0; k < RM; ++k)
                    if (k < r) g = fmaf(wu[k], h[k], g);
                const float G = sigm(g);
                float back = 0.f;   // W_dᵀ dz + W_wᵀ du at e
#pragma unroll
                for (int k = 0; k < RM; ++k)
                    if (k < r) back = fmaf(Wd[size_t(k) * K + e], q[k], back);
#pragma unroll
                for (int j = 0; j < kBranches; ++j) back = fmaf(Ww[size_t(j) * K + e], q[RM + j], back);
                const float dRh = 0.25f * (dx[t * D + c] * G + back);
                const float ri = Rs[e] * inv[i];
                V[t * K + e] = gamma[e] * ri;
                P[t * K + e] = dRh * ri;
                const float a = dRh * gamma[e];
                dR[t * K + e] = a;
                apr[i] = fmaf(a, Rs[e], apr[i]);
            }
        block_sum<kBranches>(apr, kBranches, red, tot);
#pragma unroll
        for (int i = 0; i < kBranches; ++i) {
            const float iv = inv[i], i3 = iv * iv * iv * tot[i] / float(D);
            for (int c = tid; c < D; c += kThreads) {
                const int e = i * D + c;
                dR[t * K + e] = iv * dR[t * K + e] - i3 * Rs[e];
            }
        }
    }
}

// out rows m < M: Σ over this CTA's tokens of S[t][soff + m] · B[t][j], added atomically to
// out0[m·K + j] (m < m0) or out1[(m − m0)·K + j]; or, transposed (one output), to
// out0[j·M + m]. One column j per thread, 32 tokens' small factors staged in shared memory.
template <int MM>
__global__ void __launch_bounds__(kThreads)
token_sum_kernel(int64_t N, int K, int M, const float* __restrict__ S, int s_stride, int soff,
                 const float* __restrict__ B, float* __restrict__ out0, float* __restrict__ out1,
                 int m0, bool transposed, int64_t tokens_per_cta) {
    __shared__ float sS[32][MM];
    const int j = blockIdx.x * kThreads + threadIdx.x;
    const int64_t ta = int64_t(blockIdx.y) * tokens_per_cta;
    const int64_t tb = ta + tokens_per_cta < N ? ta + tokens_per_cta : N;
    float acc[MM];
#pragma unroll
    for (int m = 0; m < MM; ++m) acc[m] = 0.f;
    for (int64_t t0 = ta; t0 < tb; t0 += 32) {
        const int nt = int(tb - t0 < 32 ? tb - t0 : 32);
        for (int e = threadIdx.x; e < nt * M; e += kThreads) {
            const int tt = e / M, m = e - tt * M;
            sS[tt][m] = S[(t0 + tt) * s_stride + soff + m];
        }
        __syncthreads();
        if (j < K) {
            for (int tt = 0; tt < nt; ++tt) {
                const float b = B[(t0 + tt) * K + j];
#pragma unroll
                for (int m = 0; m < MM; ++m)
                    if (m < M) acc[m] = fmaf(sS[tt][m], b, acc[m]);
            }
        }
        __syncthreads();
    }
    if (j < K) {
#pragma unroll
        for (int m = 0; m < MM; ++m) {
            if (m < M) {
                if (transposed) atomicAdd(&out0[size_t(j) * M + m], acc[m]);
                else if (m < m0) atomicAdd(&out0[size_t(m) * K + j], acc[m]);
                else atomicAdd(&out1[size_t(m - m0) * K + j], acc[m]);
            }
        }
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

template <typename T, int RM>
cudaError_t launch_rb(int64_t N, int D, int r, float eps, const void* R, const float* gamma,
                      const float* Wd, const float* Wu, const float* Ww, const float* dx,
                      const float* ds, float* dR, float* DG, float* V, float* P, float* S,
                      cudaStream_t st) {
    constexpr int M = RM + kBranches;
    const size_t smem = (size_t(kBranches) * D + kWarps * M + 2 * M + kBranches) * sizeof(float);
    auto kern = read_backward_kernel<T, RM>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    kern<<<grid_tokens(N), kThreads, smem, st>>>(N, D, r, eps, static_cast<const T*>(R), gamma,
                                                  Wd, Wu, Ww, dx, ds, dR, DG, V, P, S);
    return cudaGetLastError();
}

template <int MM>
cudaError_t launch_sum(int64_t N, int K, int M, const float* S, int s_stride, int soff,
                       const float* B, float* out0, float* out1, int m0, bool transposed,
                       cudaStream_t st) {
    const int gx = (K + kThreads - 1) / kThreads;
    int gy = (2 * sm_count() + gx - 1) / gx;
    const int64_t max_gy = (N + 31) / 32;
    if (gy > max_gy) gy = int(max_gy);
    if (gy < 1) gy = 1;
    const int64_t per = ((N + gy - 1) / gy + 31) / 32 * 32;
    token_sum_kernel<MM><<<dim3(gx, gy), kThreads, 0, st>>>(N, K, M, S, s_stride, soff, B, out0,
                                                            out1, m0, transposed, per);
    return cudaGetLastError();
}

}  // namespace

size_t read_backward_workspace(int64_t N, int D, int r) {
    const size_t K = size_t(kBranches) * D;
    return 3 * align256(size_t(N) * K * 4) + align256(size_t(N) * (2 * r + kBranches + 1) * 4);
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
    const int ss = 2 * r + kBranches + 1;
    cudaError_t e;
    if ((e = cudaMemsetAsync(dgamma, 0, K * 4, st)) != cudaSuccess ||
        (e = cudaMemsetAsync(dWd, 0, size_t(r) * K * 4, st)) != cudaSuccess ||
        (e = cudaMemsetAsync(dWu, 0, size_t(r) * K * 4, st)) != cudaSuccess ||
        (e = cudaMemsetAsync(dWw, 0, size_t(kBranches) * K * 4, st)) != cudaSuccess)
        return e;
    if (N == 0) return cudaSuccess;
    const bool bf = dtype == GR_BF16;
    if (r <= 16)
        e = bf ? launch_rb<__nv_bfloat16, 16>(N, D, r, eps, R, gamma, Wd, Wu, Ww, dx, ds, dR, DG,
                                              V, P, S, st)
               : launch_rb<float, 16>(N, D, r, eps, R, gamma, Wd, Wu, Ww, dx, ds, dR, DG, V, P, S,
                                      st);
    else if (r <= 32)
        e = bf ? launch_rb<__nv_bfloat16, 32>(N, D, r, eps, R, gamma, Wd, Wu, Ww, dx, ds, dR, DG,
                                              V, P, S, st)
               : launch_rb<float, 32>(N, D, r, eps, R, gamma, Wd, Wu, Ww, dx, ds, dR, DG, V, P, S,
                                      st);
    else
        e = bf ? launch_rb<__nv_bfloat16, 64>(N, D, r, eps, R, gamma, Wd, Wu, Ww, dx, ds, dR, DG,
                                              V, P, S, st)
               : launch_rb<float, 64>(N, D, r, eps, R, gamma, Wd, Wu, Ww, dx, ds, dR, DG, V, P, S,
                                      st);
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
