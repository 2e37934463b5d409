// Generic per-token GR kernel: one CTA per token row, CUDA cores, fp32 arithmetic.
//
// Serves the fp32 state path and every bf16 shape the fused tensor-core kernel does not take.
// Per token t (from "【论文解读】 Qwen3.8 Flash Next", §二.4):
//   eq write     R'_i = R_i + s_i y                       (when y is given; stored, then re-read
//                                                          at the stored precision)
//   eq rms       inv_i = 1/sqrt(mean_c R'_i[c]^2 + eps)
//   eq gate      z = (1/4) Σ_i inv_i (W_d^(i) (γ_i ⊙ R'_i)),  h = SiLU(z),  G = σ(W_u h)
//   eq use_gate  x = (1/4) Σ_i G_i ⊙ γ_i ⊙ inv_i R'_i
//   eq s         s = 2σ((1/4) Σ_i inv_i (W_w^(i) (γ_i ⊙ R'_i)))
// The projections are linear in R̂, so each branch's partial dot products are taken on the
// un-normalised row and scaled by inv_i afterwards.
#include "gr_internal.h"

namespace gr {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <typename W> __device__ __forceinline__ float wload(const W* p, size_t i) {
    return to_f32(p[i]);
}

// FOLDED: the packed W_d/W_w rows already carry gamma (bf16 path); otherwise multiply here.
template <typename T, typename W, bool FOLDED>
__global__ void __launch_bounds__(kThreads)
gr_generic_kernel(int64_t N, int D, int r, float eps, T* __restrict__ R,
                  const T* __restrict__ y, const float* __restrict__ s_prev,
                  const float* __restrict__ gamma, const W* __restrict__ wdw,
                  const W* __restrict__ wut, T* __restrict__ x, float* __restrict__ s_out) {
    extern __shared__ float smem[];
    const int K = kBranches * D;
    const int nout = r + kBranches;          // projection rows per branch: W_d then W_w
    float* Rs = smem;                         // [4][D] the (stored) state row, fp32
    float* part = Rs + K;                     // [4][nout] branch partial projections
    float* ssq = part + kBranches * nout;     // [4] sums of squares
    float* inv = ssq + kBranches;             // [4]
    float* h = inv + kBranches;               // [r]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int64_t t = blockIdx.x; t < N; t += gridDim.x) {
        T* Rt = R + t * K;
        // -- write (eq write), keep the stored value
        if (y != nullptr) {
            const float4 sv = *reinterpret_cast<const float4*>(s_prev + t * kBranches);
            const float sa[4] = {sv.x, sv.y, sv.z, sv.w};
            const T* yt = y + t * D;
            for (int e = tid; e < K; e += kThreads) {
                const int i = e / D, c = e - i * D;
                const float v = fmaf(sa[i], to_f32(yt[c]), to_f32(Rt[e]));
                const T st = from_f32<T>(v);
                Rt[e] = st;
                Rs[e] = to_f32(st);
            }
        } else {
            for (int e = tid; e < K; e += kThreads) Rs[e] = to_f32(Rt[e]);
        }
        if (x == nullptr) continue;  // write only (no shared state is reused across tokens)
        __syncthreads();

        // -- branch partials: one warp per (branch, row) dot product, plus sums of squares
        const int npairs = kBranches * nout + kBranches;
        for (int p = warp; p < npairs; p += kWarps) {
            float acc = 0.f;
            if (p < kBranches * nout) {
                const int i = p / nout, j = p - i * nout;
                const W* wrow = wdw + size_t(j) * K + size_t(i) * D;
                const float* ri = Rs + i * D;
                const float* gi = gamma + i * D;
                for (int c = lane; c < D; c += 32) {
                    float v = ri[c];
                    if (!FOLDED) v *= gi[c];
                    acc = fmaf(wload(wrow, c), v, acc);
                }
            } else {
                const float* ri = Rs + (p - kBranches * nout) * D;
                for (int c = lane; c < D; c += 32) acc = fmaf(ri[c], ri[c], acc);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) {
                if (p < kBranches * nout) part[p] = acc;
                else ssq[p - kBranches * nout] = acc;
            }
        }
        __syncthreads();
        if (tid < kBranches) inv[tid] = rsqrtf(ssq[tid] / float(D) + eps);
        __syncthreads();
        // -- bottleneck (eq gate) and write strengths (eq s)
        if (tid < nout) {
            float a = 0.f;
#pragma unroll
            for (int i = 0; i < kBranches; ++i) a = fmaf(inv[i], part[i * nout + tid], a);
            a *= 0.25f;
            if (tid < r) h[tid] = a * sigmoid_accurate(a);
            else s_out[t * kBranches + (tid - r)] = 2.0f * sigmoid_accurate(a);
        }
        __syncthreads();
        // -- up-projection, gates and combine (eq gate, eq use_gate)
        T* xt = x + t * D;
        for (int c = tid; c < D; c += kThreads) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < kBranches; ++i) {
                const int m = i * D + c;
                float g = 0.f;
                for (int k = 0; k < r; ++k) g = fmaf(wload(wut, size_t(k) * K + m), h[k], g);
                acc = fmaf(sigmoid_accurate(g) * gamma[m] * inv[i], Rs[m], acc);
            }
            xt[c] = from_f32<T>(0.25f * acc);
        }
        __syncthreads();
    }
}

template <typename T, typename W, bool FOLDED>
cudaError_t launch_t(int64_t N, int D, int r, float eps, void* R, const void* y,
                     const float* s_prev, const void* packed, void* x, float* s_out,
                     cudaStream_t st, int dtype) {
    const Layout L = make_layout(D, r, dtype);
    const char* base = static_cast<const char*>(packed);
    const size_t smem = sizeof(float) * (size_t(kBranches) * D + kBranches * (r + kBranches) +
                                         2 * kBranches + r);
    auto kern = gr_generic_kernel<T, W, FOLDED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    const int64_t cap = int64_t(sm_count()) * 4;
    const int grid = int(N < cap ? N : cap);
    kern<<<grid, kThreads, smem, st>>>(
        N, D, r, eps, static_cast<T*>(R), static_cast<const T*>(y), s_prev,
        reinterpret_cast<const float*>(base + L.gamma32),
        reinterpret_cast<const W*>(base + L.wdw), reinterpret_cast<const W*>(base + L.wut),
        static_cast<T*>(x), s_out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_generic(int64_t N, int D, int r, int dtype, float eps, void* R,
                           const void* y, const float* s_prev, const void* packed, void* x,
                           float* s_out, cudaStream_t st) {
    if (N == 0) return cudaSuccess;
    if (dtype == GR_BF16)
        return launch_t<__nv_bfloat16, __nv_bfloat16, true>(N, D, r, eps, R, y, s_prev, packed,
                                                            x, s_out, st, dtype);
    return launch_t<float, float, false>(N, D, r, eps, R, y, s_prev, packed, x, s_out, st,
                                         dtype);
}

}  // namespace gr
