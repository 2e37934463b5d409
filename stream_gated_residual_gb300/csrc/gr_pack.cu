// Packing of one GR module's parameters into the kernels' layout (gr_pack_params).
//
// Shapes from "【论文解读】 Qwen3.8 Flash Next", §二.4: gamma_i ∈ R^d per branch (eq rms),
// W_d ∈ R^{r×n_r·d}, W_u ∈ R^{n_r·d×r} (eq gate), W_w ∈ R^{n_r×n_r·d} (eq s).
#include "gr_internal.h"

namespace gr {

namespace {

template <typename W> __device__ __forceinline__ void put(W* p, size_t i, float v);
template <> __device__ __forceinline__ void put<float>(float* p, size_t i, float v) { p[i] = v; }
template <> __device__ __forceinline__ void put<__nv_bfloat16>(__nv_bfloat16* p, size_t i, float v) {
    p[i] = __float2bfloat16_rn(v);
}

// gamma32 copy, wdw = [W_d; W_w] (gamma folded when FOLD), wut = W_uᵀ.
template <typename W, bool FOLD>
__global__ void pack_generic_kernel(int D, int r, const float* __restrict__ gamma,
                                    const float* __restrict__ wd, const float* __restrict__ wu,
                                    const float* __restrict__ ww, float* __restrict__ gamma32,
                                    W* __restrict__ wdw, W* __restrict__ wut) {
    const size_t K = size_t(kBranches) * D;
    const size_t n_gamma = K;
    const size_t n_wdw = size_t(r + kBranches) * K;
    const size_t n_wut = size_t(r) * K;
    const size_t total = n_gamma + n_wdw + n_wut;
    for (size_t e = blockIdx.x * size_t(blockDim.x) + threadIdx.x; e < total;
         e += size_t(gridDim.x) * blockDim.x) {
        if (e < n_gamma) {
            gamma32[e] = gamma[e];
        } else if (e < n_gamma + n_wdw) {
            const size_t q = e - n_gamma;
            const size_t j = q / K, m = q % K;
            float v = j < size_t(r) ? wd[j * K + m] : ww[(j - r) * K + m];
            if (FOLD) v *= gamma[m];
            put<W>(wdw, q, v);
        } else {
            const size_t q = e - n_gamma - n_wdw;
            const size_t k = q / K, m = q % K;
            put<W>(wut, q, wu[m * size_t(r) + k]);
        }
    }
}

// W_u as given ([4D][r], each channel's r weights contiguous), rounded to bf16: the B operand of
// the large-rank path's up projection.
__global__ void pack_wu_kernel(size_t n, const float* __restrict__ wu,
                               __nv_bfloat16* __restrict__ out) {
    for (size_t e = blockIdx.x * size_t(blockDim.x) + threadIdx.x; e < n;
         e += size_t(gridDim.x) * blockDim.x)
        out[e] = __float2bfloat16_rn(wu[e]);
}

}  // namespace

// Fragment sections of the cluster kernel (gr_fused_bf16.cu) and the two-pass kernel
// (gr_tiled_bf16.cu).
cudaError_t launch_pack_fused(int D, int r, const float* gamma, const float* wd, const float* wu,
                              const float* ww, void* frag, cudaStream_t st);
cudaError_t launch_pack_tiled(int D, int r, const float* gamma, const float* wd, const float* wu,
                              const float* ww, void* frag, cudaStream_t st);

cudaError_t launch_pack(int D, int r, int dtype, const float* gamma, const float* wd,
                        const float* wu, const float* ww, void* packed, cudaStream_t st) {
    const Layout L = make_layout(D, r, dtype);
    char* base = static_cast<char*>(packed);
    const size_t K = size_t(kBranches) * D;
    const size_t total = K * size_t(2 * r + kBranches + 1);
    const int threads = 256;
    const size_t want = (total + threads - 1) / threads;
    const size_t cap = size_t(sm_count()) * 8;
    const int blocks = int(want < cap ? want : cap);
    float* g32 = reinterpret_cast<float*>(base + L.gamma32);
    if (dtype != GR_F32) {   // bf16 weights, gamma folded (the bf16 and FP8 paths)
        pack_generic_kernel<__nv_bfloat16, true><<<blocks, threads, 0, st>>>(
            D, r, gamma, wd, wu, ww, g32, reinterpret_cast<__nv_bfloat16*>(base + L.wdw),
            reinterpret_cast<__nv_bfloat16*>(base + L.wut));
    } else {
        pack_generic_kernel<float, false><<<blocks, threads, 0, st>>>(
            D, r, gamma, wd, wu, ww, g32, reinterpret_cast<float*>(base + L.wdw),
            reinterpret_cast<float*>(base + L.wut));
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (L.frag2_bytes) {
        e = launch_pack_tiled(D, r, gamma, wd, wu, ww, base + L.frag2, st);
        if (e != cudaSuccess) return e;
    }
    if (L.wu_bytes) {
        pack_wu_kernel<<<blocks, threads, 0, st>>>(size_t(r) * K, wu,
                                                    reinterpret_cast<__nv_bfloat16*>(base + L.wu));
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (L.frag_bytes) {
        e = dtype == GR_BF16 && fused_supported(D, r)
                ? launch_pack_fused(D, r, gamma, wd, wu, ww, base + L.frag, st)
                : launch_pack_tiled(D, r, gamma, wd, wu, ww, base + L.frag, st);
    }
    return e;
}

}  // namespace gr
