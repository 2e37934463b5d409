// Internal declarations shared by the library's translation units (not part of the C ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gr.h"

namespace gr {

constexpr int kBranches = 4;

// Layout of the packed parameter buffer written by gr_pack_params. Every section starts on a
// 256-byte boundary. `w` is the weight element size (2 for bf16, 4 for fp32).
//   gamma32 : fp32 [4][D]                      gains, used by the combine
//   wdw     : W    [r+4][4D]                   rows 0..r-1 = W_d, rows r..r+3 = W_w
//                                              (gamma folded on the bf16 path)
//   wut     : W    [r][4D]                     W_u transposed
//   wu      : bf16 [4D][r], W_u as given (each channel's r weights contiguous): only for the
//             shapes of the large-rank tensor-core path (rank_tc_supported), else 0 bytes
//   frag    : bf16 path only: the mma fragments of the weights (and gains) in the layout of the
//             tensor-core kernel that serves the shape — per-CTA slices for the cluster kernel
//             (shapes fused_supported() accepts, laid out in gr_fused_bf16.cu), else per-chunk
//             fragments for the two-pass kernel (tiled_supported(), gr_tiled_bf16.cu); 0 bytes
//             when neither takes the shape
struct Layout {
    size_t gamma32, wdw, wut, frag, total;
    size_t frag_bytes;
    // bf16 shapes of the cluster kernel also carry the two-pass kernel's fragments, which the
    // two-pass kernel uses for the tokens it takes on the SMs the clusters leave idle
    size_t frag2, frag2_bytes;
    size_t wu, wu_bytes;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Fused-kernel support and the size of its fragment section (gr_fused_bf16.cu). The fused
// kernel also needs n_tokens <= fused_max_tokens().
bool fused_supported(int D, int r);
int64_t fused_max_tokens();
// CTAs of the cluster kernel that can be resident at once on the current device (clusters ×
// cluster size; 0 if it cannot be queried).
int fused_resident_ctas(int D, int r, bool write);
size_t fused_frag_bytes(int D, int r);

// Two-pass tensor-core kernel for the bf16 shapes the cluster kernel does not take
// (gr_tiled_bf16.cu). It also needs n_tokens <= tiled_max_tokens().
bool tiled_supported(int D, int r);
int64_t tiled_max_tokens();
size_t tiled_frag_bytes(int D, int r);
// Contribution decomposition at one reader (gr_decompose.cu): per token the writers' norms
// [N][U], optional per-branch norms [N][U][4] and fractions [N][U], and with R0 the initial
// state's share [N]. Parameters fp32 as in the backward; Y [U][N][D] in the state's dtype.
cudaError_t launch_decompose(int64_t N, int D, int r, float eps, int dtype, const void* R,
                             const float* gamma, const float* Wd, const float* Wu, int U,
                             const void* Y, const float* S, const void* R0, float* norm,
                             float* bnorm, float* pi, float* a0_norm, cudaStream_t st);

// Concurrent split of a bf16 cluster-kernel shape (gr_split.cu): the tokens of the step that go
// to the two-pass kernel (a multiple of 32; 0 = no split) and the SMs it gets (*free_sms).
int64_t split_tokens(int64_t N, int D, int r, bool write, int* free_sms);
// Tokens [0, N − n2) on the cluster kernel on st, [N − n2, N) on the two-pass kernel on an
// internal stream forked from st and joined back to it.
cudaError_t launch_split_bf16(int64_t N, int64_t n2, int free_sms, int D, int r, float eps,
                              void* R, const void* y, const float* s_prev, const void* packed,
                              void* x, float* s_out, cudaStream_t st);

// The two-pass kernel on an FP8 state also needs D % 128 == 0 and D <= 8192.
bool tiled_fp8_supported(int D, int r);

// Large-rank path on the tcgen05 tensor cores (gr_rank_tc.cu): bf16 states, D a multiple of 64,
// 64 <= r <= 448 with r a multiple of 8. It needs rank_tc_workspace(N, r) bytes of device
// workspace (inv [N][4] fp32, then h [N][rank_tc_padded(r)] bf16, each 256-byte aligned).
bool rank_tc_supported(int D, int r);
int rank_tc_padded(int r);
size_t rank_tc_workspace(int64_t N, int r);
cudaError_t launch_rank_tc(int64_t N, int D, int r, float eps, void* R, const void* y,
                           const float* s_prev, const void* packed, void* x, float* s_out,
                           void* workspace, cudaStream_t st);

inline Layout make_layout(int D, int r, int dtype) {
    Layout L{};
    const size_t K = size_t(kBranches) * D;
    const size_t w = dtype == GR_F32 ? 4 : 2;   // the FP8 path computes with bf16 weights
    size_t off = 0;
    L.gamma32 = off;
    off = align256(off + K * 4);
    L.wdw = off;
    off = align256(off + size_t(r + kBranches) * K * w);
    L.wut = off;
    off = align256(off + size_t(r) * K * w);
    L.frag_bytes = dtype == GR_F32                            ? 0
                   : dtype == GR_BF16 && fused_supported(D, r) ? fused_frag_bytes(D, r)
                   : tiled_supported(D, r)                     ? tiled_frag_bytes(D, r)
                                                               : 0;
    L.frag = off;
    off = align256(off + L.frag_bytes);
    L.frag2_bytes = (dtype == GR_BF16 && fused_supported(D, r) && tiled_supported(D, r))
                        ? tiled_frag_bytes(D, r)
                        : 0;
    L.frag2 = off;
    off = align256(off + L.frag2_bytes);
    L.wu_bytes = dtype == GR_BF16 && rank_tc_supported(D, r) ? size_t(r) * K * 2 : 0;
    L.wu = off;
    off = align256(off + L.wu_bytes);
    L.total = off;
    return L;
}

// ---- launchers (return a cudaError_t from the launch) --------------------------------------

// Pack fp32 parameters into `packed` following make_layout.
cudaError_t launch_pack(int D, int r, int dtype, const float* gamma, const float* wd,
                        const float* wu, const float* ww, void* packed, cudaStream_t st);

// Generic per-token kernel: optional write (y != nullptr) then optional read (x != nullptr).
cudaError_t launch_generic(int64_t N, int D, int r, int dtype, float eps, void* R,
                           const void* y, const float* s_prev, const void* packed, void* x,
                           float* s_out, cudaStream_t st);

// Fused bf16 tensor-core kernel (write then read, or read only when y == nullptr).
cudaError_t launch_fused_bf16(int64_t N, int D, int r, float eps, void* R, const void* y,
                              const float* s_prev, const void* packed, void* x, float* s_out,
                              cudaStream_t st);

// Two-pass bf16 tensor-core kernel (write then read, or read only when y == nullptr).
// max_ctas > 0 caps the grid (the SMs left to it); the fragments come from the section the
// packed buffer has for the two-pass kernel (frag, or frag2 on a cluster-kernel shape).
// programmatic: launched as the programmatic dependent of the preceding launch on `st` (it
// starts once that grid's CTAs are all resident, and finishes only after that grid).
cudaError_t launch_tiled_bf16(int64_t N, int D, int r, float eps, void* R, const void* y,
                              const float* s_prev, const void* packed, void* x, float* s_out,
                              cudaStream_t st, int max_ctas = 0, bool programmatic = false);

// The two-pass kernel on an FP8 state (codes [N][4][D], block exponents [N][4][D/32]); y and x
// bf16; read only when y == nullptr.
cudaError_t launch_tiled_fp8(int64_t N, int D, int r, float eps, uint8_t* codes,
                             uint8_t* scales, const void* y, const float* s_prev,
                             const void* packed, void* x, float* s_out, cudaStream_t st);

// FP8 state conversions and the streaming FP8 write (gr_fp8.cu); rows = N·4 for the state.
cudaError_t launch_fp8_encode(int64_t rows, int D, int in_dtype, const void* in, uint8_t* codes,
                              uint8_t* scales, cudaStream_t st);
cudaError_t launch_fp8_decode(int64_t rows, int D, int out_dtype, const uint8_t* codes,
                              const uint8_t* scales, void* out, cudaStream_t st);
cudaError_t launch_fp8_write(int64_t N, int D, uint8_t* codes, uint8_t* scales, const void* y,
                             const float* s, cudaStream_t st);

// Backward of the read and of the write (gr_backward.cu).
size_t read_backward_workspace(int64_t N, int D, int r);
cudaError_t launch_read_backward(int64_t N, int D, int r, float eps, int dtype, const void* R,
                                 const float* gamma, const float* Wd, const float* Wu,
                                 const float* Ww, const float* dx, const float* ds, float* dR,
                                 float* dgamma, float* dWd, float* dWu, float* dWw,
                                 void* workspace, cudaStream_t st);
cudaError_t launch_write_backward(int64_t N, int D, int dtype, const float* dRp, const void* y,
                                  const float* s, float* dR, float* dy, float* ds,
                                  cudaStream_t st);

// Streaming write R += s_i * y (no read).
cudaError_t launch_write(int64_t N, int D, int dtype, void* R, const void* y, const float* s,
                         cudaStream_t st);

// Combine with given gates.
cudaError_t launch_fixed_gates(int64_t N, int D, int dtype, float eps, const void* R,
                               const float* gamma, const float* G, void* x, cudaStream_t st);

// Single-stream x += y.
cudaError_t launch_residual_add(int64_t n, int dtype, const void* y, void* x, cudaStream_t st);

// Status bits recorded by device-side bounded waits, one word per kernel unit (0 = none; -1 =
// could not be read).
int fused_status(bool clear);
int tiled_status(bool clear);

// One bounded wait that nothing satisfies (gives up after limit_cycles and sets the status).
cudaError_t launch_wait_selftest(long long limit_cycles, cudaStream_t st);

// Number of SMs of the current device (cached per device).
int sm_count();

// ---- device helpers ------------------------------------------------------------------------

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Logistic function with the accurate expf (the fp32 path's 1e-5 budget).
__device__ __forceinline__ float sigmoid_accurate(float a) { return 1.0f / (1.0f + expf(-a)); }

}  // namespace gr
