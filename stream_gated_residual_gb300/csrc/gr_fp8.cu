// FP8 branch state: encoding, decoding and the streaming write.
//
// The pages name FP8 storage of the widened state ("【论文解读】 Qwen3.8 Flash Next", §二.7) and
// leave the format open. The library's format: e4m3 codes [N][4][D]
// and one biased power-of-two exponent per 32 consecutive channels of a (token, branch) row,
// scales [N][4][D/32], scale 2^(b - 127); a block's exponent is the smallest e with
// max|v| <= 448·2^e, and codes are v/2^e rounded to the nearest e4m3 value, ties to even.
//
// One thread handles 8 channels; the four threads of a quad hold one 32-channel block, so the
// block maximum is two shuffles.
#include <cuda_fp16.h>

#include "gr_internal.h"
#include "gr_ptx.cuh"

namespace gr {
namespace {

constexpr int kThreads = 256;

template <typename T> struct In8;
template <> struct In8<__nv_bfloat16> {
    __device__ static void load(const __nv_bfloat16* p, float (&v)[8]) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __uint_as_float(w[k] << 16);
            v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    }
    __device__ static void store(__nv_bfloat16* p, const float (&v)[8]) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) w[k] = pack_bf2(v[2 * k], v[2 * k + 1]);
        *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <> struct In8<float> {
    __device__ static void load(const float* p, float (&v)[8]) {
        const float4 a = reinterpret_cast<const float4*>(p)[0];
        const float4 b = reinterpret_cast<const float4*>(p)[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
    __device__ static void store(float* p, const float (&v)[8]) {
        reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
};

// 8 values -> 8 codes of their block (the quad's shared exponent e) as one 8-byte word.
__device__ __forceinline__ uint2 encode8(const float (&v)[8], int e) {
    const float inv = pow2f(-e);
    uint32_t w[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint32_t lo = f2_to_e4m3x2(v[4 * k] * inv, v[4 * k + 1] * inv);
        const uint32_t hi = f2_to_e4m3x2(v[4 * k + 2] * inv, v[4 * k + 3] * inv);
        w[k] = lo | (hi << 16);
    }
    return make_uint2(w[0], w[1]);
}
__device__ __forceinline__ void decode8(uint2 c, int e, float (&v)[8]) {
    const float sc = pow2f(e);
    const uint32_t w[2] = {c.x, c.y};
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const float2 a = e4m3x2_to_f2(uint16_t(w[k] & 0xffffu));
        const float2 b = e4m3x2_to_f2(uint16_t(w[k] >> 16));
        v[4 * k] = a.x * sc;
        v[4 * k + 1] = a.y * sc;
        v[4 * k + 2] = b.x * sc;
        v[4 * k + 3] = b.y * sc;
    }
}
// Largest magnitude over the quad's 32 values (every lane of the warp takes part).
__device__ __forceinline__ float quad_amax(const float (&v)[8]) {
    float a = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) a = fmaxf(a, fabsf(v[k]));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    return a;
}

// Grid-stride over 8-channel items of `rows` rows of D channels; every lane of a warp runs the
// same number of iterations (the shuffles need the whole warp), items past the end idle.
#define GR_FP8_ITEMS(rows, D)                                                              \
    const int64_t n_items = int64_t(rows) * (D / 8);                                       \
    const int64_t stride = int64_t(gridDim.x) * kThreads;                                  \
    for (int64_t base = int64_t(blockIdx.x) * kThreads + (threadIdx.x & ~31);               \
         base < n_items; base += stride)

// Encode a state (bf16 or fp32 values) into codes and block exponents.
template <typename T>
__global__ void __launch_bounds__(kThreads)
fp8_encode_kernel(int64_t rows, int D, const T* __restrict__ in, uint8_t* __restrict__ codes,
                  uint8_t* __restrict__ scales) {
    const int lane = threadIdx.x & 31;
    GR_FP8_ITEMS(rows, D) {
        const int64_t it = base + lane;
        const bool on = it < n_items;
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (on) In8<T>::load(in + it * 8, v);
        const int e = fp8_block_exp(quad_amax(v));
        if (on) {
            reinterpret_cast<uint2*>(codes)[it] = encode8(v, e);
            if ((lane & 3) == 0) scales[it / 4] = uint8_t(e + 127);
        }
    }
}

// Decode codes and block exponents into bf16 or fp32 values.
template <typename T>
__global__ void __launch_bounds__(kThreads)
fp8_decode_kernel(int64_t rows, int D, const uint8_t* __restrict__ codes,
                  const uint8_t* __restrict__ scales, T* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    GR_FP8_ITEMS(rows, D) {
        const int64_t it = base + lane;
        if (it < n_items) {
            float v[8];
            decode8(reinterpret_cast<const uint2*>(codes)[it], int(scales[it / 4]) - 127, v);
            In8<T>::store(out + it * 8, v);
        }
    }
}

// eq write on an FP8 state: decode R, R' = R + s·y as one fp32 FMA per element (y bf16),
// encode R' with new block exponents, in place.
__global__ void __launch_bounds__(kThreads)
fp8_write_kernel(int64_t N, int D, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                 const __nv_bfloat16* __restrict__ y, const float* __restrict__ s) {
    const int lane = threadIdx.x & 31;
    const int d8 = D / 8;
    GR_FP8_ITEMS(N * kBranches, D) {
        const int64_t it = base + lane;
        const bool on = it < n_items;
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (on) {
            const int64_t row = it / d8;                  // token * 4 + branch
            const int c8 = int(it - row * d8);
            const int64_t t = row / kBranches;
            decode8(reinterpret_cast<const uint2*>(codes)[it], int(scales[it / 4]) - 127, v);
            float yv[8];
            In8<__nv_bfloat16>::load(y + t * D + int64_t(c8) * 8, yv);
            const float si = __ldg(s + row);
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = fmaf(si, yv[k], v[k]);
        }
        const int e = fp8_block_exp(quad_amax(v));
        if (on) {
            reinterpret_cast<uint2*>(codes)[it] = encode8(v, e);
            if ((lane & 3) == 0) scales[it / 4] = uint8_t(e + 127);
        }
    }
}
#undef GR_FP8_ITEMS

int grid_for(int64_t items) {
    const int64_t want = (items + kThreads - 1) / kThreads;
    const int64_t cap = int64_t(sm_count()) * 8;
    return int(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_fp8_encode(int64_t rows, int D, int in_dtype, const void* in, uint8_t* codes,
                              uint8_t* scales, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    const int grid = grid_for(rows * (D / 8));
    if (in_dtype == GR_BF16)
        fp8_encode_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
            rows, D, static_cast<const __nv_bfloat16*>(in), codes, scales);
    else
        fp8_encode_kernel<float><<<grid, kThreads, 0, st>>>(
            rows, D, static_cast<const float*>(in), codes, scales);
    return cudaGetLastError();
}

cudaError_t launch_fp8_decode(int64_t rows, int D, int out_dtype, const uint8_t* codes,
                              const uint8_t* scales, void* out, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    const int grid = grid_for(rows * (D / 8));
    if (out_dtype == GR_BF16)
        fp8_decode_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
            rows, D, codes, scales, static_cast<__nv_bfloat16*>(out));
    else
        fp8_decode_kernel<float><<<grid, kThreads, 0, st>>>(rows, D, codes, scales,
                                                            static_cast<float*>(out));
    return cudaGetLastError();
}

cudaError_t launch_fp8_write(int64_t N, int D, uint8_t* codes, uint8_t* scales, const void* y,
                             const float* s, cudaStream_t st) {
    if (N == 0) return cudaSuccess;
    const int grid = grid_for(N * kBranches * (D / 8));
    fp8_write_kernel<<<grid, kThreads, 0, st>>>(N, D, codes, scales,
                                                static_cast<const __nv_bfloat16*>(y), s);
    return cudaGetLastError();
}

}  // namespace gr
