// Streaming kernels: the standalone write, the fixed-gate combine, and the single-stream
// residual add used as the bandwidth reference.
#include "gr_internal.h"

namespace gr {

namespace {

constexpr int kThreads = 256;

// 8 state elements <-> fp32, for 16-byte (bf16) or 32-byte (fp32) vectors.
struct Vec8 {
    float v[8];
};

__device__ __forceinline__ Vec8 load8(const __nv_bfloat16* p) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    Vec8 r;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        r.v[2 * k] = __uint_as_float(w[k] << 16);
        r.v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
    return r;
}
__device__ __forceinline__ Vec8 load8(const float* p) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    return Vec8{{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w}};
}
// Loads of data this kernel also writes (no read-only cache path).
__device__ __forceinline__ Vec8 load8_rw(const __nv_bfloat16* p) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    Vec8 r;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        r.v[2 * k] = __uint_as_float(w[k] << 16);
        r.v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
    return r;
}
__device__ __forceinline__ Vec8 load8_rw(const float* p) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *(reinterpret_cast<const float4*>(p) + 1);
    return Vec8{{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w}};
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const Vec8& r) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(r.v[2 * k], r.v[2 * k + 1]);
        w[k] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void store8(float* p, const Vec8& r) {
    reinterpret_cast<float4*>(p)[0] = make_float4(r.v[0], r.v[1], r.v[2], r.v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(r.v[4], r.v[5], r.v[6], r.v[7]);
}

// eq write: R[t][i][c] += s[t][i] * y[t][c], 8 channels per thread and step.
template <typename T>
__global__ void __launch_bounds__(kThreads)
write_kernel(int64_t N, int D, T* __restrict__ R, const T* __restrict__ y,
             const float* __restrict__ s) {
    const int64_t row8 = int64_t(kBranches) * D / 8;  // 8-vectors per token
    const int64_t total = N * row8;
    const int d8 = D / 8;
    for (int64_t q = blockIdx.x * int64_t(kThreads) + threadIdx.x; q < total;
         q += int64_t(gridDim.x) * kThreads) {
        const int64_t t = q / row8;
        const int rem = int(q - t * row8);
        const int i = rem / d8, c8 = rem - i * d8;
        const float si = __ldg(s + t * kBranches + i);
        const Vec8 yv = load8(y + t * D + int64_t(c8) * 8);
        T* p = R + q * 8;
        Vec8 rv = load8_rw(p);
#pragma unroll
        for (int k = 0; k < 8; ++k) rv.v[k] = fmaf(si, yv.v[k], rv.v[k]);
        store8(p, rv);
    }
}

// x = (1/4) Σ_i G_i ⊙ RMSNorm(R_i; γ_i) with given G, one CTA per token.
template <typename T>
__global__ void __launch_bounds__(kThreads)
fixed_gates_kernel(int64_t N, int D, float eps, const T* __restrict__ R,
                   const float* __restrict__ gamma, const float* __restrict__ G,
                   T* __restrict__ x) {
    __shared__ float red[kThreads / 32][kBranches];
    __shared__ float inv[kBranches];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = kBranches * D;
    for (int64_t t = blockIdx.x; t < N; t += gridDim.x) {
        const T* Rt = R + t * K;
        float ss[kBranches] = {0.f, 0.f, 0.f, 0.f};
        for (int c = tid; c < D; c += kThreads) {
#pragma unroll
            for (int i = 0; i < kBranches; ++i) {
                const float v = to_f32(Rt[i * D + c]);
                ss[i] = fmaf(v, v, ss[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < kBranches; ++i) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], o);
            if (lane == 0) red[warp][i] = ss[i];
        }
        __syncthreads();
        if (tid < kBranches) {
            float a = 0.f;
            for (int w = 0; w < kThreads / 32; ++w) a += red[w][tid];
            inv[tid] = rsqrtf(a / float(D) + eps);
        }
        __syncthreads();
        for (int c = tid; c < D; c += kThreads) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < kBranches; ++i) {
                const int m = i * D + c;
                acc = fmaf(G[m] * gamma[m] * inv[i], to_f32(Rt[m]), acc);
            }
            x[t * D + c] = from_f32<T>(0.25f * acc);
        }
        __syncthreads();
    }
}

// x += y over n elements: 8-element vectors, then a scalar tail.
template <typename T>
__global__ void __launch_bounds__(kThreads)
residual_add_kernel(int64_t n, const T* __restrict__ y, T* __restrict__ x) {
    const int64_t n8 = n / 8;
    const int64_t stride = int64_t(gridDim.x) * kThreads;
    for (int64_t q = blockIdx.x * int64_t(kThreads) + threadIdx.x; q < n8; q += stride) {
        const Vec8 yv = load8(y + q * 8);
        Vec8 xv = load8_rw(x + q * 8);
#pragma unroll
        for (int k = 0; k < 8; ++k) xv.v[k] += yv.v[k];
        store8(x + q * 8, xv);
    }
    for (int64_t e = n8 * 8 + blockIdx.x * int64_t(kThreads) + threadIdx.x; e < n; e += stride)
        x[e] = from_f32<T>(to_f32(x[e]) + to_f32(y[e]));
}

int grid_for(int64_t work_items, int per_sm) {
    const int64_t want = (work_items + kThreads - 1) / kThreads;
    const int64_t cap = int64_t(sm_count()) * per_sm;
    return int(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_write(int64_t N, int D, int dtype, void* R, const void* y, const float* s,
                         cudaStream_t st) {
    if (N == 0) return cudaSuccess;
    const int grid = grid_for(N * kBranches * D / 8, 8);
    if (dtype == GR_BF16)
        write_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
            N, D, static_cast<__nv_bfloat16*>(R), static_cast<const __nv_bfloat16*>(y), s);
    else
        write_kernel<float><<<grid, kThreads, 0, st>>>(N, D, static_cast<float*>(R),
                                                       static_cast<const float*>(y), s);
    return cudaGetLastError();
}

cudaError_t launch_fixed_gates(int64_t N, int D, int dtype, float eps, const void* R,
                               const float* gamma, const float* G, void* x, cudaStream_t st) {
    if (N == 0) return cudaSuccess;
    const int64_t cap = int64_t(sm_count()) * 8;
    const int grid = int(N < cap ? N : cap);
    if (dtype == GR_BF16)
        fixed_gates_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
            N, D, eps, static_cast<const __nv_bfloat16*>(R), gamma, G,
            static_cast<__nv_bfloat16*>(x));
    else
        fixed_gates_kernel<float><<<grid, kThreads, 0, st>>>(
            N, D, eps, static_cast<const float*>(R), gamma, G, static_cast<float*>(x));
    return cudaGetLastError();
}

cudaError_t launch_residual_add(int64_t n, int dtype, const void* y, void* x, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int grid = grid_for(n / 8 + 1, 8);
    if (dtype == GR_BF16)
        residual_add_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
            n, static_cast<const __nv_bfloat16*>(y), static_cast<__nv_bfloat16*>(x));
    else
        residual_add_kernel<float><<<grid, kThreads, 0, st>>>(
            n, static_cast<const float*>(y), static_cast<float*>(x));
    return cudaGetLastError();
}

}  // namespace gr
