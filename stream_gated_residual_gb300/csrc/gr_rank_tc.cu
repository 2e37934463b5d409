// The read at the pages' own rank, r = d/8 ("【论文解读】 Qwen3.8 Flash Next", §二.4: W_d is
// r × n_r·d with r = d/8), on the 5th-generation tensor cores (tcgen05, accumulators in tensor
// memory, operands staged by TMA). At r in the hundreds the read is a dense contraction of about
// 4·r·4D flops a token, as much arithmetic as memory traffic, so the projections run as two
// GEMMs and everything else rides in their prologue and epilogue:
//
//   1. rownorm_kernel   eq write (R' = R + s_prev·y, stored bf16, as gr_write computes it) and
//                       the stored row's inv_i = 1/√(mean R'_i² + eps) into the workspace;
//                       one warp per (token, branch) row.
//   2. down_tc_kernel   [z | u] = [W_d; W_w]·γ ⊙ vec(R' ⊙ inv) for 128 tokens a CTA: TMA brings
//                       R' and the packed bf16 rows of [W_d; W_w] (γ folded) 64 channels at a
//                       time; four warps scale their token rows of each R' stage by inv_i in
//                       shared memory (eq rms), split into bf16 hi + lo; one thread issues the
//                       MMAs of both halves into a 128 × (r+4) fp32 accumulator in tensor memory;
//                       the epilogue writes h = SiLU(z/4) as bf16 into the workspace and
//                       s = 2σ(u/4) (eq gate, eq s).
//   3. up_tc_kernel     g = W_u h for 128 tokens × 4 branches × 32 channels a step (eq gate), two
//                       accumulators in tensor memory so the MMAs of one channel block overlap
//                       the epilogue of the previous one; the epilogue forms G = σ(g) and
//                       x = ¼ Σ_i G_i γ_i inv_i R'_i from a TMA copy of the block's R' (eq
//                       use_gate).
//
// Warp roles of both GEMM kernels (192 threads): warp 0 issues the TMA loads, warp 1 owns the
// tensor memory and issues the MMAs, warps 2-5 (one per tensor-memory lane quadrant) scale and
// run the epilogue. Every mbarrier wait is bounded; a wait that runs out records a status bit
// and the kernel finishes without the work.
#include <math.h>

#include "gr_internal.h"
#include "gr_ptx.cuh"
#include "gr_tc.cuh"

namespace gr {
namespace {

constexpr int kTile = 128;          // tokens per CTA: the MMA's M
constexpr int kKc = 64;             // K elements per operand stage (128-byte rows)
constexpr int kStageA = kTile * 128; // one 128-token × 64-channel bf16 stage
constexpr int kGemmThreads = 192;   // down projection: producer, MMA, 4 scaling/epilogue warps
constexpr int kUpThreads = 352;     // up projection: producer, MMA, 8 epilogue warps, R' loader
constexpr int kUpEpiWarps = 8;      // two per tensor-memory lane quadrant, 16 channels each
constexpr int kCb = 32;             // channels per branch in an up-projection block
constexpr int kMaxRankTc = 448;     // r + 4 <= 512 accumulator columns; H fits shared memory

__device__ __forceinline__ float sigm(float a) { return 1.0f / (1.0f + __expf(-a)); }
// σ(a) = ½ + ½·tanh(a/2) on the MUFU tanh (the combine's gates, as the other tensor-core paths)
__device__ __forceinline__ float sigm_fast(float a) {
    return fmaf(0.5f, tanh_approx(0.5f * a), 0.5f);
}

// ---- 1. eq write and the stored row's 1/rms --------------------------------------------------
__global__ void __launch_bounds__(256)
rownorm_kernel(int64_t N, int D, float eps, __nv_bfloat16* __restrict__ R,
               const __nv_bfloat16* __restrict__ y, const float* __restrict__ s_prev,
               float* __restrict__ inv) {
    const int lane = threadIdx.x & 31;
    const int64_t rows = N * kBranches;
    const int d8 = D / 8;
    for (int64_t row = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5); row < rows;
         row += int64_t(gridDim.x) * 8) {
        const int64_t t = row / kBranches;
        uint4* Rr = reinterpret_cast<uint4*>(R + row * D);
        const uint4* yr = y ? reinterpret_cast<const uint4*>(y + t * D) : nullptr;
        const float s = y ? s_prev[row] : 0.f;
        float ss = 0.f;
        for (int c = lane; c < d8; c += 32) {
            uint4 q = Rr[c];
            uint32_t w[4] = {q.x, q.y, q.z, q.w};
            if (y) {
                const uint4 yq = __ldg(yr + c);
                const uint32_t yw[4] = {yq.x, yq.y, yq.z, yq.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float lo = fmaf(s, __uint_as_float(yw[k] << 16),
                                          __uint_as_float(w[k] << 16));
                    const float hi = fmaf(s, __uint_as_float(yw[k] & 0xffff0000u),
                                          __uint_as_float(w[k] & 0xffff0000u));
                    w[k] = pack_bf2(lo, hi);
                }
                Rr[c] = make_uint4(w[0], w[1], w[2], w[3]);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float lo = __uint_as_float(w[k] << 16);
                const float hi = __uint_as_float(w[k] & 0xffff0000u);
                ss = fmaf(lo, lo, fmaf(hi, hi, ss));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) inv[row] = rsqrtf(ss / float(D) + eps);
    }
}

// ---- 2. down projection --------------------------------------------------------------------
// Shared memory: `stages` × {A_hi, A_lo: 128 rows × 128 B each, B: n1 rows × 128 B}, then the
// barriers. The state rows arrive in A_hi; the scaling warps leave hi = bf16(R'·inv) there and the
// rounding residual lo = bf16(R'·inv − hi) in A_lo, and both go through the MMA (the split keeps
// the down projection's inputs to about 2^-16 relative instead of bf16's 2^-8).
__host__ __device__ inline size_t down_stage_bytes(int n1) {
    return 2 * kStageA + size_t(n1) * 128;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
down_tc_kernel(const __grid_constant__ CUtensorMap tmR, const __grid_constant__ CUtensorMap tmW,
               int64_t N, int D, int r, int n1,
               int stages, const float* __restrict__ inv, __nv_bfloat16* __restrict__ h, int rp,
               float* __restrict__ s_out) {
    extern __shared__ uint8_t smraw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) &
                                             ~uintptr_t(1023));
    const size_t sb = down_stage_bytes(n1);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + stages * sb);
    uint64_t* scaled = full + 4;
    uint64_t* empty = scaled + 4;
    uint64_t* acc_full = empty + 4;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(acc_full + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = int64_t(blockIdx.x) * kTile;
    const int nk = kBranches * D / kKc, cpb = D / kKc;
    const uint32_t ncols = n1 > 256 ? 512 : 256;

    if (threadIdx.x == 0) {
        for (int s = 0; s < 4; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&scaled[s], 4);
            mbar_init(&empty[s], 1);   // the MMAs are done with the stage
        }
        mbar_init(acc_full, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(tslot, ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        if (lane == 0) {
            const uint32_t bytes = uint32_t(kStageA + size_t(n1) * 128);   // what TMA brings
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % stages;
                if (kc >= stages && !mbar_wait(&empty[s], ((kc / stages) - 1) & 1)) break;
                uint8_t* A = sm + s * sb;
                uint8_t* B = A + 2 * kStageA;
                const int half = n1 / 2;   // a box holds at most 256 rows: two boxes
                mbar_expect_tx(&full[s], bytes);
                tma_load_3d(A, &tmR, (kc % cpb) * kKc, kc / cpb, int(t0), &full[s]);
                tma_load_2d(B, &tmW, kc * kKc, 0, &full[s]);
                tma_load_2d(B + half * 128, &tmW, kc * kKc, half, &full[s]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t id0 = idesc_bf16_f32(kTile, n1 > 256 ? 256 : n1);
            const uint32_t id1 = idesc_bf16_f32(kTile, n1 > 256 ? n1 - 256 : 16);
            bool ok = true;
            for (int kc = 0; kc < nk && ok; ++kc) {
                const int s = kc % stages;
                // the stage's TMA bytes (weights too) and the scaled state rows
                ok = mbar_wait(&full[s], (kc / stages) & 1) &&
                     mbar_wait(&scaled[s], (kc / stages) & 1);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a = smem_u32(sm + s * sb), b = a + 2 * kStageA;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t acc = (kc | kk) != 0;
                    const uint64_t ah = sdesc_sw128(a + kk * 32);
                    const uint64_t al = sdesc_sw128(a + kStageA + kk * 32);
                    const uint64_t b0 = sdesc_sw128(b + kk * 32);
                    tc_mma(tmem, ah, b0, id0, acc);
                    tc_mma(tmem, al, b0, id0, 1u);
                    if (n1 > 256) {
                        const uint64_t b1 = sdesc_sw128(b + 256 * 128 + kk * 32);
                        tc_mma(tmem + 256, ah, b1, id1, acc);
                        tc_mma(tmem + 256, al, b1, id1, 1u);
                    }
                }
                tc_commit(&empty[s]);
            }
            if (ok) tc_commit(acc_full);
        }
    } else {
        // warps 2-5: lane quadrant q; thread row = token t0 + 32q + lane
        const int q = warp & 3, row = q * 32 + lane;
        const int64_t t = t0 + row;
        float iv[kBranches];
#pragma unroll
        for (int i = 0; i < kBranches; ++i) iv[i] = t < N ? inv[t * kBranches + i] : 0.f;
        bool ok = true;
        for (int kc = 0; kc < nk && ok; ++kc) {
            const int s = kc % stages;
            ok = mbar_wait(&full[s], (kc / stages) & 1);
            if (!ok) break;
            const int i = kc / cpb;
            const float m = i == 0 ? iv[0] : i == 1 ? iv[1] : i == 2 ? iv[2] : iv[3];
            uint8_t* rp8 = sm + s * sb + row * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                // logical chunk j sits at j ^ (row & 7): eight rows hit eight bank groups
                const int off = (j ^ (row & 7)) * 16;
                uint4* p = reinterpret_cast<uint4*>(rp8 + off);
                const uint4 v = *p;
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float a0 = __uint_as_float(w[k] << 16) * m;
                    const float a1 = __uint_as_float(w[k] & 0xffff0000u) * m;
                    hi[k] = pack_bf2(a0, a1);
                    lo[k] = pack_bf2(a0 - __uint_as_float(hi[k] << 16),
                                     a1 - __uint_as_float(hi[k] & 0xffff0000u));
                }
                *p = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(rp8 + kStageA + off) =
                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&scaled[s]);
        }
        // epilogue: h = SiLU(z/4) (bf16, zero in the padding up to rp), s = 2σ(u/4)
        if (ok) ok = mbar_wait(acc_full, 0);
        tc_fence_after();
        if (ok) {
            const int ncol = n1 > rp ? n1 : rp;
            for (int c0 = 0; c0 < ncol; c0 += 16) {
                float v[16];
                if (c0 < n1) {
                    tmem_ld16(tmem + (uint32_t(q * 32) << 16) + c0, v);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = 0.f;
                }
                if (t >= N) continue;
                float hv[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int col = c0 + j;
                    const float z = 0.25f * v[j];
                    hv[j] = col < r ? z * sigm(z) : 0.f;
                    if (col >= r && col < r + kBranches)
                        s_out[t * kBranches + (col - r)] = 2.0f * sigm(z);
                }
                if (c0 < rp) {
                    uint4* hp = reinterpret_cast<uint4*>(h + t * rp + c0);
                    hp[0] = make_uint4(pack_bf2(hv[0], hv[1]), pack_bf2(hv[2], hv[3]),
                                       pack_bf2(hv[4], hv[5]), pack_bf2(hv[6], hv[7]));
                    hp[1] = make_uint4(pack_bf2(hv[8], hv[9]), pack_bf2(hv[10], hv[11]),
                                       pack_bf2(hv[12], hv[13]), pack_bf2(hv[14], hv[15]));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

// ---- 3. up projection, gate and combine ------------------------------------------------------
// Shared memory: H (rp/64 stages of 128 × 128 B), nbs B stages (4 branches × 32 rows × 128 B),
// nrb R' blocks (4 branches × 128 tokens × 32 channels bf16), then the barriers. A warp of its
// own streams the R' blocks, up to nrb ahead of the epilogue, so that their HBM latency hides
// behind the blocks before.
constexpr int kUpMaxStages = 6;     // each CTA streams all of W_u: bytes in flight set its rate
constexpr int kUpMaxR = 2;
constexpr int kStageB = kBranches * kCb * 128;                 // 16 KB
constexpr int kRBlock = kBranches * kTile * kCb * 2;           // 32 KB
__host__ __device__ inline size_t up_smem_bytes(int rp, int nbs, int nrb) {
    return size_t(rp / kKc) * kStageA + size_t(nbs) * kStageB + size_t(nrb) * kRBlock + 256;
}

__global__ void __launch_bounds__(kUpThreads, 1)
up_tc_kernel(const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmU,
             const __grid_constant__ CUtensorMap tmR, int64_t N, int D, int rp, int nbs, int nrb,
             const float* __restrict__ gamma, const float* __restrict__ inv,
             __nv_bfloat16* __restrict__ x) {
    extern __shared__ uint8_t smraw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) &
                                             ~uintptr_t(1023));
    const int nkc = rp / kKc;
    uint8_t* H = sm;
    uint8_t* Bs = H + size_t(nkc) * kStageA;
    uint8_t* Rb = Bs + size_t(nbs) * kStageB;
    uint64_t* h_full = reinterpret_cast<uint64_t*>(Rb + size_t(nrb) * kRBlock);
    uint64_t* b_full = h_full + 1;
    uint64_t* b_empty = b_full + kUpMaxStages;
    uint64_t* r_full = b_empty + kUpMaxStages;
    uint64_t* r_empty = r_full + kUpMaxR;
    uint64_t* t_full = r_empty + kUpMaxR;
    uint64_t* t_empty = t_full + 2;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(t_empty + 2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = int64_t(blockIdx.x) * kTile;
    const int nb = D / kCb;

    if (threadIdx.x == 0) {
        mbar_init(h_full, 1);
        for (int s = 0; s < kUpMaxStages; ++s) {
            mbar_init(&b_full[s], 1);
            mbar_init(&b_empty[s], 1);
        }
        for (int b = 0; b < kUpMaxR; ++b) {
            mbar_init(&r_full[b], 1);
            mbar_init(&r_empty[b], kUpEpiWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&t_full[b], 1);
            mbar_init(&t_empty[b], kUpEpiWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(tslot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        if (lane == 0) {
            mbar_expect_tx(h_full, uint32_t(nkc) * kStageA);
            for (int kc = 0; kc < nkc; ++kc)
                tma_load_2d(H + kc * kStageA, &tmH, kc * kKc, int(t0), h_full);
            int it = 0;
            for (int cb = 0; cb < nb; ++cb) {
                bool ok = true;
                for (int kc = 0; kc < nkc; ++kc, ++it) {
                    const int s = it % nbs;
                    if (it >= nbs && !mbar_wait(&b_empty[s], ((it / nbs) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&b_full[s], kStageB);
                    for (int i = 0; i < kBranches; ++i)
                        tma_load_2d(Bs + s * kStageB + i * (kCb * 128), &tmU, kc * kKc,
                                    i * D + cb * kCb, &b_full[s]);
                }
                if (!ok) break;
            }
        }
    } else if (warp == 2 + kUpEpiWarps) {
        // the R' blocks of the combine, up to nrb ahead
        if (lane == 0) {
            for (int cb = 0; cb < nb; ++cb) {
                const int rb = cb % nrb;
                if (cb >= nrb && !mbar_wait(&r_empty[rb], ((cb / nrb) - 1) & 1)) break;
                mbar_expect_tx(&r_full[rb], kRBlock);
                for (int i = 0; i < kBranches; ++i)
                    tma_load_3d(Rb + rb * kRBlock + i * (kTile * kCb * 2), &tmR, cb * kCb, i,
                                int(t0), &r_full[rb]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t id = idesc_bf16_f32(kTile, kBranches * kCb);
            bool ok = mbar_wait(h_full, 0);
            int it = 0;
            for (int cb = 0; cb < nb && ok; ++cb) {
                const int buf = cb & 1;
                if (cb >= 2) ok = mbar_wait(&t_empty[buf], ((cb >> 1) - 1) & 1);
                if (!ok) break;
                tc_fence_after();
                for (int kc = 0; kc < nkc; ++kc, ++it) {
                    const int s = it % nbs;
                    ok = mbar_wait(&b_full[s], (it / nbs) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t a = smem_u32(H + kc * kStageA);
                    const uint32_t b = smem_u32(Bs + s * kStageB);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma(tmem + buf * (kBranches * kCb), sdesc_sw128(a + kk * 32),
                               sdesc_sw128(b + kk * 32), id, (kc | kk) != 0);
                    tc_commit(&b_empty[s]);
                }
                if (ok) tc_commit(&t_full[buf]);
            }
        }
    } else {
        // warps 2-9: lane quadrant q = warp % 4, channel half hh of each 32-channel block
        const int q = warp & 3, hh = (warp - 2) >> 2, row = q * 32 + lane;
        constexpr int kH = kCb / 2;   // 16 channels a warp
        const int64_t t = t0 + row;
        float iv[kBranches];
#pragma unroll
        for (int i = 0; i < kBranches; ++i) iv[i] = t < N ? inv[t * kBranches + i] : 0.f;
        bool ok = true;
        for (int cb = 0; cb < nb && ok; ++cb) {
            const int buf = cb & 1;
            const int rb = cb % nrb;
            ok = mbar_wait(&t_full[buf], (cb >> 1) & 1) && mbar_wait(&r_full[rb], (cb / nrb) & 1);
            if (!ok) break;
            tc_fence_after();
            // the four branches' 16 logits of this row, in flight together
            uint32_t g[kBranches][kH];
            const uint32_t ta = tmem + (uint32_t(q * 32) << 16) + buf * (kBranches * kCb) + hh * kH;
#pragma unroll
            for (int i = 0; i < kBranches; ++i) tmem_ld16_nowait(ta + i * kCb, g[i]);
#pragma unroll
            for (int i = 0; i < kBranches; ++i) tmem_wait_ld(g[i]);
            float acc[kH];
#pragma unroll
            for (int c = 0; c < kH; ++c) acc[c] = 0.f;
#pragma unroll
            for (int i = 0; i < kBranches; ++i) {
                const uint4* rr = reinterpret_cast<const uint4*>(
                    Rb + rb * kRBlock + i * (kTile * kCb * 2) + row * (kCb * 2) + hh * (kH * 2));
                const float4* gm =
                    reinterpret_cast<const float4*>(gamma + size_t(i) * D + cb * kCb + hh * kH);
                const float m = iv[i];
#pragma unroll
                for (int v8 = 0; v8 < kH / 8; ++v8) {
                    const uint4 u = rr[v8];
                    const float4 ga = __ldg(gm + 2 * v8), gb = __ldg(gm + 2 * v8 + 1);
                    const float gv[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int c = v8 * 8 + 2 * k;
                        acc[c] = fmaf(sigm_fast(__uint_as_float(g[i][c])) * gv[2 * k] * m,
                                      __uint_as_float(w[k] << 16), acc[c]);
                        acc[c + 1] =
                            fmaf(sigm_fast(__uint_as_float(g[i][c + 1])) * gv[2 * k + 1] * m,
                                 __uint_as_float(w[k] & 0xffff0000u), acc[c + 1]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&t_empty[buf]);
                mbar_arrive(&r_empty[rb]);
            }
            if (t < N) {
                uint4* xp = reinterpret_cast<uint4*>(x + t * D + cb * kCb + hh * kH);
#pragma unroll
                for (int v8 = 0; v8 < kH / 8; ++v8) {
                    const int c = v8 * 8;
                    xp[v8] = make_uint4(pack_bf2(0.25f * acc[c], 0.25f * acc[c + 1]),
                                        pack_bf2(0.25f * acc[c + 2], 0.25f * acc[c + 3]),
                                        pack_bf2(0.25f * acc[c + 4], 0.25f * acc[c + 5]),
                                        pack_bf2(0.25f * acc[c + 6], 0.25f * acc[c + 7]));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// ---- host side ---------------------------------------------------------------------------------

bool map_2d(CUtensorMap* m, const void* p, uint64_t inner, uint64_t outer, uint64_t row_bytes,
            uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The state [N][4][D] as (channel, branch, token), box {box_ch, 1, 128}: one branch's channels
// of 128 tokens, rows of box_ch·2 bytes.
bool map_state(CUtensorMap* m, const void* R, int64_t N, int D, uint32_t box_ch,
               CUtensorMapSwizzle sw) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(kBranches), cuuint64_t(N)};
    const cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(D) * kBranches * 2};
    const cuuint32_t box[3] = {box_ch, 1, kTile};
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(R), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Plain launch (no cluster): every CTA loads its own operands.
template <typename... KArgs, typename... Args>
cudaError_t launch_plain(void (*kern)(KArgs...), unsigned grid, int threads, size_t smem,
                         cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace

bool rank_tc_supported(int D, int r) {
    return D >= kKc && D % kKc == 0 && D <= GR_MAX_D && r >= kKc && r % 8 == 0 &&
           r <= kMaxRankTc;
}

int rank_tc_padded(int r) { return (r + kKc - 1) / kKc * kKc; }

size_t rank_tc_workspace(int64_t N, int r) {
    return align256(size_t(N) * kBranches * 4) + align256(size_t(N) * rank_tc_padded(r) * 2);
}

cudaError_t launch_rank_tc(int64_t N, int D, int r, float eps, void* R, const void* y,
                           const float* s_prev, const void* packed, void* x, float* s_out,
                           void* workspace, cudaStream_t st) {
    if (N == 0) return cudaSuccess;
    const Layout L = make_layout(D, r, GR_BF16);
    const char* base = static_cast<const char*>(packed);
    const float* gamma = reinterpret_cast<const float*>(base + L.gamma32);
    const void* wdw = base + L.wdw;
    const void* wu = base + L.wu;
    float* inv = static_cast<float*>(workspace);
    __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(workspace) +
                                                        align256(size_t(N) * kBranches * 4));
    const int rp = rank_tc_padded(r);
    const int n1 = (r + kBranches + 15) / 16 * 16;
    const int K = kBranches * D;

    // 1. write and row norms
    {
        const int64_t blocks = (N * kBranches + 7) / 8;
        const int64_t cap = int64_t(sm_count()) * 8;
        rownorm_kernel<<<unsigned(blocks < cap ? blocks : cap), 256, 0, st>>>(
            N, D, eps, static_cast<__nv_bfloat16*>(R), static_cast<const __nv_bfloat16*>(y),
            s_prev, inv);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const unsigned tiles = unsigned((N + kTile - 1) / kTile);
    // 2. down projection
    {
        CUtensorMap mR, mW;
        if (!map_state(&mR, R, N, D, kKc, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !map_2d(&mW, wdw, K, r + kBranches, size_t(K) * 2, kKc, n1 / 2,
                    CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        const size_t sb = down_stage_bytes(n1);
        int stages = int((232448 - 1024 - 256) / sb);   // within 227 KB with alignment, barriers
        stages = stages > 4 ? 4 : stages;
        if (stages < 2) return cudaErrorInvalidValue;
        const size_t smem = 1024 + stages * sb + 256;
        cudaError_t e = cudaFuncSetAttribute(down_tc_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
        if (e != cudaSuccess) return e;
        e = launch_plain(down_tc_kernel, tiles, kGemmThreads, smem, st, mR, mW, N, D, r, n1,
                         stages, static_cast<const float*>(inv), h, rp, s_out);
        if (e != cudaSuccess) return e;
    }
    // 3. up projection, gate and combine
    {
        CUtensorMap mH, mU, mR2;
        if (!map_2d(&mH, h, rp, N, size_t(rp) * 2, kKc, kTile, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !map_2d(&mU, wu, r, K, size_t(r) * 2, kKc, kCb, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !map_state(&mR2, R, N, D, kCb, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
        // two R' blocks and as many weight stages (up to 6) as the shared memory holds
        const int nrb = kUpMaxR;
        const size_t cap = 232448 - 1024;
        int nbs = kUpMaxStages;
        while (nbs > 2 && up_smem_bytes(rp, nbs, nrb) > cap) --nbs;
        if (up_smem_bytes(rp, nbs, nrb) > cap) return cudaErrorInvalidValue;
        const size_t smem = 1024 + up_smem_bytes(rp, nbs, nrb);
        cudaError_t e = cudaFuncSetAttribute(up_tc_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
        if (e != cudaSuccess) return e;
        e = launch_plain(up_tc_kernel, tiles, kUpThreads, smem, st, mH, mU, mR2, N, D, rp, nbs,
                         nrb, gamma, static_cast<const float*>(inv), static_cast<__nv_bfloat16*>(x));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace gr
