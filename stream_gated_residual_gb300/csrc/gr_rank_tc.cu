// The read at the pages' own rank, r = d/8 ("【论文解读】 Qwen3.8 Flash Next", §二.4: W_d is
// r × n_r·d with r = d/8), on the 5th-generation tensor cores (tcgen05, accumulators in tensor
// memory, operands staged by TMA). At r in the hundreds the read is a dense contraction of about
// 4·r·4D flops a token, as much arithmetic as memory traffic, so the projections run as GEMMs
// and everything else rides in their prologue and epilogue:
//
//   1. write_down_tc_kernel  one CTA per (128-token tile, branch i): the write R'_i = R_i +
//                            s_i·y (eq write, stored bf16, back to HBM by TMA store) stage by
//                            stage, each row's sum of squares, and the branch's projection
//                            P_i = [W_d; W_w]^(i)·γ_i R'_i of the unscaled stored rows (exact in
//                            bf16: one bf16 MMA) into a (r+4)-column fp32 accumulator in tensor
//                            memory; P_i and the sums of squares go to the step workspace.
//   2. gates_kernel          per token: inv_i = 1/√(ssq_i/D + eps) (eq rms), z and u = ¼ Σ_i
//                            inv_i P_i (eq gate, eq s: the normalisation is linear, so it can
//                            follow the contraction), h = SiLU(z) as bf16, s = 2σ(u).
//   3. up_tc_kernel          g = W_u h for 128 tokens × 4 branches × 32 channels a step (eq gate),
//                            two accumulators in tensor memory so the MMAs of one channel block
//                            overlap the epilogue of the previous one; the epilogue forms G = σ(g)
//                            and x = ¼ Σ_i G_i γ_i inv_i R'_i from a TMA copy of the block's R'
//                            (eq use_gate).
//
// Every mbarrier wait is bounded; a wait that runs out records a status bit and the kernel
// finishes without the work.
#include <math.h>
#include <string.h>

#include "gr_internal.h"
#include "gr_ptx.cuh"
#include "gr_tc.cuh"

namespace gr {
namespace {

constexpr int kTile = 128;          // tokens per CTA: the MMA's M
constexpr int kKc = 64;             // K elements per operand stage (128-byte rows)
constexpr int kStageA = kTile * 128; // one 128-token × 64-channel bf16 stage
constexpr int kUpThreads = 352;     // up projection: producer, MMA, 8 epilogue warps, R' loader
constexpr int kUpEpiWarps = 8;      // two per tensor-memory lane quadrant, 16 channels each
constexpr int kCb = 32;             // channels per branch in an up-projection block
constexpr int kMaxRankTc = 448;     // r + 4 <= 512 accumulator columns; H fits shared memory

__device__ __forceinline__ float sigm(float a) { return 1.0f / (1.0f + __expf(-a)); }
// σ(a) = ½ + ½·tanh(a/2) on the MUFU tanh (the combine's gates, as the other tensor-core paths)
__device__ __forceinline__ float sigm_fast(float a) {
    return fmaf(0.5f, tanh_approx(0.5f * a), 0.5f);
}

// ---- 1. eq write and each branch's down projection -----------------------------------------
// One CTA per (128-token tile, branch i): the write R'_i = R_i + s_i·y (eq write, stored bf16)
// stage by stage, each row's sum of squares, and the branch's projection of the UNSCALED stored
// rows, P_i = [W_d; W_w]^(i)·γ_i R'_i, on the tensor cores. R' is exact in bf16, so one bf16
// MMA carries it; the 1/rms factor is applied afterwards in fp32 (kernel 2), which is why each
// branch needs an accumulator of its own (a CTA of its own). R' leaves by TMA store.
//
// Shared memory: `stages` × {A: 128 rows × 128 B (R, then R' in place), Y: 128 × 128 B,
// B: n1 rows × 128 B}, then the barriers. Warps: 0 producer, 1 MMA issuer (owns the tensor
// memory), 2-5 the write and the epilogue (one per lane quadrant, thread = token row), 6 the R'
// stores (the stage is free once its MMAs are done and its store has read it).
constexpr int kWdThreads = 224;
__host__ __device__ inline size_t wd_stage_bytes(int n1) {
    return 2 * kStageA + size_t(n1) * 128;
}

template <bool WRITE>
__global__ void __launch_bounds__(kWdThreads, 1)
write_down_tc_kernel(const __grid_constant__ CUtensorMap tmR,
                     const __grid_constant__ CUtensorMap tmY,
                     const __grid_constant__ CUtensorMap tmW, int64_t N, int D, int r, int n1,
                     int stages, const float* __restrict__ s_prev, float* __restrict__ P, int ps,
                     float* __restrict__ ssq) {
    extern __shared__ uint8_t smraw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) &
                                             ~uintptr_t(1023));
    const size_t sb = wd_stage_bytes(n1);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + stages * sb);
    uint64_t* written = full + 4;
    uint64_t* empty = written + 4;
    uint64_t* acc_full = empty + 4;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(acc_full + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = int64_t(blockIdx.x >> 2) * kTile;
    const int ib = int(blockIdx.x & 3);
    const int nk = D / kKc;
    const uint32_t ncols = n1 > 256 ? 512 : 256;

    if (threadIdx.x == 0) {
        for (int s = 0; s < 4; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&written[s], 4);
            mbar_init(&empty[s], WRITE ? 2 : 1);   // the MMAs' commit (+ the store's read)
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
            const uint32_t bytes = uint32_t(kStageA + (WRITE ? kStageA : 0) + size_t(n1) * 128);
            const int half = n1 / 2;   // a box holds at most 256 rows: two boxes
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % stages;
                if (kc >= stages && !mbar_wait(&empty[s], ((kc / stages) - 1) & 1)) break;
                uint8_t* A = sm + s * sb;
                uint8_t* B = A + 2 * kStageA;
                mbar_expect_tx(&full[s], bytes);
                tma_load_3d(A, &tmR, kc * kKc, ib, int(t0), &full[s]);
                if (WRITE) tma_load_2d(A + kStageA, &tmY, kc * kKc, int(t0), &full[s]);
                tma_load_2d(B, &tmW, ib * D + kc * kKc, 0, &full[s]);
                tma_load_2d(B + half * 128, &tmW, ib * D + kc * kKc, half, &full[s]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t id0 = idesc_bf16_f32(kTile, n1 > 256 ? 256 : n1);
            const uint32_t id1 = idesc_bf16_f32(kTile, n1 > 256 ? n1 - 256 : 16);
            bool ok = true;
            for (int kc = 0; kc < nk && ok; ++kc) {
                const int s = kc % stages;
                // the stage's TMA bytes (weights too) and the rows the write warps left in place
                ok = mbar_wait(&full[s], (kc / stages) & 1) &&
                     mbar_wait(&written[s], (kc / stages) & 1);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a = smem_u32(sm + s * sb), b = a + 2 * kStageA;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t acc = (kc | kk) != 0;
                    const uint64_t ad = sdesc_sw128(a + kk * 32);
                    tc_mma(tmem, ad, sdesc_sw128(b + kk * 32), id0, acc);
                    if (n1 > 256)
                        tc_mma(tmem + 256, ad, sdesc_sw128(b + 256 * 128 + kk * 32), id1, acc);
                }
                tc_commit(&empty[s]);
            }
            if (ok) tc_commit(acc_full);
        }
    } else if (warp == 6) {
        // R' of each stage to HBM once the write warps have left it in place
        if (WRITE && lane == 0) {
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % stages;
                if (!mbar_wait(&written[s], (kc / stages) & 1)) break;
                tma_store_3d(&tmR, sm + s * sb, kc * kKc, ib, int(t0));
                bulk_commit();
                bulk_wait_read<0>();
                mbar_arrive(&empty[s]);
            }
            bulk_wait_all();
        }
    } else {
        // warps 2-5: lane quadrant q; thread row = token t0 + 32q + lane
        const int q = warp & 3, row = q * 32 + lane;
        const int64_t t = t0 + row;
        const float sv = (WRITE && t < N) ? s_prev[t * kBranches + ib] : 0.f;
        float ss = 0.f;
        bool ok = true;
        for (int kc = 0; kc < nk && ok; ++kc) {
            const int s = kc % stages;
            ok = mbar_wait(&full[s], (kc / stages) & 1);
            if (!ok) break;
            uint8_t* rp8 = sm + s * sb + row * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                // logical chunk j sits at j ^ (row & 7): eight rows hit eight bank groups
                const int off = (j ^ (row & 7)) * 16;
                uint4 v = *reinterpret_cast<const uint4*>(rp8 + off);
                uint32_t w[4] = {v.x, v.y, v.z, v.w};
                if (WRITE) {
                    const uint4 yv = *reinterpret_cast<const uint4*>(rp8 + kStageA + off);
                    const uint32_t yw[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float lo = fmaf(sv, __uint_as_float(yw[k] << 16),
                                              __uint_as_float(w[k] << 16));
                        const float hi = fmaf(sv, __uint_as_float(yw[k] & 0xffff0000u),
                                              __uint_as_float(w[k] & 0xffff0000u));
                        w[k] = pack_bf2(lo, hi);
                    }
                    *reinterpret_cast<uint4*>(rp8 + off) = make_uint4(w[0], w[1], w[2], w[3]);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float lo = __uint_as_float(w[k] << 16);
                    const float hi = __uint_as_float(w[k] & 0xffff0000u);
                    ss = fmaf(lo, lo, fmaf(hi, hi, ss));
                }
            }
            if (WRITE) fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&written[s]);
        }
        // epilogue: the branch's r + 4 projections of this row, and its sum of squares
        if (ok) ok = mbar_wait(acc_full, 0);
        tc_fence_after();
        if (ok) {
            // every lane takes part in the warp's tensor-memory loads (a row past N included);
            // only rows of real tokens are stored
            float* Prow = P + (t * kBranches + ib) * size_t(ps);
            for (int c0 = 0; c0 < n1; c0 += 16) {
                float v[16];
                tmem_ld16(tmem + (uint32_t(q * 32) << 16) + c0, v);
                if (t >= N) continue;
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4)
                    if (c0 + 4 * k4 < ps)
                        *reinterpret_cast<float4*>(Prow + c0 + 4 * k4) =
                            make_float4(v[4 * k4], v[4 * k4 + 1], v[4 * k4 + 2], v[4 * k4 + 3]);
            }
            if (t < N) ssq[t * kBranches + ib] = ss;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

// ---- 2. eq rms, eq gate (z, h) and eq s from the branches' projections ---------------------------
// One warp per token: inv_i = 1/√(ssq_i/D + eps), z = ¼ Σ_i inv_i P_i[0, r), u = ¼ Σ_i inv_i
// P_i[r, r+4); h = SiLU(z) as bf16 (zero up to rp), s = 2σ(u), and inv for the up projection.
__global__ void __launch_bounds__(256)
gates_kernel(int64_t N, int D, int r, int rp, int ps, float eps, const float* __restrict__ P,
             const float* __restrict__ ssq, __nv_bfloat16* __restrict__ h,
             float* __restrict__ inv, float* __restrict__ s_out) {
    const int lane = threadIdx.x & 31;
    for (int64_t t = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5); t < N;
         t += int64_t(gridDim.x) * 8) {
        float iv[kBranches];
#pragma unroll
        for (int i = 0; i < kBranches; ++i)
            iv[i] = rsqrtf(ssq[t * kBranches + i] / float(D) + eps);
        if (lane < kBranches) inv[t * kBranches + lane] = iv[lane];
        const float* Pt = P + t * kBranches * size_t(ps);
        for (int k = lane; k < rp || k < r + kBranches; k += 32) {
            float z = 0.f;
            if (k < r + kBranches) {
#pragma unroll
                for (int i = 0; i < kBranches; ++i) z = fmaf(iv[i], Pt[i * size_t(ps) + k], z);
                z *= 0.25f;
            }
            if (k < rp) h[t * rp + k] = __float2bfloat16_rn(k < r ? z * sigm(z) : 0.f);
            if (k >= r && k < r + kBranches) s_out[t * kBranches + (k - r)] = 2.0f * sigm(z);
        }
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

// Floats per (token, branch) row of the branches' projections: r + 4, rounded to 16 bytes.
static int rank_tc_pstride(int r) { return (r + kBranches + 3) / 4 * 4; }

// inv [N][4] fp32 | h [N][rp] bf16 | P [N][4][ps] fp32 | ssq [N][4] fp32
size_t rank_tc_workspace(int64_t N, int r) {
    return align256(size_t(N) * kBranches * 4) + align256(size_t(N) * rank_tc_padded(r) * 2) +
           align256(size_t(N) * kBranches * rank_tc_pstride(r) * 4) +
           align256(size_t(N) * kBranches * 4);
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
    const int rp = rank_tc_padded(r);
    const int ps = rank_tc_pstride(r);
    char* wsb = static_cast<char*>(workspace);
    float* inv = reinterpret_cast<float*>(wsb);
    wsb += align256(size_t(N) * kBranches * 4);
    __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(wsb);
    wsb += align256(size_t(N) * rp * 2);
    float* P = reinterpret_cast<float*>(wsb);
    wsb += align256(size_t(N) * kBranches * ps * 4);
    float* ssq = reinterpret_cast<float*>(wsb);
    const int n1 = (r + kBranches + 15) / 16 * 16;
    const int K = kBranches * D;

    const unsigned tiles = unsigned((N + kTile - 1) / kTile);
    // 1. the write and each branch's down projection: a CTA per (tile, branch)
    {
        CUtensorMap mR, mY, mW;
        memset(&mY, 0, sizeof(mY));
        if (!map_state(&mR, R, N, D, kKc, CU_TENSOR_MAP_SWIZZLE_128B) ||
            (y && !map_2d(&mY, y, D, N, size_t(D) * 2, kKc, kTile, CU_TENSOR_MAP_SWIZZLE_128B)) ||
            !map_2d(&mW, wdw, K, r + kBranches, size_t(K) * 2, kKc, n1 / 2,
                    CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        const size_t sb = wd_stage_bytes(n1);
        int stages = int((232448 - 1024 - 256) / sb);   // within 227 KB with alignment, barriers
        stages = stages > 4 ? 4 : stages;
        if (stages < 2) return cudaErrorInvalidValue;
        const size_t smem = 1024 + stages * sb + 256;
        auto kern = y ? write_down_tc_kernel<true> : write_down_tc_kernel<false>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
        if (e != cudaSuccess) return e;
        e = launch_plain(kern, tiles * kBranches, kWdThreads, smem, st, mR, mY, mW, N, D, r, n1,
                         stages, s_prev, P, ps, ssq);
        if (e != cudaSuccess) return e;
    }
    // 2. inv, z, u, h and s per token
    {
        const int64_t blocks = (N + 7) / 8;
        const int64_t cap = int64_t(sm_count()) * 8;
        gates_kernel<<<unsigned(blocks < cap ? blocks : cap), 256, 0, st>>>(
            N, D, r, rp, ps, eps, P, ssq, h, inv, s_out);
        cudaError_t e = cudaGetLastError();
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
