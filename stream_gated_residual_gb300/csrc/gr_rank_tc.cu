// The read at the pages' own rank, r = d/8 ("【论文解读】 Qwen3.8 Flash Next", §二.4: W_d is
// r × n_r·d with r = d/8), on the 5th-generation tensor cores (tcgen05, accumulators in tensor
// memory, operands staged by TMA). At r in the hundreds the read is a dense contraction of about
// 4·r·4D flops a token, as much arithmetic as memory traffic, so the projections run as GEMMs
// and everything else rides in their prologue and epilogue:
//
//   1. write_down_tc_kernel  units of (tile of <= 128 tokens, branch i) on a persistent grid: the
//                            write R'_i = R_i + s_i·y (eq write, stored bf16, back to HBM by TMA
//                            store) stage by stage, each row's sum of squares, and the branch's
//                            projection P_i = [W_d; W_w]^(i)·γ_i R'_i of the unscaled stored rows
//                            (exact in bf16: one bf16 MMA) into a (r+4)-column fp32 accumulator in
//                            tensor memory; P_i and the sums of squares go to the step workspace.
//   2. gates_kernel          per token: inv_i = 1/√(ssq_i/D + eps) (eq rms), z and u = ¼ Σ_i
//                            inv_i P_i (eq gate, eq s: the normalisation is linear, so it can
//                            follow the contraction), h/2 = ½ SiLU(z) as bf16, s = 2σ(u).
//   3. up_tc_kernel          g/2 = W_u h/2 for a tile × 4 branches × 32 channels a step (eq gate),
//                            h/2 in tensor memory as the A operand, two accumulators so the MMAs
//                            of one channel block overlap the epilogue of the previous one; the
//                            epilogue forms G = σ(g) = ½(1 + tanh(g/2)) and x = ¼ Σ_i G_i γ_i
//                            inv_i R'_i from a TMA copy of the block's R' (eq use_gate).
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

constexpr int kTile = 128;          // the MMAs' M: rows of a tile (its tokens are up to this many)
constexpr int kKc = 64;             // K elements per operand stage (128-byte rows)
constexpr int kStageA = kTile * 128; // one 128-row × 64-channel bf16 stage
// r + 4 <= 512 accumulator columns in the write pass; h/2 (r/2 columns, r rounded up to 64)
// beside the up projection's 256-column accumulator in its 512
constexpr int kMaxRankTc = 448;

__device__ __forceinline__ float sigm(float a) { return 1.0f / (1.0f + __expf(-a)); }

// ---- 1. eq write and each branch's down projection -----------------------------------------
// Units of work are (tile, branch i): the write R'_i = R_i + s_i·y (eq write, stored bf16) stage
// by stage, each row's sum of squares, and the branch's projection of the UNSCALED stored rows,
// P_i = [W_d; W_w]^(i)·γ_i R'_i, on the tensor cores. R' is exact in bf16, so one bf16 MMA
// carries it; the 1/rms factor is applied afterwards in fp32 (kernel 2), which is why each branch
// needs an accumulator of its own. R' leaves by TMA store.
// A persistent grid: CTA c takes units c, c + G, c + 2G, ... (G a multiple of 4, so the four
// branch units of a tile run side by side and share y through L2), and one ring of stages runs
// through all of them: the next unit's loads, writes and stores go on while four warps of their
// own drain the previous unit's accumulator and store its P rows; only the next unit's first
// MMA waits for that drain.
// A tile is `rows` <= 128 tokens, chosen by the host so that the units fill whole waves of SMs;
// the MMA always spans 128 rows: the rows past the tile's own (the next tile's tokens, or past N)
// are loaded but never stored, and their accumulator rows are dropped.
//
// Shared memory: `stages` × {A: 128 rows × 128 B (R, then R' in place), Y: 128 × 128 B,
// B: n1 rows × 128 B}, then the barriers and two 128-float buffers of row sums of squares.
// Warps: 0 producer, 1 MMA issuer (owns the tensor memory), 2-5 the write (one per lane quadrant,
// thread = token row), 6 the R' stores (a stage is free once its MMAs are done and its store has
// read it), 7-10 the epilogue (one per lane quadrant).
constexpr int kWdThreads = 352;
__host__ __device__ inline size_t wd_stage_bytes(int n1) {
    return 2 * kStageA + size_t(n1) * 128;
}

template <bool WRITE>
__global__ void __launch_bounds__(kWdThreads, 1)
write_down_tc_kernel(const __grid_constant__ CUtensorMap tmR,
                     const __grid_constant__ CUtensorMap tmS,
                     const __grid_constant__ CUtensorMap tmY,
                     const __grid_constant__ CUtensorMap tmW, int64_t N, int D, int r, int n1,
                     int stages, int rows, int units, const float* __restrict__ s_prev,
                     float* __restrict__ P, int ps, float* __restrict__ ssq) {
    extern __shared__ uint8_t smraw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) &
                                             ~uintptr_t(1023));
    const size_t sb = wd_stage_bytes(n1);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + stages * sb);
    uint64_t* written = full + 4;
    uint64_t* empty = written + 4;
    uint64_t* acc_full = empty + 4;      // [2]: a unit's MMAs are done
    uint64_t* acc_empty = acc_full + 2;  // the epilogue has read the accumulator
    uint64_t* ss_full = acc_empty + 1;   // [2]: a unit's sums of squares are in ssbuf
    uint64_t* ss_empty = ss_full + 2;    // [2]: the epilogue has read them
    uint32_t* tslot = reinterpret_cast<uint32_t*>(ss_empty + 2);
    float* ssbuf = reinterpret_cast<float*>(sm + stages * sb + 256);   // [2][128]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nk = D / kKc;
    const uint32_t ncols = n1 > 256 ? 512 : 256;
    const int G = int(gridDim.x);
    const int nu = units > int(blockIdx.x) ? (units - int(blockIdx.x) + G - 1) / G : 0;
    // unit j of this CTA: tile and branch, and the tile's first token
    auto unit_ib = [&](int j) { return (int(blockIdx.x) + j * G) & 3; };
    auto unit_t0 = [&](int j) { return int64_t((int(blockIdx.x) + j * G) >> 2) * rows; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < 4; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&written[s], 4);
            mbar_init(&empty[s], WRITE ? 2 : 1);   // the MMAs' commit (+ the store's read)
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&ss_full[b], 4);
            mbar_init(&ss_empty[b], 4);
        }
        mbar_init(acc_empty, 4);
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
            bool ok = true;
            for (int j = 0; j < nu && ok; ++j) {
                const int ib = unit_ib(j);
                const int t0 = int(unit_t0(j));
                for (int kc = 0; kc < nk; ++kc) {
                    const int g = j * nk + kc, s = g % stages;
                    if (g >= stages && !mbar_wait(&empty[s], ((g / stages) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    uint8_t* A = sm + s * sb;
                    uint8_t* B = A + 2 * kStageA;
                    mbar_expect_tx(&full[s], bytes);
                    tma_load_3d(A, &tmR, kc * kKc, ib, t0, &full[s]);
                    if (WRITE) tma_load_2d(A + kStageA, &tmY, kc * kKc, t0, &full[s]);
                    tma_load_2d(B, &tmW, ib * D + kc * kKc, 0, &full[s]);
                    tma_load_2d(B + half * 128, &tmW, ib * D + kc * kKc, half, &full[s]);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t id0 = idesc_bf16_f32(kTile, n1 > 256 ? 256 : n1);
            const uint32_t id1 = idesc_bf16_f32(kTile, n1 > 256 ? n1 - 256 : 16);
            bool ok = true;
            for (int j = 0; j < nu && ok; ++j) {
                // the previous unit's accumulator has been read out
                if (j > 0) ok = mbar_wait(acc_empty, (j - 1) & 1);
                for (int kc = 0; kc < nk && ok; ++kc) {
                    const int g = j * nk + kc, s = g % stages;
                    // the stage's TMA bytes (weights too) and the rows the write warps left in
                    // place
                    ok = mbar_wait(&full[s], (g / stages) & 1) &&
                         mbar_wait(&written[s], (g / stages) & 1);
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
                if (ok) tc_commit(&acc_full[j & 1]);
            }
        }
    } else if (warp == 6) {
        // R' of each stage to HBM once the write warps have left it in place. (Keeping two stores
        // in flight hands each stage back one stage later, which costs the ring a stage: slower.)
        if (WRITE && lane == 0) {
            bool ok = true;
            for (int j = 0; j < nu && ok; ++j) {
                const int ib = unit_ib(j);
                const int t0 = int(unit_t0(j));
                for (int kc = 0; kc < nk; ++kc) {
                    const int g = j * nk + kc, s = g % stages;
                    if (!mbar_wait(&written[s], (g / stages) & 1)) {
                        ok = false;
                        break;
                    }
                    tma_store_3d(&tmS, sm + s * sb, kc * kKc, ib, t0);
                    bulk_commit();
                    bulk_wait_read<0>();
                    mbar_arrive(&empty[s]);
                }
            }
            bulk_wait_all();
        }
    } else if (warp >= 7) {
        // warps 7-10: the epilogue of each unit, lane quadrant q, thread row = token t0 + 32q + lane
        const int q = warp & 3, row = q * 32 + lane;
        bool ok = true;
        for (int j = 0; j < nu && ok; ++j) {
            const int ib = unit_ib(j);
            const int64_t t = unit_t0(j) + row;
            const bool mine = row < rows && t < N;
            ok = mbar_wait(&acc_full[j & 1], (j >> 1) & 1);
            if (!ok) break;
            tc_fence_after();
            // every lane takes part in the warp's tensor-memory loads (a row past N included);
            // only rows of real tokens are stored
            float* Prow = P + (t * kBranches + ib) * size_t(ps);
            for (int c0 = 0; c0 < n1; c0 += 16) {
                float v[16];
                tmem_ld16(tmem + (uint32_t(q * 32) << 16) + c0, v);
                if (!mine) continue;
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4)
                    if (c0 + 4 * k4 < ps)
                        *reinterpret_cast<float4*>(Prow + c0 + 4 * k4) =
                            make_float4(v[4 * k4], v[4 * k4 + 1], v[4 * k4 + 2], v[4 * k4 + 3]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
            ok = mbar_wait(&ss_full[j & 1], (j >> 1) & 1);
            if (!ok) break;
            if (mine) ssq[t * kBranches + ib] = ssbuf[(j & 1) * 128 + row];
            __syncwarp();
            if (lane == 0) mbar_arrive(&ss_empty[j & 1]);
        }
    } else {
        // warps 2-5: the write; lane quadrant q; thread row = token t0 + 32q + lane
        const int q = warp & 3, row = q * 32 + lane;
        bool ok = true;
        for (int j = 0; j < nu && ok; ++j) {
            const int ib = unit_ib(j);
            const int64_t t = unit_t0(j) + row;
            const bool mine = row < rows && t < N;   // the tile's own token (the rest are ignored)
            const float sv = (WRITE && mine) ? s_prev[t * kBranches + ib] : 0.f;
            float ss = 0.f;
            for (int kc = 0; kc < nk && ok; ++kc) {
                const int g = j * nk + kc, s = g % stages;
                ok = mbar_wait(&full[s], (g / stages) & 1);
                if (!ok) break;
                uint8_t* rp8 = sm + s * sb + row * 128;
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    // logical chunk jj sits at jj ^ (row & 7): eight rows hit eight bank groups
                    const int off = (jj ^ (row & 7)) * 16;
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
            if (!ok) break;
            // the unit's sums of squares to the epilogue (its buffer free again two units on)
            if (j >= 2) ok = mbar_wait(&ss_empty[j & 1], ((j >> 1) - 1) & 1);
            if (!ok) break;
            ssbuf[(j & 1) * 128 + row] = ss;
            __syncwarp();
            if (lane == 0) mbar_arrive(&ss_full[j & 1]);
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
// P_i[r, r+4); s = 2σ(u); inv for the up projection, and h/2 = ½ SiLU(z) as bf16 (zero up to
// rp): halving is exact, so the up projection's MMAs yield g/2 exactly, the argument of the
// tanh that gives σ(g).
__global__ void __launch_bounds__(256)
gates_kernel(int64_t N, int D, int r, int rp, int ps, float eps, const float* __restrict__ P,
             const float* __restrict__ ssq, __nv_bfloat16* __restrict__ h,
             float* __restrict__ inv, float* __restrict__ s_out) {
    // the write pass's P and ssq are complete and visible past this wait; once every CTA of this
    // one-wave grid has passed it, the up projection (whose own R' loads need that grid, not this
    // one) may launch and start its weight and R' loads while these CTAs finish
    dep_wait();
    dep_launch_dependents();
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
            if (k < rp) h[t * rp + k] = __float2bfloat16_rn(k < r ? 0.5f * z * sigm(z) : 0.f);
            if (k >= r && k < r + kBranches) s_out[t * kBranches + (k - r)] = 2.0f * sigm(z);
        }
    }
}

// ---- 3. up projection, gate and combine ------------------------------------------------------
// A CTA per tile of `rows` <= 128 tokens (as in kernel 1, rows past the tile's own are computed
// and dropped). A tcgen05 MMA with M = 128 costs about the same to issue for any N up to 128 and
// only N = 256 keeps the tensor pipe busy, so a block is 64 channels of each of the 4 branches
// (N = 256). Tensor memory: the block's 256-column accumulator, then the tile's h/2 (128 rows ×
// rp bf16, two k a column) as the MMAs' A operand. The 16 epilogue warps copy their part of the
// accumulator into registers as soon as a block's MMAs are done and hand it back at once, so the
// MMAs of the next block run while they form G = σ(g) and the combine.
// Shared memory: nbs W_u stages (4 branches × 64 rows × 128 B, one k step of 64) and nrb R' half
// blocks (4 branches × 128 tokens × 32 channels bf16, 64-byte swizzled, and their γ), then the
// barriers. Warps: 0 the MMA issuer (owns the tensor memory), 2-17 the epilogue (lane quadrant
// warp % 4, 16-channel quarter (warp - 2) / 4 of the block, thread = token row), 1 the W_u stages
// (lane s owns stage slot s: one 32 KB box of the 4 branches' 64 rows in flight per lane; the
// copies one thread issues complete one after another, about an L2 round trip apiece), 18 the R'
// half blocks (one box of R' and one of γ each). The W_u lanes spin without suspending: a
// suspending wait would stop the whole warp, and with it the other lanes' copies.
constexpr int kUpThreads = 608;
constexpr int kUpEpiWarps = 16;
constexpr int kCb = 64;                                         // channels a block (per branch)
constexpr int kCh = 32;                                         // channels an R' half block
constexpr int kUpMaxStages = 6;
constexpr int kUpMaxR = 3;
constexpr int kStageB = kBranches * kCb * 128;                  // 32 KB
constexpr int kRData = kBranches * kTile * kCh * 2;             // 32 KB of R'
constexpr int kRBlock = kRData + kBranches * kCh * 4;           // + the half block's γ (fp32)
constexpr uint32_t kHCol = kBranches * kCb;                     // h's first tensor-memory column
__host__ __device__ inline size_t up_smem_bytes(int nbs, int nrb) {
    return size_t(nbs) * kStageB + size_t(nrb) * kRBlock + 256;
}

__global__ void __launch_bounds__(kUpThreads, 1)
up_tc_kernel(const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmR,
             const __grid_constant__ CUtensorMap tmG, int64_t N, int D, int rp, int nbs, int nrb,
             int rows, const __nv_bfloat16* __restrict__ h, const float* __restrict__ inv,
             __nv_bfloat16* __restrict__ x) {
    extern __shared__ uint8_t smraw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) &
                                             ~uintptr_t(1023));
    const int nkc = rp / kKc;
    uint8_t* Bs = sm;
    uint8_t* Rb = Bs + size_t(nbs) * kStageB;
    uint64_t* h_full = reinterpret_cast<uint64_t*>(Rb + size_t(nrb) * kRBlock);
    uint64_t* b_full = h_full + 1;
    uint64_t* b_empty = b_full + kUpMaxStages;
    uint64_t* r_full = b_empty + kUpMaxStages;
    uint64_t* r_empty = r_full + kUpMaxR;
    uint64_t* t_full = r_empty + kUpMaxR;
    uint64_t* t_empty = t_full + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(t_empty + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = int64_t(blockIdx.x) * rows;
    const int nb = D / kCb;

    if (threadIdx.x == 0) {
        mbar_init(h_full, 4);   // the four warps that write h's lane quadrants
        for (int s = 0; s < kUpMaxStages; ++s) {
            mbar_init(&b_full[s], 1);
            mbar_init(&b_empty[s], 1);
        }
        for (int b = 0; b < kUpMaxR; ++b) {
            mbar_init(&r_full[b], 1);
            mbar_init(&r_empty[b], kUpEpiWarps / 2);   // the 8 warps of that half of the block
        }
        mbar_init(t_full, 1);
        mbar_init(t_empty, kUpEpiWarps);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 1) {
        if (lane < nbs) {
            // stage it = cb · nkc + kc (k step kc of block cb) of slot it % nbs, from lane s
            const int total = nb * nkc;
            for (int it = lane; it < total; it += nbs) {
                if (it >= nbs && !spin_wait(&b_empty[lane], ((it / nbs) - 1) & 1)) break;
                mbar_expect_tx(&b_full[lane], kStageB);
                tma_load_3d(Bs + lane * kStageB, &tmU, (it % nkc) * kKc, (it / nkc) * kCb, 0,
                            &b_full[lane]);
            }
        }
    } else if (warp == 18) {
        if (lane == 0) {
            // the R' half blocks of the combine (and their γ), up to nrb ahead
            for (int hb = 0; hb < 2 * nb; ++hb) {
                const int rb = hb % nrb, c0 = hb * kCh;
                if (hb >= nrb && !mbar_wait(&r_empty[rb], ((hb / nrb) - 1) & 1)) break;
                mbar_expect_tx(&r_full[rb], kRBlock);
                tma_load_3d(Rb + rb * kRBlock, &tmR, c0, int(t0), 0, &r_full[rb]);
                tma_load_2d(Rb + rb * kRBlock + kRData, &tmG, c0, 0, &r_full[rb]);
            }
        }
    } else if (warp == 0) {
        if (lane == 0) {
            const uint32_t id = idesc_bf16_f32(kTile, kBranches * kCb);
            const uint64_t b0 = sdesc_sw128(smem_u32(Bs));   // + (byte offset >> 4) per stage, k
            bool ok = mbar_wait(h_full, 0);
            tc_fence_after();
            int it = 0;
            for (int cb = 0; cb < nb && ok; ++cb) {
                // the epilogue has copied the previous block's accumulator into registers
                if (cb > 0) ok = mbar_wait(t_empty, (cb - 1) & 1);
                if (!ok) break;
                tc_fence_after();
                for (int kc = 0; kc < nkc; ++kc, ++it) {
                    const int s = it % nbs;
                    ok = mbar_wait(&b_full[s], (it / nbs) & 1);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t bs = b0 + uint64_t((s * kStageB) >> 4);
                    const uint32_t a = tmem + kHCol + uint32_t(kc * (kKc / 2));
                    tc_mma_ts(tmem, a, bs, id, kc != 0);
                    tc_mma_ts(tmem, a + 8, bs + 2, id, 1u);
                    tc_mma_ts(tmem, a + 16, bs + 4, id, 1u);
                    tc_mma_ts(tmem, a + 24, bs + 6, id, 1u);
                    tc_commit(&b_empty[s]);
                }
                if (ok) tc_commit(t_full);
            }
        }
    } else {
        // warps 2-17: lane quadrant q = warp % 4, 16-channel quarter hq of each 64-channel block
        // (in R' half block hq / 2, at its 16-channel half hq % 2)
        // h and inv come from the gates kernel, this launch's programmatic predecessor
        dep_wait();
        const int q = warp & 3, hq = (warp - 2) >> 2, row = q * 32 + lane;
        constexpr int kH = 16;
        const int64_t t = t0 + row;
        const bool mine = row < rows && t < N;
        if (hq == 0) {
            // this row's h/2 into tensor memory (zeros for rows that are not the tile's own)
            const uint4* hp = reinterpret_cast<const uint4*>(h + (mine ? t : 0) * size_t(rp));
            const uint32_t ta = tmem + (uint32_t(q * 32) << 16) + kHCol;
            for (int c0 = 0; c0 < rp / 2; c0 += 16) {
                uint32_t v[16];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint4 u = mine ? __ldg(hp + c0 / 4 + k) : make_uint4(0, 0, 0, 0);
                    v[4 * k] = u.x;
                    v[4 * k + 1] = u.y;
                    v[4 * k + 2] = u.z;
                    v[4 * k + 3] = u.w;
                }
                tmem_st16(ta + uint32_t(c0), v);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(h_full);
        }
        // x = ¼ Σ_i σ(g_i) γ_i inv_i R'_i with σ(g) = ½(1 + tanh(g/2)) and the MMAs giving g/2:
        // x = Σ_i m_i w (1 + tanh(g_i/2)), w = γ_i R'_i, m_i = inv_i / 8
        float mi[kBranches];
#pragma unroll
        for (int i = 0; i < kBranches; ++i) mi[i] = mine ? 0.125f * inv[t * kBranches + i] : 0.f;
        const int half = hq >> 1, sub = hq & 1;
        bool ok = true;
        for (int cb = 0; cb < nb && ok; ++cb) {
            const int hb = 2 * cb + half, rb = hb % nrb;
            ok = mbar_wait(t_full, cb & 1);
            if (!ok) break;
            tc_fence_after();
            // the four branches' 16 logits of this row, then the accumulator goes back at once
            uint32_t g[kBranches][kH];
            const uint32_t ta = tmem + (uint32_t(q * 32) << 16) + uint32_t(hq * kH);
#pragma unroll
            for (int i = 0; i < kBranches; ++i) tmem_ld16_nowait(ta + i * kCb, g[i]);
#pragma unroll
            for (int i = 0; i < kBranches; ++i) tmem_wait_ld(g[i]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(t_empty);
            ok = mbar_wait(&r_full[rb], (hb / nrb) & 1);
            if (!ok) break;
            float acc[kH];
#pragma unroll
            for (int c = 0; c < kH; ++c) acc[c] = 0.f;
#pragma unroll
            for (int i = 0; i < kBranches; ++i) {
                const uint8_t* rbr = Rb + rb * kRBlock + i * (kTile * kCh * 2);
                const float4* gm = reinterpret_cast<const float4*>(
                    Rb + rb * kRBlock + kRData + (i * kCh + sub * kH) * 4);
                const float m = mi[i];
#pragma unroll
                for (int v8 = 0; v8 < kH / 8; ++v8) {
                    const uint4 u = *reinterpret_cast<const uint4*>(rbr + swz64(row, sub * 2 + v8));
                    const float4 ga = gm[2 * v8], gb = gm[2 * v8 + 1];
                    const float gv[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int c = v8 * 8 + 2 * k;
                        const float w0 = gv[2 * k] * __uint_as_float(w[k] << 16);
                        const float w1 = gv[2 * k + 1] * __uint_as_float(w[k] & 0xffff0000u);
                        // tanh of both logits in one MUFU op on an f16 pair (2^-11 of the logit,
                        // far inside the bf16 rounding of x); the epilogue is bound by that unit
                        uint32_t th =
                            pack_h2(__uint_as_float(g[i][c]), __uint_as_float(g[i][c + 1]));
                        asm("tanh.approx.f16x2 %0, %0;" : "+r"(th));
                        const float2 tf = __half22float2(*reinterpret_cast<const __half2*>(&th));
                        acc[c] = fmaf(m, fmaf(w0, tf.x, w0), acc[c]);
                        acc[c + 1] = fmaf(m, fmaf(w1, tf.y, w1), acc[c + 1]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&r_empty[rb]);
            if (mine) {
                uint4* xp = reinterpret_cast<uint4*>(x + t * D + cb * kCb + hq * kH);
#pragma unroll
                for (int v8 = 0; v8 < kH / 8; ++v8) {
                    const int c = v8 * 8;
                    xp[v8] = make_uint4(pack_bf2(acc[c], acc[c + 1]),
                                        pack_bf2(acc[c + 2], acc[c + 3]),
                                        pack_bf2(acc[c + 4], acc[c + 5]),
                                        pack_bf2(acc[c + 6], acc[c + 7]));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
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

// The state [N][4][D] as (channel, branch, token), box {box_ch, 1, box_tok}: one branch's
// channels of box_tok tokens, rows of box_ch·2 bytes.
bool map_state(CUtensorMap* m, const void* R, int64_t N, int D, uint32_t box_ch,
               CUtensorMapSwizzle sw, uint32_t box_tok = kTile) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(kBranches), cuuint64_t(N)};
    const cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(D) * kBranches * 2};
    const cuuint32_t box[3] = {box_ch, 1, box_tok};
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(R), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A tensor map of rank `rank` (2 or 3): dims from the innermost, byte strides of the outer dims.
bool map_nd(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* p,
            const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
            CUtensorMapSwizzle sw) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(m, dt, cuuint32_t(rank), const_cast<void*>(p), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Plain launch (no cluster): every CTA loads its own operands. `programmatic`: launched as the
// programmatic dependent of the preceding launch on the stream (it may start before that one
// ends; it waits with dep_wait before it reads that launch's results).
template <typename... KArgs, typename... Args>
cudaError_t launch_plain(void (*kern)(KArgs...), unsigned grid, int threads, size_t smem,
                         cudaStream_t st, bool programmatic, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Tokens a tile of a kernel that runs `per_tile` CTAs a tile, one CTA an SM: as few (64 to 128,
// the MMA's M) as spread the work over the whole waves that 128-token tiles would need, so that
// no wave runs part-full (at 16384 tokens on 152 SMs: 108).
int rank_tc_tile_rows(int64_t N, int per_tile, int64_t sms) {
    const int64_t ctas = (N + kTile - 1) / kTile * per_tile;
    const int64_t waves = (ctas + sms - 1) / sms;
    int64_t tiles = waves * sms / per_tile;
    tiles = tiles < 1 ? 1 : tiles;
    int64_t rows = (N + tiles - 1) / tiles;
    rows = rows < 64 ? 64 : rows;
    return int(rows > kTile ? kTile : rows);
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

    const int64_t sms = sm_count();
    // 1. the write and each branch's down projection: units (tile, branch) on a persistent grid
    {
        const int rows = rank_tc_tile_rows(N, kBranches, sms);
        const unsigned tiles = unsigned((N + rows - 1) / rows);
        CUtensorMap mR, mS, mY, mW;
        memset(&mY, 0, sizeof(mY));
        if (!map_state(&mR, R, N, D, kKc, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !map_state(&mS, R, N, D, kKc, CU_TENSOR_MAP_SWIZZLE_128B, uint32_t(rows)) ||
            (y && !map_2d(&mY, y, D, N, size_t(D) * 2, kKc, kTile, CU_TENSOR_MAP_SWIZZLE_128B)) ||
            !map_2d(&mW, wdw, K, r + kBranches, size_t(K) * 2, kKc, n1 / 2,
                    CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        const size_t sb = wd_stage_bytes(n1);
        // the stages, then 256 bytes of barriers and two 512-byte buffers of sums of squares
        int stages = int((232448 - 1024 - 1280) / sb);
        stages = stages > 4 ? 4 : stages;
        if (stages < 2) return cudaErrorInvalidValue;
        const size_t smem = 1024 + stages * sb + 1280;
        auto kern = y ? write_down_tc_kernel<true> : write_down_tc_kernel<false>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
        if (e != cudaSuccess) return e;
        // a persistent grid: a multiple of 4 CTAs (the branch units of a tile side by side)
        const int units = int(tiles) * kBranches;
        int grid = int(sms) / kBranches * kBranches;
        grid = grid < 4 ? 4 : grid;
        grid = grid > units ? units : grid;
        e = launch_plain(kern, unsigned(grid), kWdThreads, smem, st, false, mR, mS, mY, mW, N, D,
                         r, n1, stages, rows, units, s_prev, P, ps, ssq);
        if (e != cudaSuccess) return e;
    }
    // 2. inv, z, u, h and s per token
    {
        // a programmatic dependent of the write pass, which triggers nothing: the gates CTAs start
        // as the write pass's leave (triggered at the write pass's start, CTAs parked beside it
        // made the step 10 µs slower). One wave (8 CTAs of 256 threads an SM), so that every CTA
        // passes its dep_wait, and triggers the up projection's launch, without waiting for
        // another CTA to leave.
        const int64_t blocks = (N + 7) / 8;
        const int64_t cap = sms * 8;
        cudaError_t e = launch_plain(gates_kernel, unsigned(blocks < cap ? blocks : cap), 256, 0,
                                     st, true, N, D, r, rp, ps, eps, P, ssq, h, inv, s_out);
        if (e != cudaSuccess) return e;
    }
    // 3. up projection, gate and combine
    {
        const int rows = rank_tc_tile_rows(N, 1, sms);
        const unsigned tiles = unsigned((N + rows - 1) / rows);
        // W_u [4][D][r] as (k, channel, branch), box {64, 64, 4}: a k step of a block's 4 × 64
        // rows; R' [N][4][D] as (channel, token, branch), box {32, 128, 4}: [branch][token][32
        // channels]; γ [4][D] fp32, box {32, 4}
        CUtensorMap mU, mR2, mG;
        const cuuint64_t dU[3] = {cuuint64_t(r), cuuint64_t(D), cuuint64_t(kBranches)};
        const cuuint64_t sU[2] = {cuuint64_t(r) * 2, cuuint64_t(D) * r * 2};
        const cuuint32_t bU[3] = {kKc, kCb, kBranches};
        const cuuint64_t dR[3] = {cuuint64_t(D), cuuint64_t(N), cuuint64_t(kBranches)};
        const cuuint64_t sR[2] = {cuuint64_t(D) * kBranches * 2, cuuint64_t(D) * 2};
        const cuuint32_t bR[3] = {kCh, kTile, kBranches};
        const cuuint64_t dG[2] = {cuuint64_t(D), cuuint64_t(kBranches)};
        const cuuint64_t sG[1] = {cuuint64_t(D) * 4};
        const cuuint32_t bG[2] = {kCh, kBranches};
        if (!map_nd(&mU, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, wu, dU, sU, bU,
                    CU_TENSOR_MAP_SWIZZLE_128B) ||
            !map_nd(&mR2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, R, dR, sR, bR,
                    CU_TENSOR_MAP_SWIZZLE_64B) ||
            !map_nd(&mG, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, gamma, dG, sG, bG,
                    CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
        // W_u stages (up to 6) and R' half blocks (up to 3) as the shared memory holds
        const size_t cap = 232448 - 1024;
        int nbs = kUpMaxStages, nrb = kUpMaxR;
        while (up_smem_bytes(nbs, nrb) > cap && nbs > 2) {
            if (nbs > nrb + 2) --nbs;
            else if (nrb > 2) --nrb;
            else --nbs;
        }
        if (up_smem_bytes(nbs, nrb) > cap) return cudaErrorInvalidValue;
        const size_t smem = 1024 + up_smem_bytes(nbs, nrb);
        cudaError_t e = cudaFuncSetAttribute(up_tc_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
        if (e != cudaSuccess) return e;
        e = launch_plain(up_tc_kernel, tiles, kUpThreads, smem, st, true, mU, mR2, mG, N, D, rp,
                         nbs, nrb, rows, static_cast<const __nv_bfloat16*>(h),
                         static_cast<const float*>(inv), static_cast<__nv_bfloat16*>(x));
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace gr
