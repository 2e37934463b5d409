// Fused bf16 GR kernel: one sublayer's write and the next sublayer's read in one traversal of
// the state, with the low-rank projections on the tensor cores (mma.sync, bf16 in, fp32 out).
//
// What it computes, per token t, branch i, channel c ("【论文解读】 Qwen3.8 Flash Next", §二.4):
//   eq write     R'_i = R_i + s_prev_i · y                      (fp32 FMA, stored as bf16)
//   eq rms       inv_i = 1/sqrt(mean_c R'_i[c]^2 + eps)         (on the stored bf16 values)
//   eq gate      z = (1/4) Σ_i inv_i (W_d^(i)γ_i) R'_i,  h = SiLU(z),  G = σ(W_u h)
//   eq use_gate  x = (1/4) Σ_i G_i ⊙ γ_i ⊙ inv_i R'_i
//   eq s         s = 2σ((1/4) Σ_i inv_i (W_w^(i)γ_i) R'_i)
// The GR notes ("Qwen3.8-Flash-Next 架构笔记 · 06 / RESIDUAL", §5) ask that each direction
// traverse the widened state once; here write and read share one traversal: every byte of R,
// y, R', x crosses HBM once.
//
// Organisation (GB300: 152 SMs, 227 KB shared memory and 64 K registers per SM):
//   * A thread-block cluster of C = D/256 CTAs splits the channels: CTA q owns channels
//     [256q, 256q+256) of every branch.
//   * Tiles of 16 tokens (the mma M dimension) arrive by TMA (zero fill past N): R in 64-channel
//     boxes with 128-byte swizzle into a 5-buffer ring, y in 32-channel boxes with 64-byte
//     swizzle (so the A warps' reads of token rows g and g+1 hit different banks) and s_prev
//     into a 2-buffer ring. A tile's chain (load, write, exchange, combine, store) is several
//     times the period at which tiles complete, so the depth of the R ring and of the exchange
//     buffers sets the rate: both are as deep as shared memory allows.
//   * 16 warps in two roles that run concurrently on different tiles:
//     - A warps (8): warp a owns branch a%4 and 128 channels (half a/4). They form R' (written
//       back in place into the R buffer, from where a TMA store takes it to HBM), the
//       per-branch sums of squares (diagonal of R'·R'ᵀ on the tensor cores) and the down
//       projections (W_d, W_w with gamma folded; the mma fragments are resident in tensor
//       memory, which this kernel uses as storage only, so shared memory holds the ring); sum
//       the two halves; and send each token's row sums with st.async to its owner CTA.
//     - B warps (8): the CTA's owned token slots of each tile go round the B warps; for each
//       the warp gathers the token's row sums from every CTA, forms inv, h and s with warp
//       shuffles only, and sends h and inv to every CTA of the cluster. Warp b also owns 32
//       channels of all four branches and keeps its W_u fragments in registers: for each tile
//       it waits for h and inv, runs the up projection on the tensor cores in fp16 (½·W_u
//       packed as fp16; each token's h row scaled by an exact power of two that keeps it below
//       2^15, undone on the accumulator), forms σ(a) = ½ + ½·tanh(a/2), combines the
//       branches from the in-place R', stores x, and releases the R buffer for the next TMA.
//   * mbarriers carry every hand-off (TMA completion, R' ready, R buffer empty, row sums and h
//     arriving from other CTAs); there is no cluster-wide barrier in the steady state.
#include <cuda.h>
#include <string.h>

#include <type_traits>

#include "gr_internal.h"
#include "gr_ptx.cuh"
#include "gr_tc.cuh"

namespace gr {

namespace {

constexpr int kT = 16;                      // tokens per tile (mma M)
constexpr int kAW = 8, kBW = 8;             // A warps, B warps
constexpr int kThreads = (kAW + kBW) * 32;
// Register split: the block launches with 128 per thread (65,536 in all); the A warpgroups give
// 8 each back and the B warpgroups take them (2·128·120 + 2·128·136 = 65,536).
constexpr int kLaunchRegs = 128, kARegs = 120, kBRegs = 136;
static_assert(kAW % 4 == 0 && kBW % 4 == 0, "roles are whole warpgroups");
static_assert(kAW * kARegs + kBW * kBRegs == (kAW + kBW) * kLaunchRegs, "register split");
constexpr int kAThreads = kAW * 32;
constexpr int kDq = 256;                    // channels per branch per CTA
constexpr int kRStages = 5, kYStages = 2;
constexpr int kXStages = 4;                 // slots of the row-sum and h/inv exchange buffers
constexpr int kMbSlots = 32;                // 8-byte slots of the mbarrier area
// Tensor memory: the A warps' down-projection fragments, 16 columns per (A warp, 32-channel
// chunk) in the warp's lane quadrant (warp % 4); A warps a and a + 4 share a quadrant.
constexpr int kTmemCols = 128;
constexpr int kBoxCh = 64;                  // channels per TMA box (128 bytes: the swizzle span)
constexpr int kColBlocks = kDq / kBoxCh;    // 4 boxes per row slice
constexpr int kRBoxBytes = kBoxCh * 4 * kT * 2;        // [16 tok][4 br][64 ch] bf16 = 8 KB
constexpr int kRBufBytes = kColBlocks * kRBoxBytes;     // 32 KB
constexpr int kYBoxCh = 32;                             // y boxes: 64-byte rows, 64B swizzle
constexpr int kYBoxes = kDq / kYBoxCh;                  // 8 boxes per row slice
constexpr int kYBoxBytes = kYBoxCh * kT * 2;            // [16 tok][32 ch] bf16 = 1 KB
constexpr int kYBufBytes = kYBoxes * kYBoxBytes;        // 8 KB (1024-aligned: swizzle atoms)
constexpr int kSBufBytes = kT * 16;                     // s_prev rows of a tile, own small ring
constexpr int kMaxCluster = 16;
constexpr int64_t kMaxTokens = 0x7fffffff - 64;  // token indices stay in int

struct FusedShape {
    int C;            // cluster size = D / kDq
    int ntd;          // n-tiles of the down projection: ceil((r + 4) / 8)
    int half_last;    // 1 if the last down n-tile has <= 4 real rows (only lanes 0..15 stored)
    int upb;          // down-fragment units (16 B) per (A warp, 32-channel chunk)
    int rw;           // row-sum record per (token, branch): r+4 projections, sum of squares,
                      // padded to a multiple of 4 floats (16-byte records)
    int nb4;          // broadcast row per token: inv (4) then h (r values), zero padded to 8 or
                      // 24 floats (strides that keep the combine's float2/float4 reads free of
                      // bank conflicts)
    int down_bytes, up_bytes, gam_bytes, slice_bytes;
    int red_stride;   // partial row sums: [token][A warp][rw] with this token stride (floats)
    int red_bytes, recv_bytes, bcast_bytes;
    int off_gam, off_r, off_y, off_s, off_red, off_recv, off_bcast, off_mbar, smem_bytes;
};

// Packed fragment slice of one CTA: down | up | gamma. Shared memory: gamma | R ring
// (1024-aligned) | y ring | s_prev ring | red | recv[4] | bcast[4] | mbarriers. The down
// fragments go to tensor memory and the up fragments to the B warps' registers, both straight
// from global memory.
__host__ __device__ inline FusedShape fused_shape(int D, int r) {
    FusedShape s{};
    s.C = D / kDq;
    s.ntd = (r + 4 + 7) / 8;
    const int last_rows = r + 4 - 8 * (s.ntd - 1);
    s.half_last = last_rows <= 4 ? 1 : 0;
    s.upb = (s.ntd - 1) * 32 + (s.half_last ? 16 : 32);
    s.rw = round_up(r + 5, 4);
    s.nb4 = r + 4 <= 8 ? 8 : 24;
    s.down_bytes = kAW * 4 * s.upb * 16;
    s.up_bytes = kBW * 32 * 16 * 8;
    s.gam_bytes = 4 * kDq * 4;
    s.slice_bytes = s.down_bytes + s.up_bytes + s.gam_bytes;
    s.red_stride = kAW * s.rw + 8;   // floats per token: ≡ 8 (mod 32) for conflict-free access
    s.red_bytes = kT * s.red_stride * 4;
    s.recv_bytes = s.C * ((kT / s.C) * 4 * s.rw + 4) * 4;   // per source: its rows + 4 pad
    s.bcast_bytes = kT * s.nb4 * 4;
    s.off_gam = 0;
    s.off_r = round_up(s.off_gam + s.gam_bytes, 1024);
    s.off_y = s.off_r + kRStages * kRBufBytes;
    s.off_s = s.off_y + kYStages * kYBufBytes;
    s.off_red = s.off_s + kYStages * kSBufBytes;
    s.off_recv = s.off_red + round_up(s.red_bytes, 16);
    s.off_bcast = s.off_recv + kXStages * round_up(s.recv_bytes, 16);
    s.off_mbar = s.off_bcast + kXStages * round_up(s.bcast_bytes, 16);
    s.smem_bytes = s.off_mbar + round_up(8 * kMbSlots, 16);
    return s;
}

// mbarrier indices
constexpr int kMbRFull = 0;                        // [4] R tile landed (TMA)
constexpr int kMbRReady = kMbRFull + kRStages;     // [4] R' written back (8 A-warp arrivals)
constexpr int kMbREmpty = kMbRReady + kRStages;    // [4] B warps done with the R buffer (8)
constexpr int kMbYFull = kMbREmpty + kRStages;     // [2] y and s_prev landed (TMA)
constexpr int kMbWeights = kMbYFull + kYStages;    // gamma landed
constexpr int kMbRecv = kMbWeights + 1;            // [4] row sums from every CTA (owner)
constexpr int kMbBcast = kMbRecv + kXStages;       // [4] h and inv from every owner
constexpr int kMbCount = kMbBcast + kXStages;
// mbarriers, then the per-buffer counters (rdone), then the tensor-memory base address
static_assert(kMbCount * 8 + kRStages * 4 + 4 <= kMbSlots * 8, "mbarrier area");

// Named barrier among the A warps only.
__device__ __forceinline__ void a_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kAThreads) : "memory");
}

// ---- the kernel -----------------------------------------------------------------------------

template <bool WRITE, int NTD>
__global__ void __launch_bounds__(kThreads, 1)
gr_fused_kernel(const __grid_constant__ CUtensorMap tm_R, const __grid_constant__ CUtensorMap tm_y,
                int N, int D, int r, float eps, const float* __restrict__ s_prev, const char* __restrict__ frag,
                __nv_bfloat16* __restrict__ x, float* __restrict__ s_out) {
    extern __shared__ __align__(1024) char smem[];
    // This CTA is resident: a programmatic dependent (the split's two-pass share) may take the
    // SMs that the clusters leave free once every CTA of the grid is, and only then, so that it
    // cannot occupy an SM a cluster needs.
    dep_launch_dependents();
    const FusedShape S = fused_shape(D, r);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, q4 = lane & 3;
    const uint32_t crank = cluster_ctarank();
    const int C = S.C;
    const int tpc = kT / C;                     // tokens owned per CTA and tile
    // token indices fit in int: the host takes this kernel only for N <= kMaxTokens
    const int ncl = int(ncluster_x()), cid = int(cluster_id_x());
    const int ntiles = (N + kT - 1) / kT;
    const int nlocal = ntiles > cid ? (ntiles - cid + ncl - 1) / ncl : 0;
    const int nk = r + 4, rw = S.rw, nb4 = S.nb4;
    const char* slice = frag + size_t(crank) * S.slice_bytes;

    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + S.off_mbar);
    // per R buffer: count of B warps done with it (the eighth of each round refills it)
    uint32_t* rdone = reinterpret_cast<uint32_t*>(mbar + kMbCount);
    uint32_t* tslot = rdone + kRStages;   // tensor-memory base (written by tcgen05.alloc)
    auto rbuf = [&](int k) { return smem + S.off_r + int(k % kRStages) * kRBufBytes; };
    auto ybuf = [&](int k) { return smem + S.off_y + int(k % kYStages) * kYBufBytes; };
    auto sbuf = [&](int k) { return smem + S.off_s + int(k % kYStages) * kSBufBytes; };
    auto recv_ptr = [&](int p) {
        return reinterpret_cast<float*>(smem + S.off_recv + p * round_up(S.recv_bytes, 16));
    };
    auto bcast_ptr = [&](int p) {
        return reinterpret_cast<float*>(smem + S.off_bcast + p * round_up(S.bcast_bytes, 16));
    };

    if (warp == 0) {
        tmem_alloc(tslot, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < kMbCount; ++i) {
            const bool eight = (i >= kMbRReady && i < kMbRReady + kRStages) ||
                               (i >= kMbREmpty && i < kMbREmpty + kRStages);
            mbar_init(&mbar[i], eight ? 8u : 1u);
        }
        for (int i = 0; i < kRStages; ++i) rdone[i] = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    // TMA of the k-th local tile's R slice: one 4-D box {64 ch, 4 br, 16 tok, 4 blocks} = the
    // CTA's 256 channels as four 64-channel blocks (one thread).
    auto issue_r = [&](int k) {
        if (k >= nlocal) return;
        const int t0 = int((cid + k * ncl) * kT);
        uint64_t* bar = &mbar[kMbRFull + int(k % kRStages)];
        mbar_expect_tx(bar, uint32_t(kRBufBytes));
        tma_load_4d(rbuf(k), &tm_R, 0, 0, t0, int(crank) * kColBlocks, bar);
    };
    // TMA of the k-th local tile's y slice: one 3-D box {32 ch, 16 tok, 8 chunks} (lane 0, which
    // also arms the barrier) and its s_prev rows (lane 1).
    auto issue_y = [&](int k, int ln) {
        if (!WRITE || k >= nlocal) return;
        const int t0 = int((cid + k * ncl) * kT);
        const int nv = int(N - t0 < kT ? N - t0 : kT);
        uint64_t* bar = &mbar[kMbYFull + int(k % kYStages)];
        if (ln == 0) {
            mbar_expect_tx(bar, uint32_t(kYBufBytes + nv * 16));
            tma_load_3d(ybuf(k), &tm_y, 0, t0, int(crank) * kYBoxes, bar);
        }
        if (ln == 1) bulk_g2s(sbuf(k), s_prev + size_t(t0) * 4, uint32_t(nv) * 16, bar);
    };

    if (tid == 0) {
        mbar_expect_tx(&mbar[kMbWeights], uint32_t(S.gam_bytes));
        bulk_g2s(smem + S.off_gam, slice + S.down_bytes + S.up_bytes, uint32_t(S.gam_bytes),
                 &mbar[kMbWeights]);
    }
    if (warp == 0 && lane < 2) {
        if (lane == 0)
            for (int k = 0; k < kRStages; ++k) issue_r(k);
        for (int k = 0; k < kYStages; ++k) issue_y(k, lane);
    }
    cluster_sync();  // every CTA of the cluster runs before any shared::cluster access

    if (warp < kAW) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kARegs));
        // =============================== A warps ===========================================
        const int a = warp, ib = a & 3, hh = a >> 2;
        // send descriptors: float4 items it = tid, tid + 256 of the tile's 16·rw row-sum items
        // This thread's row-sum items, the same in every tile: float4 items it = tid and
        // tid + 256 of the tile's 16·rw; item it is token it / rw, branch (it % rw) / (rw/4),
        // 4 values at o, and its value is red[tok][branch][o] + red[tok][branch + 4][o].
        int s_red[2], s_off[2], s_own[2];
        bool s_has[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int it = tid + u * kAThreads;
            s_has[u] = it < kT * rw;
            const int tok = it / rw, rem4 = it - tok * rw;
            const int bi = rem4 / (rw / 4), o = 4 * (rem4 - bi * (rw / 4));
            const int owner = tok / tpc, slot = tok - owner * tpc;
            s_red[u] = tok * S.red_stride + bi * rw + o;
            // byte offset in the owner's receive slot: padded per-source rows of tpc·4·rw + 4
            s_off[u] = (int(crank) * (tpc * 4 * rw + 4) + slot * 4 * rw + 4 * rem4) * 4;
            s_own[u] = owner;
        }
        // this warp's down fragments into its tensor-memory columns: 16 per 32-channel chunk
        // j4, units (n-tile j, lane) at columns 4j .. 4j+3 (zero past the real n-tiles)
        const uint32_t ta = tmem + (uint32_t((a & 3) * 32) << 16) + uint32_t((a >> 2) * 64);
        {
            const uint4* gdown = reinterpret_cast<const uint4*>(slice);
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
                uint32_t v[16];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint4 b = make_uint4(0u, 0u, 0u, 0u);
                    const bool last_half = (j == NTD - 1) && S.half_last;
                    if (j < NTD && (!last_half || lane < 16))
                        b = gdown[(a * 4 + j4) * S.upb + j * 32 + lane];
                    v[4 * j] = b.x, v[4 * j + 1] = b.y, v[4 * j + 2] = b.z, v[4 * j + 3] = b.w;
                }
                tmem_st16(ta + uint32_t(j4 * 16), v);
            }
            tmem_wait_st();
        }
        float* red = reinterpret_cast<float*>(smem + S.off_red);   // [kT][kAW][rw], padded
        for (int k = 0; k < nlocal; ++k) {
            const int p = int(k % kXStages);
            char* rb = rbuf(k);
            const char* yb = ybuf(k);
            const char* sb = sbuf(k);
            mbar_wait(&mbar[kMbRFull + int(k % kRStages)], uint32_t((k / kRStages) & 1));
            // y of tile k+1 into the buffer of tile k-1 (free since that tile's a_sync): issued
            // once tile k's R has landed, so the y and R loads do not queue up together
            if (k >= 1 && a == 0 && lane < 2) issue_y(k - 1 + kYStages, lane);
            if (WRITE) mbar_wait(&mbar[kMbYFull + int(k % kYStages)], uint32_t((k / kYStages) & 1));

            // write (eq write) for this warp's branch and 128 channels; R' back in place.
            // All loads first: the in-place stores would otherwise order every later load.
            uint32_t Rp[2][4][4];  // [row g / g+8][chunk][channel pair]
            uint4 yv[2][4];
            float sp[2] = {0.f, 0.f};
#pragma unroll
            for (int row = 0; row < 2; ++row) {
                const int tok = g + 8 * row, brow = tok * 4 + ib;
                if (WRITE) sp[row] = *reinterpret_cast<const float*>(sb + tok * 16 + ib * 4);
#pragma unroll
                for (int j4 = 0; j4 < 4; ++j4) {
                    const int cb = hh * 2 + (j4 >> 1), cch = ((j4 & 1) << 2) | q4;
                    const uint4 rv =
                        *reinterpret_cast<const uint4*>(rb + cb * kRBoxBytes + swz(brow, cch));
                    Rp[row][j4][0] = rv.x, Rp[row][j4][1] = rv.y, Rp[row][j4][2] = rv.z,
                    Rp[row][j4][3] = rv.w;
                    if (WRITE)
                        yv[row][j4] = *reinterpret_cast<const uint4*>(
                            yb + (hh * 4 + j4) * kYBoxBytes + swz64(tok, q4));
                }
            }
            if (WRITE) {
#pragma unroll
                for (int row = 0; row < 2; ++row) {
                    const int tok = g + 8 * row, brow = tok * 4 + ib;
                    const uint64_t s2 = f2(sp[row], sp[row]);
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4) {
                        const int cb = hh * 2 + (j4 >> 1), cch = ((j4 & 1) << 2) | q4;
                        const uint32_t yw[4] = {yv[row][j4].x, yv[row][j4].y, yv[row][j4].z,
                                                yv[row][j4].w};
#pragma unroll
                        for (int m = 0; m < 4; ++m)
                            Rp[row][j4][m] = f2_to_bf2(
                                fma2(s2, bf2_to_f2(yw[m]), bf2_to_f2(Rp[row][j4][m])));
                        const uint4 o = make_uint4(Rp[row][j4][0], Rp[row][j4][1],
                                                   Rp[row][j4][2], Rp[row][j4][3]);
                        *reinterpret_cast<uint4*>(rb + cb * kRBoxBytes + swz(brow, cch)) = o;
                    }
                }
            }
            if (WRITE) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&mbar[kMbRReady + int(k % kRStages)]);

            // sums of squares (diagonal of R'·R'ᵀ) and down projections over 128 channels
            float acc[NTD][4], sq0[4], sq1[4];
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
                uint32_t bw[16];   // this chunk's down fragments, from tensor memory
                tmem_ld16_nowait(ta + uint32_t(j4 * 16), bw);
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const uint32_t a0 = Rp[0][j4][2 * ks], a1 = Rp[1][j4][2 * ks];
                    const uint32_t a2 = Rp[0][j4][2 * ks + 1], a3 = Rp[1][j4][2 * ks + 1];
                    if (j4 == 0 && ks == 0) {
                        mma_bf16_z(sq0, a0, a1, a2, a3, a0, a2);   // columns: tokens 0..7
                        mma_bf16_z(sq1, a0, a1, a2, a3, a1, a3);   // columns: tokens 8..15
                    } else {
                        mma_bf16(sq0, a0, a1, a2, a3, a0, a2);
                        mma_bf16(sq1, a0, a1, a2, a3, a1, a3);
                    }
                }
                tmem_wait_ld(bw);
#pragma unroll
                for (int j = 0; j < NTD; ++j) {
                    const uint4 b = make_uint4(bw[4 * j], bw[4 * j + 1], bw[4 * j + 2],
                                               bw[4 * j + 3]);
                    if (j4 == 0)
                        mma_bf16_z(acc[j], Rp[0][j4][0], Rp[1][j4][0], Rp[0][j4][1], Rp[1][j4][1],
                                   b.x, b.y);
                    else
                        mma_bf16(acc[j], Rp[0][j4][0], Rp[1][j4][0], Rp[0][j4][1], Rp[1][j4][1],
                                 b.x, b.y);
                    mma_bf16(acc[j], Rp[0][j4][2], Rp[1][j4][2], Rp[0][j4][3], Rp[1][j4][3], b.z,
                             b.w);
                }
            }
            // Before the row sums of tile k leave, every owner must be done with the exchange
            // slot of tile k-4 and this CTA's B warps with its h/inv slot: both follow from
            // the local combine of tile k-4 (it needed h from every owner).
            if (k >= kXStages)
                mbar_wait(&mbar[kMbREmpty + int((k - kXStages) % kRStages)],
                          uint32_t(((k - kXStages) / kRStages) & 1));
            float* r0 = red + g * S.red_stride + a * rw;
            float* r1 = red + (g + 8) * S.red_stride + a * rw;
#pragma unroll
            for (int j = 0; j < NTD; ++j) {
                const int o = 8 * j + 2 * q4;
                if (o + 1 < nk) {
                    *reinterpret_cast<float2*>(r0 + o) = make_float2(acc[j][0], acc[j][1]);
                    *reinterpret_cast<float2*>(r1 + o) = make_float2(acc[j][2], acc[j][3]);
                } else if (o < nk) {
                    r0[o] = acc[j][0], r1[o] = acc[j][2];
                }
            }
            if (q4 == (g >> 1)) {
                r0[nk] = (g & 1) ? sq0[1] : sq0[0];
                r1[nk] = (g & 1) ? sq1[3] : sq1[2];
            }
            a_sync();
            {
                const uint32_t recv_u32 = smem_u32(recv_ptr(p)), bar_u32 = smem_u32(&mbar[kMbRecv + p]);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (!s_has[u]) continue;
                    const float4 u0 = *reinterpret_cast<const float4*>(red + s_red[u]);
                    const float4 u1 = *reinterpret_cast<const float4*>(red + s_red[u] + 4 * rw);
                    st_async_v4_mapped(map_rank(recv_u32 + uint32_t(s_off[u]), uint32_t(s_own[u])),
                                       map_rank(bar_u32, uint32_t(s_own[u])), u0.x + u1.x,
                                       u0.y + u1.y, u0.z + u1.z, u0.w + u1.w);
                }
            }
            a_sync();  // red is free again
        }
        tc_fence_before();   // this warp's tensor-memory loads are done before the dealloc
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kBRegs));
        // =============================== B warps ===========================================
        const int b = warp - kAW;
        const int cb = b >> 1, cch = ((b & 1) << 2) | q4;
        __nv_bfloat16* const xg = x + size_t(g) * D + size_t(crank) * kDq + b * 32 + q4 * 8;
        // W_u fragments (pre-scaled by ½) for this warp's 32 channels: [branch*4 + n-tile]
        uint2 wu[16];
        {
            const uint4* src = reinterpret_cast<const uint4*>(slice + S.down_bytes) +
                               (b * 32 + lane) * 8;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const uint4 v = src[m];
                wu[2 * m] = make_uint2(v.x, v.y);
                wu[2 * m + 1] = make_uint2(v.z, v.w);
            }
        }
        mbar_wait(&mbar[kMbWeights], 0);
        const float* s_gam = reinterpret_cast<const float*>(smem + S.off_gam);
        const int bt = tid - kAThreads;              // 0 .. 255
        const float inv_d = 1.0f / float(D);
        int lc = 0;                                  // log2 C (C is a power of two)
        while ((1 << lc) < C) ++lc;

        // Owner step for owned token slot `slot` of local tile k, done by one warp without any
        // block-level barrier: gather the row sums of that token from every CTA (lane l holds
        // the float4 group l of the token's 4·rw values), inv_i = 1/sqrt(ssq_i/D + eps) from the
        // lanes holding the sums of squares, z and u as shuffle sums over the four branch lanes
        // of each output group, then h (eq gate), s (eq s), and the h/inv row to every CTA.
        const int rq = rw / 4;                      // float4 groups per branch record
        auto owner_slot = [&](int k, int slot) {
            const int t0 = (cid + k * ncl) * kT;
            const int p = int(k % kXStages);
            const int tok = int(crank) * tpc + slot;
            const float* recv = recv_ptr(p);
            const int srcstride = tpc * 4 * rw + 4;
            float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (lane < 4 * rq) {
                const float* base = recv + slot * 4 * rw + 4 * lane;
#pragma unroll 8
                for (int src = 0; src < C; ++src) {
                    const float4 b4 = *reinterpret_cast<const float4*>(base + src * srcstride);
                    v4.x += b4.x, v4.y += b4.y, v4.z += b4.z, v4.w += b4.w;
                }
            }
            // inv_i: the sum of squares of branch i is value nk of its record, i.e. component
            // nk & 3 of lane i·rq + nk / 4
            const int cs = nk & 3;
            const float mine = cs == 0 ? v4.x : cs == 1 ? v4.y : cs == 2 ? v4.z : v4.w;
            float inv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                inv[i] = rsqrtf(fmaf(__shfl_sync(0xffffffffu, mine, i * rq + (nk >> 2)), inv_d, eps));
            // z/u of outputs 4l .. 4l+3 = ¼ Σ_i inv_i · P[i][o]: scale by the lane's branch
            // factor, then two shuffle steps leave the branch sum in lanes l < rq
            const float sc = lane < rq ? inv[0] : lane < 2 * rq ? inv[1] : lane < 3 * rq ? inv[2]
                           : lane < 4 * rq ? inv[3] : 0.f;
            const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
            float zz[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float t = sc * vv[e];
                t += __shfl_down_sync(0xffffffffu, t, rq);
                t += __shfl_down_sync(0xffffffffu, t, 2 * rq);
                zz[e] = 0.25f * t;
            }
            // lane l < rq: h = SiLU(z) for outputs kk = 4l+e < r; s = 2σ(u) for r <= kk < r+4.
            // The four logistic values are independent (no branch between them).
            float hv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kk = 4 * lane + e;
                // σ(z) = 1/(1 + e^-z): the hardware exp2 and reciprocal are a few ulp in fp32
                const float sg = __fdividef(1.0f, 1.0f + __expf(-zz[e]));
                hv[e] = kk < r ? zz[e] * sg : 0.f;
                if (lane < rq && kk >= r && kk < nk && t0 + tok < N)
                    s_out[size_t(t0 + tok) * 4 + (kk - r)] = 2.0f * sg;
            }
            // Broadcast row of the token: inv (4), h (r values), zeros up to nb4. Lane ->
            // destination CTA lane % C (C divides 32); each round covers 32 / C float4 groups;
            // group 0 is inv, and component e of group g4 > 0 is h[4·(g4-1) + e], held in hv[e]
            // of lane g4 - 1.
            const uint32_t dst = uint32_t(lane & (C - 1));
            const uint32_t ra = map_rank(smem_u32(bcast_ptr(p) + tok * nb4), dst);
            const uint32_t rb = map_rank(smem_u32(&mbar[kMbBcast + p]), dst);
            const int ngrp = nb4 / 4, per = 32 >> lc;
            for (int g0 = 0; g0 < ngrp; g0 += per) {
                const int g4 = g0 + (lane >> lc);
                float v[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float hj = __shfl_sync(0xffffffffu, hv[e], (g4 - 1) & 31);
                    v[e] = g4 == 0 ? inv[e] : (4 * (g4 - 1) + e < r ? hj : 0.f);
                }
                if (g4 < ngrp) st_async_v4_mapped(ra + 16u * uint32_t(g4), rb, v[0], v[1], v[2], v[3]);
            }
        };

        // Up projection (eq gate), gates, combine (eq use_gate) and x for local tile k; then the
        // R buffer is released and refilled with tile k+5.
        auto combine = [&](int k) {
            const int t0 = (cid + k * ncl) * kT;
            const int p = int(k % kXStages);
            const char* rb = rbuf(k);
            mbar_wait(&mbar[kMbBcast + p], uint32_t((k / kXStages) & 1));
            mbar_wait(&mbar[kMbRReady + int(k % kRStages)], uint32_t((k / kRStages) & 1));
            // R' of this tile (written back in place by the A warps) goes to HBM by one TMA
            // store (B warp 0, lane 0); the box is clipped to the N tokens
            if (WRITE && b == 0 && lane == 0) {
                tma_store_4d(&tm_R, rb, 0, 0, t0, int(crank) * kColBlocks);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
            const float* bc = bcast_ptr(p);
            // h as fp16 A fragments (11 significant bits, as the packed ½·W_u), each token's row
            // scaled by an exact power of two that keeps it below 2^15; the scale is undone on
            // the fp32 accumulator
            uint32_t ah[4];
            float2 hv2[4];
            float ma = 0.f, mb = 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int tk = g + 8 * (m & 1), kc = 2 * q4 + 8 * (m >> 1);
                // h[kc], h[kc+1] (zero past r: the row is zero padded after h)
                hv2[m] = kc < r ? *reinterpret_cast<const float2*>(bc + tk * nb4 + 4 + kc)
                                : make_float2(0.f, 0.f);
                const float mm = fmaxf(fabsf(hv2[m].x), fabsf(hv2[m].y));
                if (m & 1) mb = fmaxf(mb, mm);
                else ma = fmaxf(ma, mm);
            }
            // the four lanes of a quad hold the whole row of a token
            ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
            ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
            const int ea = min(max(((__float_as_int(ma) >> 23) & 0xff) - 127 - 14, 0), 126);
            const int eb = min(max(((__float_as_int(mb) >> 23) & 0xff) - 127 - 14, 0), 126);
            const float sa = __int_as_float((127 - ea) << 23), sb = __int_as_float((127 - eb) << 23);
            const float ua = __int_as_float((127 + ea) << 23), ub = __int_as_float((127 + eb) << 23);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float sc = (m & 1) ? sb : sa;
                ah[m] = pack_h2(hv2[m].x * sc, hv2[m].y * sc);
            }
            uint64_t xacc2[2][4];   // [row][channel pair], packed fp32 pairs
#pragma unroll
            for (int row = 0; row < 2; ++row)
#pragma unroll
                for (int j = 0; j < 4; ++j) xacc2[row][j] = f2(0.f, 0.f);
            const float4 iv0 = *reinterpret_cast<const float4*>(bc + g * nb4);
            const float4 iv1 = *reinterpret_cast<const float4*>(bc + (g + 8) * nb4);
            const float inv0s[4] = {iv0.x, iv0.y, iv0.z, iv0.w};
            const float inv1s[4] = {iv1.x, iv1.y, iv1.z, iv1.w};
            // SCALED: some token row of the warp was scaled down (ea or eb > 0) and its logits
            // are scaled back; otherwise every scale is 1 and the code path has no multiplies
            // for it (the same result: a product with 1 is exact)
            auto gate_combine = [&](auto scaled) {
                constexpr bool SCALED = decltype(scaled)::value;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float inv0 = inv0s[i], inv1 = inv1s[i];
                const uint4 r0 = *reinterpret_cast<const uint4*>(rb + cb * kRBoxBytes +
                                                                 swz(g * 4 + i, cch));
                const uint4 r1 = *reinterpret_cast<const uint4*>(rb + cb * kRBoxBytes +
                                                                 swz((g + 8) * 4 + i, cch));
                const uint32_t q0[4] = {r0.x, r0.y, r0.z, r0.w};
                const uint32_t q1[4] = {r1.x, r1.y, r1.z, r1.w};
                const float4 gA = *reinterpret_cast<const float4*>(s_gam + i * kDq + b * 32 + q4 * 8);
                const float4 gB =
                    *reinterpret_cast<const float4*>(s_gam + i * kDq + b * 32 + q4 * 8 + 4);
                const float gm[8] = {gA.x, gA.y, gA.z, gA.w, gB.x, gB.y, gB.z, gB.w};
                const uint64_t inv0_2 = f2(inv0, inv0), inv1_2 = f2(inv1, inv1);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float c[4];
                    mma_f16_z(c, ah[0], ah[1], ah[2], ah[3], wu[i * 4 + j].x, wu[i * 4 + j].y);
                    if constexpr (SCALED) {
                        c[0] *= ua;
                        c[1] *= ua;
                        c[2] *= ub;
                        c[3] *= ub;
                    }
                    const uint64_t gm2 = f2(gm[2 * j], gm[2 * j + 1]);
                    const uint64_t u0 = mul2(gm2, bf2_to_f2(q0[j]));   // γ·R' (row g)
                    const uint64_t u1 = mul2(gm2, bf2_to_f2(q1[j]));   // γ·R' (row g+8)
                    // G·u = ½u + ½·tanh(·)·u; the ½ is applied once at the end
                    const uint64_t w0 = fma2(f2(tanh_approx(c[0]), tanh_approx(c[1])), u0, u0);
                    const uint64_t w1 = fma2(f2(tanh_approx(c[2]), tanh_approx(c[3])), u1, u1);
                    xacc2[0][j] = fma2(inv0_2, w0, xacc2[0][j]);
                    xacc2[1][j] = fma2(inv1_2, w1, xacc2[1][j]);
                }
            }
            };
            if (__all_sync(0xffffffffu, (ea | eb) == 0)) gate_combine(std::false_type{});
            else gate_combine(std::true_type{});
            // the buffer is released only after the TMA store has read it
            if (WRITE && b == 0 && lane == 0)
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&mbar[kMbREmpty + int(k % kRStages)]);
            const uint64_t eighth = f2(0.125f, 0.125f);
#pragma unroll
            for (int row = 0; row < 2; ++row) {
                const int tok = g + 8 * row;
                if (t0 + tok < N) {
                    __nv_bfloat16* dst = xg + (size_t(t0) + row * 8) * size_t(D);
                    *reinterpret_cast<uint4*>(dst) = make_uint4(
                        f2_to_bf2(mul2(eighth, xacc2[row][0])), f2_to_bf2(mul2(eighth, xacc2[row][1])),
                        f2_to_bf2(mul2(eighth, xacc2[row][2])), f2_to_bf2(mul2(eighth, xacc2[row][3])));
                }
            }
            // refill: the last B warp done with this buffer loads R of tile k+5 into it (lane 0);
            // no other warp waits for it
            if (k + kRStages < nlocal) {
                uint32_t last = 0;
                if (lane == 0) last = (atomicAdd(&rdone[k % kRStages], 1u) & (kBW - 1)) == kBW - 1;
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last && lane == 0) {
                    mbar_wait(&mbar[kMbREmpty + int(k % kRStages)], uint32_t((k / kRStages) & 1));
                    issue_r(k + kRStages);
                }
            }
        };

        for (int k = 0; k < nlocal; ++k) {
            const int p = int(k % kXStages);
            if (bt == 0) {
                mbar_expect_tx(&mbar[kMbRecv + p], uint32_t(C * tpc * 4 * rw * 4));
                mbar_expect_tx(&mbar[kMbBcast + p], uint32_t(kT * nb4 * 4));
            }
            // owned slot j of tile k goes to B warp (k·tpc + j) mod 8, so the owner work
            // rotates over the warps
            const int first = (b - k * tpc) & (kBW - 1);
            if (first < tpc) {
                mbar_wait(&mbar[kMbRecv + p], uint32_t((k / kXStages) & 1));
                for (int slot = first; slot < tpc; slot += kBW) owner_slot(k, slot);
            }
            if (k > 0) combine(k - 1);
        }
        if (nlocal > 0) combine(nlocal - 1);
        // the R' stores must be complete before the CTA leaves
        if (WRITE && b == 0 && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }
    cluster_sync();  // no CTA leaves while shared::cluster traffic to it may be in flight
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Fragment section: for CTA slice q, [down | up | gamma].
//   down: [A warp a][32-channel chunk j4][upb units of 16 B]: unit (n-tile j, lane) holds
//         W'[8j + lane/4][8 channels 128·(a/4) + 32·j4 + 8·(lane%4) ...] of branch a%4, where
//         rows 0..r-1 are W_d, rows r..r+3 are W_w (gamma folded) and the rest are zero.
//   up:   [B warp b][lane][branch i][n-tile j] 8 B: ½·W_u[i·D + c][k] for the channel
//         c = 256q + 32b + 8·(g/2) + 2j + g%2 (g = lane/4) and k = 2·(lane%4) + {0, 1, 8, 9}.
//   gamma: fp32 [4][256] of this CTA's channels.
__global__ void pack_fused_kernel(int D, int r, const float* __restrict__ gamma,
                                  const float* __restrict__ wd, const float* __restrict__ wu,
                                  const float* __restrict__ ww, char* __restrict__ frag) {
    const FusedShape S = fused_shape(D, r);
    const int K = 4 * D;
    const int n_down = kAW * 4 * S.upb;           // 16-byte units per slice
    const int n_up = kBW * 32 * 16;               // 8-byte units per slice
    const int n_gam = 4 * kDq;                    // floats per slice
    const int per_slice = n_down + n_up + n_gam;
    const int64_t total = int64_t(S.C) * per_slice;
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int q = int(e / per_slice);
        int u = int(e - int64_t(q) * per_slice);
        char* slice = frag + size_t(q) * S.slice_bytes;
        if (u < n_down) {
            const int aj = u / S.upb, rest = u - aj * S.upb;   // aj = A warp * 4 + chunk
            const int j = rest >> 5, lane = rest & 31;
            const int a = aj >> 2, j4 = aj & 3;
            const int i = a & 3, hh = a >> 2;
            const int n = 8 * j + (lane >> 2);
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(slice + size_t(u) * 16);
            for (int c8 = 0; c8 < 8; ++c8) {
                const int m = i * D + q * kDq + hh * 128 + j4 * 32 + (lane & 3) * 8 + c8;
                float v = 0.f;
                if (n < r) v = wd[size_t(n) * K + m] * gamma[m];
                else if (n < r + 4) v = ww[size_t(n - r) * K + m] * gamma[m];
                dst[c8] = __float2bfloat16_rn(v);
            }
        } else if ((u -= n_down) < n_up) {
            const int nt = u & 15, rest = u >> 4;       // nt = branch*4 + n-tile
            const int lane = rest & 31, bw = rest >> 5;
            const int i = nt >> 2, j = nt & 3;
            const int gg = lane >> 2, qq = lane & 3;
            const int m = i * D + q * kDq + bw * 32 + 8 * (gg >> 1) + 2 * j + (gg & 1);
            const int kk[4] = {2 * qq, 2 * qq + 1, 2 * qq + 8, 2 * qq + 9};
            __half* dst = reinterpret_cast<__half*>(slice + S.down_bytes + size_t(u) * 8);
            for (int t = 0; t < 4; ++t) {
                const float v = kk[t] < r ? 0.5f * wu[size_t(m) * r + kk[t]] : 0.f;
                dst[t] = __float2half_rn(fminf(fmaxf(v, -65504.f), 65504.f));
            }
        } else {
            u -= n_up;
            const int i = u / kDq, cl = u - i * kDq;
            reinterpret_cast<float*>(slice + S.down_bytes + S.up_bytes)[u] =
                gamma[i * D + q * kDq + cl];
        }
    }
}

// ---- host side ------------------------------------------------------------------------------

// R as a 4-D tensor {channel within a 64-channel block, branch, token, block}; box
// {64, 4, 16, 4} (one CTA's 256 channels of a tile), 128-byte swizzle on the 128-byte rows.
bool make_map_R(CUtensorMap* m, const void* R, int64_t N, int D) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {cuuint64_t(kBoxCh), 4, cuuint64_t(N), cuuint64_t(D / kBoxCh)};
    const cuuint64_t strides[3] = {cuuint64_t(D) * 2, cuuint64_t(D) * 8, cuuint64_t(kBoxCh) * 2};
    const cuuint32_t box[4] = {kBoxCh, 4, kT, kColBlocks};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(R), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// y as a 3-D tensor {channel within a 32-channel chunk, token, chunk}; box {32, 16, 8} (one
// CTA's 256 channels of a tile), 64-byte swizzle on the 64-byte rows.
bool make_map_y(CUtensorMap* m, const void* y, int64_t N, int D) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {cuuint64_t(kYBoxCh), cuuint64_t(N), cuuint64_t(D / kYBoxCh)};
    const cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(kYBoxCh) * 2};
    const cuuint32_t box[3] = {kYBoxCh, kT, kYBoxes};
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(y), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

struct ClusterCache {
    int max_clusters[2][4][5];  // [WRITE][NTD][log2 C], 0 = not queried
    int smem_set[2][4];         // [WRITE][NTD]: dynamic shared memory granted (attributes set)
};
ClusterCache g_cluster_cache[64];

// Kernel attributes and the launch configuration (all but grid and stream) of one
// instantiation, and the number of its clusters that can be resident at once (queried once per
// device and cached).
template <bool WRITE, int NTD>
cudaError_t prepare_t(const FusedShape& S, cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr,
                      int& max_clusters) {
    auto kern = gr_fused_kernel<WRITE, NTD>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    ClusterCache& cc = g_cluster_cache[dev & 63];
    // the attributes are checked and set once per device and instantiation (the largest shared
    // memory so far), not on every launch
    if (cc.smem_set[WRITE ? 1 : 0][NTD] < S.smem_bytes) {
        // the register split assumes this launch size; anything else could stall setmaxnreg.inc
        cudaFuncAttributes fa;
        if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
        if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S.smem_bytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        cc.smem_set[WRITE ? 1 : 0][NTD] = S.smem_bytes;
    }
    cfg = cudaLaunchConfig_t{};
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(S.C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = size_t(S.smem_bytes);
    int lc = 0;
    while ((1 << lc) < S.C) ++lc;
    int& maxc = cc.max_clusters[WRITE ? 1 : 0][NTD][lc];
    if (maxc == 0) {
        cfg.gridDim = dim3(unsigned(S.C * 64));
        int n = 0;
        if ((e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg)) != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        maxc = n;
    }
    max_clusters = maxc;
    return cudaSuccess;
}

template <bool WRITE, int NTD>
cudaError_t launch_t(int64_t N, int D, int r, float eps, void* R, const void* y,
                     const float* s_prev, const char* frag, void* x, float* s_out,
                     cudaStream_t st) {
    const FusedShape S = fused_shape(D, r);
    CUtensorMap mR, my;
    memset(&my, 0, sizeof(my));
    if (!make_map_R(&mR, R, N, D)) return cudaErrorInvalidValue;
    if (WRITE && !make_map_y(&my, y, N, D)) return cudaErrorInvalidValue;
    auto kern = gr_fused_kernel<WRITE, NTD>;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    int maxc = 0;
    cudaError_t e = prepare_t<WRITE, NTD>(S, cfg, attr, maxc);
    if (e != cudaSuccess) return e;
    cfg.stream = st;
    const int64_t ntiles = (N + kT - 1) / kT;
    const int64_t ncl = ntiles < maxc ? ntiles : maxc;
    cfg.gridDim = dim3(unsigned(ncl * S.C));
    if (N > kMaxTokens) return cudaErrorInvalidValue;
    return cudaLaunchKernelEx(&cfg, kern, mR, my, int(N), D, r, eps, s_prev, frag,
                              static_cast<__nv_bfloat16*>(x), s_out);
}

template <bool WRITE>
int max_ctas_w(int D, int r) {
    const FusedShape S = fused_shape(D, r);
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    int maxc = 0;
    cudaError_t e = cudaErrorInvalidValue;
    switch (S.ntd) {
        case 1: e = prepare_t<WRITE, 1>(S, cfg, attr, maxc); break;
        case 2: e = prepare_t<WRITE, 2>(S, cfg, attr, maxc); break;
        case 3: e = prepare_t<WRITE, 3>(S, cfg, attr, maxc); break;
        default: break;
    }
    return e == cudaSuccess ? maxc * S.C : 0;
}

template <bool WRITE>
cudaError_t launch_w(int64_t N, int D, int r, float eps, void* R, const void* y,
                     const float* s_prev, const char* frag, void* x, float* s_out,
                     cudaStream_t st) {
    switch (fused_shape(D, r).ntd) {
        case 1: return launch_t<WRITE, 1>(N, D, r, eps, R, y, s_prev, frag, x, s_out, st);
        case 2: return launch_t<WRITE, 2>(N, D, r, eps, R, y, s_prev, frag, x, s_out, st);
        case 3: return launch_t<WRITE, 3>(N, D, r, eps, R, y, s_prev, frag, x, s_out, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool fused_supported(int D, int r) {
    if (D % kDq != 0 || r < 1 || r > 16) return false;
    const int C = D / kDq;
    if (C < 1 || C > kMaxCluster || (kT % C) != 0) return false;
    return fused_shape(D, r).smem_bytes <= 227 * 1024;
}

int64_t fused_max_tokens() { return kMaxTokens; }

int fused_resident_ctas(int D, int r, bool write) {
    if (!fused_supported(D, r)) return 0;
    return write ? max_ctas_w<true>(D, r) : max_ctas_w<false>(D, r);
}

namespace {
// Self-test of the bounded waits: one thread waits on an mbarrier that nothing arrives at, with
// the fused kernel's wait helper and a short limit; the wait gives up and sets the status word.
__global__ void wait_selftest_kernel(long long limit) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1u);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_wait(&bar, 0u, limit);   // phase 0 never completes
    }
}
}  // namespace

cudaError_t launch_wait_selftest(long long limit_cycles, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(limit_cycles);
    return cudaGetLastError();
}

int fused_status(bool clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_wait_status, sizeof(v)) != cudaSuccess) return -1;
    if (clear && v) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(g_wait_status, &z, sizeof(z)) != cudaSuccess) return -1;
    }
    return int(v);
}

size_t fused_frag_bytes(int D, int r) {
    const FusedShape S = fused_shape(D, r);
    return size_t(S.C) * size_t(S.slice_bytes);
}

cudaError_t launch_pack_fused(int D, int r, const float* gamma, const float* wd, const float* wu,
                              const float* ww, void* frag, cudaStream_t st) {
    const int64_t units = int64_t(fused_frag_bytes(D, r)) / 8;
    const int threads = 256;
    const int64_t want = (units + threads - 1) / threads;
    const int64_t cap = int64_t(sm_count()) * 8;
    pack_fused_kernel<<<int(want < cap ? want : cap), threads, 0, st>>>(
        D, r, gamma, wd, wu, ww, static_cast<char*>(frag));
    return cudaGetLastError();
}

cudaError_t launch_fused_bf16(int64_t N, int D, int r, float eps, void* R, const void* y,
                              const float* s_prev, const void* packed, void* x, float* s_out,
                              cudaStream_t st) {
    if (N == 0) return cudaSuccess;
    const Layout L = make_layout(D, r, GR_BF16);
    const char* frag = static_cast<const char*>(packed) + L.frag;
    if (y != nullptr)
        return launch_w<true>(N, D, r, eps, R, y, s_prev, frag, x, s_out, st);
    return launch_w<false>(N, D, r, eps, R, y, s_prev, frag, x, s_out, st);
}

}  // namespace gr
