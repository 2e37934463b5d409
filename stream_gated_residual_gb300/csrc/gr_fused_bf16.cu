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
// Organisation (GB300: 152 SMs, 227 KB shared memory per CTA):
//   * A thread-block cluster of C = D/256 CTAs splits the channels: CTA q owns channels
//     [256q, 256q+256) of every branch and keeps that slice of the packed weights (mma
//     fragments, gamma folded into W_d and W_w) and of gamma resident in shared memory.
//   * Tiles of 16 tokens (the mma M dimension) stream through a 3-stage ring of shared-memory
//     buffers filled by TMA tensor copies (128-byte swizzle, 9 copies per tile) completing on
//     mbarriers.
//   * 8 warps per CTA; warp w owns 32 channels of each branch. A thread holds 8 channels of two
//     token rows per branch; those registers are directly the A fragments of mma.m16n8k16 once
//     the K index is permuted consistently with the packed B fragments. The same registers as
//     B operand give R'·R'ᵀ, whose diagonal is the per-branch sum of squares.
//   * The per-token row reductions (4 sums of squares and 4·(r+4) partial projections) are
//     summed over warps in shared memory, then sent with st.async to the token's owner CTA
//     (completing on the owner's mbarrier), which forms inv, h and s and sends h and inv to
//     every CTA of the cluster the same way. No cluster-wide barrier in the steady state.
//   * The up-projection runs on the tensor cores with h split into bf16 hi + lo parts (about 16
//     significant bits), and σ(a) = ½ + ½·tanh(a/2) with W_u pre-scaled by ½ (exact in bf16).
#include <cuda.h>
#include <string.h>

#include "gr_internal.h"

namespace gr {

namespace {

constexpr int kT = 16;                      // tokens per tile (mma M)
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kDq = kWarps * 32;            // channels per branch per CTA
constexpr int kStages = 3;
constexpr int kBoxCh = 64;                  // channels per TMA box (128 bytes: the swizzle span)
constexpr int kColBlocks = kDq / kBoxCh;    // 4 boxes per row slice
constexpr int kRBoxBytes = kBoxCh * 4 * kT * 2;   // [16 tok][4 br][64 ch] bf16 = 8 KB
constexpr int kYBoxBytes = kBoxCh * kT * 2;       // [16 tok][64 ch] bf16 = 2 KB
constexpr int kYOff = kColBlocks * kRBoxBytes;    // 32 KB
constexpr int kSOff = kYOff + kColBlocks * kYBoxBytes;  // 40 KB
constexpr int kLoadBytes = kSOff + kT * 16;
constexpr int kMaxCluster = 16;
constexpr long long kWaitLimit = 4000000000LL;  // clock cycles before a wait gives up (~2 s)

// Bit 0: an mbarrier wait of the fused kernel ran out (the data it waited for never came).
__device__ unsigned int g_fused_status;

__host__ __device__ inline int round_up(int x, int a) { return (x + a - 1) / a * a; }

struct FusedShape {
    int C;            // cluster size = D / kDq
    int ntd;          // n-tiles of the down projection: ceil((r + 4) / 8)
    int half_last;    // 1 if the last down n-tile has <= 4 real rows (only lanes 0..15 stored)
    int upb;          // down-fragment units (16 B) per (warp, branch)
    int rw;           // reduction row per (token, branch): r+4 projections, sum of squares; even
    int nb4;          // broadcast row per token: h (r values) then inv (4), padded to 4 floats
    int down_bytes, up_bytes, gam_bytes, slice_bytes;
    int stage_bytes, recv_bytes, bcast_bytes;
    int off_up, off_gam, off_stage, off_recv, off_bcast, off_out, off_mbar, smem_bytes;
};

// Shared-memory layout: down | up | gamma | kStages stages (1024-aligned) | recv[2] | bcast[2]
// | out (an owner's outgoing h/inv rows) | mbarriers (stage_full[kStages], weights_full,
// recv_full[2], bcast_full[2]).
// The first three form one CTA's slice of the packed fragment section, in the same order.
__host__ __device__ inline FusedShape fused_shape(int D, int r) {
    FusedShape s{};
    s.C = D / kDq;
    s.ntd = (r + 4 + 7) / 8;
    const int last_rows = r + 4 - 8 * (s.ntd - 1);
    s.half_last = last_rows <= 4 ? 1 : 0;
    s.upb = (s.ntd - 1) * 32 + (s.half_last ? 16 : 32);
    s.rw = round_up(r + 5, 2);
    s.nb4 = round_up(r + 4, 4);
    s.down_bytes = kWarps * 4 * s.upb * 16;
    s.up_bytes = kWarps * 4 * 4 * 32 * 8;
    s.gam_bytes = 4 * kDq * 4;
    s.slice_bytes = s.down_bytes + s.up_bytes + s.gam_bytes;
    const int red_bytes = kWarps * kT * 4 * s.rw * 4;        // cross-warp partials
    s.stage_bytes = round_up(kLoadBytes > red_bytes ? kLoadBytes : red_bytes, 1024);
    s.recv_bytes = kT * 4 * s.rw * 4;
    s.bcast_bytes = kT * s.nb4 * 4;
    s.off_up = s.down_bytes;
    s.off_gam = s.off_up + s.up_bytes;
    s.off_stage = round_up(s.off_gam + s.gam_bytes, 1024);
    s.off_recv = s.off_stage + kStages * s.stage_bytes;
    s.off_bcast = s.off_recv + 2 * round_up(s.recv_bytes, 16);
    s.off_out = s.off_bcast + 2 * round_up(s.bcast_bytes, 16);
    s.off_mbar = s.off_out + round_up(s.bcast_bytes, 16);
    s.smem_bytes = s.off_mbar + 8 * (kStages + 5);
    return s;
}

// ---- PTX wrappers ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t ncluster_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
// Bounded wait on phase `parity` (acquire at cluster scope, so data that remote CTAs delivered
// with complete_tx is visible); records a status bit and returns false if it runs out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    const uint32_t a = smem_u32(bar);
    const long long t0 = clock64();
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n"
            " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
        if (clock64() - t0 > kWaitLimit) {
            atomicOr(&g_fused_status, 1u);
            return false;
        }
    }
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ uint32_t map_rank(uint32_t local_addr, uint32_t rank) {
    uint32_t ra;
    asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
    return ra;
}
// 16 bytes into CTA `rank`'s shared memory at the same offset as `local_addr`, completing
// 16 transaction bytes on that CTA's mbarrier at the offset of `local_bar`.
__device__ __forceinline__ void st_async_v4(uint32_t local_addr, uint32_t local_bar,
                                            uint32_t rank, float a, float b, float c, float d) {
    const uint32_t ra = map_rank(local_addr, rank), rb = map_rank(local_bar, rank);
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, "
        "[%5];" ::"r"(ra),
        "f"(a), "f"(b), "f"(c), "f"(d), "r"(rb)
        : "memory");
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&b);
}

// ---- the kernel -----------------------------------------------------------------------------
//
// Per tile k of this cluster, every CTA runs
//   A(k)  wait for the stage; write R' (eq write); sums of squares and down projections on
//         the tensor cores; sum the partials over the 8 warps; st.async each token's sums
//         to its owner CTA (completing on the owner's recv_full mbarrier); refill the stage.
//   B(k-1) wait for h and inv of tile k-1 (bcast_full); up projection, gates, combine, x.
//   C(k)  as owner: wait for the partial sums of its tokens from all CTAs; form inv, h and s
//         (eq rms, gate, s); write s; st.async h and inv to every CTA of the cluster.
// B trails A by one tile so that the owners' round trip of tile k is hidden behind A(k+1);
// the R' registers of tile k-1 stay live across A(k). recv and bcast are double-buffered by
// tile parity: a CTA can run at most one tile ahead of the slowest CTA in its cluster, because
// C(k) needs every CTA's A(k).

template <bool WRITE, int NTD>
__global__ void __launch_bounds__(kThreads, 1)
gr_fused_kernel(const __grid_constant__ CUtensorMap tm_R, const __grid_constant__ CUtensorMap tm_y,
                int64_t N, int D, int r, float eps, __nv_bfloat16* __restrict__ R,
                const float* __restrict__ s_prev, const char* __restrict__ frag,
                __nv_bfloat16* __restrict__ x, float* __restrict__ s_out) {
    extern __shared__ __align__(1024) char smem[];
    const FusedShape S = fused_shape(D, r);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, q4 = lane & 3;
    const uint32_t crank = cluster_ctarank();
    const int C = S.C;
    const int tpc = kT / C;                     // tokens owned per CTA and tile
    const int64_t ncl = ncluster_x(), cid = cluster_id_x();
    const int64_t ntiles = (N + kT - 1) / kT;
    const int nk = r + 4, rw = S.rw, nb4 = S.nb4;

    const uint4* s_down = reinterpret_cast<const uint4*>(smem);
    const uint2* s_up = reinterpret_cast<const uint2*>(smem + S.off_up);
    const float* s_gam = reinterpret_cast<const float*>(smem + S.off_gam);
    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + S.off_mbar);
    uint64_t* stage_full = mbar;                 // [kStages]
    uint64_t* weights_full = mbar + kStages;
    uint64_t* recv_full = mbar + kStages + 1;    // [2]
    uint64_t* bcast_full = mbar + kStages + 3;   // [2]
    auto stage_ptr = [&](int st) { return smem + S.off_stage + st * S.stage_bytes; };
    auto recv_ptr = [&](int p) {
        return reinterpret_cast<float*>(smem + S.off_recv + p * round_up(S.recv_bytes, 16));
    };
    auto bcast_ptr = [&](int p) {
        return reinterpret_cast<float*>(smem + S.off_bcast + p * round_up(S.bcast_bytes, 16));
    };

    if (tid == 0) {
        for (int i = 0; i < kStages + 5; ++i) mbar_init(&mbar[i], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // Stage fill for the k-th tile of this cluster: 4 R boxes [16 tok][4 br][64 ch] (lane 0 of
    // warps 0..3), 4 y boxes [16 tok][64 ch] (lane 0 of warps 4..7), s_prev rows (warp 0,
    // lane 1); warp 0 lane 0 arms the stage barrier. Rows past N are zero-filled by the TMA
    // unit. Spreading the copies over warps keeps each warp's issue latency short.
    auto issue_tile = [&](int64_t k) {
        const int64_t tile = cid + k * ncl;
        if (tile >= ntiles) return;
        const int st = int(k % kStages);
        char* sb = stage_ptr(st);
        const int t0 = int(tile * kT);
        const int nv = int(N - t0 < kT ? N - t0 : kT);
        const int c0 = int(crank) * kDq;
        if (warp == 0 && lane == 0)
            mbar_expect_tx(&stage_full[st],
                           uint32_t(kColBlocks * kRBoxBytes +
                                    (WRITE ? kColBlocks * kYBoxBytes + nv * 16 : 0)));
        if (lane == 0 && warp < kColBlocks) {
            tma_load_3d(sb + warp * kRBoxBytes, &tm_R, c0 + warp * kBoxCh, 0, t0,
                        &stage_full[st]);
        } else if (WRITE && lane == 0 && warp < 2 * kColBlocks) {
            const int yb = warp - kColBlocks;
            tma_load_2d(sb + kYOff + yb * kYBoxBytes, &tm_y, c0 + yb * kBoxCh, t0,
                        &stage_full[st]);
        } else if (WRITE && lane == 1 && warp == 0) {
            bulk_g2s(sb + kSOff, s_prev + size_t(t0) * 4, uint32_t(nv) * 16, &stage_full[st]);
        }
    };

    if (tid == 0) {
        mbar_expect_tx(weights_full, uint32_t(S.slice_bytes));
        bulk_g2s(smem, frag + size_t(crank) * S.slice_bytes, uint32_t(S.slice_bytes),
                 weights_full);
    }
    for (int k = 0; k < kStages; ++k) issue_tile(k);
    cluster_sync();  // every CTA of the cluster runs before any shared::cluster access
    mbar_wait(weights_full, 0);

    // This thread's 16-byte chunk in the swizzled boxes: column block cb, chunk cch (channels
    // 32·warp + 8·q4 ... +7 of the CTA slice); box row `row` keeps chunk c at c ^ (row & 7).
    const int cb = warp >> 1, cch = ((warp & 1) << 2) | q4;

    uint32_t Rp[4][2][4];      // R' of the current tile (bf16 pairs): [branch][row][pair]
    uint32_t Rq[4][2][4];      // R' of the previous tile, for its phase B
    int64_t t0_prev = 0;

    // Phase B of a tile: up projection (eq gate), gates, combine (eq use_gate), store x.
    auto phase_b = [&](int64_t kb, int64_t t0b) {
        const int p = int(kb & 1);
        mbar_wait(&bcast_full[p], uint32_t((kb >> 1) & 1));
        const float* bc = bcast_ptr(p);
        uint32_t ahi[4], alo[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int tk = g + 8 * (m & 1), kc = 2 * q4 + 8 * (m >> 1);
            const float h0 = kc < r ? bc[tk * nb4 + kc] : 0.f;
            const float h1 = kc + 1 < r ? bc[tk * nb4 + kc + 1] : 0.f;
            const float h0h = __bfloat162float(__float2bfloat16_rn(h0));
            const float h1h = __bfloat162float(__float2bfloat16_rn(h1));
            ahi[m] = pack_bf2(h0h, h1h);
            alo[m] = pack_bf2(h0 - h0h, h1 - h1h);
        }
        float xacc[2][8];
#pragma unroll
        for (int row = 0; row < 2; ++row)
#pragma unroll
            for (int e = 0; e < 8; ++e) xacc[row][e] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float inv0 = bc[g * nb4 + r + i], inv1 = bc[(g + 8) * nb4 + r + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint2 b = s_up[((warp * 4 + i) * 4 + j) * 32 + lane];
                float c[4] = {0.f, 0.f, 0.f, 0.f};
                mma_bf16(c, ahi[0], ahi[1], ahi[2], ahi[3], b.x, b.y);
                mma_bf16(c, alo[0], alo[1], alo[2], alo[3], b.x, b.y);
                const float2 gm =
                    *reinterpret_cast<const float2*>(s_gam + i * kDq + warp * 32 + q4 * 8 + 2 * j);
                const float a00 = gm.x * inv0 * bf_lo(Rq[i][0][j]);
                const float a01 = gm.y * inv0 * bf_hi(Rq[i][0][j]);
                const float a10 = gm.x * inv1 * bf_lo(Rq[i][1][j]);
                const float a11 = gm.y * inv1 * bf_hi(Rq[i][1][j]);
                // G·a = ½a + ½·tanh(·)·a; the ½ is applied once at the end
                xacc[0][2 * j] += fmaf(tanh_approx(c[0]), a00, a00);
                xacc[0][2 * j + 1] += fmaf(tanh_approx(c[1]), a01, a01);
                xacc[1][2 * j] += fmaf(tanh_approx(c[2]), a10, a10);
                xacc[1][2 * j + 1] += fmaf(tanh_approx(c[3]), a11, a11);
            }
        }
#pragma unroll
        for (int row = 0; row < 2; ++row) {
            const int tok = g + 8 * row;
            if (t0b + tok < N) {
                __nv_bfloat16* dst =
                    x + size_t(t0b + tok) * D + size_t(crank) * kDq + warp * 32 + q4 * 8;
                *reinterpret_cast<uint4*>(dst) = make_uint4(
                    pack_bf2(0.125f * xacc[row][0], 0.125f * xacc[row][1]),
                    pack_bf2(0.125f * xacc[row][2], 0.125f * xacc[row][3]),
                    pack_bf2(0.125f * xacc[row][4], 0.125f * xacc[row][5]),
                    pack_bf2(0.125f * xacc[row][6], 0.125f * xacc[row][7]));
            }
        }
    };

    int64_t k = 0;
    for (;; ++k) {
        const int64_t tile = cid + k * ncl;
        if (tile >= ntiles) break;
        const int st = int(k % kStages);
        const int p = int(k & 1);
        char* sb = stage_ptr(st);
        const int64_t t0 = tile * kT;
        const int nv = int(N - t0 < kT ? N - t0 : kT);
        mbar_wait(&stage_full[st], uint32_t((k / kStages) & 1));

        // ---- A(k): write (eq write), sums of squares, down projections ----------------------
#pragma unroll
        for (int row = 0; row < 2; ++row) {
            const int tok = g + 8 * row;
            float yf[8], sp[4] = {0.f, 0.f, 0.f, 0.f};
            if (WRITE) {
                const float4 s4 = *reinterpret_cast<const float4*>(sb + kSOff + tok * 16);
                sp[0] = s4.x, sp[1] = s4.y, sp[2] = s4.z, sp[3] = s4.w;
                const uint4 yv = *reinterpret_cast<const uint4*>(
                    sb + kYOff + cb * kYBoxBytes + tok * 128 + ((cch ^ (tok & 7)) << 4));
                const uint32_t yw[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
                for (int m = 0; m < 4; ++m) yf[2 * m] = bf_lo(yw[m]), yf[2 * m + 1] = bf_hi(yw[m]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int brow = tok * 4 + i;
                const uint4 rv = *reinterpret_cast<const uint4*>(
                    sb + cb * kRBoxBytes + brow * 128 + ((cch ^ (brow & 7)) << 4));
                const uint32_t rw4[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    uint32_t v = rw4[m];
                    if (WRITE)
                        v = pack_bf2(fmaf(sp[i], yf[2 * m], bf_lo(v)),
                                     fmaf(sp[i], yf[2 * m + 1], bf_hi(v)));
                    Rp[i][row][m] = v;
                }
                if (WRITE && tok < nv) {
                    __nv_bfloat16* dst = R + (size_t(t0 + tok) * 4 + i) * size_t(D) +
                                         size_t(crank) * kDq + warp * 32 + q4 * 8;
                    *reinterpret_cast<uint4*>(dst) =
                        make_uint4(Rp[i][row][0], Rp[i][row][1], Rp[i][row][2], Rp[i][row][3]);
                }
            }
        }
        __syncthreads();  // every warp has read the stage; it becomes the partial-sum buffer
        float* red = reinterpret_cast<float*>(sb);  // [kWarps][kT][4][rw]
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float* r0 = red + ((warp * kT + g) * 4 + i) * rw;
            float* r1 = red + ((warp * kT + g + 8) * 4 + i) * rw;
            // down projections (rows: W_d then W_w, gamma folded)
#pragma unroll
            for (int j = 0; j < NTD; ++j) {
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
                uint4 b = make_uint4(0u, 0u, 0u, 0u);
                const bool last_half = (j == NTD - 1) && S.half_last;
                if (!last_half || lane < 16) b = s_down[(warp * 4 + i) * S.upb + j * 32 + lane];
                mma_bf16(acc, Rp[i][0][0], Rp[i][1][0], Rp[i][0][1], Rp[i][1][1], b.x, b.y);
                mma_bf16(acc, Rp[i][0][2], Rp[i][1][2], Rp[i][0][3], Rp[i][1][3], b.z, b.w);
                const int o = 8 * j + 2 * q4;
                if (o + 1 < nk) {
                    *reinterpret_cast<float2*>(r0 + o) = make_float2(acc[0], acc[1]);
                    *reinterpret_cast<float2*>(r1 + o) = make_float2(acc[2], acc[3]);
                } else if (o < nk) {
                    r0[o] = acc[0], r1[o] = acc[2];
                }
            }
            // sums of squares: diagonal of R'·R'ᵀ over this warp's 32 channels
            float sq0[4] = {0.f, 0.f, 0.f, 0.f}, sq1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const uint32_t a0 = Rp[i][0][2 * ks], a1 = Rp[i][1][2 * ks];
                const uint32_t a2 = Rp[i][0][2 * ks + 1], a3 = Rp[i][1][2 * ks + 1];
                mma_bf16(sq0, a0, a1, a2, a3, a0, a2);   // columns: tokens 0..7
                mma_bf16(sq1, a0, a1, a2, a3, a1, a3);   // columns: tokens 8..15
            }
            if (q4 == (g >> 1)) {
                r0[nk] = (g & 1) ? sq0[1] : sq0[0];
                r1[nk] = (g & 1) ? sq1[3] : sq1[2];
            }
        }
        __syncthreads();
        {
            const int nval = kT * 4 * rw;            // a multiple of 4
            const uint32_t recv_u32 = smem_u32(recv_ptr(p));
            for (int v = 4 * tid; v < nval; v += 4 * kThreads) {
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int w = 0; w < kWarps; ++w) {
                    const float4 b = *reinterpret_cast<const float4*>(red + w * nval + v);
                    a.x += b.x, a.y += b.y, a.z += b.z, a.w += b.w;
                }
                const int tok = v / (4 * rw), rest = v - tok * 4 * rw;
                const int owner = tok / tpc, slot = tok - owner * tpc;
                st_async_v4(recv_u32 + uint32_t(((int(crank) * tpc + slot) * 4 * rw + rest) * 4),
                            smem_u32(&recv_full[p]), uint32_t(owner), a.x, a.y, a.z, a.w);
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();  // the stage is free: refill it with tile k + kStages
        issue_tile(k + kStages);

        // ---- B(k-1) -------------------------------------------------------------------------
        if (k > 0) phase_b(k - 1, t0_prev);

        // ---- C(k): owner ---------------------------------------------------------------------
        if (tid == 0) {
            mbar_expect_tx(&recv_full[p], uint32_t(C * tpc * 4 * rw * 4));
            mbar_expect_tx(&bcast_full[p], uint32_t(kT * nb4 * 4));
        }
        mbar_wait(&recv_full[p], uint32_t((k >> 1) & 1));
        {
            float* recv = recv_ptr(p);              // [C][tpc][4][rw]
            const int nown = tpc * 4 * rw;          // a multiple of 4
            // sum over the C sources: 4 threads per 4-value group, each a quarter of the sources
            for (int v = tid; v < nown; v += kThreads) {
                const int grp = v >> 2, qtr = v & 3;
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int src = qtr; src < C; src += 4) {
                    const float4 b =
                        *reinterpret_cast<const float4*>(recv + src * nown + 4 * grp);
                    a.x += b.x, a.y += b.y, a.z += b.z, a.w += b.w;
                }
                // nown is a multiple of 4, so the four lanes of a group are active together
                const unsigned mask = __activemask();
#pragma unroll
                for (int o = 1; o < 4; o <<= 1) {
                    a.x += __shfl_xor_sync(mask, a.x, o);
                    a.y += __shfl_xor_sync(mask, a.y, o);
                    a.z += __shfl_xor_sync(mask, a.z, o);
                    a.w += __shfl_xor_sync(mask, a.w, o);
                }
                if (qtr == 0) *reinterpret_cast<float4*>(recv + 4 * grp) = a;
            }
            __syncthreads();
            // one output per thread: h_k = SiLU(z_k) (k < r), else s written and inv kept
            float* outrow = reinterpret_cast<float*>(smem + S.off_out);   // [tpc][nb4]
            for (int v = tid; v < tpc * nb4; v += kThreads) {
                const int slot = v / nb4, kk = v - slot * nb4;
                const int tok = int(crank) * tpc + slot;
                const float* P = recv + slot * 4 * rw;
                float out = 0.f;
                if (kk < nk) {
                    float inv[4], a = 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        inv[i] = rsqrtf(P[i * rw + nk] / float(D) + eps);
                        a = fmaf(inv[i], P[i * rw + kk], a);
                    }
                    a *= 0.25f;
                    if (kk < r) {
                        out = a * sigmoid_accurate(a);
                    } else {
                        if (t0 + tok < N)
                            s_out[(t0 + tok) * 4 + (kk - r)] = 2.0f * sigmoid_accurate(a);
                        out = inv[kk - r];
                    }
                }
                outrow[v] = out;
            }
            __syncthreads();
            const uint32_t bc_u32 = smem_u32(bcast_ptr(p));
            const int ngrp = nb4 / 4;
            // one thread per (owned token, group of 4 outputs, destination CTA)
            for (int v = tid; v < tpc * ngrp * C; v += kThreads) {
                const int dst = v % C, rem = v / C;
                const int slot = rem / ngrp, g4 = rem - slot * ngrp;
                const int tok = int(crank) * tpc + slot;
                const float4 o4 = *reinterpret_cast<const float4*>(outrow + slot * nb4 + 4 * g4);
                st_async_v4(bc_u32 + uint32_t((tok * nb4 + 4 * g4) * 4),
                            smem_u32(&bcast_full[p]), uint32_t(dst), o4.x, o4.y, o4.z, o4.w);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int row = 0; row < 2; ++row)
#pragma unroll
                for (int m = 0; m < 4; ++m) Rq[i][row][m] = Rp[i][row][m];
        t0_prev = t0;
    }
    if (k > 0) phase_b(k - 1, t0_prev);
    cluster_sync();  // no CTA leaves while shared::cluster traffic to it may be in flight
}

// Fragment section: for CTA slice q, [down | up | gamma] (the kernel's shared-memory order).
__global__ void pack_fused_kernel(int D, int r, const float* __restrict__ gamma,
                                  const float* __restrict__ wd, const float* __restrict__ wu,
                                  const float* __restrict__ ww, char* __restrict__ frag) {
    const FusedShape S = fused_shape(D, r);
    const int K = 4 * D;
    const int n_down = kWarps * 4 * S.upb;        // 16-byte units per slice
    const int n_up = kWarps * 4 * 4 * 32;         // 8-byte units per slice
    const int n_gam = 4 * kDq;                    // floats per slice
    const int per_slice = n_down + n_up + n_gam;
    const int64_t total = int64_t(S.C) * per_slice;
    for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int q = int(e / per_slice);
        int u = int(e - int64_t(q) * per_slice);
        char* slice = frag + size_t(q) * S.slice_bytes;
        if (u < n_down) {
            const int wi = u / S.upb, rest = u - wi * S.upb;   // wi = warp*4 + branch
            const int j = rest >> 5, lane = rest & 31;
            const int w = wi >> 2, i = wi & 3;
            const int n = 8 * j + (lane >> 2);
            __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(slice + size_t(u) * 16);
            for (int c8 = 0; c8 < 8; ++c8) {
                const int m = i * D + q * kDq + w * 32 + (lane & 3) * 8 + c8;
                float v = 0.f;
                if (n < r) v = wd[size_t(n) * K + m] * gamma[m];
                else if (n < r + 4) v = ww[size_t(n - r) * K + m] * gamma[m];
                dst[c8] = __float2bfloat16_rn(v);
            }
        } else if ((u -= n_down) < n_up) {
            const int lane = u & 31, rest = u >> 5;
            const int j = rest & 3, wi = rest >> 2;
            const int w = wi >> 2, i = wi & 3;
            const int gg = lane >> 2, qq = lane & 3;
            const int m = i * D + q * kDq + w * 32 + 8 * (gg >> 1) + 2 * j + (gg & 1);
            const int kk[4] = {2 * qq, 2 * qq + 1, 2 * qq + 8, 2 * qq + 9};
            __nv_bfloat16* dst =
                reinterpret_cast<__nv_bfloat16*>(slice + S.off_up + size_t(u) * 8);
            for (int t = 0; t < 4; ++t)
                dst[t] = __float2bfloat16_rn(kk[t] < r ? 0.5f * wu[size_t(m) * r + kk[t]] : 0.f);
        } else {
            u -= n_up;
            const int i = u / kDq, cl = u - i * kDq;
            reinterpret_cast<float*>(slice + S.off_gam)[u] = gamma[i * D + q * kDq + cl];
        }
    }
}

// ---- host side ------------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// R as a 3-D tensor {channel, branch, token}; box {64, 4, 16}, 128-byte swizzle.
bool make_map_R(CUtensorMap* m, const void* R, int64_t N, int D) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {cuuint64_t(D), 4, cuuint64_t(N)};
    const cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(D) * 8};
    const cuuint32_t box[3] = {kBoxCh, 4, kT};
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(R), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// y as a 2-D tensor {channel, token}; box {64, 16}, 128-byte swizzle.
bool make_map_y(CUtensorMap* m, const void* y, int64_t N, int D) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(N)};
    const cuuint64_t strides[1] = {cuuint64_t(D) * 2};
    const cuuint32_t box[2] = {kBoxCh, kT};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(y), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

struct ClusterCache {
    int max_clusters[2][4][5];  // [WRITE][NTD][log2 C], 0 = not queried
};
ClusterCache g_cluster_cache[64];

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
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         S.smem_bytes);
    if (e != cudaSuccess) return e;
    if (S.C > 8) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(S.C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = size_t(S.smem_bytes);
    cfg.stream = st;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    int lc = 0;
    while ((1 << lc) < S.C) ++lc;
    int& maxc = g_cluster_cache[dev & 63].max_clusters[WRITE ? 1 : 0][NTD][lc];
    if (maxc == 0) {
        cfg.gridDim = dim3(unsigned(S.C * 64));
        int n = 0;
        if ((e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg)) != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        maxc = n;
    }
    const int64_t ntiles = (N + kT - 1) / kT;
    const int64_t ncl = ntiles < maxc ? ntiles : maxc;
    cfg.gridDim = dim3(unsigned(ncl * S.C));
    return cudaLaunchKernelEx(&cfg, kern, mR, my, N, D, r, eps, static_cast<__nv_bfloat16*>(R),
                              s_prev, frag, static_cast<__nv_bfloat16*>(x), s_out);
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

int fused_status(bool clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_fused_status, sizeof(v)) != cudaSuccess) return -1;
    if (clear && v) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(g_fused_status, &z, sizeof(z)) != cudaSuccess) return -1;
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
