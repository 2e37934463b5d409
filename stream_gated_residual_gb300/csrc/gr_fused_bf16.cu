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
//     buffers filled by cp.async.bulk copies completing on mbarriers.
//   * 8 warps per CTA; warp w owns 32 channels of each branch. A thread holds 8 channels of two
//     token rows per branch; those registers are directly the A fragments of
//     mma.m16n8k16 once the K index is permuted consistently with the packed B fragments.
//   * The per-token row reductions (4 sums of squares and 4·(r+4) partial projections) are
//     summed over warps in shared memory, then sent through distributed shared memory to the
//     token's owner CTA, which forms inv, h and s and broadcasts h and inv to the cluster.
//   * The up-projection runs on the tensor cores with h split into bf16 hi + lo parts (about 16
//     significant bits), and σ(a) = ½ + ½·tanh(a/2) with W_u pre-scaled by ½ (exact in bf16).
#include "gr_internal.h"

namespace gr {

namespace {

constexpr int kT = 16;                      // tokens per tile (mma M)
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kDq = kWarps * 32;            // channels per branch per CTA
constexpr int kStages = 3;
constexpr int kRowBytes = kDq * 2;          // one token-branch row slice, bf16
constexpr int kRowStride = kRowBytes + 16;  // staggers banks between token rows
constexpr int kMaxCluster = 16;
constexpr long long kWaitLimit = 4000000000LL;  // clock cycles before a wait gives up (~2 s)

// Bit 0: an mbarrier wait of the fused kernel ran out (the data it waited for never came).
__device__ unsigned int g_fused_status;

struct FusedShape {
    int C;            // cluster size = D / kDq
    int ntd;          // n-tiles of the down projection: ceil((r + 4) / 8)
    int rw;           // reduction row per (token, branch): r + 4 projections + 1 sum of squares
    int down_bytes;   // kWarps·4·ntd·32 lanes·16 B
    int up_bytes;     // kWarps·4·4·32 lanes·8 B
    int gam_bytes;    // 4·kDq fp32
    int slice_bytes;  // one CTA's share of the packed fragment section
    int stage_bytes;
    int off_up, off_gam, off_stage, off_recv, off_bcast, off_mbar, smem_bytes;
};

__host__ __device__ inline int round_up(int x, int a) { return (x + a - 1) / a * a; }

__host__ __device__ inline FusedShape fused_shape(int D, int r) {
    FusedShape s{};
    s.C = D / kDq;
    s.ntd = (r + 4 + 7) / 8;
    s.rw = r + 4 + 1;
    s.down_bytes = kWarps * 4 * s.ntd * 32 * 16;
    s.up_bytes = kWarps * 4 * 4 * 32 * 8;
    s.gam_bytes = 4 * kDq * 4;
    s.slice_bytes = s.down_bytes + s.up_bytes + s.gam_bytes;
    const int load_bytes = kT * 5 * kRowStride + kT * 16;   // R rows, y rows, s_prev
    const int red_bytes = kWarps * kT * 4 * s.rw * 4;        // cross-warp partials
    s.stage_bytes = round_up(load_bytes > red_bytes ? load_bytes : red_bytes, 128);
    s.off_up = s.down_bytes;
    s.off_gam = s.off_up + s.up_bytes;
    s.off_stage = s.off_gam + s.gam_bytes;
    s.off_recv = s.off_stage + kStages * s.stage_bytes;
    s.off_bcast = s.off_recv + round_up(kT * 4 * s.rw * 4, 16);
    s.off_mbar = s.off_bcast + round_up(kT * (r + 4) * 4, 16);
    s.smem_bytes = s.off_mbar + 8 * (kStages + 1);
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
// Bounded wait on phase `parity`; records a status bit and returns false if it runs out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    const uint32_t a = smem_u32(bar);
    const long long t0 = clock64();
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
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
__device__ __forceinline__ void st_cluster(uint32_t local_addr, uint32_t rank, float v) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local_addr), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(ra), "f"(v) : "memory");
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
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

template <bool WRITE, int NTD>
__global__ void __launch_bounds__(kThreads, 1)
gr_fused_kernel(int64_t N, int D, int r, float eps, __nv_bfloat16* __restrict__ R,
                const __nv_bfloat16* __restrict__ y, const float* __restrict__ s_prev,
                const char* __restrict__ frag, __nv_bfloat16* __restrict__ x,
                float* __restrict__ s_out) {
    extern __shared__ __align__(1024) char smem[];
    const FusedShape S = fused_shape(D, r);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, q4 = lane & 3;
    const uint32_t crank = cluster_ctarank();
    const int C = S.C;
    const int tpc = kT / C;                     // tokens owned per CTA and tile
    const int64_t ncl = ncluster_x(), cid = cluster_id_x();
    const int64_t ntiles = (N + kT - 1) / kT;
    const int nk = r + 4;

    const uint4* s_down = reinterpret_cast<const uint4*>(smem);
    const uint2* s_up = reinterpret_cast<const uint2*>(smem + S.off_up);
    const float* s_gam = reinterpret_cast<const float*>(smem + S.off_gam);
    float* recv = reinterpret_cast<float*>(smem + S.off_recv);     // [C][tpc][4][rw]
    float* bcast = reinterpret_cast<float*>(smem + S.off_bcast);   // [kT][r+4]: h, inv
    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + S.off_mbar);
    auto stage_ptr = [&](int st) { return smem + S.off_stage + st * S.stage_bytes; };

    if (tid == 0) {
        for (int st = 0; st <= kStages; ++st) mbar_init(&mbar[st], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // Stage fill for the k-th tile of this cluster (warp 0, all lanes).
    auto issue_tile = [&](int64_t k) {
        const int64_t tile = cid + k * ncl;
        if (tile >= ntiles) return;
        const int st = int(k % kStages);
        char* sb = stage_ptr(st);
        const int64_t t0 = tile * kT;
        const int nv = int(N - t0 < kT ? N - t0 : kT);
        const uint32_t bytes = uint32_t(nv) * (4 * kRowBytes + (WRITE ? kRowBytes + 16 : 0));
        if (lane == 0) mbar_expect_tx(&mbar[st], bytes);
        __syncwarp();
        const int ncopy = nv * 4 + (WRITE ? nv + 1 : 0);
        const size_t cofs = size_t(crank) * kDq;
        for (int c = lane; c < ncopy; c += 32) {
            if (c < nv * 4) {
                const int j = c >> 2, i = c & 3;
                bulk_g2s(sb + (j * 4 + i) * kRowStride,
                         R + (size_t(t0 + j) * 4 + i) * size_t(D) + cofs, kRowBytes, &mbar[st]);
            } else if (c < nv * 5) {
                const int j = c - nv * 4;
                bulk_g2s(sb + (kT * 4 + j) * kRowStride, y + size_t(t0 + j) * D + cofs,
                         kRowBytes, &mbar[st]);
            } else {
                bulk_g2s(sb + kT * 5 * kRowStride, s_prev + t0 * 4, uint32_t(nv) * 16,
                         &mbar[st]);
            }
        }
    };

    if (tid == 0) {
        mbar_expect_tx(&mbar[kStages], uint32_t(S.slice_bytes));
        bulk_g2s(smem, frag + size_t(crank) * S.slice_bytes, uint32_t(S.slice_bytes),
                 &mbar[kStages]);
    }
    if (warp == 0)
        for (int k = 0; k < kStages; ++k) issue_tile(k);
    cluster_sync();  // every CTA of the cluster runs before any shared::cluster access
    mbar_wait(&mbar[kStages], 0);

    const int cofs_b = (warp * 32 + q4 * 8) * 2;  // this thread's byte offset in a row slice
    const uint32_t recv_u32 = smem_u32(recv);
    const uint32_t bcast_u32 = smem_u32(bcast);

    for (int64_t k = 0;; ++k) {
        const int64_t tile = cid + k * ncl;
        if (tile >= ntiles) break;
        const int st = int(k % kStages);
        const uint32_t par = uint32_t((k / kStages) & 1);
        char* sb = stage_ptr(st);
        const int64_t t0 = tile * kT;
        const int nv = int(N - t0 < kT ? N - t0 : kT);
        mbar_wait(&mbar[st], par);

        // ---- phase A: write (eq write), sums of squares, down projections -------------------
        uint32_t Rp[4][2][4];  // stored R' (bf16 pairs): [branch][row g / g+8][channel pair]
        float ssq[2][4];
#pragma unroll
        for (int row = 0; row < 2; ++row) {
            const int tok = g + 8 * row;
            float yf[8], sp[4] = {0.f, 0.f, 0.f, 0.f};
            if (WRITE) {
                const float4 s4 = *reinterpret_cast<const float4*>(sb + kT * 5 * kRowStride +
                                                                   tok * 16);
                sp[0] = s4.x, sp[1] = s4.y, sp[2] = s4.z, sp[3] = s4.w;
                const uint4 yv =
                    *reinterpret_cast<const uint4*>(sb + (kT * 4 + tok) * kRowStride + cofs_b);
                const uint32_t yw[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
                for (int m = 0; m < 4; ++m) yf[2 * m] = bf_lo(yw[m]), yf[2 * m + 1] = bf_hi(yw[m]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 rv =
                    *reinterpret_cast<const uint4*>(sb + (tok * 4 + i) * kRowStride + cofs_b);
                const uint32_t rw4[4] = {rv.x, rv.y, rv.z, rv.w};
                float a = 0.f;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    uint32_t p = rw4[m];
                    if (WRITE)
                        p = pack_bf2(fmaf(sp[i], yf[2 * m], bf_lo(p)),
                                     fmaf(sp[i], yf[2 * m + 1], bf_hi(p)));
                    Rp[i][row][m] = p;
                    const float v0 = bf_lo(p), v1 = bf_hi(p);
                    a = fmaf(v0, v0, a);
                    a = fmaf(v1, v1, a);
                }
                ssq[row][i] = a;
                if (WRITE && tok < nv) {
                    __nv_bfloat16* dst = R + (size_t(t0 + tok) * 4 + i) * size_t(D) +
                                         size_t(crank) * kDq + warp * 32 + q4 * 8;
                    *reinterpret_cast<uint4*>(dst) =
                        make_uint4(Rp[i][row][0], Rp[i][row][1], Rp[i][row][2], Rp[i][row][3]);
                }
            }
        }
        float acc[4][NTD][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int j = 0; j < NTD; ++j) {
                acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;
                const uint4 b = s_down[((warp * 4 + i) * NTD + j) * 32 + lane];
                mma_bf16(acc[i][j], Rp[i][0][0], Rp[i][1][0], Rp[i][0][1], Rp[i][1][1], b.x, b.y);
                mma_bf16(acc[i][j], Rp[i][0][2], Rp[i][1][2], Rp[i][0][3], Rp[i][1][3], b.z, b.w);
            }
        }
#pragma unroll
        for (int row = 0; row < 2; ++row)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                ssq[row][i] += __shfl_xor_sync(0xffffffffu, ssq[row][i], 1);
                ssq[row][i] += __shfl_xor_sync(0xffffffffu, ssq[row][i], 2);
            }

        // ---- row reductions: over warps (shared memory), then to the owner CTA (DSMEM) -------
        __syncthreads();  // every warp has read the stage; it becomes the partial-sum buffer
        float* red = reinterpret_cast<float*>(sb);  // [kWarps][kT][4][rw]
        const int rw = S.rw;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < NTD; ++j) {
                const int o = 8 * j + 2 * q4;
                float* r0 = red + ((warp * kT + g) * 4 + i) * rw;
                float* r1 = red + ((warp * kT + g + 8) * 4 + i) * rw;
                if (o < nk) r0[o] = acc[i][j][0], r1[o] = acc[i][j][2];
                if (o + 1 < nk) r0[o + 1] = acc[i][j][1], r1[o + 1] = acc[i][j][3];
            }
        if (q4 == 0)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                red[((warp * kT + g) * 4 + i) * rw + nk] = ssq[0][i];
                red[((warp * kT + g + 8) * 4 + i) * rw + nk] = ssq[1][i];
            }
        __syncthreads();
        const int nval = kT * 4 * rw;
        for (int v = tid; v < nval; v += kThreads) {
            float a = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) a += red[w * nval + v];
            const int tok = v / (4 * rw), rest = v - tok * 4 * rw;
            const int owner = tok / tpc, slot = tok - owner * tpc;
            st_cluster(recv_u32 + uint32_t(((crank * tpc + slot) * 4 * rw + rest) * 4),
                       uint32_t(owner), a);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        cluster_sync();  // #1: partials are at their owners; this stage is free again
        if (warp == 0) issue_tile(k + kStages);

        // ---- owner: inv, h (eq gate), s (eq s) for its tokens; broadcast h and inv ----------
        const int nown = tpc * 4 * rw;
        for (int v = tid; v < nown; v += kThreads) {
            float a = 0.f;
            for (int src = 0; src < C; ++src) a += recv[src * nown + v];
            recv[v] = a;
        }
        __syncthreads();
        for (int v = tid; v < tpc * nk; v += kThreads) {
            const int slot = v / nk, kk = v - slot * nk;
            const int tok = int(crank) * tpc + slot;
            const float* P = recv + slot * 4 * rw;
            float inv[4], a = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                inv[i] = rsqrtf(P[i * rw + nk] / float(D) + eps);
                a = fmaf(inv[i], P[i * rw + kk], a);
            }
            a *= 0.25f;
            float out;
            if (kk < r) {
                out = a * sigmoid_accurate(a);  // h = SiLU(z)
            } else {
                if (t0 + tok < N) s_out[(t0 + tok) * 4 + (kk - r)] = 2.0f * sigmoid_accurate(a);
                out = inv[kk - r];
            }
            const uint32_t la = bcast_u32 + uint32_t((tok * nk + kk) * 4);
            for (int dst = 0; dst < C; ++dst) st_cluster(la, uint32_t(dst), out);
        }
        cluster_sync();  // #2: h and inv of every token of the tile are in every CTA

        // ---- phase B: up projection (eq gate), gates, combine (eq use_gate) ----------------
        uint32_t ahi[4], alo[4];
        {
            const int kq[4][2] = {{g, 2 * q4}, {g + 8, 2 * q4}, {g, 2 * q4 + 8}, {g + 8, 2 * q4 + 8}};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int tk = kq[m][0], kc = kq[m][1];
                const float h0 = kc < r ? bcast[tk * nk + kc] : 0.f;
                const float h1 = kc + 1 < r ? bcast[tk * nk + kc + 1] : 0.f;
                const float h0h = __bfloat162float(__float2bfloat16_rn(h0));
                const float h1h = __bfloat162float(__float2bfloat16_rn(h1));
                ahi[m] = pack_bf2(h0h, h1h);
                alo[m] = pack_bf2(h0 - h0h, h1 - h1h);
            }
        }
        float xacc[2][8];
#pragma unroll
        for (int row = 0; row < 2; ++row)
#pragma unroll
            for (int e = 0; e < 8; ++e) xacc[row][e] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float inv0 = bcast[g * nk + r + i], inv1 = bcast[(g + 8) * nk + r + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint2 b = s_up[((warp * 4 + i) * 4 + j) * 32 + lane];
                float c[4] = {0.f, 0.f, 0.f, 0.f};
                mma_bf16(c, ahi[0], ahi[1], ahi[2], ahi[3], b.x, b.y);
                mma_bf16(c, alo[0], alo[1], alo[2], alo[3], b.x, b.y);
                const float2 gm =
                    *reinterpret_cast<const float2*>(s_gam + i * kDq + warp * 32 + q4 * 8 + 2 * j);
                const float G0 = fmaf(0.5f, tanh_approx(c[0]), 0.5f);
                const float G1 = fmaf(0.5f, tanh_approx(c[1]), 0.5f);
                const float G2 = fmaf(0.5f, tanh_approx(c[2]), 0.5f);
                const float G3 = fmaf(0.5f, tanh_approx(c[3]), 0.5f);
                xacc[0][2 * j] = fmaf(G0 * gm.x * inv0, bf_lo(Rp[i][0][j]), xacc[0][2 * j]);
                xacc[0][2 * j + 1] = fmaf(G1 * gm.y * inv0, bf_hi(Rp[i][0][j]), xacc[0][2 * j + 1]);
                xacc[1][2 * j] = fmaf(G2 * gm.x * inv1, bf_lo(Rp[i][1][j]), xacc[1][2 * j]);
                xacc[1][2 * j + 1] = fmaf(G3 * gm.y * inv1, bf_hi(Rp[i][1][j]), xacc[1][2 * j + 1]);
            }
        }
#pragma unroll
        for (int row = 0; row < 2; ++row) {
            const int tok = g + 8 * row;
            if (t0 + tok < N) {
                __nv_bfloat16* dst =
                    x + size_t(t0 + tok) * D + size_t(crank) * kDq + warp * 32 + q4 * 8;
                *reinterpret_cast<uint4*>(dst) = make_uint4(
                    pack_bf2(0.25f * xacc[row][0], 0.25f * xacc[row][1]),
                    pack_bf2(0.25f * xacc[row][2], 0.25f * xacc[row][3]),
                    pack_bf2(0.25f * xacc[row][4], 0.25f * xacc[row][5]),
                    pack_bf2(0.25f * xacc[row][6], 0.25f * xacc[row][7]));
            }
        }
    }
}

// Fragment section: for CTA slice q, [down | up | gamma] (see the kernel's smem layout).
__global__ void pack_fused_kernel(int D, int r, const float* __restrict__ gamma,
                                  const float* __restrict__ wd, const float* __restrict__ wu,
                                  const float* __restrict__ ww, char* __restrict__ frag) {
    const FusedShape S = fused_shape(D, r);
    const int K = 4 * D;
    const int n_down = kWarps * 4 * S.ntd * 32;   // 16-byte units per slice
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
            const int lane = u & 31, rest = u >> 5;
            const int j = rest % S.ntd, wi = rest / S.ntd;   // wi = warp*4 + branch
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

struct ClusterCache {
    int max_clusters[2][4][5];  // [WRITE][NTD][log2 C], 0 = not queried
};
ClusterCache g_cluster_cache[64];

template <bool WRITE, int NTD>
cudaError_t launch_t(int64_t N, int D, int r, float eps, void* R, const void* y,
                     const float* s_prev, const char* frag, void* x, float* s_out,
                     cudaStream_t st) {
    const FusedShape S = fused_shape(D, r);
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
    return cudaLaunchKernelEx(&cfg, kern, N, D, r, eps, static_cast<__nv_bfloat16*>(R),
                              static_cast<const __nv_bfloat16*>(y), s_prev, frag,
                              static_cast<__nv_bfloat16*>(x), s_out);
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
