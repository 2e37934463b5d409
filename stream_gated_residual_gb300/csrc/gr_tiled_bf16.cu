// Two-pass bf16 GR kernel for the shapes the cluster kernel (gr_fused_bf16.cu) does not take:
// any D that is a multiple of 64 and 1 <= r <= 32, e.g. D = 7168 with r = 32.
//
// What it computes is the same fused step as the cluster kernel, from "【论文解读】 Qwen3.8
// Flash Next", §二.4: the write R' = R + s_prev·y (eq write), then the read of R': per-branch
// RMS (eq rms), the low-rank gate (eq gate), the write strengths s = 2σ(u) (eq s) and the gated
// combine x = (1/n_r)·Σ_i G_i ⊙ R̂_i (eq use_gate).
//
// Design. One CTA owns a tile of 32 tokens across all D channels; the CTAs are persistent
// (one per SM, tiles handed out round-robin). Each tile takes two passes over its channels in
// 64-channel chunks:
//   pass 1 (forward over the chunks): TMA-load R [4 branches][32 tokens][64 ch] and y
//     [32][64]; the write R' = RNE(R + s·y) in registers, stored back in place and sent to HBM by
//     a TMA store per (branch, 16-token m-tile); per-(token, branch) sums of R'² in registers;
//     the down projection [W_d; W_w]·R' on the tensor cores (mma.sync m16n8k16, bf16 in, fp32
//     accumulate). Warp (branch, m-tile, k-half) takes two of the chunk's four 16-channel
//     k-steps and accumulates over all chunks; the B fragments (γ folded) stream from L2
//     through a weight ring.
//   owner step (once per tile): inv_i = 1/sqrt(ms_i + eps); z = ¼Σ_i inv_i·P_i, h = SiLU(z)
//     and u = ¼Σ_i inv_i·Q_i, s = 2σ(u) — through shared memory, no cluster needed.
//   pass 2 (backward over the chunks, so the R' chunks written last are read first, while
//     some are still in L2): TMA-load R' again; the up projection W_u·h on the tensor cores
//     in fp16 (½·W_u packed as fp16; each token's h row scaled by an exact power of two that
//     keeps it below 2^15, undone on the fp32 accumulator), σ as ½ + ½·tanh, and the combine.
//     fp16 carries 11 significant bits for both operands, so one mma per k-step suffices
//     (the cluster kernel does the same). Warp
//     (m-tile, 8-channel group) covers the four branches of its channels; x leaves through a
//     per-warp TMA store.
// The price is one more read of R' than the single traversal (about 40% more HBM traffic at
// D = 7168); in exchange the tile needs no cluster and the weights never have to fit on chip.
//
// Roles: warps 0..15 compute, warp 16 (one lane) produces: it fills the state ring (R/R' + y,
// 20 KB a stage) and the weight ring, and before pass 2 of a tile it waits until the compute
// warps report pass 1's R' stores complete. Sixteen compute warps (rather than eight) are there
// for latency hiding: each step of a chunk is a short dependent chain of shared-memory loads,
// conversions and mma. Every mbarrier wait is bounded; a wait that runs out sets this unit's
// status word and a CTA-wide abort flag, after which the CTA's waits return at once and the CTA
// finishes without blocking (its outputs are then invalid).
#include <cuda.h>
#include <string.h>

#include <type_traits>

#include "gr_internal.h"
#include "gr_ptx.cuh"

namespace gr {
namespace {

constexpr int kTT = 32;                           // tokens per tile
constexpr int kCh = 64;                           // channels per chunk
constexpr int kCW = 16;                           // compute warps
constexpr int kCThreads = kCW * 32;
constexpr int kThreadsT = kCThreads + 32;         // + the producer warp
constexpr int kSStages = 7;                       // state ring depth
constexpr int kWStages = 3;                       // weight ring depth
constexpr int kYChunk = kTT * kCh * 2;              // 4 KB: y [32][64] bf16, 128B-swizzled
constexpr int kXBuf = 16 * 8 * 2;                 // per warp: x [16 tok][8 ch], unswizzled
constexpr int kXBufs = 4;                         // x buffers per warp (stores in flight)
constexpr int kMaxTiledRank = 32;
constexpr int kMaxFp8D = 8192;                    // the tile's block exponents: 4·D bytes on chip

// Compile-time sizes for NTD = ceil((r+4)/8) down-projection n-tiles and KSU = ceil(r/16)
// up-projection k-steps, for a bf16 state or an FP8 state (e4m3 codes; the tile's block
// exponents [32 tok][4][D/32] then sit at the end of shared memory, 4·D bytes).
template <int NTD, int KSU, bool FP8> struct TiledCfg {
    // R chunk [4][32][64]: bf16 with 128-byte rows (128B swizzle) or e4m3 codes with 64-byte
    // rows (64B swizzle)
    static constexpr int kRChunk = kBranches * kTT * kCh * (FP8 ? 1 : 2);
    static constexpr int kStateStage = kRChunk + kYChunk;
    static constexpr int kNP = 8 * NTD;                        // padded r + 4
    static constexpr int kHP = 16 * KSU;                       // padded r
    static constexpr int kDownChunk = kBranches * 4 * NTD * 256;  // [i][ks][nt][lane] uint2
    static constexpr int kUpFrag = 32 * KSU * 256;             // [co][i][lane][ks] uint2 (fp16)
    static constexpr int kUpChunk = kUpFrag + kBranches * kCh * 4;  // + gamma/8 [4][64] fp32
    static constexpr int kWStage = kDownChunk > kUpChunk ? kDownChunk : kUpChunk;
    static constexpr int off_state = 0;
    static constexpr int off_w = off_state + kSStages * kStateStage;
    static constexpr int off_x = off_w + kWStages * kWStage;
    // the owner step's partial sums [k-half][4][32][kNP] live in the state ring: between the
    // end of a tile's pass 1 and the owner step's completion no state fill is in flight or issued
    static constexpr int off_red = off_state;
    static constexpr int kRedBytes = 2 * kBranches * kTT * kNP * 4;
    static_assert(kRedBytes <= kSStages * kStateStage, "partial sums must fit in the state ring");
    static constexpr int off_ssq = off_x + kCW * kXBufs * kXBuf;
    static constexpr int off_h = off_ssq + 2 * kBranches * kTT * 4;
    static constexpr int off_inv = off_h + kTT * kHP * 4;
    static constexpr int off_bar = off_inv + kBranches * kTT * 4;
    static constexpr int kBars = 2 * kSStages + 2 * kWStages + 1;
    static constexpr int off_abort = off_bar + kBars * 8;
    // 16-byte vector copies move the block exponents in and out: keep the buffer aligned
    static constexpr int off_scl = (off_abort + 16 + 127) / 128 * 128;
    static_assert(off_scl % 16 == 0, "exponent buffer must be 16-byte aligned");
    // + 4·D bytes of block exponents on the FP8 path, + slack for the 1 KB alignment
    static int smem_bytes(int D) {
        return off_scl + (FP8 ? kBranches * kTT * scl_stride(D) : 0) + 1024;
    }
    // Row stride of the on-chip exponents [32 tok][4 br] rows of D/32 bytes: padded to 4 mod 8
    // bytes so that the rows 4g + i a warp reads together (g = 0..7) fall on 8 different banks.
    static __host__ __device__ int scl_stride(int D) {
        const int nblk = D / 32;   // a multiple of 4 (D % 128 == 0)
        return nblk % 8 == 0 ? nblk + 4 : nblk;
    }
};

// Bounded wait: one non-blocking test first (the common case: the data is there), then the
// bounded wait, which gives up at once after any wait of this CTA has run out.
__device__ __forceinline__ bool twait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (done) return true;
    if (*abort) return false;
    if (mbar_wait(bar, parity)) return true;
    *abort = 1u;
    return false;
}

// Position in a ring of S stages: the stage index and the parity of the round through the ring.
template <int S> struct RingPos {
    int st = 0;
    uint32_t ph = 0;
    __device__ __forceinline__ void next() {
        if (++st == S) {
            st = 0;
            ph ^= 1u;
        }
    }
};

__device__ __forceinline__ uint32_t lds32(const char* p) {
    return *reinterpret_cast<const uint32_t*>(p);
}
__device__ __forceinline__ void sts32(char* p, uint32_t v) { *reinterpret_cast<uint32_t*>(p) = v; }
__device__ __forceinline__ uint16_t lds16(const char* p) {
    return *reinterpret_cast<const uint16_t*>(p);
}
__device__ __forceinline__ void sts16(char* p, uint16_t v) { *reinterpret_cast<uint16_t*>(p) = v; }

template <bool WRITE, int NTD, int KSU, bool FP8>
__global__ void __launch_bounds__(kThreadsT, 1)
gr_tiled_kernel(const __grid_constant__ CUtensorMap tm_R,   // R/R' loads, box {64, 32, 4, 1}
                const __grid_constant__ CUtensorMap tm_Rs,  // R' stores, box {64, 16, 1, 1}
                const __grid_constant__ CUtensorMap tm_y,   // y loads, box {64, 32}
                const __grid_constant__ CUtensorMap tm_x,   // x stores, box {8, 16}
                int N, int D, int r, float eps, const float* __restrict__ s_prev,
                const char* __restrict__ frag, float* __restrict__ s_out,
                uint8_t* __restrict__ scales) {              // FP8: block exponents [N][4][D/32]
    using C = TiledCfg<NTD, KSU, FP8>;
    constexpr int kRChunk = C::kRChunk;
    constexpr int kStateStage = C::kStateStage;
    extern __shared__ uint8_t smem_raw[];
    char* smem = reinterpret_cast<char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int J = D / kCh;
    const int ntiles = (N + kTT - 1) / kTT;
    const char* down_frag = frag;                                   // J chunks of kDownChunk
    const char* up_frag = frag + size_t(J) * C::kDownChunk;         // J chunks of kUpChunk

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::off_bar);
    uint64_t* sfull = bars;
    uint64_t* sempty = bars + kSStages;
    uint64_t* wfull = bars + 2 * kSStages;
    uint64_t* wempty = bars + 2 * kSStages + kWStages;
    uint64_t* t1done = bars + 2 * kSStages + 2 * kWStages;
    volatile uint32_t* abort = reinterpret_cast<volatile uint32_t*>(smem + C::off_abort);
    float* red = reinterpret_cast<float*>(smem + C::off_red);   // [k-half][4][32][kNP]
    float* ssqb = reinterpret_cast<float*>(smem + C::off_ssq);  // [k-half][4][32]
    float* hbuf = reinterpret_cast<float*>(smem + C::off_h);    // [32][kHP]
    float* invb = reinterpret_cast<float*>(smem + C::off_inv);  // [4][32]
    uint8_t* scl = reinterpret_cast<uint8_t*>(smem + C::off_scl);  // FP8: [32 tok][4][D/32]
    const int nblk = D / 32;
    const int sst = C::scl_stride(D);   // bytes between the exponent rows on chip
    auto sbuf = [&](int st) { return smem + C::off_state + st * kStateStage; };
    auto wbuf = [&](int st) { return smem + C::off_w + st * C::kWStage; };

    if (tid == 0) {
        for (int s = 0; s < kSStages; ++s) {
            mbar_init(&sfull[s], 1u);
            mbar_init(&sempty[s], uint32_t(kCW));
        }
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(&wfull[s], 1u);
            mbar_init(&wempty[s], uint32_t(kCW));
        }
        mbar_init(t1done, 1u);
        *abort = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // h columns r .. kHP-1 stay zero (the padded k of the up projection)
    for (int e = tid; e < kTT * C::kHP; e += kThreadsT) hbuf[e] = 0.f;
    __syncthreads();

    if (warp == kCW) {
        // ================================ producer =============================================
        if (lane != 0) return;
        RingPos<kSStages> sp;   // next fill of each ring; a stage is refilled once the compute
        RingPos<kWStages> wp;   // warps released the previous round's fill (after the first round)
        bool s_wrapped = false, w_wrapped = false;
        uint32_t nt_local = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++nt_local) {
            const int t0 = tile * kTT;
            for (int pass = 0; pass < 2; ++pass) {
                if (pass == 1) {
                    // pass 2 reads back the R' that pass 1 stored through the async proxy, and
                    // its fills reuse the ring the owner step borrowed for its partial sums
                    twait(t1done, nt_local & 1u, abort);
                    fence_async_global();
                }
                for (int jj = 0; jj < J; ++jj) {
                    const int j = pass == 0 ? jj : J - 1 - jj;
                    {   // state: R (pass 1) or R' (pass 2) chunk j, plus y chunk j in pass 1
                        const int st = sp.st;
                        if (s_wrapped) twait(&sempty[st], sp.ph ^ 1u, abort);
                        char* b = sbuf(st);
                        const bool with_y = WRITE && pass == 0;
                        mbar_expect_tx(&sfull[st], uint32_t(kRChunk + (with_y ? kYChunk : 0)));
                        tma_load_4d(b, &tm_R, 0, t0, 0, j, &sfull[st]);
                        if (with_y) tma_load_2d(b + kRChunk, &tm_y, j * kCh, t0, &sfull[st]);
                        sp.next();
                        s_wrapped |= sp.st == 0;
                    }
                    {   // weights: down-projection fragments (pass 1) or W_u fragments + γ/8
                        const int st = wp.st;
                        if (w_wrapped) twait(&wempty[st], wp.ph ^ 1u, abort);
                        const uint32_t bytes = uint32_t(pass == 0 ? C::kDownChunk : C::kUpChunk);
                        const char* src = pass == 0 ? down_frag + size_t(j) * C::kDownChunk
                                                    : up_frag + size_t(j) * C::kUpChunk;
                        mbar_expect_tx(&wfull[st], bytes);
                        bulk_g2s(wbuf(st), src, bytes, &wfull[st]);
                        wp.next();
                        w_wrapped |= wp.st == 0;
                    }
                }
            }
        }
        // drain: the last fill of every stage has landed before the CTA may exit (stage s was
        // last filled in the current round if s < the next fill's index, else in the previous)
        for (int s = 0; s < kSStages; ++s)
            if (s < sp.st || s_wrapped) mbar_wait(&sfull[s], s < sp.st ? sp.ph : sp.ph ^ 1u);
        for (int s = 0; s < kWStages; ++s)
            if (s < wp.st || w_wrapped) mbar_wait(&wfull[s], s < wp.st ? wp.ph : wp.ph ^ 1u);
        return;
    }

    // ================================== compute warps ==========================================
    const int g = lane >> 2, q = lane & 3;
    // pass 1: branch ib, m-tile mt, k-half kh (k-steps 2kh and 2kh+1 of every chunk); the two
    // k-halves of one (branch, m-tile) meet at named barrier 2 + pair before its R' store
    const int ib = warp & 3, mt = (warp >> 2) & 1, kh = warp >> 3, pair = warp & 7;
    // pass 2: m-tile mt2, 8-channel group co of the chunk
    const int mt2 = warp & 1, co = warp >> 1;
    const float inv_d = 1.0f / float(D);
    char* xb0 = smem + C::off_x + warp * kXBufs * kXBuf;
    RingPos<kSStages> sr;   // next chunk to consume on each ring
    RingPos<kWStages> wr;
    uint32_t xc = 0;

    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int t0 = tile * kTT;
        if constexpr (FP8) {
            // The tile's block exponents, [32 tok][4][D/32], contiguous in HBM, into padded rows
            // on chip with 4-byte loads (D % 128 == 0: every row is a whole number of words).
            // The first barrier waits until no warp still reads the previous tile's exponents
            // in its pass 2.
            named_sync(1, kCThreads);
            const int nv = min(kTT, N - t0);
            const int wpr = nblk / 4;   // words per row
            const int nw = nv * kBranches * wpr;
            const uint32_t* src = reinterpret_cast<const uint32_t*>(scales + size_t(t0) * (D / 8));
            for (int e = tid; e < nw; e += kCThreads) {
                const int row = e / wpr, w = e - row * wpr;
                *reinterpret_cast<uint32_t*>(scl + row * sst + 4 * w) = src[e];
            }
            named_sync(1, kCThreads);
        }
        // ---------------------------------- pass 1 --------------------------------------------
        float spa = 0.f, spb = 0.f;   // s_prev of tokens g and g+8 of the m-tile, branch ib
        if (WRITE) {
            const int ta = t0 + 16 * mt + g, tb = ta + 8;
            if (ta < N) spa = s_prev[size_t(ta) * 4 + ib];
            if (tb < N) spb = s_prev[size_t(tb) * 4 + ib];
        }
        const uint64_t sa2 = f2(spa, spa), sb2 = f2(spb, spb);
        float acc[NTD][4];
#pragma unroll
        for (int n = 0; n < NTD; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        uint64_t ssa = f2(0.f, 0.f), ssb = f2(0.f, 0.f);
        const int rowa = ib * kTT + 16 * mt + g, rowb = rowa + 8;  // rows of the R box
        const int ya = 16 * mt + g, yb = ya + 8;                     // rows of the y box
        int prev_st = -1;
        for (int j = 0; j < J; ++j) {
            const int st = sr.st;
            twait(&sfull[st], sr.ph, abort);
            twait(&wfull[wr.st], wr.ph, abort);
            char* rb = sbuf(st);
            const char* ybuf = rb + kRChunk;
            const uint2* wd = reinterpret_cast<const uint2*>(wbuf(wr.st)) + ib * 4 * NTD * 32;
            if constexpr (!FP8) {
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const int ks = 2 * kh + kk;
                    uint32_t a[4];
                    const int o[4] = {swz(rowa, 2 * ks) + 4 * q, swz(rowb, 2 * ks) + 4 * q,
                                      swz(rowa, 2 * ks + 1) + 4 * q, swz(rowb, 2 * ks + 1) + 4 * q};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint32_t v = lds32(rb + o[e]);
                        if (WRITE) {
                            const int yo = swz((e & 1) ? yb : ya, 2 * ks + (e >> 1)) + 4 * q;
                            const uint64_t yy = bf2_to_f2(lds32(ybuf + yo));
                            v = f2_to_bf2(fma2(yy, (e & 1) ? sb2 : sa2, bf2_to_f2(v)));
                            sts32(rb + o[e], v);
                        }
                        const uint64_t f = bf2_to_f2(v);
                        if (e & 1) ssb = fma2(f, f, ssb);
                        else ssa = fma2(f, f, ssa);
                        a[e] = v;
                    }
#pragma unroll
                    for (int n = 0; n < NTD; ++n) {
                        const uint2 b = wd[(ks * NTD + n) * 32 + lane];
                        mma_bf16(acc[n], a[0], a[1], a[2], a[3], b.x, b.y);
                    }
                }
            } else {
                // FP8: this warp's two k-steps are exactly one 32-channel block (2j + kh) of its
                // rows; the four lanes of a quad hold the block. Decode R with the old exponent,
                // write in fp32, pick the new exponent from the block maximum, encode in place.
                uint8_t* ea_p = scl + ((16 * mt + g) * kBranches + ib) * sst + 2 * j + kh;
                uint8_t* eb_p = ea_p + 8 * kBranches * sst;
                const float da = pow2f(int(*ea_p) - 127), db = pow2f(int(*eb_p) - 127);
                float2 v[2][4];
                // byte offset of the code pair (row a or b, channels 2q, 2q+1 (+8)) in the box
                auto code_off = [&](int kk, int e) {
                    return swz64((e & 1) ? rowb : rowa, 2 * kh + kk) + 2 * q + 8 * (e >> 1);
                };
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const int ks = 2 * kh + kk;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float2 w = e4m3x2_to_f2(lds16(rb + code_off(kk, e)));
                        const float d = (e & 1) ? db : da;
                        w.x *= d;
                        w.y *= d;
                        if (WRITE) {
                            const int yo = swz((e & 1) ? yb : ya, 2 * ks + (e >> 1)) + 4 * q;
                            float yx, yy;
                            unf2(bf2_to_f2(lds32(ybuf + yo)), yx, yy);
                            const float sv = (e & 1) ? spb : spa;
                            w.x = fmaf(sv, yx, w.x);
                            w.y = fmaf(sv, yy, w.y);
                        }
                        v[kk][e] = w;
                    }
                }
                if (WRITE) {
                    float ma = 0.f, mb = 0.f;
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float m = fmaxf(fabsf(v[kk][e].x), fabsf(v[kk][e].y));
                            if (e & 1) mb = fmaxf(mb, m);
                            else ma = fmaxf(ma, m);
                        }
                    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
                    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
                    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
                    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
                    const int na = fp8_block_exp(ma), nb = fp8_block_exp(mb);
                    const float ia = pow2f(-na), ib_ = pow2f(-nb);
                    const float ua = pow2f(na), ub = pow2f(nb);
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float i_ = (e & 1) ? ib_ : ia, u_ = (e & 1) ? ub : ua;
                            const uint16_t code = f2_to_e4m3x2(v[kk][e].x * i_, v[kk][e].y * i_);
                            sts16(rb + code_off(kk, e), code);
                            float2 w = e4m3x2_to_f2(code);   // the stored value, for the read
                            w.x *= u_;
                            w.y *= u_;
                            v[kk][e] = w;
                        }
                    // every lane of the quad has read the old exponent (it fed the maximum)
                    if (q == 0) {
                        *ea_p = uint8_t(na + 127);
                        *eb_p = uint8_t(nb + 127);
                    }
                }
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const int ks = 2 * kh + kk;
                    uint32_t a[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint64_t f = f2(v[kk][e].x, v[kk][e].y);
                        if (e & 1) ssb = fma2(f, f, ssb);
                        else ssa = fma2(f, f, ssa);
                        a[e] = pack_bf2(v[kk][e].x, v[kk][e].y);   // exact: 4 significant bits
                    }
#pragma unroll
                    for (int n = 0; n < NTD; ++n) {
                        const uint2 b = wd[(ks * NTD + n) * 32 + lane];
                        mma_bf16(acc[n], a[0], a[1], a[2], a[3], b.x, b.y);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&wempty[wr.st]);
            if (WRITE) {
                // both k-halves of this (branch, m-tile) have written R' back before its store
                fence_async_shared();
                named_sync(2 + pair, 64);
                if (kh == 1) {
                    if (lane == 0) mbar_arrive(&sempty[st]);
                } else if (lane == 0) {
                    // an m-tile wholly past the last token has nothing to store (empty group)
                    if (t0 + 16 * mt < N)
                        tma_store_4d(&tm_Rs, rb + (ib * kTT + 16 * mt) * kCh * (FP8 ? 1 : 2), 0,
                                     t0 + 16 * mt, ib, j);
                    bulk_commit();
                    // the previous chunk's stage is free once its store has read it
                    bulk_wait_read<1>();
                    if (prev_st >= 0) mbar_arrive(&sempty[prev_st]);
                }
            } else if (lane == 0) {
                mbar_arrive(&sempty[st]);
            }
            prev_st = st;
            sr.next();
            wr.next();
        }
        if (WRITE && lane == 0 && kh == 0) {
            bulk_wait_all();           // every R' store of the tile has reached global memory
            fence_async_global();
            if (prev_st >= 0) mbar_arrive(&sempty[prev_st]);
        }
        // ---------------------------------- owner step ----------------------------------------
        // every warp is done with pass 1's stages and every store has read them: the partial
        // sums may now overwrite the ring
        named_sync(1, kCThreads);
        if constexpr (FP8 && WRITE) {
            // the tile's new block exponents go back to HBM (pass 2 reads them from here)
            const int nv = min(kTT, N - t0);
            const int wpr = nblk / 4;
            const int nw = nv * kBranches * wpr;
            uint32_t* dst = reinterpret_cast<uint32_t*>(scales + size_t(t0) * (D / 8));
            for (int e = tid; e < nw; e += kCThreads) {
                const int row = e / wpr, w = e - row * wpr;
                dst[e] = *reinterpret_cast<const uint32_t*>(scl + row * sst + 4 * w);
            }
        }
        {
            float s0, s1, s2, s3;
            unf2(ssa, s0, s1);
            unf2(ssb, s2, s3);
            float qa = s0 + s1, qb = s2 + s3;
            qa += __shfl_xor_sync(0xffffffffu, qa, 1);
            qa += __shfl_xor_sync(0xffffffffu, qa, 2);
            qb += __shfl_xor_sync(0xffffffffu, qb, 1);
            qb += __shfl_xor_sync(0xffffffffu, qb, 2);
            const int ra_row = ib * kTT + 16 * mt + g;
            float* ra = red + (kh * kBranches * kTT + ra_row) * C::kNP;
            float* rb_ = ra + 8 * C::kNP;
#pragma unroll
            for (int n = 0; n < NTD; ++n) {
                *reinterpret_cast<float2*>(ra + n * 8 + 2 * q) = make_float2(acc[n][0], acc[n][1]);
                *reinterpret_cast<float2*>(rb_ + n * 8 + 2 * q) = make_float2(acc[n][2], acc[n][3]);
            }
            if (q == 0) {
                ssqb[kh * kBranches * kTT + ra_row] = qa;
                ssqb[kh * kBranches * kTT + ra_row + 8] = qb;
            }
        }
        named_sync(1, kCThreads);
        {
            const int nk = r + 4;
            for (int it = tid; it < kTT * nk; it += kCThreads) {
                const int tok = it / nk, n = it - tok * nk;
                float z = 0.f;
#pragma unroll
                for (int i = 0; i < kBranches; ++i) {
                    const int row = i * kTT + tok;
                    const float inv =
                        rsqrtf((ssqb[row] + ssqb[kBranches * kTT + row]) * inv_d + eps);
                    z = fmaf(inv, red[row * C::kNP + n] + red[(kBranches * kTT + row) * C::kNP + n],
                             z);
                    if (n == 0) invb[row] = inv;
                }
                z *= 0.25f;
                const float sg = __fdividef(1.0f, 1.0f + __expf(-z));
                if (n < r) hbuf[tok * C::kHP + n] = z * sg;
                else if (t0 + tok < N) s_out[size_t(t0 + tok) * 4 + (n - r)] = 2.0f * sg;
            }
        }
        named_sync(1, kCThreads);
        // the partial sums are consumed: the producer may start pass 2's fills
        if (tid == 0) mbar_arrive(t1done);
        // ---------------------------------- pass 2 --------------------------------------------
        uint32_t ah[KSU][4];     // fp16 A fragments of the scaled h
        uint64_t unscale_a, unscale_b;   // 2^e of tokens g and g+8, as fp32 pairs
        bool unit_scale;                 // every row of the warp unscaled (e = 0)
        {
            const float* ha = hbuf + (16 * mt2 + g) * C::kHP;
            const float* hb = ha + 8 * C::kHP;
            float2 v[KSU][4];
            float ma = 0.f, mb = 0.f;
#pragma unroll
            for (int ks = 0; ks < KSU; ++ks) {
                v[ks][0] = *reinterpret_cast<const float2*>(ha + ks * 16 + 2 * q);
                v[ks][1] = *reinterpret_cast<const float2*>(hb + ks * 16 + 2 * q);
                v[ks][2] = *reinterpret_cast<const float2*>(ha + ks * 16 + 2 * q + 8);
                v[ks][3] = *reinterpret_cast<const float2*>(hb + ks * 16 + 2 * q + 8);
                ma = fmaxf(ma, fmaxf(fmaxf(fabsf(v[ks][0].x), fabsf(v[ks][0].y)),
                                     fmaxf(fabsf(v[ks][2].x), fabsf(v[ks][2].y))));
                mb = fmaxf(mb, fmaxf(fmaxf(fabsf(v[ks][1].x), fabsf(v[ks][1].y)),
                                     fmaxf(fabsf(v[ks][3].x), fabsf(v[ks][3].y))));
            }
            // the four lanes of a quad hold the whole row of a token
            ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
            ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
            // e = max(0, exponent(max) - 14): the scaled row stays below 2^15 (fp16 max 65504)
            const int ea = min(max(((__float_as_int(ma) >> 23) & 0xff) - 127 - 14, 0), 126);
            const int eb = min(max(((__float_as_int(mb) >> 23) & 0xff) - 127 - 14, 0), 126);
            const float sa = __int_as_float((127 - ea) << 23), sb = __int_as_float((127 - eb) << 23);
            const float ua = __int_as_float((127 + ea) << 23), ub = __int_as_float((127 + eb) << 23);
            unscale_a = f2(ua, ua);
            unscale_b = f2(ub, ub);
            unit_scale = __all_sync(0xffffffffu, (ea | eb) == 0);
#pragma unroll
            for (int ks = 0; ks < KSU; ++ks)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float sc = (e & 1) ? sb : sa;
                    ah[ks][e] = pack_h2(v[ks][e].x * sc, v[ks][e].y * sc);
                }
        }
        float inv2[kBranches][2];
#pragma unroll
        for (int i = 0; i < kBranches; ++i) {
            inv2[i][0] = invb[i * kTT + 16 * mt2 + g];
            inv2[i][1] = invb[i * kTT + 16 * mt2 + g + 8];
        }
        const int ch = co * 8 + 2 * q;   // this thread's channel pair within the chunk
        // SCALED: some token row of the warp was scaled down and its logits are scaled back;
        // otherwise every scale is 1 and the chunk loop has no multiplies for it (a product
        // with 1 is exact, so both paths give the same result)
        auto pass2 = [&](auto scaled) {
        constexpr bool SCALED = decltype(scaled)::value;
        for (int jj = 0; jj < J; ++jj) {
            const int j = J - 1 - jj;
            const int st = sr.st;
            twait(&sfull[st], sr.ph, abort);
            twait(&wfull[wr.st], wr.ph, abort);
            const char* rb = sbuf(st);
            const char* wb = wbuf(wr.st);
            const uint2* wu = reinterpret_cast<const uint2*>(wb) + co * kBranches * 32 * KSU;
            const float* gam = reinterpret_cast<const float*>(wb + C::kUpFrag);  // [4][64], γ/8
            char* xb = xb0 + int(xc % kXBufs) * kXBuf;
            // the x buffer is free once the store issued from it kXBufs chunks ago has read it
            if (lane == 0) bulk_wait_read<kXBufs - 1>();
            __syncwarp();
            // all of the chunk's mma first, then the combine in packed fp32 pairs
            float cg4[kBranches][4];
#pragma unroll
            for (int i = 0; i < kBranches; ++i) {
                const uint2 b = wu[(i * 32 + lane) * KSU];
                mma_f16_z(cg4[i], ah[0][0], ah[0][1], ah[0][2], ah[0][3], b.x, b.y);
            }
#pragma unroll
            for (int ks = 1; ks < KSU; ++ks)
#pragma unroll
                for (int i = 0; i < kBranches; ++i) {
                    const uint2 b = wu[(i * 32 + lane) * KSU + ks];
                    mma_f16(cg4[i], ah[ks][0], ah[ks][1], ah[ks][2], ah[ks][3], b.x, b.y);
                }
            uint64_t xa = f2(0.f, 0.f), xbv = f2(0.f, 0.f);
            const uint64_t one2 = f2(1.0f, 1.0f);
#pragma unroll
            for (int i = 0; i < kBranches; ++i) {
                const float2 gm = *reinterpret_cast<const float2*>(gam + i * kCh + ch);
                const uint64_t g2 = f2(gm.x, gm.y);
                const int row = i * kTT + 16 * mt2 + g;
                uint64_t rpa, rpb;   // R' of tokens g and g+8 at this thread's channel pair
                if constexpr (!FP8) {
                    rpa = bf2_to_f2(lds32(rb + swz(row, co) + 4 * q));
                    rpb = bf2_to_f2(lds32(rb + swz(row + 8, co) + 4 * q));
                } else {
                    const int off = (co & 1) * 8 + 2 * q;
                    const uint8_t* ep =
                        scl + ((16 * mt2 + g) * kBranches + i) * sst + 2 * j + (co >> 2);
                    const float da = pow2f(int(ep[0]) - 127);
                    const float db = pow2f(int(ep[8 * kBranches * sst]) - 127);
                    const float2 wa = e4m3x2_to_f2(lds16(rb + swz64(row, co >> 1) + off));
                    const float2 wb = e4m3x2_to_f2(lds16(rb + swz64(row + 8, co >> 1) + off));
                    rpa = f2(wa.x * da, wa.y * da);
                    rpb = f2(wb.x * db, wb.y * db);
                }
                const uint64_t ra = mul2(rpa, mul2(g2, f2(inv2[i][0], inv2[i][0])));
                const uint64_t rbv = mul2(rpb, mul2(g2, f2(inv2[i][1], inv2[i][1])));
                float a0 = cg4[i][0], a1 = cg4[i][1], b0 = cg4[i][2], b1 = cg4[i][3];
                if constexpr (SCALED) {
                    unf2(mul2(f2(a0, a1), unscale_a), a0, a1);
                    unf2(mul2(f2(b0, b1), unscale_b), b0, b1);
                }
                const uint64_t ta = add2(f2(tanh_approx(a0), tanh_approx(a1)), one2);
                const uint64_t tb = add2(f2(tanh_approx(b0), tanh_approx(b1)), one2);
                xa = fma2(ta, ra, xa);
                xbv = fma2(tb, rbv, xbv);
            }
            sts32(xb + g * 16 + 4 * q, f2_to_bf2(xa));
            sts32(xb + (g + 8) * 16 + 4 * q, f2_to_bf2(xbv));
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sempty[st]);
                mbar_arrive(&wempty[wr.st]);
            }
            fence_async_shared();
            __syncwarp();
            if (lane == 0) {
                if (t0 + 16 * mt2 < N) tma_store_2d(&tm_x, xb, j * kCh + co * 8, t0 + 16 * mt2);
                bulk_commit();
            }
            sr.next();
            wr.next();
            ++xc;
        }
        };
        if (unit_scale) pass2(std::false_type{});
        else pass2(std::true_type{});
    }
    if (lane == 0) bulk_wait_all();
    // As the programmatic dependent of a cluster-kernel launch (the concurrent split), this grid
    // completes only after that grid has: work after the call in the stream then follows both.
    dep_wait();
}

// ---- packing ---------------------------------------------------------------------------------

// Fragment section of the tiled kernel: J chunks of down-projection B fragments (bf16, γ
// folded), then J chunks of W_u B fragments (fp16, ×½, clamped to ±65504) each followed by γ/8
// of the chunk's channels.
template <int NTD, int KSU>
__global__ void pack_tiled_kernel(int D, int r, const float* __restrict__ gamma,
                                  const float* __restrict__ wd, const float* __restrict__ wu,
                                  const float* __restrict__ ww, char* __restrict__ frag) {
    using C = TiledCfg<NTD, KSU, false>;   // the fragment layout is the same for both states
    const int J = D / kCh;
    const size_t K = size_t(kBranches) * D;
    const int n_down = kBranches * 4 * NTD * 32;      // uint2 units per chunk
    const int n_up = 32 * KSU * 32;                   // uint2 units per chunk
    const int n_gam = kBranches * kCh;                // floats per chunk
    const size_t per_chunk = size_t(n_down + n_up + n_gam);
    const size_t total = per_chunk * J;
    for (size_t e = blockIdx.x * size_t(blockDim.x) + threadIdx.x; e < total;
         e += size_t(gridDim.x) * blockDim.x) {
        const int j = int(e / per_chunk);
        int u = int(e - size_t(j) * per_chunk);
        if (u < n_down) {
            // u = ((i*4 + ks)*NTD + nt)*32 + lane
            const int lane = u & 31, rest = u >> 5;
            const int nt = rest % NTD, iks = rest / NTD;
            const int ks = iks & 3, i = iks >> 2;
            const int n = nt * 8 + (lane >> 2);
            const size_t m0 = size_t(i) * D + size_t(j) * kCh + ks * 16 + 2 * (lane & 3);
            const int koff[4] = {0, 1, 8, 9};
            __nv_bfloat16* dst =
                reinterpret_cast<__nv_bfloat16*>(frag + size_t(j) * C::kDownChunk) + size_t(u) * 4;
            for (int t = 0; t < 4; ++t) {
                const size_t m = m0 + koff[t];
                float v = 0.f;
                if (n < r) v = wd[size_t(n) * K + m] * gamma[m];
                else if (n < r + 4) v = ww[size_t(n - r) * K + m] * gamma[m];
                dst[t] = __float2bfloat16_rn(v);
            }
        } else if ((u -= n_down) < n_up) {
            // u = ((co*4 + i)*32 + lane)*KSU + ks
            const int ks = u % KSU, rest = u / KSU;
            const int lane = rest & 31, r2 = rest >> 5;
            const int i = r2 & 3, co = r2 >> 2;
            const size_t m = size_t(i) * D + size_t(j) * kCh + co * 8 + (lane >> 2);
            const int k0 = ks * 16 + 2 * (lane & 3);
            const int kk[4] = {k0, k0 + 1, k0 + 8, k0 + 9};
            __half* dst = reinterpret_cast<__half*>(frag + size_t(J) * C::kDownChunk +
                                                    size_t(j) * C::kUpChunk) +
                          size_t(u) * 4;
            for (int t = 0; t < 4; ++t) {
                const float v = kk[t] < r ? 0.5f * wu[m * size_t(r) + kk[t]] : 0.f;
                dst[t] = __float2half_rn(fminf(fmaxf(v, -65504.f), 65504.f));
            }
        } else {
            u -= n_up;
            const int i = u / kCh, c = u - i * kCh;
            float* dst = reinterpret_cast<float*>(frag + size_t(J) * C::kDownChunk +
                                                  size_t(j) * C::kUpChunk + C::kUpFrag);
            dst[u] = 0.125f * gamma[size_t(i) * D + size_t(j) * kCh + c];
        }
    }
}

// ---- host side ---------------------------------------------------------------------------------

// R as {channel within a 64-channel chunk, token, branch, chunk}: the box {64, tok_box, br_box, 1}
// lands as rows (branch, token) of 64 elements: 128 bytes of bf16 (128-byte swizzle) or 64 bytes
// of e4m3 codes (64-byte swizzle).
bool make_map_R(CUtensorMap* m, const void* R, int64_t N, int D, int tok_box, int br_box,
                bool fp8) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t es_b = fp8 ? 1 : 2;
    const cuuint64_t dims[4] = {cuuint64_t(kCh), cuuint64_t(N), 4, cuuint64_t(D / kCh)};
    const cuuint64_t strides[3] = {cuuint64_t(D) * 4 * es_b, cuuint64_t(D) * es_b,
                                   cuuint64_t(kCh) * es_b};
    const cuuint32_t box[4] = {cuuint32_t(kCh), cuuint32_t(tok_box), cuuint32_t(br_box), 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
               const_cast<void*>(R), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               fp8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// A [N, D] bf16 matrix (y or x) with box {box_ch, box_tok}.
bool make_map_nd(CUtensorMap* m, const void* p, int64_t N, int D, int box_ch, int box_tok,
                 CUtensorMapSwizzle sw) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cuuint64_t(D), cuuint64_t(N)};
    const cuuint64_t strides[1] = {cuuint64_t(D) * 2};
    const cuuint32_t box[2] = {cuuint32_t(box_ch), cuuint32_t(box_tok)};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Largest dynamic shared memory already granted to each instantiation, per device (the attribute
// is set once, not on every launch).
template <bool WRITE, int NTD, int KSU, bool FP8> int g_smem_set[64];

template <bool WRITE, int NTD, int KSU, bool FP8>
cudaError_t launch_t(int64_t N, int D, int r, float eps, void* R, uint8_t* scales, const void* y,
                     const float* s_prev, const char* frag, void* x, float* s_out,
                     cudaStream_t st, int max_ctas, bool programmatic) {
    using C = TiledCfg<NTD, KSU, FP8>;
    CUtensorMap mR, mRs, my, mx;
    memset(&mRs, 0, sizeof(mRs));
    memset(&my, 0, sizeof(my));
    if (!make_map_R(&mR, R, N, D, kTT, kBranches, FP8)) return cudaErrorInvalidValue;
    if (WRITE && !make_map_R(&mRs, R, N, D, 16, 1, FP8)) return cudaErrorInvalidValue;
    if (WRITE && !make_map_nd(&my, y, N, D, kCh, kTT, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (!make_map_nd(&mx, x, N, D, 8, 16, CU_TENSOR_MAP_SWIZZLE_NONE)) return cudaErrorInvalidValue;
    auto kern = gr_tiled_kernel<WRITE, NTD, KSU, FP8>;
    const int smem = C::smem_bytes(D);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int& granted = g_smem_set<WRITE, NTD, KSU, FP8>[dev & 63];
    if (granted < smem) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        granted = smem;
    }
    const int64_t ntiles = (N + kTT - 1) / kTT;
    int64_t grid = ntiles < sm_count() ? ntiles : sm_count();
    if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
    // as a programmatic dependent of the preceding launch on the stream (the split's cluster
    // kernel): its CTAs start once that grid's CTAs are all resident, and it finishes after it
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(kThreadsT);
    cfg.dynamicSmemBytes = size_t(smem);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, mR, mRs, my, mx, int(N), D, r, eps, s_prev, frag,
                              s_out, scales);
}

template <int NTD, int KSU, bool FP8>
cudaError_t launch_k(int64_t N, int D, int r, float eps, void* R, uint8_t* scales, const void* y,
                     const float* s_prev, const char* frag, void* x, float* s_out,
                     cudaStream_t st, int max_ctas = 0, bool programmatic = false) {
    return y ? launch_t<true, NTD, KSU, FP8>(N, D, r, eps, R, scales, y, s_prev, frag, x, s_out,
                                             st, max_ctas, programmatic)
             : launch_t<false, NTD, KSU, FP8>(N, D, r, eps, R, scales, y, s_prev, frag, x, s_out,
                                              st, max_ctas, programmatic);
}

}  // namespace

bool tiled_supported(int D, int r) {
    return D >= kCh && D % kCh == 0 && r >= 1 && r <= kMaxTiledRank;
}

int64_t tiled_max_tokens() { return int64_t(0x7fffffff) - kTT; }

// The two instantiations: r <= 12 (NTD 2, KSU 1) is served by NTD 3; r <= 16 by (3, 1); r <= 32
// by (5, 2). Padded rows and k columns are zero in the packed fragments.
static void tiled_cfg(int r, int& ntd, int& ksu) {
    if (r <= 16) { ntd = 3; ksu = 1; }
    else { ntd = 5; ksu = 2; }
}

size_t tiled_frag_bytes(int D, int r) {
    int ntd, ksu;
    tiled_cfg(r, ntd, ksu);
    const size_t J = size_t(D / kCh);
    using C3 = TiledCfg<3, 1, false>;
    using C5 = TiledCfg<5, 2, false>;
    return ntd == 3 ? J * (C3::kDownChunk + C3::kUpChunk) : J * (C5::kDownChunk + C5::kUpChunk);
}

cudaError_t launch_pack_tiled(int D, int r, const float* gamma, const float* wd, const float* wu,
                              const float* ww, void* frag, cudaStream_t st) {
    int ntd, ksu;
    tiled_cfg(r, ntd, ksu);
    const size_t total = tiled_frag_bytes(D, r) / 8 + 1;
    const int threads = 256;
    const size_t want = (total + threads - 1) / threads;
    const size_t cap = size_t(sm_count()) * 8;
    const int blocks = int(want < cap ? want : cap);
    if (ntd == 3)
        pack_tiled_kernel<3, 1><<<blocks, threads, 0, st>>>(D, r, gamma, wd, wu, ww,
                                                            static_cast<char*>(frag));
    else
        pack_tiled_kernel<5, 2><<<blocks, threads, 0, st>>>(D, r, gamma, wd, wu, ww,
                                                            static_cast<char*>(frag));
    return cudaGetLastError();
}

cudaError_t launch_tiled_bf16(int64_t N, int D, int r, float eps, void* R, const void* y,
                              const float* s_prev, const void* packed, void* x, float* s_out,
                              cudaStream_t st, int max_ctas, bool programmatic) {
    if (!tiled_supported(D, r) || N < 1 || N > tiled_max_tokens()) return cudaErrorInvalidValue;
    const Layout L = make_layout(D, r, GR_BF16);
    const char* frag = static_cast<const char*>(packed) + (L.frag2_bytes ? L.frag2 : L.frag);
    int ntd, ksu;
    tiled_cfg(r, ntd, ksu);
    if (ntd == 3)
        return launch_k<3, 1, false>(N, D, r, eps, R, nullptr, y, s_prev, frag, x, s_out, st,
                                     max_ctas, programmatic);
    return launch_k<5, 2, false>(N, D, r, eps, R, nullptr, y, s_prev, frag, x, s_out, st,
                                 max_ctas, programmatic);
}

bool tiled_fp8_supported(int D, int r) {
    return tiled_supported(D, r) && D % 128 == 0 && D <= kMaxFp8D;
}

cudaError_t launch_tiled_fp8(int64_t N, int D, int r, float eps, uint8_t* codes,
                             uint8_t* scales, const void* y, const float* s_prev,
                             const void* packed, void* x, float* s_out, cudaStream_t st) {
    if (!tiled_fp8_supported(D, r) || N < 1 || N > tiled_max_tokens())
        return cudaErrorInvalidValue;
    const Layout L = make_layout(D, r, GR_FP8);
    const char* frag = static_cast<const char*>(packed) + L.frag;
    int ntd, ksu;
    tiled_cfg(r, ntd, ksu);
    if (ntd == 3)
        return launch_k<3, 1, true>(N, D, r, eps, codes, scales, y, s_prev, frag, x, s_out, st);
    return launch_k<5, 2, true>(N, D, r, eps, codes, scales, y, s_prev, frag, x, s_out, st);
}

int tiled_status(bool clear) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_wait_status, sizeof(v)) != cudaSuccess) return -1;
    if (clear && v) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(g_wait_status, &z, sizeof(z)) != cudaSuccess) return -1;
    }
    return int(v);
}

}  // namespace gr
