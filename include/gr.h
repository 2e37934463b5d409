/*
 * gr.h — C ABI of the GB300 Gated Residual (GR) read/write library (libgr_gb300.so).
 *
 * What the calls compute (all per token t, branch i, channel c; n_r = 4 branches):
 *   "【论文解读】 Qwen3.8 Flash Next" (wkq9411.github.io), §二.4 Gated Residual:
 *     eq rms      R̂_i = RMSNorm(R_i; γ_i) = R_i · γ_i / sqrt(mean_c R_i[c]^2 + eps)
 *     eq gate     G = unvec σ(W_u SiLU((1/n_r) W_d vec R̂))
 *     eq use_gate x = (1/n_r) Σ_i G_i ⊙ R̂_i
 *     eq s        s = 2σ((1/n_r) W_w vec R̂)
 *     eq write    R'_i = R_i + s_i · y
 *   "Qwen3.8-Flash-Next 架构笔记 · 06 / RESIDUAL" (cbphcr.github.io) §2–§3 give the same
 *   formulas at n_r = 4, and §5 asks that the read and the write each traverse the widened
 *   state once; gr_write_then_read fuses one sublayer's write with the next sublayer's read so
 *   that each state byte crosses HBM once per sublayer.
 *
 * Conventions shared by every call:
 *   - Tensor pointers are DEVICE pointers owned by the caller (unless a call says HOST). The
 *     library never allocates or frees memory.
 *   - Calls are asynchronous on the caller's CUDA stream, passed as `void*` (cudaStream_t;
 *     NULL = the legacy default stream). Results are ready when the stream has reached them.
 *   - Layouts are row-major and dense:
 *       R   [N][4][D]  state (token, branch, channel), dtype shape->state_dtype
 *       y   [N][D]     sublayer output F(x), state dtype
 *       x   [N][D]     block input for the next sublayer, state dtype
 *       s   [N][4]     write strengths, fp32
 *       gamma [4][D], W_d [r][4D], W_u [4D][r], W_w [4][4D], fp32 (vec index = i*D + c)
 *   - Arithmetic is fp32. bf16 stores round to nearest even. On the bf16 path the weights are
 *     used as bf16 with gamma folded into W_d and W_w (see gr_pack_params); the combine uses
 *     gamma in fp32. The read after a fused write uses the stored (rounded) state.
 *   - Every call validates its arguments on the host first. On any validation error it returns
 *     a negative status, launches nothing and touches no output. A status of GR_E_CUDA means a
 *     launch or copy failed; the CUDA error is not cleared from the runtime.
 *   - n_tokens == 0 is valid and does nothing; the tensor pointers may then be NULL.
 */
#ifndef GR_GB300_H
#define GR_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GR_API_VERSION 1
#define GR_MAX_D 12288   /* largest d_model (one token's fp32 state row must fit on chip) */
#define GR_MAX_RANK 64      /* largest rank of every path but the large-rank one            */
#define GR_MAX_RANK_TC 448  /* largest rank of the large-rank tensor-core path (bf16 states,
                               d_model a multiple of 64, rank a multiple of 8, rank >= 64)    */

/* Status codes. */
enum {
    GR_OK = 0,
    GR_E_NULL = -1,        /* a required pointer is NULL                                        */
    GR_E_SHAPE = -2,       /* n_tokens < 0, d_model not a multiple of 8 in [8, GR_MAX_D],      */
                           /* or n_branch != 4                                                 */
    GR_E_DTYPE = -3,       /* unknown state dtype                                               */
    GR_E_ALIGN = -4,       /* a device pointer is not 16-byte aligned                           */
    GR_E_RANK = -5,        /* rank outside [1, 64], and outside the large-rank path's shapes    */
    GR_E_PARAMS = -6,      /* params not packed by gr_pack_params, or packed for another shape  */
    GR_E_SIZE = -7,        /* a caller-provided buffer is smaller than the call needs           */
    GR_E_ALIAS = -8,       /* an output overlaps an input in a way the call forbids             */
    GR_E_CUDA = -9,        /* a CUDA launch or copy failed                                      */
    GR_E_DEVICE = -10,     /* no usable CUDA device (this build runs on sm_103a only)           */
    GR_E_EPS = -11,        /* eps negative or not finite                                        */
    GR_E_TIMEOUT = -12,    /* a kernel's bounded device-side wait ran out (see gr_device_status) */
    GR_E_NOMEM = -13       /* the device could not commit the fixed workspace of
                              gr_write_then_read_host_static (its memory is taken)               */
};

/* Storage dtype of R, y and x. GR_FP8 is the FP8 branch state (see the FP8 section below): R is
 * e4m3 codes plus block exponents, y and x are bf16. */
typedef enum { GR_F32 = 0, GR_BF16 = 1, GR_FP8 = 2 } gr_dtype;

/* Problem shape. n_branch must be 4; d_model a multiple of 8 in [8, GR_MAX_D]; 1 <= rank <= 64. */
typedef struct gr_shape {
    int64_t n_tokens;    /* N: flattened tokens ([B,S,D] or [B,1,D] -> N rows) */
    int32_t d_model;     /* D: block width */
    int32_t n_branch;    /* n_r: must be 4 */
    int32_t rank;        /* r: gate bottleneck rank */
    int32_t state_dtype; /* gr_dtype of R, y, x */
    float eps;           /* RMSNorm epsilon (the pages give none; 1e-6 is the usual value) */
} gr_shape;

/* Packed parameters of one sublayer's GR module. Filled by gr_pack_params; the caller owns the
 * device buffer `packed` and keeps it alive while calls that use these params are in flight. */
typedef struct gr_params {
    const void* packed;  /* device buffer written by gr_pack_params */
    int32_t d_model, n_branch, rank, state_dtype;
    uint64_t tag;        /* GR_PARAMS_TAG once packed */
} gr_params;

#define GR_PARAMS_TAG 0x47523330304B5031ull

/* Version of this ABI (GR_API_VERSION). */
int gr_api_version(void);

/* Human-readable text for a status code (static storage; never NULL). */
const char* gr_status_string(int status);

/* Name of the kernel path a read or fused step takes for `shape` (static string, never NULL):
 * "fused_bf16" (cluster tensor-core kernel: bf16, D in {256, 512, 1024, 2048, 4096}, r <= 16),
 * "fused_bf16+tiled_bf16" (the same shapes when n_tokens is large enough that a share of the
 * tokens also runs on the two-pass kernel, concurrently, on the SMs the clusters leave idle;
 * this form needs the device, so without one the plain "fused_bf16" is reported),
 * "tiled_bf16" (two-pass tensor-core kernel: the other bf16 shapes with D % 64 == 0, r <= 32),
 * "tc_bf16" (the large-rank path on the tcgen05 tensor cores: bf16, D % 64 == 0,
 * 64 <= r <= GR_MAX_RANK_TC, r % 8 == 0), "tiled_fp8" (the two-pass kernel on an FP8 state),
 * "generic" (one CTA per token), or "invalid". Host only. */
const char* gr_kernel_path(const gr_shape* shape);

/* Bytes of device memory gr_pack_params needs for `shape` (host only; no CUDA call).
 * Returns GR_OK and sets *bytes, or a validation status. shape->n_tokens is ignored. */
int gr_packed_size(const gr_shape* shape, size_t* bytes);

/* Lay the fp32 parameters of one GR module out for the kernels (Digest §二.4 shapes:
 * gamma [4][D], W_d [r][4D], W_u [4D][r], W_w [4][4D]; all DEVICE pointers, fp32, 16-byte
 * aligned). `packed` is a DEVICE buffer of at least gr_packed_size() bytes, 256-byte aligned.
 * On the bf16 path the packed weights are bf16 (nearest even) with gamma folded into W_d and
 * W_w (W[k][i*D+c]·gamma[i][c] in fp32, then rounded); gamma is also kept in fp32 for the combine. On
 * the fp32 path the weights stay fp32 and nothing is folded. Runs on `stream`; the inputs may
 * be freed once the stream has passed the call. Fills *out on success. */
int gr_pack_params(const gr_shape* shape, const float* gamma, const float* w_down,
                   const float* w_up, const float* w_write, void* packed, size_t packed_bytes,
                   gr_params* out, void* stream);

/* The read (eq rms, eq gate, eq use_gate, eq s) of a chain's first sublayer:
 * R [N][4][D] -> x [N][D] and s [N][4]. R is only read. x and s must not overlap R. */
int gr_read(const gr_shape* shape, const void* R, const gr_params* params, void* x, float* s,
            void* stream);

/* ---- the pages' own rank, r = d/8 (large-rank path) ------------------------------------------
 * "【论文解读】 Qwen3.8 Flash Next", §二.4 sets W_d ∈ R^{r × n_r·d} with r = d/8 (320 at d = 2560).
 * bf16 states with d_model a multiple of 64 and a rank r with 64 <= r <= GR_MAX_RANK_TC,
 * r % 8 == 0 (and at most 2^31 - 2^16 tokens a call), run on the tcgen05 tensor cores
 * ("tc_bf16" in gr_kernel_path): three launches
 * (the write with each branch's projection [W_d; W_w]·γ_i of its unscaled stored rows, as a GEMM
 * a (128-token tile, branch); the per-token gates, which apply each branch's 1/rms to those
 * projections; the up projection as a GEMM with the gate and combine in its epilogue). Its
 * numerics: the down projection's inputs are the stored bf16 rows and the packed bf16 weights,
 * the 1/rms factors are applied afterwards in fp32, h is rounded to bf16 for the up projection,
 * W_u is bf16; fp32 accumulation throughout. It needs a device workspace between its launches,
 * so these shapes take the _ws entries below; gr_read and gr_write_then_read return GR_E_SIZE
 * for them and the host-buffer entries GR_E_RANK. */

/* Bytes of device workspace a read or fused step of this shape needs on the large-rank path, each
 * part rounded up to 256: N·16 (each row's 1/rms), N·round_up(r, 64)·2 (h in bf16),
 * N·16·round_up(r + 4, 4) (the four branches' r + 4 projections in fp32) and N·16 (each row's
 * sum of squares); 0 for every other shape. */
int gr_step_workspace_size(const gr_shape* shape, size_t* bytes);

/* gr_read and gr_write_then_read with a caller-owned DEVICE workspace (256-byte aligned, at
 * least gr_step_workspace_size bytes, not overlapping the call's other buffers; may be NULL
 * with 0 bytes when the size is 0). Same contracts otherwise; every shape the library takes. */
int gr_read_ws(const gr_shape* shape, const void* R, const gr_params* params, void* x, float* s,
               void* workspace, size_t workspace_bytes, void* stream);
int gr_write_then_read_ws(const gr_shape* shape, void* R, const void* y, const float* s_prev,
                          const gr_params* next, void* x, float* s_next, void* workspace,
                          size_t workspace_bytes, void* stream);

/* The write (eq write) of a chain's last sublayer: R[t][i][:] += s[t][i] · y[t][:], in place. */
int gr_write(const gr_shape* shape, void* R, const void* y, const float* s, void* stream);

/* One sublayer's write fused with the next sublayer's read, in one traversal of the state:
 *   R[t][i][:] = R[t][i][:] + s_prev[t][i] · y[t][:]            (eq write, in place)
 *   x, s_next  = read of the written (stored) R with `next`       (eq rms … eq s)
 * y and x may be the same buffer (F's input/output buffer), and s_prev and s_next may be the
 * same buffer: each token's y and s_prev are read before its x and s_next are written. Apart
 * from those two exact matches, x and s_next must not overlap R, y, s_prev or each other.
 * On the "fused_bf16+tiled_bf16" path (here and in gr_read) the trailing share of the tokens
 * runs on an internal per-device stream that first waits for the work already queued on
 * `stream`, and `stream` then waits for it, so the call stays ordered on `stream`; that stream
 * and two events are created on the first such call (CUDA graph capture of the call captures
 * the fork and the join). */
int gr_write_then_read(const gr_shape* shape, void* R, const void* y, const float* s_prev,
                       const gr_params* next, void* x, float* s_next, void* stream);

/* The combine of eq use_gate with caller-given gates: x = (1/4) Σ_i G_i ⊙ RMSNorm(R_i; γ_i),
 * G [4][D] fp32 broadcast over tokens, gamma [4][D] fp32. No gate prediction, no s. Used to
 * check reductions that need gates σ cannot produce (one-hot reads: GR as Pre-Norm,
 * Digest §二.2 and §二.4). */
int gr_read_fixed_gates(const gr_shape* shape, const void* R, const float* gamma,
                        const float* G, void* x, void* stream);

/* Single-stream residual add x[e] += y[e], e < n, in `dtype` (the plain residual
 * x_{l+1} = x_l + F(x_l) of "Residual" §1): the bandwidth reference for the GR kernels.
 * n >= 0; pointers 16-byte aligned. */
int gr_residual_add_ref(int64_t n, int32_t dtype, const void* y, void* x, void* stream);

/* Device-side status of the kernels that use bounded waits (every wait of the fused kernel on
 * its mbarriers gives up after a time limit instead of spinning forever). Synchronises the current
 * device, then returns GR_OK, GR_E_TIMEOUT if a wait ran out since the last clear (the outputs of
 * that call are not valid), or GR_E_CUDA. `clear` != 0 resets the status. */
int gr_device_status(int clear);

/* Self-test of the failure-detection path (the pages have no counterpart): launches one thread
 * that waits, with the fused kernel's bounded-wait helper, on an mbarrier that nothing arrives
 * at. After limit_cycles (1 .. 4e9 SM clock cycles; else GR_E_SIZE, nothing launched) the wait
 * gives up, sets the device status word and the kernel returns, so gr_device_status() reports
 * GR_E_TIMEOUT until cleared. No fault, trap or hang is involved. Asynchronous on `stream`. */
int gr_selftest_bounded_wait(int64_t limit_cycles, void* stream);

/* Bytes of device workspace gr_write_then_read_host needs for `shape`. */
int gr_host_workspace_size(const gr_shape* shape, size_t* bytes);

/* gr_write_then_read on HOST buffers (pinned memory gives asynchronous copies): copies R, y and
 * s_prev into `workspace` (DEVICE, >= gr_host_workspace_size bytes, 256-byte aligned), runs the
 * fused step there, copies R', x and s_next back into R_host, x_host and s_next_host, and
 * synchronises `stream` before returning. Host buffers must not overlap.
 * The work is split into up to 16 token chunks (at least 1024 tokens each): each chunk's
 * host-to-device copies run on an internal stream, its step on `stream`, its device-to-host
 * copies on a second internal stream (both created once per device), ordered by events, so
 * copies in both directions overlap the steps. The copies into the workspace start after the
 * work already queued on `stream`. Calls for the same device are serialised (they share the
 * internal streams). */
int gr_write_then_read_host(const gr_shape* shape, void* R_host, const void* y_host,
                            const float* s_prev_host, const gr_params* next, void* x_host,
                            float* s_next_host, void* workspace, size_t workspace_bytes,
                            void* stream);

/* Size of the fixed device workspace of gr_write_then_read_host_static (32 MiB). */
#define GR_STATIC_WORKSPACE_BYTES (32u << 20)

/* gr_write_then_read_host without a caller-provided workspace: the same step on HOST buffers,
 * staged through a fixed device workspace of GR_STATIC_WORKSPACE_BYTES that the library holds
 * in a file-scope device array. The pages have no counterpart. It serves callers that cannot
 * allocate device memory themselves:
 *   - a plain host program with no device allocator of its own (only host arrays to pass);
 *   - a process whose device memory is already reserved by another allocator (a framework's
 *     caching allocator, a serving engine's preallocated pool), where an extra cudaMalloc can
 *     fail or fragment the pool;
 *   - a latency-bound loop (decode), where cudaFree would synchronise the whole device.
 * It calls no cudaMalloc or cudaFree and creates no stream or event. Its device memory is a
 * fixed-size array, held by every device that loads it until the process exits. When the device
 * commits that memory depends on CUDA's module loading: with lazy loading (the default) at the
 * first call of this entry on the device, with CUDA_MODULE_LOADING=EAGER when the library's
 * module loads with the context. A process whose allocator takes the device's memory first
 * should therefore make one call (or set EAGER) before its pool grows.
 *   - Returns GR_E_SIZE, without touching anything, when gr_host_workspace_size(shape) exceeds
 *     GR_STATIC_WORKSPACE_BYTES (for example N > 682 tokens at D = 4096, bf16).
 *   - The first call on a device looks the workspace's device address up once
 *     (cudaGetSymbolAddress); make that first call outside any stream capture. If the device
 *     cannot commit the memory there, the call returns GR_E_NOMEM (GR_E_CUDA for any other
 *     failure), clears the CUDA runtime's error, touches nothing, and the next call tries again.
 *   - Shapes that the device entries split between the cluster kernel and the two-pass kernel
 *     (gr_kernel_path "fused_bf16+tiled_bf16") run on the cluster kernel alone here (on a GB300
 *     no shape that fits the workspace is split anyway). Their R' is bit-identical to
 *     gr_write_then_read_host's; x and s agree within the bf16 tolerance.
 *   - Nothing in the workspace has to start at zero (each call writes all it reads).
 *   - All calls on a device share the one workspace: calls that overlap in time (on different
 *     streams or host threads) race on it. Run them one after another.
 *   - Runs on `stream` (copies in, step, copies out) and synchronises it before returning. */
int gr_write_then_read_host_static(const gr_shape* shape, void* R_host, const void* y_host,
                                   const float* s_prev_host, const gr_params* next, void* x_host,
                                   float* s_next_host, void* stream);

/* ---- backward (training) ------------------------------------------------------------------------
 * The gradients of the read and the write by the chain rule through eq rms, eq gate, eq use_gate,
 * eq s and eq write ("【论文解读】 Qwen3.8 Flash Next", §二.4), in fp32 on CUDA cores. States (R,
 * y) in shape->state_dtype (GR_BF16 or GR_F32), parameters and every gradient fp32, all DEVICE
 * pointers, 16-byte aligned. Ranks 1 … GR_MAX_RANK (GR_E_RANK above). */

/* Bytes of device workspace gr_read_backward needs: 3·N·4·D·4 bytes of per-token factors of
 * the parameter gradients, N·(2r+5)·4 more, and r·4·D·4 for W_u transposed, each part rounded
 * up to 256 bytes. */
int gr_read_backward_workspace_size(const gr_shape* shape, size_t* bytes);

/* Backward of the read of R [N][4][D] with the fp32 parameters gamma [4][D], W_d [r][4D],
 * W_u [4D][r], W_w [4][4D] (unpacked), given dL/dx [N][D] and dL/ds [N][4]:
 *   dR [N][4][D]   dL/dR (overwritten)
 *   dgamma, dw_down, dw_up, dw_write   the parameter gradients summed over the N tokens, in the
 *                                      parameters' shapes (overwritten)
 * `workspace` (>= gr_read_backward_workspace_size bytes, 256-byte aligned) holds per-token
 * factors between the two kernels. Outputs must not overlap the inputs, the workspace or each
 * other. Asynchronous on `stream`; the parameter gradients are reduced with fp32 atomics, so their
 * last bits may differ from run to run. */
int gr_read_backward(const gr_shape* shape, const void* R, const float* gamma,
                     const float* w_down, const float* w_up, const float* w_write,
                     const float* dx, const float* ds, float* dR, float* dgamma, float* dw_down,
                     float* dw_up, float* dw_write, void* workspace, size_t workspace_bytes,
                     void* stream);

/* Backward of the write R' = R + s_i·y given dL/dR' [N][4][D]: dR = dL/dR' (dR may be the same
 * buffer as dR_next), dy [N][D] = Σ_i s_i dL/dR'_i, ds [N][4] with ds_i = Σ_c dL/dR'_i[c] y[c].
 * y in the state dtype; s and every gradient fp32. */
int gr_write_backward(const gr_shape* shape, const float* dR_next, const void* y, const float* s,
                      float* dR, float* dy, float* ds, void* stream);

/* ---- contribution decomposition (analysis) ----------------------------------------------------
 * "【论文解读】 Qwen3.8 Flash Next", §二.6 (eq auv and the fractions π): GR never mixes branches,
 * so the input of block v splits exactly into the initial state's share and one term per earlier
 * writer u, a_{u→v} = ¼ Σ_i G_i^(v) ⊙ γ_i ⊙ s_i^(u) y^(u) / rms(R_i^(v)). For one reader v:
 *   R        [N][4][D]  the state block v reads (R^(v)), in shape->state_dtype (GR_BF16/GR_F32)
 *   gamma, w_down, w_up, w_write   block v's parameters, fp32, unpacked (as gr_read_backward);
 *                      w_write is accepted for symmetry and not read (s plays no part here)
 *   n_writers U >= 0, y [U][N][D] the writers' outputs (state dtype), s [U][N][4] fp32 their
 *                      write strengths
 *   R0       [N][4][D]  the initial state (state dtype), or NULL
 * Outputs (fp32, overwritten; the gates are recomputed in fp32 from R):
 *   norm        [N][U]     ‖a_{u→v}‖₂ over the token's D channels (required when U > 0)
 *   branch_norm [N][U][4]  ‖a_{u→v,i}‖₂, branch i's share (or NULL)
 *   pi          [N][U]     π_uv = ‖a_{u→v}‖ / Σ_u' ‖a_{u'→v}‖, per token; 0 where that sum is 0
 *                          (or NULL)
 *   a0_norm     [N]        ‖a_{0→v}‖₂, a_{0→v} = ¼ Σ_i G_i ⊙ γ_i ⊙ R0_i / rms(R_i) (required
 *                          with R0, ignored without)
 * All DEVICE pointers, 16-byte aligned; outputs must not overlap the inputs or each other.
 * 0 <= U <= GR_MAX_WRITERS; ranks 1 … GR_MAX_RANK (GR_E_RANK above). Asynchronous on
 * `stream`. Errors: as the other calls. */
#define GR_MAX_WRITERS 65536
int gr_decompose(const gr_shape* shape, const void* R, const float* gamma, const float* w_down,
                 const float* w_up, const float* w_write, int32_t n_writers, const void* y,
                 const float* s, const void* R0, float* norm, float* branch_norm, float* pi,
                 float* a0_norm, void* stream);

/* ---- FP8 branch state ------------------------------------------------------------------------
 * "【论文解读】 Qwen3.8 Flash Next", §二.7 stores the widened state in FP8 and fixes no format.
 * This library's FP8 state is two DEVICE arrays:
 *   codes  [N][4][D]     uint8, OCP FP8 E4M3 ("e4m3fn": bias 7, 3 fraction bits, largest
 *                        finite 448, no infinities; 0x7F/0xFF are NaN)
 *   scales [N][4][D/32]  uint8 biased exponents b: channels 32k..32k+31 of row (t, i) have the
 *                        scale 2^(b - 127)
 * Element (t, i, c) is decode(codes[t][i][c]) · 2^(scales[t][i][c/32] - 127). A block of 32 values
 * v is encoded with the smallest e such that max|v| <= 448·2^e (e clamped to [-127, 127]; an
 * all-zero block gets e = -127) and codes v/2^e rounded to the nearest e4m3 value, ties to even.
 * The FP8 write decodes R, forms R + s·y as one fp32 fused multiply-add and encodes the result;
 * the read uses the decoded stored values. y and x are bf16, s fp32; params are packed with
 * state_dtype GR_FP8 (bf16 weights, as on the bf16 path).
 * Shapes: state_dtype GR_FP8, d_model a multiple of 128 in [128, 8192], rank 1..32 for the read
 * calls (encode, decode and write take any multiple of 32 up to GR_MAX_D). codes, scales, y, x
 * and s must be 16-byte aligned. Inputs with NaN or infinite values have no FP8 encoding; their
 * blocks come out undefined. */

/* Encode a state R [N][4][D] given in `in_dtype` (GR_BF16 or GR_F32) into codes and scales. */
int gr_fp8_encode(const gr_shape* shape, const void* R, int32_t in_dtype, uint8_t* codes,
                  uint8_t* scales, void* stream);

/* Decode codes and scales into R [N][4][D] in `out_dtype` (GR_BF16: rounded to nearest even;
 * GR_F32: exact). */
int gr_fp8_decode(const gr_shape* shape, const uint8_t* codes, const uint8_t* scales, void* R,
                  int32_t out_dtype, void* stream);

/* gr_read on an FP8 state: x [N][D] bf16 and s [N][4] fp32. codes and scales are only read. */
int gr_read_fp8(const gr_shape* shape, const uint8_t* codes, const uint8_t* scales,
                const gr_params* params, void* x, float* s, void* stream);

/* gr_write on an FP8 state, in place: R[t][i][:] += s[t][i] · y[t][:] (y bf16), re-encoded. */
int gr_write_fp8(const gr_shape* shape, uint8_t* codes, uint8_t* scales, const void* y,
                 const float* s, void* stream);

/* gr_write_then_read on an FP8 state: the write in place (codes and scales), then the read of
 * the stored state with `next` into x (bf16) and s_next. The aliasing rules are those of
 * gr_write_then_read, with codes and scales in the place of R. */
int gr_write_then_read_fp8(const gr_shape* shape, uint8_t* codes, uint8_t* scales,
                           const void* y, const float* s_prev, const gr_params* next, void* x,
                           float* s_next, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GR_GB300_H */
