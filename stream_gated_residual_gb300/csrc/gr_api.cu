// C ABI of the GR library: host-side validation, dispatch to the kernels, status codes.
// Declarations and the contract of every entry point are in include/gr.h.
#include <math.h>
#include <string.h>

#include <mutex>

#include "gr_internal.h"

namespace gr {

namespace {

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];        // 0 = not queried yet
int g_device_ok[kMaxDevices];       // 0 = unknown, 1 = sm_103, -1 = unusable

int current_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return -1;
    return (d >= 0 && d < kMaxDevices) ? d : -1;
}

// The build targets sm_103a only; refuse other devices before launching anything.
int check_device() {
    const int d = current_device();
    if (d < 0) return GR_E_DEVICE;
    if (g_device_ok[d] == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) {
            return GR_E_DEVICE;
        }
        g_sm_count[d] = sms;
        g_device_ok[d] = (major == 10 && minor == 3) ? 1 : -1;
    }
    return g_device_ok[d] == 1 ? GR_OK : GR_E_DEVICE;
}

// Per-device objects of the pipelined host entry: a stream for the host-to-device copies, one
// for the device-to-host copies and two events per chunk, created on first use; the mutex
// serialises the calls that share them.
constexpr int kHostChunks = 16;
struct HostPipe {
    std::mutex mu;
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t loaded[kHostChunks] = {}, computed[kHostChunks] = {};
    cudaEvent_t start = nullptr, copied = nullptr;
};
HostPipe g_host_pipe[kMaxDevices];

bool host_pipe_init(HostPipe& hp) {
    if (hp.ready) return true;
    if (cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) != cudaSuccess)
        return false;
    for (int i = 0; i < kHostChunks; ++i)
        if (cudaEventCreateWithFlags(&hp.loaded[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp.computed[i], cudaEventDisableTiming) != cudaSuccess)
            return false;
    if (cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.copied, cudaEventDisableTiming) != cudaSuccess)
        return false;
    hp.ready = true;
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return na && nb && a0 < b0 + nb && b0 < a0 + na;
}

// Shape checks of the bf16/fp32 calls; fp8_ok also admits GR_FP8 (the calls that only pack or
// describe parameters), whose width must be a multiple of 32.
int validate_shape(const gr_shape* s, bool fp8_ok = false) {
    if (!s) return GR_E_NULL;
    if (s->n_tokens < 0 || s->n_branch != kBranches || s->d_model < 8 || s->d_model % 8 != 0 ||
        s->d_model > GR_MAX_D)
        return GR_E_SHAPE;
    if (s->state_dtype == GR_FP8 && fp8_ok) {
        if (s->d_model % 32 != 0) return GR_E_SHAPE;
    } else if (s->state_dtype != GR_F32 && s->state_dtype != GR_BF16) {
        return GR_E_DTYPE;
    }
    // ranks above GR_MAX_RANK only on the large-rank tensor-core path (bf16 states)
    if (s->rank < 1 || s->rank > GR_MAX_RANK_TC) return GR_E_RANK;
    if (s->rank > GR_MAX_RANK &&
        !(s->state_dtype == GR_BF16 && rank_tc_supported(s->d_model, s->rank)))
        return GR_E_RANK;
    if (!(s->eps >= 0.0f) || !isfinite(s->eps)) return GR_E_EPS;
    return GR_OK;
}

int validate_params(const gr_shape* s, const gr_params* p) {
    if (!p) return GR_E_NULL;
    if (p->tag != GR_PARAMS_TAG || !p->packed) return GR_E_PARAMS;
    if (p->d_model != s->d_model || p->n_branch != s->n_branch || p->rank != s->rank ||
        p->state_dtype != s->state_dtype)
        return GR_E_PARAMS;
    return GR_OK;
}

// Shape checks of the FP8-state calls: state_dtype GR_FP8, D a multiple of 32; the calls that
// read through the two-pass kernel (tensor_core) also need D % 128 == 0, D <= 8192, r <= 32.
int validate_fp8(const gr_shape* s, bool tensor_core) {
    if (!s) return GR_E_NULL;
    if (s->state_dtype != GR_FP8) return GR_E_DTYPE;
    int st = validate_shape(s, true);
    if (st) return st;
    if (tensor_core) {
        if (!tiled_fp8_supported(s->d_model, 1)) return GR_E_SHAPE;
        if (!tiled_fp8_supported(s->d_model, s->rank)) return GR_E_RANK;
        if (s->n_tokens > tiled_max_tokens()) return GR_E_SHAPE;
    }
    return GR_OK;
}

size_t elem_size(int dtype) { return dtype == GR_BF16 ? 2 : 4; }

int status_of(cudaError_t e) { return e == cudaSuccess ? GR_OK : GR_E_CUDA; }

// Which kernel runs a read (or fused step) for this shape.
bool use_fused(const gr_shape* s) {
    return s->state_dtype == GR_BF16 && fused_supported(s->d_model, s->rank) &&
           s->n_tokens <= fused_max_tokens();
}

// The large-rank tensor-core path (gr_rank_tc.cu) takes precedence over the generic kernel. Its
// TMA coordinates are 32-bit: tokens up to kRankTcMaxTokens.
constexpr int64_t kRankTcMaxTokens = 0x7fff0000;
bool use_rank_tc(const gr_shape* s) {
    return s->state_dtype == GR_BF16 && rank_tc_supported(s->d_model, s->rank);
}

bool use_tiled(const gr_shape* s) {
    return s->state_dtype == GR_BF16 && !fused_supported(s->d_model, s->rank) &&
           tiled_supported(s->d_model, s->rank) && s->n_tokens <= tiled_max_tokens();
}

// allow_split = false keeps a cluster-kernel step on the cluster kernel alone (the host entries'
// chunks, which are below the split's token threshold anyway).
int run_step(const gr_shape* s, void* R, const void* y, const float* s_prev,
             const gr_params* p, void* x, float* s_out, cudaStream_t st,
             void* ws = nullptr, size_t ws_bytes = 0, bool allow_split = true) {
    if (s->n_tokens == 0) return GR_OK;
    cudaError_t e;
    if (use_rank_tc(s)) {
        if (s->n_tokens > kRankTcMaxTokens) return GR_E_SHAPE;   // 32-bit TMA token coordinate
        if (!ws || ws_bytes < rank_tc_workspace(s->n_tokens, s->rank)) return GR_E_SIZE;
        return status_of(launch_rank_tc(s->n_tokens, s->d_model, s->rank, s->eps, R, y, s_prev,
                                         p->packed, x, s_out, ws, st));
    }
    int free_sms = 0;
    const int64_t n2 =
        use_fused(s) && allow_split
            ? split_tokens(s->n_tokens, s->d_model, s->rank, y != nullptr, &free_sms)
            : 0;
    if (n2 > 0)
        return status_of(launch_split_bf16(s->n_tokens, n2, free_sms, s->d_model, s->rank,
                                           s->eps, R, y, s_prev, p->packed, x, s_out, st));
    if (use_fused(s))
        e = launch_fused_bf16(s->n_tokens, s->d_model, s->rank, s->eps, R, y, s_prev, p->packed,
                              x, s_out, st);
    else if (use_tiled(s))
        e = launch_tiled_bf16(s->n_tokens, s->d_model, s->rank, s->eps, R, y, s_prev, p->packed,
                              x, s_out, st);
    else
        e = launch_generic(s->n_tokens, s->d_model, s->rank, s->state_dtype, s->eps, R, y,
                           s_prev, p->packed, x, s_out, st);
    return status_of(e);
}

}  // namespace

int sm_count() {
    const int d = current_device();
    if (d < 0) return 1;
    if (g_sm_count[d] == 0) {
        int sms = 1;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d);
        g_sm_count[d] = sms > 0 ? sms : 1;
    }
    return g_sm_count[d];
}

}  // namespace gr

namespace gr {
namespace {

// The workspace of a step (large-rank path only): 256-byte aligned, big enough, and clear of the
// step's other buffers.
int check_step_ws(const gr_shape* s, const void* ws, size_t ws_bytes, const void* const* bufs,
                  const size_t* sizes, int nbufs) {
    if (!use_rank_tc(s)) return GR_OK;
    const size_t need = rank_tc_workspace(s->n_tokens, s->rank);
    if (!ws || ws_bytes < need) return GR_E_SIZE;
    if (!aligned256(ws)) return GR_E_ALIGN;
    for (int b = 0; b < nbufs; ++b)
        if (overlaps(ws, need, bufs[b], sizes[b])) return GR_E_ALIAS;
    return GR_OK;
}

int read_impl(const gr_shape* shape, const void* R, const gr_params* params, void* x, float* s,
              void* ws, size_t ws_bytes, void* stream) {
    int st = validate_shape(shape);
    if (st) return st;
    if ((st = validate_params(shape, params))) return st;
    if (shape->n_tokens == 0) return GR_OK;
    if (!R || !x || !s) return GR_E_NULL;
    if (!aligned16(R) || !aligned16(x) || !aligned16(s)) return GR_E_ALIGN;
    const size_t es = elem_size(shape->state_dtype);
    const size_t N = size_t(shape->n_tokens), D = size_t(shape->d_model);
    const size_t nR = N * kBranches * D * es, nx = N * D * es, ns = N * kBranches * 4;
    if (overlaps(x, nx, R, nR) || overlaps(s, ns, R, nR) || overlaps(x, nx, s, ns))
        return GR_E_ALIAS;
    const void* bufs[3] = {R, x, s};
    const size_t sizes[3] = {nR, nx, ns};
    if ((st = check_step_ws(shape, ws, ws_bytes, bufs, sizes, 3))) return st;
    if ((st = check_device())) return st;
    return run_step(shape, const_cast<void*>(R), nullptr, nullptr, params, x, s,
                    static_cast<cudaStream_t>(stream), ws, ws_bytes);
}

int write_then_read_impl(const gr_shape* shape, void* R, const void* y, const float* s_prev,
                         const gr_params* next, void* x, float* s_next, void* ws,
                         size_t ws_bytes, void* stream) {
    int st = validate_shape(shape);
    if (st) return st;
    if ((st = validate_params(shape, next))) return st;
    if (shape->n_tokens == 0) return GR_OK;
    if (!R || !y || !s_prev || !x || !s_next) return GR_E_NULL;
    if (!aligned16(R) || !aligned16(y) || !aligned16(s_prev) || !aligned16(x) ||
        !aligned16(s_next))
        return GR_E_ALIGN;
    const size_t es = elem_size(shape->state_dtype);
    const size_t N = size_t(shape->n_tokens), D = size_t(shape->d_model);
    const size_t nR = N * kBranches * D * es, ny = N * D * es, ns = N * kBranches * 4;
    if (overlaps(R, nR, y, ny) || overlaps(R, nR, s_prev, ns) || overlaps(x, ny, R, nR) ||
        overlaps(s_next, ns, R, nR) || overlaps(x, ny, s_next, ns) ||
        overlaps(x, ny, s_prev, ns) || overlaps(s_next, ns, y, ny) ||
        (x != y && overlaps(x, ny, y, ny)) || (s_next != s_prev && overlaps(s_next, ns, s_prev, ns)))
        return GR_E_ALIAS;
    const void* bufs[5] = {R, y, s_prev, x, s_next};
    const size_t sizes[5] = {nR, ny, ns, ny, ns};
    if ((st = check_step_ws(shape, ws, ws_bytes, bufs, sizes, 5))) return st;
    if ((st = check_device())) return st;
    return run_step(shape, R, y, s_prev, next, x, s_next, static_cast<cudaStream_t>(stream), ws,
                    ws_bytes);
}

}  // namespace
}  // namespace gr

using namespace gr;

extern "C" {

int gr_api_version(void) { return GR_API_VERSION; }

const char* gr_status_string(int status) {
    switch (status) {
        case GR_OK: return "ok";
        case GR_E_NULL: return "a required pointer is NULL";
        case GR_E_SHAPE: return "bad shape (n_tokens < 0, d_model not a multiple of 8 in [8, 12288], or n_branch != 4)";
        case GR_E_DTYPE: return "unknown state dtype";
        case GR_E_ALIGN: return "a pointer is not aligned as the call requires";
        case GR_E_RANK: return "rank outside [1, 64]";
        case GR_E_PARAMS: return "params not packed by gr_pack_params or packed for another shape";
        case GR_E_SIZE: return "a caller-provided buffer is too small";
        case GR_E_ALIAS: return "an output overlaps an input";
        case GR_E_CUDA: return "a CUDA launch or copy failed";
        case GR_E_DEVICE: return "no usable sm_103 CUDA device";
        case GR_E_EPS: return "eps negative or not finite";
        case GR_E_TIMEOUT: return "a bounded device-side wait ran out";
        case GR_E_NOMEM: return "the device could not commit the library's fixed workspace";
        default: return "unknown status";
    }
}

const char* gr_kernel_path(const gr_shape* shape) {
    if (shape && shape->state_dtype == GR_FP8)
        return validate_fp8(shape, true) == GR_OK ? "tiled_fp8" : "invalid";
    if (validate_shape(shape) != GR_OK) return "invalid";
    if (use_rank_tc(shape)) return "tc_bf16";
    if (use_fused(shape))
        return split_tokens(shape->n_tokens, shape->d_model, shape->rank, true, nullptr) > 0
                   ? "fused_bf16+tiled_bf16"
                   : "fused_bf16";
    return use_tiled(shape) ? "tiled_bf16" : "generic";
}

int gr_packed_size(const gr_shape* shape, size_t* bytes) {
    int st = validate_shape(shape, true);
    if (st) return st;
    if (!bytes) return GR_E_NULL;
    *bytes = make_layout(shape->d_model, shape->rank, shape->state_dtype).total;
    return GR_OK;
}

int gr_pack_params(const gr_shape* shape, const float* gamma, const float* w_down,
                   const float* w_up, const float* w_write, void* packed, size_t packed_bytes,
                   gr_params* out, void* stream) {
    int st = validate_shape(shape, true);
    if (st) return st;
    if (!gamma || !w_down || !w_up || !w_write || !packed || !out) return GR_E_NULL;
    if (!aligned16(gamma) || !aligned16(w_down) || !aligned16(w_up) || !aligned16(w_write) ||
        !aligned256(packed))
        return GR_E_ALIGN;
    const Layout L = make_layout(shape->d_model, shape->rank, shape->state_dtype);
    if (packed_bytes < L.total) return GR_E_SIZE;
    const size_t K = size_t(kBranches) * shape->d_model;
    const size_t r = size_t(shape->rank);
    if (overlaps(packed, L.total, gamma, K * 4) || overlaps(packed, L.total, w_down, r * K * 4) ||
        overlaps(packed, L.total, w_up, r * K * 4) ||
        overlaps(packed, L.total, w_write, kBranches * K * 4))
        return GR_E_ALIAS;
    if ((st = check_device())) return st;
    cudaError_t e = launch_pack(shape->d_model, shape->rank, shape->state_dtype, gamma, w_down,
                                w_up, w_write, packed, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return GR_E_CUDA;
    out->packed = packed;
    out->d_model = shape->d_model;
    out->n_branch = shape->n_branch;
    out->rank = shape->rank;
    out->state_dtype = shape->state_dtype;
    out->tag = GR_PARAMS_TAG;
    return GR_OK;
}

int gr_step_workspace_size(const gr_shape* shape, size_t* bytes) {
    int st = validate_shape(shape);
    if (st) return st;
    if (!bytes) return GR_E_NULL;
    *bytes = use_rank_tc(shape) ? rank_tc_workspace(shape->n_tokens, shape->rank) : 0;
    return GR_OK;
}

int gr_read(const gr_shape* shape, const void* R, const gr_params* params, void* x, float* s,
            void* stream) {
    return read_impl(shape, R, params, x, s, nullptr, 0, stream);
}

int gr_read_ws(const gr_shape* shape, const void* R, const gr_params* params, void* x, float* s,
               void* workspace, size_t workspace_bytes, void* stream) {
    return read_impl(shape, R, params, x, s, workspace, workspace_bytes, stream);
}

int gr_write(const gr_shape* shape, void* R, const void* y, const float* s, void* stream) {
    int st = validate_shape(shape);
    if (st) return st;
    if (shape->n_tokens == 0) return GR_OK;
    if (!R || !y || !s) return GR_E_NULL;
    if (!aligned16(R) || !aligned16(y) || !aligned16(s)) return GR_E_ALIGN;
    const size_t es = elem_size(shape->state_dtype);
    const size_t N = size_t(shape->n_tokens), D = size_t(shape->d_model);
    const size_t nR = N * kBranches * D * es;
    if (overlaps(R, nR, y, N * D * es) || overlaps(R, nR, s, N * kBranches * 4))
        return GR_E_ALIAS;
    if ((st = check_device())) return st;
    return status_of(launch_write(shape->n_tokens, shape->d_model, shape->state_dtype, R, y, s,
                                  static_cast<cudaStream_t>(stream)));
}

int gr_write_then_read(const gr_shape* shape, void* R, const void* y, const float* s_prev,
                       const gr_params* next, void* x, float* s_next, void* stream) {
    return write_then_read_impl(shape, R, y, s_prev, next, x, s_next, nullptr, 0, stream);
}

int gr_write_then_read_ws(const gr_shape* shape, void* R, const void* y, const float* s_prev,
                          const gr_params* next, void* x, float* s_next, void* workspace,
                          size_t workspace_bytes, void* stream) {
    return write_then_read_impl(shape, R, y, s_prev, next, x, s_next, workspace, workspace_bytes,
                                stream);
}

int gr_read_fixed_gates(const gr_shape* shape, const void* R, const float* gamma,
                        const float* G, void* x, void* stream) {
    int st = validate_shape(shape);
    if (st) return st;
    if (shape->n_tokens == 0) return GR_OK;
    if (!R || !gamma || !G || !x) return GR_E_NULL;
    if (!aligned16(R) || !aligned16(x)) return GR_E_ALIGN;
    const size_t es = elem_size(shape->state_dtype);
    const size_t N = size_t(shape->n_tokens), D = size_t(shape->d_model);
    if (overlaps(x, N * D * es, R, N * kBranches * D * es)) return GR_E_ALIAS;
    if ((st = check_device())) return st;
    return status_of(launch_fixed_gates(shape->n_tokens, shape->d_model, shape->state_dtype,
                                        shape->eps, R, gamma, G, x,
                                        static_cast<cudaStream_t>(stream)));
}

int gr_residual_add_ref(int64_t n, int32_t dtype, const void* y, void* x, void* stream) {
    if (n < 0) return GR_E_SHAPE;
    if (dtype != GR_F32 && dtype != GR_BF16) return GR_E_DTYPE;
    if (n == 0) return GR_OK;
    if (!y || !x) return GR_E_NULL;
    if (!aligned16(y) || !aligned16(x)) return GR_E_ALIGN;
    if (overlaps(x, size_t(n) * elem_size(dtype), y, size_t(n) * elem_size(dtype)))
        return GR_E_ALIAS;
    int st = check_device();
    if (st) return st;
    return status_of(launch_residual_add(n, dtype, y, x, static_cast<cudaStream_t>(stream)));
}

// ---- backward ---------------------------------------------------------------------------------

int gr_read_backward_workspace_size(const gr_shape* shape, size_t* bytes) {
    int st = validate_shape(shape);
    if (st) return st;
    if (shape->rank > GR_MAX_RANK) return GR_E_RANK;
    if (!bytes) return GR_E_NULL;
    *bytes = read_backward_workspace(shape->n_tokens, shape->d_model, shape->rank);
    return GR_OK;
}

int gr_read_backward(const gr_shape* shape, const void* R, const float* gamma,
                     const float* w_down, const float* w_up, const float* w_write,
                     const float* dx, const float* ds, float* dR, float* dgamma, float* dw_down,
                     float* dw_up, float* dw_write, void* workspace, size_t workspace_bytes,
                     void* stream) {
    int st = validate_shape(shape);
    if (st) return st;
    if (shape->rank > GR_MAX_RANK) return GR_E_RANK;
    if (shape->n_tokens == 0) return GR_OK;
    const void* in[8] = {R, gamma, w_down, w_up, w_write, dx, ds, workspace};
    const void* out[5] = {dR, dgamma, dw_down, dw_up, dw_write};
    for (const void* p : in)
        if (!p) return GR_E_NULL;
    for (const void* p : out)
        if (!p) return GR_E_NULL;
    for (const void* p : in)
        if (!aligned16(p)) return GR_E_ALIGN;
    for (const void* p : out)
        if (!aligned16(p)) return GR_E_ALIGN;
    if (!aligned256(workspace)) return GR_E_ALIGN;
    const size_t N = size_t(shape->n_tokens), D = size_t(shape->d_model), r = size_t(shape->rank);
    const size_t K = kBranches * D;
    const size_t need = read_backward_workspace(shape->n_tokens, shape->d_model, shape->rank);
    if (workspace_bytes < need) return GR_E_SIZE;
    const size_t in_n[8] = {N * K * elem_size(shape->state_dtype), K * 4, r * K * 4, r * K * 4,
                            kBranches * K * 4, N * D * 4, N * kBranches * 4, need};
    const size_t out_n[5] = {N * K * 4, K * 4, r * K * 4, r * K * 4, kBranches * K * 4};
    for (int a = 0; a < 5; ++a) {
        for (int b = 0; b < 8; ++b)
            if (overlaps(out[a], out_n[a], in[b], in_n[b])) return GR_E_ALIAS;
        for (int b = a + 1; b < 5; ++b)
            if (overlaps(out[a], out_n[a], out[b], out_n[b])) return GR_E_ALIAS;
    }
    for (int b = 0; b < 7; ++b)
        if (overlaps(workspace, need, in[b], in_n[b])) return GR_E_ALIAS;
    if ((st = check_device())) return st;
    return status_of(launch_read_backward(shape->n_tokens, shape->d_model, shape->rank,
                                          shape->eps, shape->state_dtype, R, gamma, w_down, w_up,
                                          w_write, dx, ds, dR, dgamma, dw_down, dw_up, dw_write,
                                          workspace, static_cast<cudaStream_t>(stream)));
}

int gr_write_backward(const gr_shape* shape, const float* dR_next, const void* y, const float* s,
                      float* dR, float* dy, float* ds, void* stream) {
    int st = validate_shape(shape);
    if (st) return st;
    if (shape->n_tokens == 0) return GR_OK;
    if (!dR_next || !y || !s || !dR || !dy || !ds) return GR_E_NULL;
    if (!aligned16(dR_next) || !aligned16(y) || !aligned16(s) || !aligned16(dR) ||
        !aligned16(dy) || !aligned16(ds))
        return GR_E_ALIGN;
    const size_t N = size_t(shape->n_tokens), D = size_t(shape->d_model);
    const size_t nR = N * kBranches * D * 4, ny = N * D * elem_size(shape->state_dtype);
    const size_t nd = N * D * 4, ns = N * kBranches * 4;
    if ((dR != dR_next && overlaps(dR, nR, dR_next, nR)) || overlaps(dR, nR, y, ny) ||
        overlaps(dR, nR, s, ns) || overlaps(dy, nd, dR_next, nR) || overlaps(dy, nd, y, ny) ||
        overlaps(dy, nd, s, ns) || overlaps(dy, nd, dR, nR) || overlaps(ds, ns, dR_next, nR) ||
        overlaps(ds, ns, y, ny) || overlaps(ds, ns, s, ns) || overlaps(ds, ns, dR, nR) ||
        overlaps(ds, ns, dy, nd))
        return GR_E_ALIAS;
    if ((st = check_device())) return st;
    return status_of(launch_write_backward(shape->n_tokens, shape->d_model, shape->state_dtype,
                                           dR_next, y, s, dR, dy, ds,
                                           static_cast<cudaStream_t>(stream)));
}

// ---- contribution decomposition -----------------------------------------------------------

int gr_decompose(const gr_shape* shape, const void* R, const float* gamma, const float* w_down,
                 const float* w_up, const float* w_write, int32_t n_writers, const void* y,
                 const float* s, const void* R0, float* norm, float* branch_norm, float* pi,
                 float* a0_norm, void* stream) {
    int st = validate_shape(shape);
    if (st) return st;
    if (shape->rank > GR_MAX_RANK) return GR_E_RANK;
    if (n_writers < 0 || n_writers > GR_MAX_WRITERS) return GR_E_SHAPE;
    if (!R || !gamma || !w_down || !w_up || !w_write) return GR_E_NULL;
    const size_t U = size_t(n_writers);
    if (U > 0 && (!y || !s || !norm)) return GR_E_NULL;
    if (R0 && !a0_norm) return GR_E_NULL;
    if (shape->n_tokens == 0 || (U == 0 && !R0)) return GR_OK;
    const void* in[8] = {R, gamma, w_down, w_up, w_write, U ? y : nullptr, U ? s : nullptr, R0};
    float* out[4] = {U ? norm : nullptr, U ? branch_norm : nullptr, U ? pi : nullptr,
                     R0 ? a0_norm : nullptr};
    for (const void* p : in)
        if (p && !aligned16(p)) return GR_E_ALIGN;
    for (const float* p : out)
        if (p && !aligned16(p)) return GR_E_ALIGN;
    const size_t N = size_t(shape->n_tokens), D = size_t(shape->d_model), r = size_t(shape->rank);
    const size_t K = kBranches * D, es = elem_size(shape->state_dtype);
    const size_t in_n[8] = {N * K * es, K * 4, r * K * 4, r * K * 4, kBranches * K * 4,
                            U * N * D * es, U * N * kBranches * 4, N * K * es};
    const size_t out_n[4] = {N * U * 4, N * U * kBranches * 4, N * U * 4, N * 4};
    for (int a = 0; a < 4; ++a) {
        if (!out[a]) continue;
        for (int b = 0; b < 8; ++b)
            if (in[b] && overlaps(out[a], out_n[a], in[b], in_n[b])) return GR_E_ALIAS;
        for (int b = a + 1; b < 4; ++b)
            if (out[b] && overlaps(out[a], out_n[a], out[b], out_n[b])) return GR_E_ALIAS;
    }
    if ((st = check_device())) return st;
    return status_of(launch_decompose(shape->n_tokens, shape->d_model, shape->rank, shape->eps,
                                      shape->state_dtype, R, gamma, w_down, w_up, int(U),
                                      U ? y : nullptr, U ? s : nullptr, R0, out[0], out[1],
                                      out[2], out[3], static_cast<cudaStream_t>(stream)));
}

// ---- FP8 branch state ------------------------------------------------------------------------

int gr_fp8_encode(const gr_shape* shape, const void* R, int32_t in_dtype, uint8_t* codes,
                  uint8_t* scales, void* stream) {
    int st = validate_fp8(shape, false);
    if (st) return st;
    if (in_dtype != GR_BF16 && in_dtype != GR_F32) return GR_E_DTYPE;
    if (shape->n_tokens == 0) return GR_OK;
    if (!R || !codes || !scales) return GR_E_NULL;
    if (!aligned16(R) || !aligned16(codes) || !aligned16(scales)) return GR_E_ALIGN;
    const size_t n = size_t(shape->n_tokens) * kBranches * size_t(shape->d_model);
    if (overlaps(R, n * elem_size(in_dtype), codes, n) ||
        overlaps(R, n * elem_size(in_dtype), scales, n / 32) || overlaps(codes, n, scales, n / 32))
        return GR_E_ALIAS;
    if ((st = check_device())) return st;
    return status_of(launch_fp8_encode(shape->n_tokens * kBranches, shape->d_model, in_dtype, R,
                                       codes, scales, static_cast<cudaStream_t>(stream)));
}

int gr_fp8_decode(const gr_shape* shape, const uint8_t* codes, const uint8_t* scales, void* R,
                  int32_t out_dtype, void* stream) {
    int st = validate_fp8(shape, false);
    if (st) return st;
    if (out_dtype != GR_BF16 && out_dtype != GR_F32) return GR_E_DTYPE;
    if (shape->n_tokens == 0) return GR_OK;
    if (!R || !codes || !scales) return GR_E_NULL;
    if (!aligned16(R) || !aligned16(codes) || !aligned16(scales)) return GR_E_ALIGN;
    const size_t n = size_t(shape->n_tokens) * kBranches * size_t(shape->d_model);
    if (overlaps(R, n * elem_size(out_dtype), codes, n) ||
        overlaps(R, n * elem_size(out_dtype), scales, n / 32))
        return GR_E_ALIAS;
    if ((st = check_device())) return st;
    return status_of(launch_fp8_decode(shape->n_tokens * kBranches, shape->d_model, out_dtype,
                                       codes, scales, R, static_cast<cudaStream_t>(stream)));
}

int gr_read_fp8(const gr_shape* shape, const uint8_t* codes, const uint8_t* scales,
                const gr_params* params, void* x, float* s, void* stream) {
    int st = validate_fp8(shape, true);
    if (st) return st;
    if ((st = validate_params(shape, params))) return st;
    if (shape->n_tokens == 0) return GR_OK;
    if (!codes || !scales || !x || !s) return GR_E_NULL;
    if (!aligned16(codes) || !aligned16(scales) || !aligned16(x) || !aligned16(s))
        return GR_E_ALIGN;
    const size_t N = size_t(shape->n_tokens), D = size_t(shape->d_model);
    const size_t nc = N * kBranches * D, nb = nc / 32, nx = N * D * 2, ns = N * kBranches * 4;
    if (overlaps(x, nx, codes, nc) || overlaps(x, nx, scales, nb) || overlaps(s, ns, codes, nc) ||
        overlaps(s, ns, scales, nb) || overlaps(x, nx, s, ns))
        return GR_E_ALIAS;
    if ((st = check_device())) return st;
    return status_of(launch_tiled_fp8(shape->n_tokens, shape->d_model, shape->rank, shape->eps,
                                      const_cast<uint8_t*>(codes), const_cast<uint8_t*>(scales),
                                      nullptr, nullptr, params->packed, x, s,
                                      static_cast<cudaStream_t>(stream)));
}

int gr_write_fp8(const gr_shape* shape, uint8_t* codes, uint8_t* scales, const void* y,
                 const float* s, void* stream) {
    int st = validate_fp8(shape, false);
    if (st) return st;
    if (shape->n_tokens == 0) return GR_OK;
    if (!codes || !scales || !y || !s) return GR_E_NULL;
    if (!aligned16(codes) || !aligned16(scales) || !aligned16(y) || !aligned16(s))
        return GR_E_ALIGN;
    const size_t N = size_t(shape->n_tokens), D = size_t(shape->d_model);
    const size_t nc = N * kBranches * D, nb = nc / 32, ny = N * D * 2, ns = N * kBranches * 4;
    if (overlaps(codes, nc, scales, nb) || overlaps(codes, nc, y, ny) ||
        overlaps(codes, nc, s, ns) || overlaps(scales, nb, y, ny) || overlaps(scales, nb, s, ns))
        return GR_E_ALIAS;
    if ((st = check_device())) return st;
    return status_of(launch_fp8_write(shape->n_tokens, shape->d_model, codes, scales, y, s,
                                      static_cast<cudaStream_t>(stream)));
}

int gr_write_then_read_fp8(const gr_shape* shape, uint8_t* codes, uint8_t* scales,
                           const void* y, const float* s_prev, const gr_params* next, void* x,
                           float* s_next, void* stream) {
    int st = validate_fp8(shape, true);
    if (st) return st;
    if ((st = validate_params(shape, next))) return st;
    if (shape->n_tokens == 0) return GR_OK;
    if (!codes || !scales || !y || !s_prev || !x || !s_next) return GR_E_NULL;
    if (!aligned16(codes) || !aligned16(scales) || !aligned16(y) || !aligned16(s_prev) ||
        !aligned16(x) || !aligned16(s_next))
        return GR_E_ALIGN;
    const size_t N = size_t(shape->n_tokens), D = size_t(shape->d_model);
    const size_t nc = N * kBranches * D, nb = nc / 32, ny = N * D * 2, ns = N * kBranches * 4;
    const void* state[2] = {codes, scales};
    const size_t sz[2] = {nc, nb};
    if (overlaps(codes, nc, scales, nb)) return GR_E_ALIAS;
    for (int k = 0; k < 2; ++k)
        if (overlaps(state[k], sz[k], y, ny) || overlaps(state[k], sz[k], s_prev, ns) ||
            overlaps(state[k], sz[k], x, ny) || overlaps(state[k], sz[k], s_next, ns))
            return GR_E_ALIAS;
    if (overlaps(x, ny, s_next, ns) || overlaps(x, ny, s_prev, ns) ||
        overlaps(s_next, ns, y, ny) || (x != y && overlaps(x, ny, y, ny)) ||
        (s_next != s_prev && overlaps(s_next, ns, s_prev, ns)))
        return GR_E_ALIAS;
    if ((st = check_device())) return st;
    return status_of(launch_tiled_fp8(shape->n_tokens, shape->d_model, shape->rank, shape->eps,
                                      codes, scales, y, s_prev, next->packed, x, s_next,
                                      static_cast<cudaStream_t>(stream)));
}

int gr_device_status(int clear) {
    int st = check_device();
    if (st) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return GR_E_CUDA;
    const int v = fused_status(clear != 0), w = tiled_status(clear != 0);
    if (v < 0 || w < 0) return GR_E_CUDA;
    return (v | w) ? GR_E_TIMEOUT : GR_OK;
}

int gr_selftest_bounded_wait(int64_t limit_cycles, void* stream) {
    if (limit_cycles < 1 || limit_cycles > 4000000000LL) return GR_E_SIZE;
    int st = check_device();
    if (st) return st;
    return status_of(launch_wait_selftest(static_cast<long long>(limit_cycles),
                                          static_cast<cudaStream_t>(stream)));
}

int gr_host_workspace_size(const gr_shape* shape, size_t* bytes) {
    int st = validate_shape(shape);
    if (st) return st;
    if (!bytes) return GR_E_NULL;
    const size_t es = elem_size(shape->state_dtype);
    const size_t N = size_t(shape->n_tokens), D = size_t(shape->d_model);
    *bytes = align256(N * kBranches * D * es) + align256(N * D * es) * 2 +
             align256(N * kBranches * 4) * 2;
    return GR_OK;
}

int gr_write_then_read_host(const gr_shape* shape, void* R_host, const void* y_host,
                            const float* s_prev_host, const gr_params* next, void* x_host,
                            float* s_next_host, void* workspace, size_t workspace_bytes,
                            void* stream) {
    int st = validate_shape(shape);
    if (st) return st;
    if ((st = validate_params(shape, next))) return st;
    if (use_rank_tc(shape)) return GR_E_RANK;   // the large-rank path has device entries only
    if (shape->n_tokens == 0) return GR_OK;
    if (!R_host || !y_host || !s_prev_host || !x_host || !s_next_host || !workspace)
        return GR_E_NULL;
    if (!aligned256(workspace)) return GR_E_ALIGN;
    size_t need = 0;
    gr_host_workspace_size(shape, &need);
    if (workspace_bytes < need) return GR_E_SIZE;
    const size_t es = elem_size(shape->state_dtype);
    const size_t N = size_t(shape->n_tokens), D = size_t(shape->d_model);
    const size_t nR = N * kBranches * D * es, ny = N * D * es, ns = N * kBranches * 4;
    if (overlaps(R_host, nR, y_host, ny) || overlaps(R_host, nR, x_host, ny) ||
        overlaps(x_host, ny, y_host, ny) || overlaps(s_prev_host, ns, s_next_host, ns) ||
        overlaps(R_host, nR, s_next_host, ns) || overlaps(x_host, ny, s_next_host, ns))
        return GR_E_ALIAS;
    if ((st = check_device())) return st;
    if (N == 0) return GR_OK;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    char* w = static_cast<char*>(workspace);
    char* dR = w;
    char* dy = w + align256(nR);
    char* dx = w + align256(nR) + align256(ny);
    char* dsp = w + align256(nR) + 2 * align256(ny);
    char* dsn = w + align256(nR) + 2 * align256(ny) + align256(ns);
    char* hR = static_cast<char*>(R_host);
    const char* hy = static_cast<const char*>(y_host);
    const char* hsp = reinterpret_cast<const char*>(s_prev_host);
    char* hx = static_cast<char*>(x_host);
    char* hsn = reinterpret_cast<char*>(s_next_host);
    // Token chunks of at least 1024 (a multiple of 16): chunk i's host-to-device copies run on
    // one internal stream, its step on `stream` after them, its device-to-host copies on a second
    // internal stream after the step, so both copy directions and the steps overlap.
    const size_t nchunk = N >= 2 * 1024 ? (N / 1024 < kHostChunks ? N / 1024 : kHostChunks) : 1;
    const size_t per = ((N + nchunk - 1) / nchunk + 15) / 16 * 16;
    HostPipe& hp = g_host_pipe[current_device()];
    std::lock_guard<std::mutex> lock(hp.mu);
    if (!host_pipe_init(hp)) return GR_E_CUDA;
    // the copies into the workspace wait for the work already queued on `stream`
    if (cudaEventRecord(hp.start, cs) != cudaSuccess ||
        cudaStreamWaitEvent(hp.h2d, hp.start, 0) != cudaSuccess)
        return GR_E_CUDA;
    const size_t bR = kBranches * D * es, by = D * es, bs = kBranches * 4;  // bytes per token
    for (size_t c = 0, t = 0; t < N; ++c, t += per) {
        const size_t n = N - t < per ? N - t : per;
        if (cudaMemcpyAsync(dR + t * bR, hR + t * bR, n * bR, cudaMemcpyHostToDevice, hp.h2d) !=
                cudaSuccess ||
            cudaMemcpyAsync(dy + t * by, hy + t * by, n * by, cudaMemcpyHostToDevice, hp.h2d) !=
                cudaSuccess ||
            cudaMemcpyAsync(dsp + t * bs, hsp + t * bs, n * bs, cudaMemcpyHostToDevice, hp.h2d) !=
                cudaSuccess ||
            cudaEventRecord(hp.loaded[c], hp.h2d) != cudaSuccess ||
            cudaStreamWaitEvent(cs, hp.loaded[c], 0) != cudaSuccess)
            return GR_E_CUDA;
        gr_shape sc = *shape;
        sc.n_tokens = int64_t(n);
        st = run_step(&sc, dR + t * bR, dy + t * by, reinterpret_cast<const float*>(dsp + t * bs),
                      next, dx + t * by, reinterpret_cast<float*>(dsn + t * bs), cs);
        if (st) return st;
        if (cudaEventRecord(hp.computed[c], cs) != cudaSuccess ||
            cudaStreamWaitEvent(hp.d2h, hp.computed[c], 0) != cudaSuccess ||
            cudaMemcpyAsync(hR + t * bR, dR + t * bR, n * bR, cudaMemcpyDeviceToHost, hp.d2h) !=
                cudaSuccess ||
            cudaMemcpyAsync(hx + t * by, dx + t * by, n * by, cudaMemcpyDeviceToHost, hp.d2h) !=
                cudaSuccess ||
            cudaMemcpyAsync(hsn + t * bs, dsn + t * bs, n * bs, cudaMemcpyDeviceToHost,
                            hp.d2h) != cudaSuccess)
            return GR_E_CUDA;
    }
    // the caller's stream covers the read-back too
    if (cudaEventRecord(hp.copied, hp.d2h) != cudaSuccess ||
        cudaStreamWaitEvent(cs, hp.copied, 0) != cudaSuccess)
        return GR_E_CUDA;
    return status_of(cudaStreamSynchronize(cs));
}

}  // extern "C"

// ---- gr_write_then_read_host_static: the host-buffer step with a fixed device workspace ----

namespace gr {
namespace {

// The device workspace of gr_write_then_read_host_static, the host-buffer step for callers that
// cannot allocate device memory (a host program with no device allocator, a process whose
// memory a pool already holds, a decode loop that cannot take cudaFree's device-wide
// synchronisation): file scope, module lifetime, the same layout gr_write_then_read_host uses in
// its caller-provided workspace. Nothing in it has to start at zero: every byte a call reads was
// written earlier in the same call. Calls that overlap in time race on it.
static __device__ __align__(256) unsigned char g_static_ws[GR_STATIC_WORKSPACE_BYTES];
void* g_static_ws_addr[kMaxDevices];  // device address, looked up once per device
std::mutex g_static_mu;

}  // namespace
}  // namespace gr

extern "C" {

int gr_write_then_read_host_static(const gr_shape* shape, void* R_host, const void* y_host,
                                   const float* s_prev_host, const gr_params* next, void* x_host,
                                   float* s_next_host, void* stream) {
    int st = validate_shape(shape);
    if (st) return st;
    if ((st = validate_params(shape, next))) return st;
    if (use_rank_tc(shape)) return GR_E_RANK;   // the large-rank path has device entries only
    if (shape->n_tokens == 0) return GR_OK;
    if (!R_host || !y_host || !s_prev_host || !x_host || !s_next_host) return GR_E_NULL;
    size_t need = 0;
    gr_host_workspace_size(shape, &need);
    if (need > size_t(GR_STATIC_WORKSPACE_BYTES)) return GR_E_SIZE;
    const size_t es = elem_size(shape->state_dtype);
    const size_t N = size_t(shape->n_tokens), D = size_t(shape->d_model);
    const size_t nR = N * kBranches * D * es, ny = N * D * es, ns = N * kBranches * 4;
    if (overlaps(R_host, nR, y_host, ny) || overlaps(R_host, nR, x_host, ny) ||
        overlaps(x_host, ny, y_host, ny) || overlaps(s_prev_host, ns, s_next_host, ns) ||
        overlaps(R_host, nR, s_next_host, ns) || overlaps(x_host, ny, s_next_host, ns))
        return GR_E_ALIAS;
    if ((st = check_device())) return st;
    const int dev = current_device();
    {
        std::lock_guard<std::mutex> lock(g_static_mu);
        if (!g_static_ws_addr[dev]) {
            // under lazy module loading (CUDA's default) this is where the device commits the
            // array's memory; a device whose memory is taken fails here with an allocation error
            const cudaError_t e = cudaGetSymbolAddress(&g_static_ws_addr[dev], g_static_ws);
            if (e != cudaSuccess) {
                g_static_ws_addr[dev] = nullptr;
                cudaGetLastError();   // not a sticky error: clear it for the caller's next call
                return e == cudaErrorMemoryAllocation ? GR_E_NOMEM : GR_E_CUDA;
            }
        }
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    char* w = static_cast<char*>(g_static_ws_addr[dev]);
    void* dR = w;
    void* dy = w + align256(nR);
    void* dx = w + align256(nR) + align256(ny);
    float* dsp = reinterpret_cast<float*>(w + align256(nR) + 2 * align256(ny));
    float* dsn = reinterpret_cast<float*>(w + align256(nR) + 2 * align256(ny) + align256(ns));
    if (cudaMemcpyAsync(dR, R_host, nR, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        cudaMemcpyAsync(dy, y_host, ny, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        cudaMemcpyAsync(dsp, s_prev_host, ns, cudaMemcpyHostToDevice, cs) != cudaSuccess)
        return GR_E_CUDA;
    // the cluster kernel alone (no shape that fits the workspace reaches the split's threshold)
    st = run_step(shape, dR, dy, dsp, next, dx, dsn, cs, nullptr, 0, false);
    if (st) return st;
    if (cudaMemcpyAsync(R_host, dR, nR, cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
        cudaMemcpyAsync(x_host, dx, ny, cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
        cudaMemcpyAsync(s_next_host, dsn, ns, cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        return GR_E_CUDA;
    return status_of(cudaStreamSynchronize(cs));
}

}  // extern "C"
