// Concurrent split of a large cluster-kernel step. The cluster kernel fills only the SMs its
// resident clusters take (7 clusters of 16 = 112 of 152 SMs at D = 4096); the two-pass kernel
// takes a share of the tokens on the rest. Both go on the caller's stream: the two-pass kernel is
// the cluster kernel's programmatic dependent, so its CTAs start only once every cluster is
// resident (they cannot take an SM a cluster needs) and its grid completes only after the
// cluster kernel's (work after the call waits for both).
#include "gr_internal.h"

namespace gr {

namespace {

// The share is k whole rounds of 32-token tiles on the free SMs, with k chosen to minimise the
// later of the two finish times. Time model, in units of the cluster kernel's period per
// 16-token tile and cluster (about 2.2 µs, nearly independent of D since each CTA always owns
// 256 channels): a two-pass tile of 32 tokens takes kTiledTilePerChannel · D of them (about
// 115 µs at D = 4096). At the prefill shape this gives 2560 of 16384 tokens to 40 SMs, the best
// split measured there.
constexpr double kTiledTilePerChannel = 0.0122;

}  // namespace

int64_t split_tokens(int64_t n_tokens, int D, int r, bool write, int* free_sms) {
    if (!fused_supported(D, r) || !tiled_supported(D, r)) return 0;
    const double rho = kTiledTilePerChannel * D;   // one two-pass round
    // cheap bound first (no device query): one two-pass round must fit in the cluster kernel's
    // time even with a single cluster of 16 per 16 SMs' worth of the device
    if (double(n_tokens) < 16.0 * 4.0 * rho) return 0;
    const int fused_ctas = fused_resident_ctas(D, r, write);
    const int clusters = fused_ctas / (D / 256);
    const int free = sm_count() - fused_ctas;
    if (fused_ctas <= 0 || clusters <= 0 || free < 1) return 0;
    const double N = double(n_tokens);
    double best = N / (16.0 * clusters);   // no split
    int64_t best_n2 = 0;
    for (int k = 1; k * rho < best; ++k) {
        const int64_t n2 = int64_t(32) * k * free;
        if (n2 >= n_tokens) break;
        const double t_f = (N - double(n2)) / (16.0 * clusters);
        const double t = t_f > k * rho ? t_f : k * rho;
        if (t < best) {
            best = t;
            best_n2 = n2;
        }
    }
    if (best_n2 > 0 && free_sms) *free_sms = free;
    return best_n2;
}

cudaError_t launch_split_bf16(int64_t N, int64_t n2, int free_sms, int D, int r, float eps,
                              void* R, const void* y, const float* s_prev, const void* packed,
                              void* x, float* s_out, cudaStream_t st) {
    // tokens [0, n1) on the cluster kernel, [n1, N) on the two-pass kernel, both on `st`
    const int64_t n1 = N - n2;
    const size_t Dz = size_t(D);
    char* R2 = static_cast<char*>(R) + size_t(n1) * kBranches * Dz * 2;
    const char* y2 = y ? static_cast<const char*>(y) + size_t(n1) * Dz * 2 : nullptr;
    const float* sp2 = s_prev ? s_prev + size_t(n1) * kBranches : nullptr;
    char* x2 = static_cast<char*>(x) + size_t(n1) * Dz * 2;
    float* so2 = s_out + size_t(n1) * kBranches;
    cudaError_t e = launch_fused_bf16(n1, D, r, eps, R, y, s_prev, packed, x, s_out, st);
    if (e != cudaSuccess) return e;
    return launch_tiled_bf16(n2, D, r, eps, R2, y2, sp2, packed, x2, so2, st, free_sms, true);
}

}  // namespace gr
