// Fused bf16 write→read kernel (tensor cores). Not enabled yet: every shape takes the
// generic kernel.
#include "gr_internal.h"

namespace gr {

bool fused_supported(int, int) { return false; }
size_t fused_frag_down_bytes(int, int) { return 0; }
size_t fused_frag_up_bytes(int, int) { return 0; }

cudaError_t launch_pack_fused(int, int, const float*, const float*, const float*, const float*,
                              void*, void*, cudaStream_t) {
    return cudaSuccess;
}

cudaError_t launch_fused_bf16(int64_t, int, int, float, void*, const void*, const float*,
                              const void*, void*, float*, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace gr
