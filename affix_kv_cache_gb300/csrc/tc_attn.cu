// tc_attn.cu -- tensor-core attention kernels (placeholder until the tcgen05 path lands).
#include "tc_attn.cuh"

namespace acache {

bool tc_supported(const AttnArgs&) { return false; }

int launch_tc_slot_attention(const AttnArgs&, int, int, const void*, int, const int32_t*,
                             const void*, const void*, int64_t, void*, int32_t*, cudaStream_t) {
    return ACACHE_ERR_UNSUPPORTED;
}
int launch_tc_probe_pass_a(const AttnArgs&, int, int, int, int, const void*, const void*,
                           const void*, const void*, const void*, void*, float*, float*,
                           int32_t*, cudaStream_t) {
    return ACACHE_ERR_UNSUPPORTED;
}
int launch_tc_probe_pass_b(const AttnArgs&, int, int, int, const int32_t*, int, const void*,
                           const void*, const float*, const float*, float*, int32_t*,
                           cudaStream_t) {
    return ACACHE_ERR_UNSUPPORTED;
}

}  // namespace acache
