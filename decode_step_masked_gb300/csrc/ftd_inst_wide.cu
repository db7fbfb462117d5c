// ftd_inst_wide.cu -- tensor-core decode kernels for kv heads shared by 32 or 64
// query rows (multi-query and wide grouped-query caches).
#include "ftd_decode_wide_tc.cuh"

namespace ftd {
template <typename CT, bool MQ>
static TcKernelInfo pick_wide(int G) {
    return G == 64 ? wide_kernel_info<CT, 64, MQ>() : wide_kernel_info<CT, 32, MQ>();
}

TcKernelInfo select_wide(bool bf16, int G, bool multi_token) {
    if (bf16) return multi_token ? pick_wide<__nv_bfloat16, true>(G) : pick_wide<__nv_bfloat16, false>(G);
    return multi_token ? pick_wide<__half, true>(G) : pick_wide<__half, false>(G);
}
}  // namespace ftd
