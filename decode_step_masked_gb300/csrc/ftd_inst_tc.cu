// ftd_inst_tc.cu -- tensor-core decode kernels for fp16 / bf16 caches whose kv
// heads carry 8 or 16 query rows (grouped heads, or several new tokens).
#include "ftd_decode_gqa_tc.cuh"

namespace ftd {
template <typename CT, bool MQ>
static TcKernelInfo pick_g(int G) {
    return G == 16 ? tc_kernel_info<CT, 16, MQ>() : tc_kernel_info<CT, 8, MQ>();
}

TcKernelInfo select_tc(bool bf16, int G, bool multi_token) {
    if (bf16) return multi_token ? pick_g<__nv_bfloat16, true>(G) : pick_g<__nv_bfloat16, false>(G);
    return multi_token ? pick_g<__half, true>(G) : pick_g<__half, false>(G);
}
}  // namespace ftd
