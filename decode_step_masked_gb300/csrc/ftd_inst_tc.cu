// ftd_inst_tc.cu -- tensor-core decode kernels for grouped-query fp16 / bf16 caches.
#include "ftd_decode_gqa_tc.cuh"

namespace ftd {
TcKernelInfo select_tc(bool bf16, int G) {
    if (bf16) return G == 16 ? tc_kernel_info<__nv_bfloat16, 16>() : tc_kernel_info<__nv_bfloat16, 8>();
    return G == 16 ? tc_kernel_info<__half, 16>() : tc_kernel_info<__half, 8>();
}
}  // namespace ftd
