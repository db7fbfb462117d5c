// ftd_inst_tc_i8.cu -- tensor-core decode kernels for INT8 caches whose kv heads
// carry a multiple of 8 query rows (codes converted to fp16 on chip).
#include "ftd_decode_gqa_tc.cuh"

namespace ftd {
TcKernelInfo select_tc_i8(bool multi_token) {
    return multi_token ? tc_kernel_info<int8_t, 8, true>() : tc_kernel_info<int8_t, 8, false>();
}
}  // namespace ftd
