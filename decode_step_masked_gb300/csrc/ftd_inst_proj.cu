// ftd_inst_proj.cu -- the output-projection kernels (bf16 and fp16 operands).
#include "ftd_out_proj.cuh"

namespace ftd {
ProjKernelInfo select_proj(bool bf16) {
    return ProjKernelInfo{bf16 ? reinterpret_cast<const void*>(&out_proj_kernel<true>)
                               : reinterpret_cast<const void*>(&out_proj_kernel<false>)};
}
}  // namespace ftd
