// ftd_inst_bf16.cu -- decode-step kernels for bf16 caches (one translation unit per
// cache type so the build compiles them in parallel).
#include "ftd_decode_splitk.cuh"

namespace ftd {
KernelInfo select_bf16(int D, int G) { return select_kernel<__nv_bfloat16>(D, G); }
}  // namespace ftd
