// ftd_inst_i8.cu -- decode-step kernels for i8 caches (one translation unit per
// cache type so the build compiles them in parallel).
#include "ftd_decode_splitk.cuh"

namespace ftd {
KernelInfo select_i8(int D, int G) { return select_kernel<int8_t>(D, G); }
}  // namespace ftd
