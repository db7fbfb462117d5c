// ftd_inst_f16.cu -- decode-step kernels for f16 caches (one translation unit per
// cache type so the build compiles them in parallel).
#include "ftd_decode_splitk.cuh"

namespace ftd {
KernelInfo select_f16(int D, int G) { return select_kernel<__half>(D, G); }
}  // namespace ftd
