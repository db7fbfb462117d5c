// ftd_inst_f32.cu -- decode-step kernels for f32 caches (one translation unit per
// cache type so the build compiles them in parallel).
#include "ftd_decode_splitk.cuh"

namespace ftd {
KernelInfo select_f32(int D, int G) { return select_kernel<float>(D, G); }
}  // namespace ftd
