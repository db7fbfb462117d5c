// ftd_debug.cu -- test hooks of the C ABI (include/ftd.h): a kernel that lets
// the next launch on its stream start at once and writes seq_lens late, so
// that the decode kernels' re-planning path (lengths changed after they were
// first read) runs on demand.
#include <cuda_runtime.h>

#include "../../include/ftd.h"
#include "ftd_common.cuh"

namespace ftd {
void set_last_error(const char* msg);
void note_launch();

namespace {
__global__ void late_lengths_kernel(const int32_t* src, int32_t* dst, int n, long long delay_cycles) {
    grid_dep_launch();  // the next launch may start now and read dst before it is written
    if (threadIdx.x == 0) {
        const long long t0 = clock64();
        while (clock64() - t0 < delay_cycles) {
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
}
}  // namespace
}  // namespace ftd

extern "C" ftd_status ftd_debug_late_lengths(const int32_t* src, int32_t* dst, int n, int delay_us, void* stream) {
    ftd::set_last_error("");
    if (!src || !dst || n < 1 || n > ftd::kMaxBatch || delay_us < 0 || delay_us > 1000000) {
        ftd::set_last_error("ftd_debug_late_lengths: src, dst, 1 <= n <= 1024 and 0 <= delay_us <= 1e6 required");
        return FTD_ERR_INVALID_ARG;
    }
    int dev = 0, khz = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev) != cudaSuccess) {
        cudaGetLastError();
        khz = 2100000;
    }
    const long long cycles = static_cast<long long>(delay_us) * (khz / 1000);
    ftd::late_lengths_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(src, dst, n, cycles);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        ftd::set_last_error(cudaGetErrorString(e));
        return FTD_ERR_CUDA;
    }
    ftd::note_launch();
    return FTD_OK;
}
