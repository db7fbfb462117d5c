// ftd_internal.cuh -- host-side helpers shared by the library's entry points
// (ftd_api.cu and ftd_noalloc.cu); hidden, not part of the C ABI.
#pragma once

#include <cuda.h>

#include "../../include/ftd.h"
#include "ftd_decode_wide_tc.cuh"

namespace ftd {
// The tensor-core kernel a configuration runs (tki.fn null: the CUDA-core
// kernel), with its query-row blocks per kv head (nhb) and real rows per block.
struct TcChoice {
    TcKernelInfo tki;
    int nhb;
    int qblk;
};
TcChoice choose_tc(const ftd_config& c);

// What a valid configuration runs: the CUDA-core kernel's block of G query rows
// (nhb blocks per kv head) and its instantiation, the tensor-core choice, and
// the number of cache rows (of head_dim elements) the caches hold.
struct Plan {
    int G, nhb;
    KernelInfo ki;
    TcChoice tcc;
    size_t rows;
    // output projection (proj_dim > 0): tokens per step, tokens per block of the
    // projection kernel, blocks, feature tiles of 128 and K chunks of 64
    int tokens, ntb, nblk, mtiles, kch;
};
// Every check of a configuration (sizes, dtypes, options, 32-bit index bounds);
// FTD_OK and the plan, or a status and a message in msg.
ftd_status plan_config(const ftd_config& c, Plan* plan, char* msg, size_t n);

// Null and alignment checks of a decode call's pointers.
ftd_status check_pointers(const ftd_config& c, const void* q, const void* k_new, const void* v_new, const void* bias,
                          const int32_t* seq_lens, const void* k_cache, const void* v_cache, const float* scales,
                          const void* out, char* msg, size_t n);

// Limit of the kernels' pipeline waits in SM cycles (cfg.wait_limit_us, or the default).
long long wait_cycles_for(const ftd_config& c, int dev);

// Tensor map of a [rows][128] cache view for the tensor-core kernel; false when
// the driver entry point is missing or the encoding fails.
bool encode_tc_cache_map(CUtensorMap* map, void* base, ftd_dtype dt, size_t rows);
}  // namespace ftd
