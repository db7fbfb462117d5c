// ftd_internal.cuh -- host-side helpers shared by the library's entry points
// (ftd_api.cu and ftd_noalloc.cu); hidden, not part of the C ABI.
#pragma once

#include <cuda.h>

#include "../../include/ftd.h"
#include "ftd_decode_gqa_tc.cuh"

namespace ftd {
// The tensor-core kernel a configuration runs (tki.fn null: the CUDA-core
// kernel), with its query-row blocks per kv head (nhb) and real rows per block.
struct TcChoice {
    TcKernelInfo tki;
    int nhb;
    int qblk;
};
TcChoice choose_tc(const ftd_config& c);

// Tensor map of a [rows][128] cache view for the tensor-core kernel; false when
// the driver entry point is missing or the encoding fails.
bool encode_tc_cache_map(CUtensorMap* map, void* base, ftd_dtype dt, size_t rows);
}  // namespace ftd
