// ftd_common.cuh -- device helpers shared by the decode-step kernels (sm_103a).
//
// Inline PTX for the pieces CUDA C++ does not expose directly: shared-memory
// mbarriers, the bulk-copy engine (cp.async.bulk, global -> shared, completing
// on an mbarrier) and the proxy fence that orders ordinary shared-memory
// accesses before the copy engine reuses a buffer.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace ftd {

// Sticky device error bits (read and cleared by ftd_get_error).
constexpr uint32_t kErrSeqOverflow = 1u;
constexpr uint32_t kErrTimeout = 2u;

// A wait on a copy gives up after this many SM clock cycles (about 2 s).
constexpr long long kWaitLimitCycles = 4000000000LL;

constexpr int kMaxBatch = 1024;
constexpr int kWarps = 8;               // warps per CTA, each an independent worker
constexpr int kThreads = kWarps * 32;

enum QkvType : int { kF32 = 0, kF16 = 1, kBF16 = 2 };

// Arguments of one decode step, resolved by the host entry point.
struct DecodeParams {
    const void* q;        // [B][Hq][D]  qkv dtype
    const void* k_new;    // [B][Hkv][D] qkv dtype
    const void* v_new;    // [B][Hkv][D] qkv dtype
    const void* bias;     // [(Hq+2Hkv)*D] qkv dtype or nullptr
    unsigned char* k_cache;  // [B][Hkv][Lmax][D] cache dtype
    unsigned char* v_cache;
    float* k_scales;      // [B][Hkv][Lmax] (int8 caches)
    float* v_scales;
    const int32_t* seq_lens;  // [B]
    float* out;           // [B][Hq][D]
    float* ws;            // split-K partial slots
    uint32_t* counters;   // one arrival counter per segment, zero between launches
    uint32_t* err;        // sticky error word
    int B, Hq, Hkv, Lmax, group, nhb;
    int qkv_dtype;
    float qscale;         // softmax scale * log2(e): scores live in the log2 domain
};

// ---------------------------------------------------------------- PTX
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// One contiguous global -> shared copy; completes `bytes` of the barrier's
// transaction count.  dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of a barrier; after kWaitLimitCycles raise the
// timeout bit and return false instead of spinning forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint32_t* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitLimitCycles) {
            atomicOr(err, kErrTimeout);
            return false;
        }
    }
    return true;
}

// ------------------------------------------------------------ small loads
__device__ __forceinline__ float ld_qkv(const void* p, int dt, size_t i) {
    if (dt == kF32) return __ldg(static_cast<const float*>(p) + i);
    if (dt == kF16) return __half2float(static_cast<const __half*>(p)[i]);
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

}  // namespace ftd
