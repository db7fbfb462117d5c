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
constexpr uint32_t kErrBadPage = 4u;

// Most new tokens per slot in one step (speculative verification runs).
constexpr int kMaxQLen = 64;

// Default limit of a pipeline wait (a wait on a copy, an MMA or another role of
// the block), in SM clock cycles: about 2 s.  A context can set a shorter one.
constexpr long long kWaitLimitCycles = 4000000000LL;
// Limit of a drain wait after an abort (the copies and MMAs a block still has in
// flight before it exits).  It never takes the context's shorter pipeline limit:
// a bulk copy must not land in shared memory after the block has left.
constexpr long long kDrainLimitCycles = 4000000000LL;

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
    void* out;            // [B][Hq][D], out_dtype
    float* ws;            // split-K partial slots
    uint32_t* counters;   // one arrival counter per segment, zero between launches
    uint32_t* err;        // sticky error word
    int B, Hq, Hkv, Lmax, group, nhb;
    int qkv_dtype;
    float qscale;         // softmax scale * log2(e): scores live in the log2 domain
    int out_dtype;        // kF32 / kF16 / kBF16
    int window;           // > 0: attend only the last `window` positions
    int nq;               // new tokens per slot (q [B][nq][Hq][D]); query rows per kv head = nq * group
    int qblk;             // query rows per tensor-core block (<= its G; the rest of the block is zero)
    // paged cache: page p of the pool holds rows [p][Hkv][page_size][D];
    // block_table[b * pages_per_seq + i] is the page of positions [i*page_size, (i+1)*page_size)
    const int32_t* block_table;  // nullptr: contiguous [B][Hkv][Lmax][D] cache
    int pages_per_seq, page_shift, num_pages;  // page_size = 1 << page_shift
    long long wait_cycles;  // limit of a pipeline wait (kWaitLimitCycles unless the context sets one)
    int stall;              // test hook: block 0 never issues its first tile copy (see ftd_debug_stall_next)
    // Output projection (ftd_decode_mha_proj): the final stores also write each output
    // value, as out holds it, split into a high and a low part of the projection's
    // operand type (proj_dt, kF16 or kBF16), into two planes laid out like out.
    void* proj_hi;          // nullptr: no projection
    void* proj_lo;
    int proj_dt;
};

// First visible position of a slot with L cached tokens (the window start).
__device__ __forceinline__ int window_start(int L, int window) {
    const int ctx = L + 1;
    return (window > 0 && ctx > window) ? ctx - window : 0;
}

// Query row qi of a kv head (qi = head block * G + j, token-major: qi = token * group + head in
// group) -> its token, and its row in q / out ([B][nq][Hq] rows of D elements).
__device__ __forceinline__ int q_token(const DecodeParams& p, int qi) { return qi / p.group; }
__device__ __forceinline__ size_t q_row(const DecodeParams& p, int b, int kvh, int qi) {
    const int tok = qi / p.group;
    return (static_cast<size_t>(b) * p.nq + tok) * p.Hq + kvh * p.group + (qi - tok * p.group);
}

// Row index (in cache rows of D elements) of position `pos` of (slot b, kv head),
// contiguous or through the block table.  A page outside [0, num_pages) raises
// the bad-page error and returns -1 (the caller then skips the access).
__device__ __forceinline__ long long cache_row(const DecodeParams& p, int b, int kvh, int pos, int page) {
    if (!p.block_table) return (static_cast<long long>(b) * p.Hkv + kvh) * p.Lmax + pos;
    if (page < 0 || page >= p.num_pages) return -1;
    return ((static_cast<long long>(page) * p.Hkv + kvh) << p.page_shift) + (pos & ((1 << p.page_shift) - 1));
}

__device__ __forceinline__ int page_of(const DecodeParams& p, int b, int pos) {
    return p.block_table ? __ldg(p.block_table + static_cast<size_t>(b) * p.pages_per_seq + (pos >> p.page_shift))
                         : 0;
}

// Block-table entries a copy issuer holds: the entry of the current page and,
// loaded one page early, the next one, so a tile that starts a page seldom
// waits for a table load.
struct PageCursor {
    int key = -1, val = 0, nkey = -1, nval = 0;
    __device__ __forceinline__ int page(const DecodeParams& p, int b, int t0) {
        if (!p.block_table) return 0;
        const int i = t0 >> p.page_shift;
        const int k = b * p.pages_per_seq + i;
        if (k != key) {
            val = k == nkey ? nval : __ldg(p.block_table + k);
            key = k;
            if (i + 1 < p.pages_per_seq) {
                nkey = k + 1;
                nval = __ldg(p.block_table + k + 1);
            }
        }
        return val;
    }
};

// ---------------------------------------------------------------- output
__device__ __forceinline__ void st_out1(void* out, size_t i, float v, int dt) {
    if (dt == kF32) static_cast<float*>(out)[i] = v;
    else if (dt == kF16) static_cast<__half*>(out)[i] = __float2half_rn(v);
    else static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
}

// Four consecutive outputs starting at element i (i a multiple of 4).
__device__ __forceinline__ void st_out4(void* out, size_t i, float a, float b, float c, float d, int dt) {
    if (dt == kF32) {
        *reinterpret_cast<float4*>(static_cast<float*>(out) + i) = make_float4(a, b, c, d);
    } else if (dt == kF16) {
        const __half2 x = __floats2half2_rn(a, b), y = __floats2half2_rn(c, d);
        uint2 u;
        memcpy(&u.x, &x, 4);
        memcpy(&u.y, &y, 4);
        *reinterpret_cast<uint2*>(static_cast<__half*>(out) + i) = u;
    } else {
        const __nv_bfloat162 x = __floats2bfloat162_rn(a, b), y = __floats2bfloat162_rn(c, d);
        uint2 u;
        memcpy(&u.x, &x, 4);
        memcpy(&u.y, &y, 4);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + i) = u;
    }
}

// The value out holds after storing v in out_dtype.
__device__ __forceinline__ float as_stored(float v, int dt) {
    if (dt == kF16) return __half2float(__float2half_rn(v));
    if (dt == kBF16) return __bfloat162float(__float2bfloat16_rn(v));
    return v;
}

// x as a high and a low part of type kF16 / kBF16 (x ~ hi + lo, about 16 mantissa bits), as bit patterns.
__device__ __forceinline__ void split_hilo(float x, int dt, uint16_t& hi, uint16_t& lo) {
    if (dt == kF16) {
        const __half h = __float2half_rn(x);
        hi = __half_as_ushort(h);
        lo = __half_as_ushort(__float2half_rn(x - __half2float(h)));
    } else {
        const __nv_bfloat16 h = __float2bfloat16_rn(x);
        hi = __bfloat16_as_ushort(h);
        lo = __bfloat16_as_ushort(__float2bfloat16_rn(x - __bfloat162float(h)));
    }
}

// Final stores of the step: out, and the projection planes when there is a projection.
__device__ __forceinline__ void store_out1(const DecodeParams& p, size_t i, float v) {
    st_out1(p.out, i, v, p.out_dtype);
    if (p.proj_hi) {
        uint16_t hi, lo;
        split_hilo(as_stored(v, p.out_dtype), p.proj_dt, hi, lo);
        static_cast<uint16_t*>(p.proj_hi)[i] = hi;
        static_cast<uint16_t*>(p.proj_lo)[i] = lo;
    }
}

__device__ __forceinline__ void store_out4(const DecodeParams& p, size_t i, float a, float b, float c, float d) {
    st_out4(p.out, i, a, b, c, d, p.out_dtype);
    if (p.proj_hi) {
        const float v[4] = {a, b, c, d};
        uint16_t hi[4], lo[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) split_hilo(as_stored(v[k], p.out_dtype), p.proj_dt, hi[k], lo[k]);
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.proj_hi) + i) =
            make_uint2(hi[0] | (static_cast<uint32_t>(hi[1]) << 16), hi[2] | (static_cast<uint32_t>(hi[3]) << 16));
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.proj_lo) + i) =
            make_uint2(lo[0] | (static_cast<uint32_t>(lo[1]) << 16), lo[2] | (static_cast<uint32_t>(lo[3]) << 16));
    }
}

// Zero n outputs starting at element i (i and n multiples of 8), by all threads of a block.
__device__ __forceinline__ void zero_out(void* out, size_t i, int n, int dt) {
    const int eb = dt == kF32 ? 4 : 2;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<unsigned char*>(out) + i * eb);
    for (int k = threadIdx.x; k < n * eb / 16; k += blockDim.x) dst[k] = make_uint4(0u, 0u, 0u, 0u);
}

// zero_out of the step's outputs: out, and the projection planes when there is a projection.
__device__ __forceinline__ void zero_outputs(const DecodeParams& p, size_t i, int n) {
    zero_out(p.out, i, n, p.out_dtype);
    if (p.proj_hi) {
        zero_out(p.proj_hi, i, n, kF16);
        zero_out(p.proj_lo, i, n, kF16);
    }
}

// ---------------------------------------------------------------- PTX
// Programmatic dependent launch.  grid_dep_wait blocks until the grid this
// launch was allowed to overlap has finished and its writes are visible (it
// returns at once after an ordinary launch); every global read of the step's
// inputs comes after it.  grid_dep_launch lets the next launch on the stream
// start placing its blocks on SMs this grid frees; those blocks then wait in
// their own grid_dep_wait.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Split-K arrival on a segment counter: an acquire-release add at GPU scope.
// The release publishes the partial that the calling warp or block stored
// before it (those stores are ordered before the caller by a warp or block
// barrier); the acquire orders the merge reads that follow, which the caller
// extends to its warp or block with another barrier.  Unlike a full fence it
// does not wait for every outstanding memory operation of the thread.
__device__ __forceinline__ uint32_t arrive_acq_rel(uint32_t* ctr, uint32_t n) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(ctr), "r"(n) : "memory");
    return old;
}

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

// L2 policy for the K/V stream: each cache row is read once per step, so its
// lines go first when L2 needs room.  The step's small operands (q, k_new,
// v_new, the split-K partials and counters) then stay resident and their loads
// hit L2 instead of waiting behind the stream in HBM.
__device__ __forceinline__ uint64_t l2_stream_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// L2 policy for small operands many blocks read (the output projection's
// activation planes): their lines stay in L2 ahead of streamed data.
__device__ __forceinline__ uint64_t l2_keep_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// bulk_g2s with an L2 cache policy (l2_stream_policy) for the streamed cache rows.
// L2 prefetch of `bytes` contiguous global bytes (16-byte aligned start, size a
// multiple of 16).  A hint: L2 is the coherence point, so lines another kernel is
// still writing are never served stale.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                              uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
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

// Wait for phase `parity` of a barrier; after `limit` SM cycles raise the
// timeout bit and return false instead of spinning forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint32_t* err, long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) {
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
