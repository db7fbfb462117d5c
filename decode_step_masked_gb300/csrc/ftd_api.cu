// ftd_api.cu -- the C ABI declared in include/ftd.h.
//
// Host side only: argument checks, the single pool allocation made at init
// (the pre-allocated KV-cache buffer of "FasterTransformer source analysis",
// framerc.cn, section 3.2), kernel selection and launch.  Every step of the
// decode path itself runs in the kernels of ftd_decode_splitk.cuh.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "../../include/ftd.h"
#include "ftd_decode_splitk.cuh"
#include "ftd_decode_gqa_tc.cuh"
#include "ftd_internal.cuh"
#include "ftd_decode_wide_tc.cuh"
#include "ftd_out_proj.cuh"

namespace {

thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches{0};
// Live contexts in the order they were initialised; the last one is the current
// context of ftd_decode_mha_current.  The lock also covers that call's launch,
// so ftd_destroy cannot free a context under it.
std::mutex g_live_mutex;
std::vector<ftd_ctx*> g_live;

ftd_status fail(ftd_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
ftd_status fail(ftd_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

ftd_status cuda_fail(cudaError_t e, const char* what) {
    if (e == cudaErrorMemoryAllocation) return fail(FTD_ERR_OOM, "%s: %s", what, cudaGetErrorString(e));
    return fail(FTD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int elem_bytes(ftd_dtype d) {
    switch (d) {
        case FTD_F32: return 4;
        case FTD_F16: return 2;
        case FTD_BF16: return 2;
        case FTD_I8: return 1;
    }
    return 0;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// cuTensorMapEncodeTiled, fetched once through the runtime (no link against libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// 2-D view of a [B][Hkv][Lmax][128] cache as rows of 128 elements, read in
// boxes of 128 rows with the 128-byte swizzle: 64 columns per box for fp16/bf16
// (the tensor-core operand layout), whole 128-byte rows for INT8 (the kernel
// converts those to the operand layout itself).
bool encode_cache_map(CUtensorMap* map, void* base, ftd_dtype dt, size_t rows) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const bool i8 = dt == FTD_I8;
    const cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(i8 ? 128 : 128 * 2)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(i8 ? 128 : 64), 128};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType ty = i8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                      : (dt == FTD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    return fn(map, ty, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D view [rows][cols] of a half-precision matrix (cols contiguous), read in boxes of
// 64 columns x box_rows rows with the 128-byte swizzle, rows past the end read as zero:
// the output projection's weight W [F][K] and its activation planes [tokens][K].
bool encode_rows_map(CUtensorMap* map, const void* base, bool bf16, size_t rows, size_t cols, int box_rows) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
              const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The projection's workspace is one partial slot of ntb x 128 floats per tile and per
// CTA; configurations that would need more than this are refused.
constexpr size_t kMaxProjWorkspace = static_cast<size_t>(256) << 20;

}  // namespace

namespace ftd {
// fp16/bf16 caches with head_dim 128 whose kv heads carry a multiple of 4 query
// rows (group x new tokens) use the tensor-core kernel, in blocks of 16 or 8
// rows (blocks of 4 fill half of an 8-column block, since the MMA needs N >= 16
// with the hi/lo split), or its wide variant in blocks of 64 or 32 rows when the
// rows are a multiple of 32.  INT8 caches with head_dim 128 and a multiple of 8
// query rows per kv head use its INT8 variant, in blocks of 8.
// cfg.kernel == FTD_KERNEL_CUDA_CORE selects the CUDA-core kernel instead.
// Internal to the library (hidden), shared by ftd_init and the no-allocation
// entry point; tki.fn is null when the CUDA-core kernel runs.
__attribute__((visibility("hidden"))) TcChoice choose_tc(const ftd_config& c) {
    TcChoice r{};
    r.nhb = 1;
    r.qblk = 8;
    const int rows_q = (c.q_len > 1 ? c.q_len : 1) * (c.n_q_heads / c.n_kv_heads);
    const bool forced = c.kernel == FTD_KERNEL_CUDA_CORE;
    const bool want_tc = (c.cache_dtype == FTD_F16 || c.cache_dtype == FTD_BF16) && c.head_dim == 128 &&
                         rows_q % 4 == 0 && !forced;
    const bool want_tc_i8 = c.cache_dtype == FTD_I8 && c.head_dim == 128 && rows_q % 8 == 0 && !forced;
    if ((want_tc || want_tc_i8) && encode_tiled()) {
        if (want_tc && rows_q % 32 == 0) {
            // 32 or more query rows per kv head: the wide kernel, all rows of a block of
            // 32 or 64 in one pass per tile
            r.qblk = rows_q % 64 == 0 ? 64 : 32;
            r.tki = select_wide(c.cache_dtype == FTD_BF16, r.qblk, c.q_len > 1);
        } else {
            const int Gt = (rows_q % 16 == 0 && !want_tc_i8) ? 16 : 8;
            r.qblk = rows_q % 8 == 0 ? Gt : 4;
            r.tki = want_tc_i8 ? select_tc_i8(c.q_len > 1) : select_tc(c.cache_dtype == FTD_BF16, Gt, c.q_len > 1);
        }
        r.nhb = rows_q / r.qblk;
    }
    return r;
}

__attribute__((visibility("hidden"))) bool encode_tc_cache_map(CUtensorMap* map, void* base, ftd_dtype dt,
                                                               size_t rows) {
    return encode_cache_map(map, base, dt, rows);
}

// Checks of a configuration shared by every entry point that takes one (ftd_init
// and the no-allocation entry point), and the kernel plan it implies.  On failure
// the message goes to msg.
__attribute__((visibility("hidden"))) ftd_status plan_config(const ftd_config& c, Plan* pl, char* msg, size_t n) {
    auto bad = [&](ftd_status st, const char* fmt, auto... a) {
        if constexpr (sizeof...(a) == 0) snprintf(msg, n, "%s", fmt);
        else snprintf(msg, n, fmt, a...);
        return st;
    };
    if (c.max_batch < 1 || c.max_batch > kMaxBatch)
        return bad(FTD_ERR_INVALID_ARG, "max_batch %d outside 1..%d", c.max_batch, kMaxBatch);
    if (c.n_kv_heads < 1 || c.n_q_heads < c.n_kv_heads || c.n_q_heads % c.n_kv_heads != 0)
        return bad(FTD_ERR_INVALID_ARG, "n_q_heads %d must be a positive multiple of n_kv_heads %d", c.n_q_heads,
                   c.n_kv_heads);
    if (c.max_len < 16 || c.max_len % 16 != 0)
        return bad(FTD_ERR_INVALID_ARG, "max_len %d must be a positive multiple of 16", c.max_len);
    if (c.head_dim <= 0) return bad(FTD_ERR_INVALID_ARG, "head_dim %d", c.head_dim);
    if (c.head_dim != 64 && c.head_dim != 128)
        return bad(FTD_ERR_UNSUPPORTED, "head_dim %d not built (64 or 128)", c.head_dim);
    if (c.qkv_dtype != FTD_F32 && c.qkv_dtype != FTD_F16 && c.qkv_dtype != FTD_BF16)
        return bad(FTD_ERR_UNSUPPORTED, "qkv_dtype %d (F32, F16 or BF16)", static_cast<int>(c.qkv_dtype));
    if (c.cache_dtype != FTD_F32 && c.cache_dtype != FTD_F16 && c.cache_dtype != FTD_BF16 &&
        c.cache_dtype != FTD_I8)
        return bad(FTD_ERR_UNSUPPORTED, "cache_dtype %d", static_cast<int>(c.cache_dtype));
    if (!(c.softmax_scale >= 0.f) || !std::isfinite(c.softmax_scale))
        return bad(FTD_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");
    if (c.out_dtype != FTD_F32 && c.out_dtype != FTD_F16 && c.out_dtype != FTD_BF16)
        return bad(FTD_ERR_UNSUPPORTED, "out_dtype %d (F32, F16 or BF16)", static_cast<int>(c.out_dtype));
    if (c.window < 0) return bad(FTD_ERR_INVALID_ARG, "window %d must be >= 0", c.window);
    if (c.q_len < 0 || c.q_len > kMaxQLen)
        return bad(FTD_ERR_INVALID_ARG, "q_len %d outside 0..%d", c.q_len, kMaxQLen);
    const bool paged = c.page_size != 0;
    if (paged && (c.page_size < 128 || (c.page_size & (c.page_size - 1)) != 0 || c.num_pages < 1))
        return bad(FTD_ERR_INVALID_ARG, "page_size %d must be a power of two >= 128 with num_pages %d >= 1",
                   c.page_size, c.num_pages);
    if (c.kernel != FTD_KERNEL_AUTO && c.kernel != FTD_KERNEL_CUDA_CORE)
        return bad(FTD_ERR_INVALID_ARG, "kernel %d (FTD_KERNEL_AUTO or FTD_KERNEL_CUDA_CORE)", c.kernel);
    if (c.wait_limit_us < 0) return bad(FTD_ERR_INVALID_ARG, "wait_limit_us %d must be >= 0", c.wait_limit_us);
    if (c.proj_dim < 0 || c.proj_dim % 128 != 0 || c.proj_dim > 65536)
        return bad(FTD_ERR_INVALID_ARG, "proj_dim %d must be 0 or a positive multiple of 128 up to 65536", c.proj_dim);
    if (c.proj_dim > 0 && c.qkv_dtype != FTD_F16 && c.qkv_dtype != FTD_BF16)
        return bad(FTD_ERR_UNSUPPORTED, "the output projection needs an F16 or BF16 qkv_dtype (its weight's type)");

    const int g = c.n_q_heads / c.n_kv_heads;
    const int nq = c.q_len > 1 ? c.q_len : 1;
    const int rows_q = nq * g;  // query rows per kv head: every new token's heads of the group
    int G = 8;
    while (rows_q % G) G >>= 1;
    KernelInfo ki{};
    switch (c.cache_dtype) {
        case FTD_F32: ki = select_f32(c.head_dim, G); break;
        case FTD_F16: ki = select_f16(c.head_dim, G); break;
        case FTD_BF16: ki = select_bf16(c.head_dim, G); break;
        case FTD_I8: ki = select_i8(c.head_dim, G); break;
    }
    if (!ki.fn) return bad(FTD_ERR_UNSUPPORTED, "no kernel for this configuration");
    const size_t Hkv = static_cast<size_t>(c.n_kv_heads);
    const size_t rows = paged ? static_cast<size_t>(c.num_pages) * Hkv * c.page_size
                              : static_cast<size_t>(c.max_batch) * Hkv * c.max_len;
    if (rows >= (static_cast<size_t>(1) << 31)) return bad(FTD_ERR_UNSUPPORTED, "cache too large for 32-bit row indices");
    const TcChoice tcc = choose_tc(c);
    // the kernel's tile space (tiles of T rows per segment) and its weighted length (a few
    // tiles more per segment) are indexed with 32-bit integers
    const int T = tcc.tki.fn ? tc::TM : ki.T;
    const long long nhb = tcc.tki.fn ? tcc.nhb : rows_q / G;
    const long long segs = static_cast<long long>(c.max_batch) * c.n_kv_heads * nhb;
    const long long tiles = segs * ((c.max_len + T - 1) / T);
    if (tiles + 8 * segs >= (1LL << 31)) return bad(FTD_ERR_UNSUPPORTED, "cache too large for 32-bit tile indices");
    pl->G = G;
    pl->nhb = rows_q / G;
    pl->ki = ki;
    pl->tcc = tcc;
    pl->rows = rows;
    pl->tokens = c.max_batch * nq;
    pl->ntb = pl->nblk = pl->mtiles = pl->kch = 0;
    if (c.proj_dim > 0) {
        if (!encode_tiled()) return bad(FTD_ERR_UNSUPPORTED, "the output projection needs the tensor-map driver entry point");
        const int t16 = (pl->tokens + 15) / 16 * 16;
        pl->ntb = t16 < op::kMaxNtb ? t16 : op::kMaxNtb;
        pl->nblk = (pl->tokens + pl->ntb - 1) / pl->ntb;
        pl->mtiles = c.proj_dim / op::MT;
        pl->kch = c.n_q_heads * c.head_dim / op::KCH;
        const size_t ws = (static_cast<size_t>(pl->nblk) * pl->mtiles + 1024) * pl->ntb * op::MT * sizeof(float);
        if (ws > kMaxProjWorkspace)
            return bad(FTD_ERR_UNSUPPORTED, "output projection of %d tokens x %d features needs %zu MB of workspace",
                       pl->tokens, c.proj_dim, ws >> 20);
    }
    return FTD_OK;
}

// Pointer checks of a decode call, shared by every decode entry point.  Device
// pointers: caches, scales (INT8) and out 16-byte aligned; q, k_new, v_new and the
// bias aligned to their element size; seq_lens 4-byte aligned.
__attribute__((visibility("hidden"))) ftd_status check_pointers(const ftd_config& c, const void* q, const void* k_new,
                                                                const void* v_new, const void* bias,
                                                                const int32_t* seq_lens, const void* k_cache,
                                                                const void* v_cache, const float* scales,
                                                                const void* out, char* msg, size_t n) {
    if (!q || !k_new || !v_new || !seq_lens || !out || !k_cache || !v_cache) {
        snprintf(msg, n, "q, k_new, v_new, seq_lens, out and the caches must be non-NULL");
        return FTD_ERR_INVALID_ARG;
    }
    const bool i8 = c.cache_dtype == FTD_I8;
    if (i8 && !scales) {
        snprintf(msg, n, "an INT8 cache needs its scales");
        return FTD_ERR_INVALID_ARG;
    }
    if (!aligned16(k_cache) || !aligned16(v_cache) || (i8 && !aligned16(scales)) || !aligned16(out)) {
        snprintf(msg, n, "caches, scales and out must be 16-byte aligned");
        return FTD_ERR_INVALID_ARG;
    }
    const uintptr_t qmask = static_cast<uintptr_t>(elem_bytes(c.qkv_dtype) - 1);
    if ((reinterpret_cast<uintptr_t>(q) & qmask) || (reinterpret_cast<uintptr_t>(k_new) & qmask) ||
        (reinterpret_cast<uintptr_t>(v_new) & qmask) || (reinterpret_cast<uintptr_t>(bias) & qmask) ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3u)) {
        snprintf(msg, n, "q, k_new, v_new, bias, seq_lens must be naturally aligned");
        return FTD_ERR_INVALID_ARG;
    }
    return FTD_OK;
}

// Pipeline wait limit in SM cycles: wait_limit_us at the device's peak SM clock, or the default.
__attribute__((visibility("hidden"))) long long wait_cycles_for(const ftd_config& c, int dev) {
    if (c.wait_limit_us <= 0) return kWaitLimitCycles;
    int khz = 0;
    if (cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev) != cudaSuccess || khz <= 0) {
        cudaGetLastError();
        khz = 2100000;
    }
    const long long cyc = static_cast<long long>(c.wait_limit_us) * (khz / 1000);
    return cyc < kWaitLimitCycles ? cyc : kWaitLimitCycles;
}

// Internal to the library (hidden): used by the no-allocation entry point so its
// failures show in ftd_last_error() and its launches in ftd_kernel_launches().
__attribute__((visibility("hidden"))) void set_last_error(const char* msg) { g_last_error = msg; }
__attribute__((visibility("hidden"))) void note_launch() { g_launches.fetch_add(1); }
}  // namespace ftd

struct ftd_ctx {
    ftd_config cfg;
    int device = 0;
    int grid = 0;
    int G = 1, nhb = 1;
    ftd::KernelInfo ki{};
    bool use_tc = false;       // grouped-query fp16/bf16 caches run on the tensor cores
    ftd::TcKernelInfo tki{};
    int tc_nhb = 1;
    int tc_qblk = 8;         // real query rows per tensor-core block
    CUtensorMap tmk;  // the type carries its own alignment
    CUtensorMap tmv;
    const void* tm_k_base = nullptr;
    const void* tm_v_base = nullptr;
    float qscale = 0.f;
    void* pool = nullptr;
    size_t pool_bytes = 0;
    unsigned char* k_cache = nullptr;
    unsigned char* v_cache = nullptr;
    float* scales = nullptr;
    float* ws = nullptr;
    uint32_t* counters = nullptr;
    size_t n_counters = 0;
    uint32_t* err = nullptr;
    void* st_q = nullptr;
    void* st_k = nullptr;
    void* st_v = nullptr;
    void* st_bias = nullptr;
    int32_t* st_lens = nullptr;
    void* st_out = nullptr;
    // ftd_decode_mha_host: the host buffers of the last call, and their device
    // addresses when they are GPU-addressable pinned memory (null otherwise)
    const void* hp[6] = {};
    void* hd[6] = {};
    size_t q_bytes = 0, kv_new_bytes = 0, bias_bytes = 0, out_bytes = 0;
    size_t rows = 0;         // cache rows (of head_dim elements) in the pool
    int nq = 1;              // new tokens per slot per step
    bool paged = false;
    int pages_per_seq = 0;
    cudaStream_t last_stream = nullptr;
    long long wait_cycles = 0;  // limit of the kernels' pipeline waits
    int stall_calls = 0;        // ftd_debug_stall_next: calls left that withhold a copy
    // output projection (proj_dim > 0)
    ftd::Plan plan{};
    const void* proj_fn = nullptr;
    int proj_smem = 0;
    void* proj_hi = nullptr;    // activation planes [tokens][Hq * D], qkv dtype
    void* proj_lo = nullptr;
    float* proj_ws = nullptr;
    uint32_t* proj_counters = nullptr;
    size_t n_proj_counters = 0;
    CUtensorMap tmph;
    CUtensorMap tmpl;
    CUtensorMap tmw;
    const void* tm_w_base = nullptr;
};

extern "C" {

const char* ftd_status_str(ftd_status s) {
    switch (s) {
        case FTD_OK: return "FTD_OK";
        case FTD_ERR_INVALID_ARG: return "FTD_ERR_INVALID_ARG";
        case FTD_ERR_UNSUPPORTED: return "FTD_ERR_UNSUPPORTED";
        case FTD_ERR_OOM: return "FTD_ERR_OOM";
        case FTD_ERR_CUDA: return "FTD_ERR_CUDA";
        case FTD_ERR_SEQ_OVERFLOW: return "FTD_ERR_SEQ_OVERFLOW";
        case FTD_ERR_DEVICE_TIMEOUT: return "FTD_ERR_DEVICE_TIMEOUT";
        case FTD_ERR_BAD_PAGE: return "FTD_ERR_BAD_PAGE";
    }
    return "FTD_ERR_UNKNOWN";
}

const char* ftd_last_error(void) { return g_last_error.c_str(); }

uint64_t ftd_kernel_launches(void) { return g_launches.load(); }

ftd_status ftd_init(const ftd_config* cfg, void* stream, ftd_ctx** out) {
    g_last_error.clear();
    if (!out) return fail(FTD_ERR_INVALID_ARG, "ftd_init: out is NULL");
    *out = nullptr;
    if (!cfg) return fail(FTD_ERR_INVALID_ARG, "ftd_init: cfg is NULL");
    const ftd_config c = *cfg;
    ftd::Plan plan{};
    char msg[256];
    const ftd_status pst = ftd::plan_config(c, &plan, msg, sizeof msg);
    if (pst != FTD_OK) return fail(pst, "%s", msg);
    const bool paged = c.page_size != 0;
    const int nq = c.q_len > 1 ? c.q_len : 1;
    const int G = plan.G, nhb = plan.nhb;
    const ftd::KernelInfo ki = plan.ki;

    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    e = cudaFuncSetAttribute(ki.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ki.smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");

    const int grid = sms;  // one persistent CTA per SM
    const size_t B = c.max_batch, Hq = c.n_q_heads, Hkv = c.n_kv_heads, D = c.head_dim;
    // cache rows of D elements: [B][Hkv][Lmax] contiguous, or [num_pages][Hkv][page_size] paged
    const size_t rows = plan.rows;
    const size_t cache_bytes = rows * D * elem_bytes(c.cache_dtype);
    const size_t scale_bytes = c.cache_dtype == FTD_I8 ? 2 * rows * sizeof(float) : 0;

    const ftd::TcChoice tcc = plan.tcc;
    const ftd::TcKernelInfo tki = tcc.tki;
    const int tc_nhb = tcc.nhb, tc_qblk = tcc.qblk;
    if (tki.fn) {
        e = cudaFuncSetAttribute(tki.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, tki.smem);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute (tensor-core kernel)");
    }
    const bool use_tc = tki.fn != nullptr;
    const size_t n_seg = use_tc ? B * Hkv * tc_nhb : B * Hkv * nhb;
    const size_t n_slots = n_seg + static_cast<size_t>(grid) * (use_tc ? 1 : ki.warps);
    const size_t ws_bytes = n_slots * (use_tc ? tki.slot_floats : ki.slot_floats) * sizeof(float);
    const int qeb = elem_bytes(c.qkv_dtype);

    ftd_ctx* ctx = new (std::nothrow) ftd_ctx();
    if (!ctx) return fail(FTD_ERR_OOM, "host allocation of the context failed");
    ctx->cfg = c;
    ctx->device = dev;
    ctx->grid = grid;
    ctx->G = G;
    ctx->nhb = nhb;
    ctx->ki = ki;
    ctx->use_tc = use_tc;
    ctx->tki = tki;
    ctx->tc_nhb = tc_nhb;
    ctx->tc_qblk = tc_qblk;
    const float scale = c.softmax_scale > 0.f ? c.softmax_scale : 1.0f / sqrtf(static_cast<float>(D));
    ctx->qscale = scale * 1.4426950408889634f;
    ctx->nq = nq;
    ctx->q_bytes = B * nq * Hq * D * qeb;
    ctx->kv_new_bytes = B * nq * Hkv * D * qeb;
    ctx->bias_bytes = (Hq + 2 * Hkv) * D * qeb;
    ctx->out_bytes = B * nq * Hq * D * static_cast<size_t>(elem_bytes(c.out_dtype));
    ctx->rows = rows;
    ctx->paged = paged;
    ctx->pages_per_seq = paged ? (c.max_len + c.page_size - 1) / c.page_size : 0;
    ctx->n_counters = n_seg;
    ctx->wait_cycles = ftd::wait_cycles_for(c, dev);

    size_t off = 0;
    auto carve = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    const size_t o_k = carve(cache_bytes), o_v = carve(cache_bytes), o_s = carve(scale_bytes);
    const size_t o_cnt = carve(n_seg * sizeof(uint32_t)), o_err = carve(sizeof(uint32_t));
    const bool proj = c.proj_dim > 0;
    const size_t n_pcnt = proj ? static_cast<size_t>(plan.nblk) * plan.mtiles : 0;
    const size_t o_pcnt = carve(n_pcnt * sizeof(uint32_t));
    const size_t zero_end = off;  // caches, scales, counters and the error word start at zero
    const size_t o_ws = carve(ws_bytes);
    const size_t plane_bytes = proj ? static_cast<size_t>(plan.tokens) * Hq * D * 2 : 0;
    const size_t o_ph = carve(plane_bytes), o_pl = carve(plane_bytes);
    const size_t o_pws = carve(proj ? (n_pcnt + static_cast<size_t>(grid)) * plan.ntb * ftd::op::MT * sizeof(float) : 0);
    const size_t o_q = carve(ctx->q_bytes), o_kn = carve(ctx->kv_new_bytes), o_vn = carve(ctx->kv_new_bytes);
    const size_t o_b = carve(ctx->bias_bytes), o_l = carve(B * sizeof(int32_t)), o_o = carve(ctx->out_bytes);
    ctx->pool_bytes = off;

    e = cudaMalloc(&ctx->pool, ctx->pool_bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        delete ctx;
        return cuda_fail(e, "cudaMalloc of the cache pool");
    }
    unsigned char* base = static_cast<unsigned char*>(ctx->pool);
    ctx->k_cache = base + o_k;
    ctx->v_cache = base + o_v;
    ctx->scales = scale_bytes ? reinterpret_cast<float*>(base + o_s) : nullptr;
    ctx->counters = reinterpret_cast<uint32_t*>(base + o_cnt);
    ctx->err = reinterpret_cast<uint32_t*>(base + o_err);
    ctx->ws = reinterpret_cast<float*>(base + o_ws);
    ctx->st_q = base + o_q;
    ctx->st_k = base + o_kn;
    ctx->st_v = base + o_vn;
    ctx->st_bias = base + o_b;
    ctx->st_lens = reinterpret_cast<int32_t*>(base + o_l);
    ctx->st_out = base + o_o;
    ctx->last_stream = static_cast<cudaStream_t>(stream);
    ctx->plan = plan;
    if (proj) {
        ctx->proj_hi = base + o_ph;
        ctx->proj_lo = base + o_pl;
        ctx->proj_ws = reinterpret_cast<float*>(base + o_pws);
        ctx->proj_counters = reinterpret_cast<uint32_t*>(base + o_pcnt);
        ctx->n_proj_counters = n_pcnt;
        ctx->proj_fn = ftd::select_proj(c.qkv_dtype == FTD_BF16).fn;
        ctx->proj_smem = ftd::op::smem_bytes(plan.ntb);
        const bool bf = c.qkv_dtype == FTD_BF16;
        // the limit for the largest token block, so contexts of every size can launch the kernel
        e = cudaFuncSetAttribute(ctx->proj_fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 ftd::op::kStageBudget + 2048);
        if (e != cudaSuccess || !encode_rows_map(&ctx->tmph, ctx->proj_hi, bf, plan.tokens, Hq * D, plan.ntb) ||
            !encode_rows_map(&ctx->tmpl, ctx->proj_lo, bf, plan.tokens, Hq * D, plan.ntb)) {
            cudaFree(ctx->pool);
            delete ctx;
            return e != cudaSuccess ? cuda_fail(e, "cudaFuncSetAttribute (projection kernel)")
                                    : fail(FTD_ERR_CUDA, "cuTensorMapEncodeTiled failed for the projection planes");
        }
    }

    e = cudaMemsetAsync(ctx->pool, 0, zero_end, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaFree(ctx->pool);
        delete ctx;
        return cuda_fail(e, "cudaMemsetAsync of the cache pool");
    }
    *out = ctx;
    {
        std::lock_guard<std::mutex> lock(g_live_mutex);
        g_live.push_back(ctx);
    }
    return FTD_OK;
}

ftd_status ftd_cache_ptrs(ftd_ctx* ctx, void** k_cache, void** v_cache, float** scales) {
    if (!ctx) return fail(FTD_ERR_INVALID_ARG, "ftd_cache_ptrs: ctx is NULL");
    if (k_cache) *k_cache = ctx->k_cache;
    if (v_cache) *v_cache = ctx->v_cache;
    if (scales) *scales = ctx->scales;
    return FTD_OK;
}

// Launch with programmatic stream serialisation: when the previous operation on
// the stream is a kernel, this grid's blocks may be placed while it drains and
// wait in griddepcontrol.wait (the kernels' grid_dep_wait) for its completion,
// which hides the launch gap between back-to-back decode steps.
static cudaError_t launch_overlapped(const void* fn, int grid, int threads, int smem, void** args,
                                     cudaStream_t stream) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

static ftd_status launch_decode(ftd_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                                const void* bias, void* k_cache, void* v_cache, const int32_t* block_table,
                                const int32_t* seq_lens, float* scales, void* out, cudaStream_t stream,
                                bool proj = false) {
    if (!k_cache) k_cache = ctx->k_cache;
    if (!v_cache) v_cache = ctx->v_cache;
    const bool i8 = ctx->cfg.cache_dtype == FTD_I8;
    if (i8 && !scales) scales = ctx->scales;
    char msg[160];
    const ftd_status cst = ftd::check_pointers(ctx->cfg, q, k_new, v_new, bias, seq_lens, k_cache, v_cache, scales,
                                               out, msg, sizeof msg);
    if (cst != FTD_OK) return fail(cst, "%s", msg);

    const ftd_config& c = ctx->cfg;
    ftd::DecodeParams p{};
    p.q = q;
    p.k_new = k_new;
    p.v_new = v_new;
    p.bias = bias;
    p.k_cache = static_cast<unsigned char*>(k_cache);
    p.v_cache = static_cast<unsigned char*>(v_cache);
    if (ctx->paged && (!block_table || (reinterpret_cast<uintptr_t>(block_table) & 3u)))
        return fail(FTD_ERR_INVALID_ARG, "a paged context needs a 4-byte aligned block table");
    const size_t plane = ctx->rows;
    p.k_scales = i8 ? scales : nullptr;
    p.v_scales = i8 ? scales + plane : nullptr;
    p.seq_lens = seq_lens;
    p.out = out;
    p.ws = ctx->ws;
    p.counters = ctx->counters;
    p.err = ctx->err;
    p.B = c.max_batch;
    p.Hq = c.n_q_heads;
    p.Hkv = c.n_kv_heads;
    p.Lmax = c.max_len;
    p.group = c.n_q_heads / c.n_kv_heads;
    p.nhb = ctx->nhb;
    p.qkv_dtype = static_cast<int>(c.qkv_dtype);
    p.qscale = ctx->qscale;
    p.out_dtype = static_cast<int>(c.out_dtype);
    p.window = c.window;
    p.nq = ctx->nq;
    p.block_table = ctx->paged ? block_table : nullptr;
    p.pages_per_seq = ctx->pages_per_seq;
    p.page_shift = 0;
    while (ctx->paged && (1 << p.page_shift) < c.page_size) ++p.page_shift;
    p.num_pages = c.num_pages;
    p.wait_cycles = ctx->wait_cycles;
    p.proj_hi = proj ? ctx->proj_hi : nullptr;
    p.proj_lo = proj ? ctx->proj_lo : nullptr;
    p.proj_dt = c.qkv_dtype == FTD_BF16 ? ftd::kBF16 : ftd::kF16;
    p.stall = 0;
    if (ctx->stall_calls > 0) {
        p.stall = 1;
        --ctx->stall_calls;
    }

    cudaError_t e;
    if (ctx->use_tc) {
        const size_t rows = ctx->rows;
        if (ctx->tm_k_base != k_cache) {
            if (!encode_cache_map(&ctx->tmk, k_cache, c.cache_dtype, rows))
                return fail(FTD_ERR_CUDA, "cuTensorMapEncodeTiled failed for k_cache");
            ctx->tm_k_base = k_cache;
        }
        if (ctx->tm_v_base != v_cache) {
            if (!encode_cache_map(&ctx->tmv, v_cache, c.cache_dtype, rows))
                return fail(FTD_ERR_CUDA, "cuTensorMapEncodeTiled failed for v_cache");
            ctx->tm_v_base = v_cache;
        }
        p.nhb = ctx->tc_nhb;
        p.qblk = ctx->tc_qblk;
        void* args[] = {&ctx->tmk, &ctx->tmv, &p};
        e = launch_overlapped(ctx->tki.fn, ctx->grid, ctx->tki.threads, ctx->tki.smem, args, stream);
    } else {
        void* args[] = {&p};
        e = launch_overlapped(ctx->ki.fn, ctx->grid, ctx->ki.warps * 32, ctx->ki.smem, args, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
    g_launches.fetch_add(1);
    ctx->last_stream = stream;
    return FTD_OK;
}

ftd_status ftd_decode_mha(ftd_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                          const void* qkv_bias, void* k_cache, void* v_cache, const int32_t* seq_lens,
                          float* scales, void* out, void* stream) {
    g_last_error.clear();
    if (!ctx) return fail(FTD_ERR_INVALID_ARG, "ftd_decode_mha: ctx is NULL");
    if (ctx->paged) return fail(FTD_ERR_INVALID_ARG, "the context is paged: use ftd_decode_mha_paged");
    return launch_decode(ctx, q, k_new, v_new, qkv_bias, k_cache, v_cache, nullptr, seq_lens, scales, out,
                         static_cast<cudaStream_t>(stream));
}

ftd_status ftd_decode_mha_current(const void* q, const void* k_new, const void* v_new, const void* qkv_bias,
                                  void* k_cache, void* v_cache, const int32_t* seq_lens, float* scales, void* out,
                                  void* stream) {
    std::lock_guard<std::mutex> lock(g_live_mutex);  // ftd_destroy waits until the launch is done
    ftd_ctx* ctx = g_live.empty() ? nullptr : g_live.back();
    if (!ctx) return fail(FTD_ERR_INVALID_ARG, "ftd_decode_mha_current: no context (ftd_init first)");
    return ftd_decode_mha(ctx, q, k_new, v_new, qkv_bias, k_cache, v_cache, seq_lens, scales, out, stream);
}

ftd_status ftd_decode_mha_paged(ftd_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                                const void* qkv_bias, void* k_pages, void* v_pages, const int32_t* block_table,
                                const int32_t* seq_lens, float* scales, void* out, void* stream) {
    g_last_error.clear();
    if (!ctx) return fail(FTD_ERR_INVALID_ARG, "ftd_decode_mha_paged: ctx is NULL");
    if (!ctx->paged) return fail(FTD_ERR_INVALID_ARG, "the context is not paged (page_size 0)");
    return launch_decode(ctx, q, k_new, v_new, qkv_bias, k_pages, v_pages, block_table, seq_lens, scales, out,
                         static_cast<cudaStream_t>(stream));
}

ftd_status ftd_decode_mha_proj(ftd_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                               const void* qkv_bias, void* k_cache, void* v_cache, const int32_t* seq_lens,
                               float* scales, void* out, const void* w_o, void* y, void* stream) {
    g_last_error.clear();
    if (!ctx) return fail(FTD_ERR_INVALID_ARG, "ftd_decode_mha_proj: ctx is NULL");
    if (ctx->cfg.proj_dim <= 0) return fail(FTD_ERR_INVALID_ARG, "the context has no output projection (proj_dim 0)");
    if (ctx->paged) return fail(FTD_ERR_INVALID_ARG, "ftd_decode_mha_proj serves contiguous caches only");
    if (!w_o || !y || !aligned16(w_o) || !aligned16(y))
        return fail(FTD_ERR_INVALID_ARG, "w_o and y must be non-NULL and 16-byte aligned");
    const ftd_config& c = ctx->cfg;
    const ftd::Plan& pl = ctx->plan;
    if (ctx->tm_w_base != w_o) {
        if (!encode_rows_map(&ctx->tmw, w_o, c.qkv_dtype == FTD_BF16, static_cast<size_t>(c.proj_dim),
                             static_cast<size_t>(c.n_q_heads) * c.head_dim, ftd::op::MT))
            return fail(FTD_ERR_CUDA, "cuTensorMapEncodeTiled failed for w_o");
        ctx->tm_w_base = w_o;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const ftd_status st = launch_decode(ctx, q, k_new, v_new, qkv_bias, k_cache, v_cache, nullptr, seq_lens, scales,
                                        out, s, true);
    if (st != FTD_OK) return st;
    ftd::ProjParams pp{};
    pp.y = y;
    pp.ws = ctx->proj_ws;
    pp.counters = ctx->proj_counters;
    pp.err = ctx->err;
    pp.tokens = pl.tokens;
    pp.ntb = pl.ntb;
    pp.nblk = pl.nblk;
    pp.mtiles = pl.mtiles;
    pp.kch = pl.kch;
    pp.out_dtype = static_cast<int>(c.out_dtype);
    pp.wait_cycles = ctx->wait_cycles;
    void* args[] = {&ctx->tmw, &ctx->tmph, &ctx->tmpl, &pp};
    const cudaError_t e = launch_overlapped(ctx->proj_fn, ctx->grid, ftd::op::kThreads, ctx->proj_smem, args, s);
    if (e != cudaSuccess) return cuda_fail(e, "projection kernel launch");
    g_launches.fetch_add(1);
    return FTD_OK;
}

// Device address of host pointer p when the GPU can address it (pinned and mapped), else null.
static void* device_alias(const void* p) {
    if (!p) return nullptr;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

ftd_status ftd_decode_mha_host(ftd_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                               const void* qkv_bias, void* k_cache, void* v_cache, const int32_t* seq_lens,
                               float* scales, void* out, void* stream) {
    g_last_error.clear();
    if (!ctx) return fail(FTD_ERR_INVALID_ARG, "ftd_decode_mha_host: ctx is NULL");
    if (ctx->paged) return fail(FTD_ERR_INVALID_ARG, "ftd_decode_mha_host serves contiguous caches only");
    if (!q || !k_new || !v_new || !seq_lens || !out)
        return fail(FTD_ERR_INVALID_ARG, "q, k_new, v_new, seq_lens and out must be non-NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t B = ctx->cfg.max_batch;
    cudaError_t e;

    // Pinned, GPU-addressable host buffers (looked up once per set of pointers): the
    // decode kernel reads the inputs in place (on Grace systems across NVLink-C2C;
    // each q, k_new and v_new row is read by the few workers of its segment) and
    // writes out straight to the host, so a step is one launch and no copy call.
    const void* hp[6] = {q, k_new, v_new, qkv_bias, seq_lens, out};
    bool same = true;
    for (int i = 0; i < 6; ++i) same = same && hp[i] == ctx->hp[i];
    if (!same) {
        for (int i = 0; i < 6; ++i) {
            ctx->hp[i] = hp[i];
            ctx->hd[i] = device_alias(hp[i]);
        }
    }
    bool direct = true;
    for (int i = 0; i < 6; ++i) {
        if (i == 3 && !qkv_bias) continue;
        const uintptr_t a = reinterpret_cast<uintptr_t>(ctx->hd[i]);
        direct = direct && a != 0 && (a & (i == 4 ? 3u : 15u)) == 0;
    }
    if (direct) {
        ftd_status st = launch_decode(ctx, ctx->hd[0], ctx->hd[1], ctx->hd[2], qkv_bias ? ctx->hd[3] : nullptr,
                                      k_cache, v_cache, nullptr, static_cast<const int32_t*>(ctx->hd[4]), scales,
                                      ctx->hd[5], s);
        if (st != FTD_OK) return st;
        e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
        return FTD_OK;
    }

    // Pageable (or unaligned) host buffers: copies through the staging buffers.
    if ((e = cudaMemcpyAsync(ctx->st_q, q, ctx->q_bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(ctx->st_k, k_new, ctx->kv_new_bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(ctx->st_v, v_new, ctx->kv_new_bytes, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(ctx->st_lens, seq_lens, B * sizeof(int32_t), cudaMemcpyHostToDevice, s)) !=
            cudaSuccess)
        return cuda_fail(e, "host-to-device copy of the step inputs");
    if (qkv_bias) {
        e = cudaMemcpyAsync(ctx->st_bias, qkv_bias, ctx->bias_bytes, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy of the bias");
    }
    ftd_status st = launch_decode(ctx, ctx->st_q, ctx->st_k, ctx->st_v, qkv_bias ? ctx->st_bias : nullptr,
                                  k_cache, v_cache, nullptr, ctx->st_lens, scales, ctx->st_out, s);
    if (st != FTD_OK) return st;
    e = cudaMemcpyAsync(out, ctx->st_out, ctx->out_bytes, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy of the output");
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    return FTD_OK;
}

ftd_status ftd_get_error(ftd_ctx* ctx) {
    g_last_error.clear();
    if (!ctx) return fail(FTD_ERR_INVALID_ARG, "ftd_get_error: ctx is NULL");
    cudaError_t e = cudaStreamSynchronize(ctx->last_stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    uint32_t h = 0;
    e = cudaMemcpy(&h, ctx->err, sizeof h, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (!h) return FTD_OK;
    e = cudaMemset(ctx->err, 0, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
    if (h & ftd::kErrTimeout) {
        // an abandoned launch may have left segment counters part-way; restart them
        e = cudaMemset(ctx->counters, 0, ctx->n_counters * sizeof(uint32_t));
        if (e == cudaSuccess && ctx->n_proj_counters)
            e = cudaMemset(ctx->proj_counters, 0, ctx->n_proj_counters * sizeof(uint32_t));
        if (e != cudaSuccess) return cuda_fail(e, "clearing the split-K counters");
        return fail(FTD_ERR_DEVICE_TIMEOUT, "a decode kernel gave up waiting for a copy");
    }
    if (h & ftd::kErrBadPage)
        return fail(FTD_ERR_BAD_PAGE, "a block-table entry was outside [0, num_pages); those slots are undefined");
    return fail(FTD_ERR_SEQ_OVERFLOW, "some seq_lens[b] + q_len > max_len; those slots were skipped");
}

ftd_status ftd_debug_stall_next(ftd_ctx* ctx, int calls) {
    g_last_error.clear();
    if (!ctx) return fail(FTD_ERR_INVALID_ARG, "ftd_debug_stall_next: ctx is NULL");
    if (calls < 0) return fail(FTD_ERR_INVALID_ARG, "ftd_debug_stall_next: calls %d must be >= 0", calls);
    ctx->stall_calls = calls;
    return FTD_OK;
}

void ftd_destroy(ftd_ctx* ctx) {
    if (!ctx) return;
    {
        std::lock_guard<std::mutex> lock(g_live_mutex);
        for (size_t i = 0; i < g_live.size(); ++i)
            if (g_live[i] == ctx) {
                g_live.erase(g_live.begin() + static_cast<long>(i));
                break;
            }
    }
    cudaDeviceSynchronize();
    cudaFree(ctx->pool);
    delete ctx;
}

}  // extern "C"
