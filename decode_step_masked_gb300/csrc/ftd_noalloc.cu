// ftd_noalloc.cu -- ftd_decode_mha_noalloc: the decode step without a context
// and without any device allocation.
//
// Who needs it: callers that are not allowed to call cudaMalloc at all, such
// as a plugin running inside a host runtime that owns every byte of device
// memory through its own allocator, or a latency-critical serving loop where
// an allocation (which can synchronise the device and can fail under
// fragmentation) is forbidden after start-up.  They pass the caches, inputs
// and output they already own; the only other memory the step needs -- the
// split-K partials, the per-segment arrival counters and the device error
// word -- lives in g_scratch below, a fixed array in the library's own device
// image that every GPU holds from the moment it loads the library until the
// process exits.
//
// The array is shared by every call on a device and keeps the previous call's
// contents, so each call clears the counters and the error word it needs at
// zero (cudaMemsetAsync on the caller's stream, no allocation).  Calls whose
// kernels overlap in time on one GPU race on the array and give wrong
// results: issue them on one stream, or order their streams with events.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <mutex>
#include <set>

#include "../../include/ftd.h"
#include "ftd_decode_splitk.cuh"
#include "ftd_internal.cuh"

namespace {

// Scratch of the no-allocation entry point (see FTD_NOALLOC_SCRATCH_BYTES).
static __device__ __align__(256) unsigned char g_scratch[FTD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Per-device set-up, done once with the device current: the device address of
// g_scratch (in host code the symbol is only a host-side stand-in, never a
// device address), the SM count, and the kernels whose shared-memory limit
// has been raised on that device.
struct DeviceState {
    bool ready = false;
    unsigned char* scratch = nullptr;
    int sms = 0;
    std::set<const void*> configured;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];

// Host-side failures are described through ftd_last_error(), like every entry point.
ftd_status reject(ftd_status s, const char* msg) {
    char buf[384];
    snprintf(buf, sizeof buf, "ftd_decode_mha_noalloc: %s", msg);
    ftd::set_last_error(buf);
    return s;
}

}  // namespace

extern "C" ftd_status ftd_decode_mha_noalloc(const ftd_config* cfg, const void* q, const void* k_new,
                                             const void* v_new, const void* qkv_bias, void* k_cache,
                                             void* v_cache, const int32_t* seq_lens, float* scales,
                                             void* out, uint32_t* device_err, void* stream) {
    ftd::set_last_error("");
    if (!cfg) return reject(FTD_ERR_INVALID_ARG, "cfg is NULL");
    const ftd_config c = *cfg;
    // the same checks and kernel choice as ftd_init and ftd_decode_mha
    ftd::Plan plan{};
    char msg[256];
    ftd_status st = ftd::plan_config(c, &plan, msg, sizeof msg);
    if (st != FTD_OK) return reject(st, msg);
    if (c.page_size != 0) return reject(FTD_ERR_INVALID_ARG, "paged caches need a context (ftd_init)");
    st = ftd::check_pointers(c, q, k_new, v_new, qkv_bias, seq_lens, k_cache, v_cache, scales, out, msg, sizeof msg);
    if (st != FTD_OK) return reject(st, msg);
    const bool i8 = c.cache_dtype == FTD_I8;
    const int g = c.n_q_heads / c.n_kv_heads;
    const int nq = c.q_len > 1 ? c.q_len : 1;
    const int nhb = plan.nhb;
    const ftd::KernelInfo ki = plan.ki;
    const ftd::TcChoice tcc = plan.tcc;
    const bool use_tc = tcc.tki.fn != nullptr;
    const void* fn = use_tc ? tcc.tki.fn : ki.fn;
    const int smem = use_tc ? tcc.tki.smem : ki.smem;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return reject(FTD_ERR_CUDA, "cudaGetDevice failed");
    DeviceState* ds = &g_devices[dev];
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (!ds->ready) {
            void* p = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
            if (e != cudaSuccess || p == nullptr) return reject(FTD_ERR_CUDA, cudaGetErrorString(e));
            int sms = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess || sms <= 0) return reject(FTD_ERR_CUDA, "cudaDeviceGetAttribute failed");
            ds->scratch = static_cast<unsigned char*>(p);
            ds->sms = sms;
            ds->ready = true;
        }
        if (!ds->configured.count(fn)) {
            if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
                return reject(FTD_ERR_CUDA, "cudaFuncSetAttribute failed");
            ds->configured.insert(fn);
        }
    }

    // Scratch layout: [error word | counters | split-K partial slots], 256-byte aligned parts.
    const size_t n_seg = static_cast<size_t>(c.max_batch) * c.n_kv_heads * (use_tc ? tcc.nhb : nhb);
    const size_t n_slots = n_seg + static_cast<size_t>(ds->sms) * (use_tc ? 1 : ki.warps);
    const size_t cnt_off = 256;
    const size_t ws_off = cnt_off + (n_seg * sizeof(uint32_t) + 255) / 256 * 256;
    const size_t need =
        ws_off + n_slots * static_cast<size_t>(use_tc ? tcc.tki.slot_floats : ki.slot_floats) * sizeof(float);
    if (need > FTD_NOALLOC_SCRATCH_BYTES) {
        char buf[256];
        snprintf(buf, sizeof buf,
                 "this configuration needs %zu bytes of scratch, more than the %u-byte static array; "
                 "use ftd_init / ftd_decode_mha instead",
                 need, static_cast<unsigned>(FTD_NOALLOC_SCRATCH_BYTES));
        return reject(FTD_ERR_INVALID_ARG, buf);
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ds->scratch, 0, ws_off, s) != cudaSuccess)
        return reject(FTD_ERR_CUDA, "clearing the scratch counters failed");

    ftd::DecodeParams p{};
    p.q = q;
    p.k_new = k_new;
    p.v_new = v_new;
    p.bias = qkv_bias;
    p.k_cache = static_cast<unsigned char*>(k_cache);
    p.v_cache = static_cast<unsigned char*>(v_cache);
    const size_t plane = static_cast<size_t>(c.max_batch) * c.n_kv_heads * c.max_len;
    p.k_scales = i8 ? scales : nullptr;
    p.v_scales = i8 ? scales + plane : nullptr;
    p.seq_lens = seq_lens;
    p.out = out;
    p.ws = reinterpret_cast<float*>(ds->scratch + ws_off);
    p.counters = reinterpret_cast<uint32_t*>(ds->scratch + cnt_off);
    p.err = device_err ? device_err : reinterpret_cast<uint32_t*>(ds->scratch);
    p.B = c.max_batch;
    p.Hq = c.n_q_heads;
    p.Hkv = c.n_kv_heads;
    p.Lmax = c.max_len;
    p.group = g;
    p.nhb = nhb;
    p.qkv_dtype = static_cast<int>(c.qkv_dtype);
    const float scale = c.softmax_scale > 0.f ? c.softmax_scale : 1.0f / sqrtf(static_cast<float>(c.head_dim));
    p.qscale = scale * 1.4426950408889634f;
    p.out_dtype = static_cast<int>(c.out_dtype);
    p.window = c.window;
    p.nq = nq;
    p.wait_cycles = ftd::wait_cycles_for(c, dev);
    p.stall = 0;

    cudaError_t e;
    if (use_tc) {
        // tensor maps of the caller's caches, encoded per call on the host (no allocation)
        CUtensorMap tmk, tmv;
        const size_t rows = static_cast<size_t>(c.max_batch) * c.n_kv_heads * c.max_len;
        if (!ftd::encode_tc_cache_map(&tmk, k_cache, c.cache_dtype, rows) ||
            !ftd::encode_tc_cache_map(&tmv, v_cache, c.cache_dtype, rows))
            return reject(FTD_ERR_CUDA, "cuTensorMapEncodeTiled failed for the caches");
        p.nhb = tcc.nhb;
        p.qblk = tcc.qblk;
        void* args[] = {&tmk, &tmv, &p};
        e = cudaLaunchKernel(fn, dim3(ds->sms), dim3(tcc.tki.threads), args, static_cast<size_t>(smem), s);
    } else {
        void* args[] = {&p};
        e = cudaLaunchKernel(fn, dim3(ds->sms), dim3(ki.warps * 32), args, static_cast<size_t>(smem), s);
    }
    if (e != cudaSuccess) return reject(FTD_ERR_CUDA, cudaGetErrorString(e));
    ftd::note_launch();
    return FTD_OK;
}
