/*
 * ftd.h -- C ABI of the GB300 masked multi-head attention decode step.
 *
 * One call performs one decode step of masked multi-head attention for every
 * slot of a continuous batch, entirely in hand-written sm_103a kernels:
 *
 *   1. fused QKV bias add           q' = q + b_q, k' = k_new + b_k, v' = v_new + b_v
 *                                   (FasterTransformer practice notes, lpnh.cn,
 *                                   section 2.1: the projection output is split
 *                                   into Q/K/V and the bias is added in the fused
 *                                   attention kernel, with no extra HBM round trip)
 *   2. KV-cache append              K[b, h, L_b, :] = round(k'), V likewise
 *                                   (lpnh.cn section 2.2: a pre-allocated cache the
 *                                   new K/V is appended to at every token;
 *                                   "FasterTransformer source analysis",
 *                                   framerc.cn, section 3.2: one buffer sized for
 *                                   the preset maximum length, shared by offset)
 *   3. scores over the whole cache  s_t = scale * q' . K[t],  t = 0 .. L_b
 *   4. masked, stable softmax       p = softmax(s) over t <= L_b (the current
 *                                   position; nothing after it is visible)
 *   5. weighted sum                 o = sum_t p_t V[t]
 *   6. split-K merge                partial (max, sum, o) of several thread
 *                                   blocks combined by log-sum-exp ("10 tricks
 *                                   for Transformer throughput", pptc.cn,
 *                                   section 2.2: online softmax statistics, no
 *                                   N x N matrix in memory)
 *
 * with ragged per-slot lengths (intelliparadigm.com section 3.2, continuous
 * batching), grouped / multi-query heads (pptc.cn section 3.4: query head h
 * reads kv head h / (Hq / Hkv)) and an INT8 cache with an fp32 scale per
 * (slot, kv head, position) (pptc.cn section 3.1).
 *
 * Four options the pages name next to the step:
 *  - out_dtype F16 / BF16: the output is rounded once, to nearest even, from
 *    the fp32 result, in the precision the following projection reads
 *    (lpnh.cn section 2.1: the fused kernels run in half precision).
 *  - window W > 0: sliding-window attention, slot b attends to positions
 *    max(0, L_b + 1 - W) .. L_b only (pptc.cn section 3.1: keep only the
 *    recent part of the history in the cache).
 *  - page_size > 0: a paged cache (intelliparadigm.com section 5.1: the cache
 *    cut into fixed pages, e.g. 256 tokens each; framerc.cn section 3.2:
 *    fixed-size blocks mapped like a virtual-memory page table): the cache is
 *    a pool of pages and a per-slot block table maps positions to pages;
 *    served by ftd_decode_mha_paged.
 *  - q_len T > 1: T new tokens per slot in one step, as a speculative
 *    verification pass checks a run of draft tokens (pptc.cn section 4.3).
 *    Token j of slot b is appended at position L_b + j and its query attends
 *    to positions 0 .. L_b + j (with a window, the last W of them).  The
 *    caller then advances seq_lens[b] by the number of tokens it accepts;
 *    rows written past that are overwritten by the next step.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - B = max_batch, Hq = n_q_heads, Hkv = n_kv_heads, D = head_dim,
 *    Lmax = max_len.  L_b = seq_lens[b] is the number of tokens already in
 *    the cache for slot b; the new token is written at position L_b and
 *    attends to positions 0 .. L_b inclusive.
 *  - Layouts are dense and row-major (T = q_len, 1 unless set):
 *        q      [B][T][Hq][D]     qkv dtype
 *        k_new  [B][T][Hkv][D]    qkv dtype      v_new likewise
 *        bias   [(Hq + 2*Hkv)*D]  qkv dtype, the q part, then k, then v
 *        cache  [B][Hkv][Lmax][D] cache dtype    (k_cache, v_cache)
 *        scales [2][B][Hkv][Lmax] fp32, plane 0 for K and plane 1 for V
 *                                 (INT8 caches only)
 *        out    [B][T][Hq][D]     out_dtype (fp32 unless the config says)
 *    A paged context replaces the cache and scale layouts by
 *        pages  [num_pages][Hkv][page_size][D]  cache dtype (k_pages, v_pages)
 *        scales [2][num_pages][Hkv][page_size]  fp32 (INT8 caches only)
 *        block_table [B][ceil(Lmax / page_size)] int32: entry i of slot b is
 *               the page holding positions i*page_size .. (i+1)*page_size - 1.
 *  - Slots with seq_lens[b] < 0 are inactive: their cache is untouched and
 *    their output is zero.  seq_lens[b] + T > Lmax is an overflow: the slot is
 *    skipped the same way and a sticky device error is raised, which
 *    ftd_get_error() reports as FTD_ERR_SEQ_OVERFLOW.  Nothing traps.
 *  - Device pointers must be 16-byte aligned.  All device work goes to the
 *    caller's stream (a cudaStream_t passed as void*; NULL = legacy default
 *    stream) and is asynchronous; the decode entry points never allocate.
 *  - The caller advances seq_lens after a step; the library never writes it.
 *  - Errors found on the host return synchronously and leave the device
 *    untouched.  ftd_last_error() describes the most recent one.
 */
#ifndef FTD_H
#define FTD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FTD_OK = 0,
    FTD_ERR_INVALID_ARG = 1,     /* null pointer, bad size, misaligned pointer */
    FTD_ERR_UNSUPPORTED = 2,     /* dtype / head_dim combination not built */
    FTD_ERR_OOM = 3,             /* ftd_init could not allocate its pool */
    FTD_ERR_CUDA = 4,            /* a CUDA runtime call failed */
    FTD_ERR_SEQ_OVERFLOW = 5,    /* some seq_lens[b] + q_len > max_len in a past call */
    FTD_ERR_DEVICE_TIMEOUT = 6,  /* a kernel gave up waiting for a copy (bounded wait) */
    FTD_ERR_BAD_PAGE = 7         /* a block-table entry read in a past call was outside [0, num_pages) */
} ftd_status;

typedef enum { FTD_F32 = 0, FTD_F16 = 1, FTD_BF16 = 2, FTD_I8 = 3 } ftd_dtype;

typedef struct {
    int max_batch;       /* B, 1 .. 1024 */
    int n_q_heads;       /* Hq, a multiple of n_kv_heads */
    int n_kv_heads;      /* Hkv >= 1 (Hkv == Hq: MHA, Hkv == 1: MQA) */
    int head_dim;        /* D: 64 or 128 */
    int max_len;         /* Lmax: a multiple of 16 */
    ftd_dtype qkv_dtype;   /* q, k_new, v_new, bias: F32, F16 or BF16 */
    ftd_dtype cache_dtype; /* F32, F16, BF16 or I8 */
    float softmax_scale;   /* 0 selects 1/sqrt(head_dim) */
    /* Options; an all-zero tail gives the plain step (fp32 out, full context,
     * contiguous cache). */
    ftd_dtype out_dtype;   /* F32 (0), F16 or BF16 */
    int window;            /* 0: whole context; W > 0: the last W positions */
    int page_size;         /* 0: contiguous cache; else a power of two >= 128 */
    int num_pages;         /* pages in the pool when page_size > 0 */
    int q_len;             /* new tokens per slot per step, 0 or 1 .. 64 (0 = 1) */
    int kernel;            /* FTD_KERNEL_AUTO (0): the library's choice;
                              FTD_KERNEL_CUDA_CORE (1): the CUDA-core split-K kernel
                              for every configuration (the tensor-core kernel is
                              otherwise taken for head_dim 128 caches whose kv heads
                              carry a multiple of 4 query rows, 8 for INT8) */
    int proj_dim;          /* 0: no output projection; F > 0 (a multiple of 128): the
                              context also serves ftd_decode_mha_proj, y = out . W_o^T
                              with W_o [F][n_q_heads * head_dim] (F16 / BF16 qkv only) */
    int wait_limit_us;     /* 0: a kernel's bounded waits give up after about 2 s;
                              else after this many microseconds (measured in SM clock
                              cycles at the device's peak clock), raising
                              FTD_ERR_DEVICE_TIMEOUT.  The drain of copies still in
                              flight after such an abort always keeps the 2 s limit. */
} ftd_config;

enum { FTD_KERNEL_AUTO = 0, FTD_KERNEL_CUDA_CORE = 1 };

typedef struct ftd_ctx ftd_ctx;

/*
 * ftd_init -- validate cfg and pre-allocate the cache pool.
 * One cudaMalloc on the current device holds the K and V caches (zeroed; for
 * a paged context, num_pages pages of each),
 * the INT8 scale planes, the split-K workspace, the sticky error word and the
 * staging buffers of ftd_decode_mha_host.  Zeroing runs on `stream`.
 * The pool is the pre-allocated buffer of framerc.cn section 3.2 (allocated
 * once for max_batch x max_len, requests share it by offset, no resize).
 * On success *out owns the pool until ftd_destroy.  Returns INVALID_ARG,
 * UNSUPPORTED, OOM or CUDA on failure, with *out set to NULL.
 */
ftd_status ftd_init(const ftd_config* cfg, void* stream, ftd_ctx** out);

/*
 * ftd_cache_ptrs -- device addresses of the context's own pool: the K and V
 * caches [B][Hkv][Lmax][D] (pages for a paged context) and the INT8 scale
 * planes, i.e. the per-sequence cache pointers of the decoding state that
 * intelliparadigm.com section 3.2 keeps for each request, and the buffer that
 * framerc.cn section 3.2 pre-allocates once.  Any output pointer may be NULL.
 * *scales is NULL unless the cache is INT8.  The caller may fill the cache
 * (prefill) through these pointers.  Returns INVALID_ARG for a NULL ctx.
 */
ftd_status ftd_cache_ptrs(ftd_ctx* ctx, void** k_cache, void** v_cache, float** scales);

/*
 * ftd_decode_mha -- one decode step for all max_batch slots (device buffers).
 *   q, k_new, v_new : device, caller-owned, qkv dtype, layouts above.
 *   qkv_bias        : device or NULL (no bias).
 *   k_cache, v_cache: device caches with the layout above, read and appended
 *                     to in place; NULL selects the context's own pool.
 *   seq_lens        : device int32 [B]; read only.
 *   scales          : device fp32 [2][B][Hkv][Lmax] for INT8 caches (NULL
 *                     selects the pool's planes); ignored otherwise.
 *   out             : device [B][T][Hq][D] of out_dtype; every element is written.
 *   stream          : cudaStream_t as void*.
 * Launches one kernel; no host synchronisation and no allocation.  Two calls
 * on the same context must not overlap in time (they share the workspace):
 * issue them on one stream, or order their streams with events.
 * The kernel is launched with programmatic dependent launch: it may start
 * while the preceding kernel on the stream finishes, if that kernel allows
 * it (this library's decode kernels do, right after their own start).  Before
 * it waits for that kernel it reads only seq_lens, to plan its work and to
 * prefetch cache lines into L2 (always safe); after the wait it reads seq_lens
 * again and re-plans if they changed, so a preceding kernel may write seq_lens
 * (for example the caller's seq_lens += accepted kernel).
 * A paged context (page_size > 0) is refused with INVALID_ARG.
 */
ftd_status ftd_decode_mha(ftd_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                          const void* qkv_bias, void* k_cache, void* v_cache,
                          const int32_t* seq_lens, float* scales, void* out, void* stream);

/*
 * ftd_decode_mha_current -- ftd_decode_mha with the specified ten-argument
 * signature (no context handle): it runs on the most recently initialised
 * context that has not been destroyed (destroying it makes the one initialised
 * before it current again), and returns FTD_ERR_INVALID_ARG when there is
 * none.  It holds a library lock while it launches, so an ftd_destroy in
 * another thread waits for it.  For a process that holds one context; with
 * several, pass the handle to ftd_decode_mha instead.
 */
ftd_status ftd_decode_mha_current(const void* q, const void* k_new, const void* v_new, const void* qkv_bias,
                                  void* k_cache, void* v_cache, const int32_t* seq_lens, float* scales,
                                  void* out, void* stream);

/*
 * ftd_decode_mha_paged -- ftd_decode_mha over a paged cache (intelliparadigm.com
 * section 5.1, framerc.cn section 3.2: the cache is cut into fixed-size pages
 * and a block table maps each slot's positions to pages, so the pool holds
 * the pages in use rather than max_batch x max_len).
 *   k_pages, v_pages: device pages [num_pages][Hkv][page_size][D]; NULL
 *                     selects the context's own pool.
 *   block_table     : device int32 [B][ceil(max_len / page_size)], read only;
 *                     only entries covering positions 0 .. L_b of active
 *                     slots are read (the window start's page and on, when a
 *                     window is set).  The new token goes to position L_b of
 *                     its page.  Pages must not be shared between the
 *                     positions that two slots write.
 *   scales          : device fp32 [2][num_pages][Hkv][page_size] (INT8), NULL
 *                     selects the pool's planes.
 * Other arguments as in ftd_decode_mha.  An entry outside [0, num_pages)
 * raises a sticky device error (FTD_ERR_BAD_PAGE from ftd_get_error); the
 * kernel then reads nothing through it and writes no cache row for it, and
 * the output of that slot is undefined.  Refused (INVALID_ARG) on a context
 * without pages.
 */
ftd_status ftd_decode_mha_paged(ftd_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                                const void* qkv_bias, void* k_pages, void* v_pages,
                                const int32_t* block_table, const int32_t* seq_lens, float* scales,
                                void* out, void* stream);

/*
 * ftd_decode_mha_proj -- ftd_decode_mha followed, in the same call and on the
 * same stream, by the output projection of the step's result (the fused
 * kernels hand their output straight to the next projection in half
 * precision, "FasterTransformer practice", lpnh.cn, section 2.1):
 *     y[b][t][f] = sum_k W_o[f][k] * out[b][t][k],   k < n_q_heads * head_dim,
 * out taken as stored (its out_dtype) and flattened over heads.  The decode
 * kernel's final stores also write each output value as a high and a low half
 * of W_o's type into two planes of the context, so the product keeps about 16
 * mantissa bits of an fp32 out; a second kernel, a tcgen05 GEMM that reads W_o
 * once, starts while the decode kernel's last blocks finish (programmatic
 * dependent launch) and writes y.
 *   w_o : device [proj_dim][n_q_heads * head_dim] in the qkv dtype (F16 or
 *         BF16; the layout of a linear layer's weight), 16-byte aligned, read only.
 *   y   : device [B][T][proj_dim] of out_dtype, 16-byte aligned; every element
 *         is written (zero for inactive and overflowing slots).
 * Other arguments as in ftd_decode_mha; out is written as well.  Needs a
 * context with proj_dim > 0 and a contiguous cache (INVALID_ARG otherwise).
 * Launches two kernels; no host synchronisation and no allocation.
 */
ftd_status ftd_decode_mha_proj(ftd_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                               const void* qkv_bias, void* k_cache, void* v_cache, const int32_t* seq_lens,
                               float* scales, void* out, const void* w_o, void* y, void* stream);

/*
 * ftd_decode_mha_host -- the same step for callers whose per-step inputs live
 * in host memory (the host input-id update, kernel launches and device-to-host
 * read of the output that one decode step makes in lmnt.cn section 3.3).  q, k_new, v_new, qkv_bias (nullable), seq_lens and out are
 * HOST pointers; the caches stay on the device as in ftd_decode_mha (NULL =
 * the pool).  When every one of them is pinned, GPU-addressable memory
 * (cudaHostAlloc / cudaHostRegister; 16-byte aligned, seq_lens 4-byte) the
 * decode kernel reads the inputs in place and writes out straight into the
 * host buffer (one launch, no copy calls; on Grace systems both cross
 * NVLink-C2C).  The buffers must not change until the call returns.
 * Otherwise the inputs are copied in and out is copied back with
 * cudaMemcpyAsync.  Either way the call synchronises `stream` before it
 * returns, so out is valid on return.  Contiguous contexts only.
 */
ftd_status ftd_decode_mha_host(ftd_ctx* ctx, const void* q, const void* k_new, const void* v_new,
                               const void* qkv_bias, void* k_cache, void* v_cache,
                               const int32_t* seq_lens, float* scales, void* out, void* stream);

/*
 * ftd_get_error -- synchronise the stream of the context's last call, then
 * read and clear the sticky device error word.  A sequence that outgrows the
 * pre-allocated length is an error the caller must see, not a silent
 * overwrite (framerc.cn section 3.2; lmnt.cn section 5.2); the kernels skip
 * such a slot and set the word instead of trapping.  Returns FTD_OK,
 * FTD_ERR_SEQ_OVERFLOW, FTD_ERR_BAD_PAGE, FTD_ERR_DEVICE_TIMEOUT or
 * FTD_ERR_CUDA (the most serious first when several bits are set).  After a
 * timeout it also resets the split-K counters, so the next call starts clean.
 */
ftd_status ftd_get_error(ftd_ctx* ctx);

/* ftd_destroy -- free the pool (synchronises the device first).  NULL is a
 * no-op.  The context must not be in use by another thread's call; if it is
 * the current context of ftd_decode_mha_current, the most recently initialised
 * of the remaining live contexts becomes current. */
void ftd_destroy(ftd_ctx* ctx);

/* ftd_status_str -- static name of a status code. */
const char* ftd_status_str(ftd_status s);

/* ftd_last_error -- text of the most recent host-side error in this thread ("" if none). */
const char* ftd_last_error(void);

/* ftd_kernel_launches -- number of kernels this library has launched in this
 * process (every decode call adds one; host-side failures add none). */
uint64_t ftd_kernel_launches(void);

/*
 * ftd_debug_stall_next -- test hook for the bounded-wait error path; the pages
 * have no counterpart.  The next `calls` decode calls on ctx withhold the first
 * tile copy of block 0, so that block's waits run out after the context's
 * wait_limit_us, it drains what it has in flight and returns, and
 * ftd_get_error reports FTD_ERR_DEVICE_TIMEOUT (and resets the counters).
 * Outputs of such a call are undefined.  Nothing faults and nothing hangs:
 * every wait is bounded.  calls = 0 cancels.
 */
ftd_status ftd_debug_stall_next(ftd_ctx* ctx, int calls);

/*
 * ftd_debug_late_lengths -- test hook for the decode kernels' re-planning path;
 * the pages have no counterpart.  Launches, on `stream`, one small kernel that
 * at once allows the next launch on the stream to start (programmatic
 * dependent launch), waits about delay_us microseconds and then copies n int32
 * lengths from src to dst (both device pointers).  A decode call issued right
 * after it on the same stream with seq_lens = dst therefore plans its split
 * from the old lengths and must notice, after its wait, that they changed.
 * n is 1 .. 1024 and delay_us 0 .. 1e6; the kernel's wait is bounded by delay_us.
 */
ftd_status ftd_debug_late_lengths(const int32_t* src, int32_t* dst, int n, int delay_us, void* stream);

/* Size of the fixed device array that ftd_decode_mha_noalloc uses as scratch. */
#define FTD_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * ftd_decode_mha_noalloc -- the decode step of ftd_decode_mha for callers that
 * must not allocate device memory.  The pages describe nothing like it: it
 * exists for callers that cannot call cudaMalloc at all -- a plugin inside a
 * host runtime whose own allocator owns all device memory, or a serving loop
 * that forbids allocation (which can synchronise the device or fail) after
 * start-up -- and so cannot create a context with ftd_init.
 *
 *   cfg              : shape, dtypes and options, same rules as ftd_init,
 *                      except that page_size must be 0 (contiguous caches).
 *   q ... out        : as in ftd_decode_mha, all caller-owned device memory;
 *                      k_cache and v_cache are required (there is no pool), and
 *                      so are scales for an INT8 cache.
 *   device_err       : device uint32, or NULL.  When given, the kernel ORs its
 *                      error bits into it (1 = some seq_lens[b] + q_len > max_len,
 *                      2 = a bounded wait gave up); the caller reads and clears
 *                      it.  When NULL those bits are dropped (overflowing slots
 *                      still get a zero output).
 *   stream           : cudaStream_t as void*.
 *
 * It allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * It runs the kernel ftd_decode_mha would run for the same config; for the
 * tensor-core kernel it encodes the caches' tensor maps on the host at every
 * call (a context caches them), so its results are ftd_decode_mha's bytes.
 * Its split-K partials, counters and error word live in one static device
 * array of FTD_NOALLOC_SCRATCH_BYTES (8 MiB) that every GPU loading the
 * library holds until the process exits.  A configuration that needs more is
 * rejected with FTD_ERR_INVALID_ARG, and ftd_last_error() gives the bytes it
 * needs.  The need is one partial slot per segment (max_batch * n_kv_heads *
 * query-row blocks per kv head) plus, per SM, one slot per worker: the CUDA-core
 * kernel's warps per block (8, or 12 for INT8 caches with blocks of at most 2
 * query rows), or 1 for the tensor-core kernel; a slot holds (2 + head_dim)
 * floats per query row of a block, plus counters and the error word.
 * The first call on each device does a one-time set-up with that device
 * current (it looks up the array's device address and raises the kernel's
 * shared-memory limit); make that first call before any stream capture.
 * Every call clears the counters and error word it uses at the start, on
 * `stream`.  All calls share the one array: calls whose kernels overlap in
 * time on the same GPU race and give wrong results, so issue them on one
 * stream or order them with events.
 */
ftd_status ftd_decode_mha_noalloc(const ftd_config* cfg, const void* q, const void* k_new,
                                  const void* v_new, const void* qkv_bias, void* k_cache,
                                  void* v_cache, const int32_t* seq_lens, float* scales, void* out,
                                  uint32_t* device_err, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FTD_H */
