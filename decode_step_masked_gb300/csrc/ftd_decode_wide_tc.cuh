// ftd_decode_wide_tc.cuh -- decode step for kv heads shared by many query rows
// (multi-query and wide grouped-query caches: 32 or 64 query rows per kv head,
// group x new tokens), on the tensor cores (tcgen05 + TMEM + TMA, sm_103a).
//
// With MQA every query head reads the same K/V ("10 tricks", pptc.cn, section
// 3.4): 64 query rows per cached row are 64 dot products and 64 weights per
// element, a real dense contraction.  The 8- and 16-row kernel of
// ftd_decode_gqa_tc.cuh would stream such a kv head once per 16 rows and pay
// its per-tile chain (score MMA, softmax, P.V MMA, reading O back) each time.
// Here one 128-row tile serves all G rows of a block at once:
//
//   S^T [128 x G]  = K_tile [128 x D] . Qhi^T + K_tile . Qlo^T        (two S buffers in TMEM)
//   O^T [D x G]   += V_tile^T [D x 128] . Phi^T + V_tile^T . Plo^T   (one O accumulator in TMEM)
//
// q and the weights are each carried as a hi / lo pair of 16-bit values (about 16
// mantissa bits, as in the narrow kernel); the two MMAs of a pair accumulate into
// the same TMEM columns, so the softmax reads one value per score and per output.
// The weights are stored MN-major (each key row holds its G hi and G lo weights
// contiguously), so the thread that owns a key row writes them with 16-byte stores.
// O stays in TMEM for the whole piece: the softmax keeps its running reference m
// per query row and only when a score passes it by more than 2^8 does it move m
// and rescale that row's O column in TMEM (tcgen05.ld / st); the P.V MMAs
// accumulate into O across the tiles of a piece, and O is read once, at the end.
//
// Roles (320 threads, one persistent CTA per SM):
//   warp 0     TMA producer: 128-row K and V tiles into a 2-stage ring whose K
//              and V halves are refilled separately (K after the score MMA);
//   warp 1     TMEM allocation, the append of the new rows, the MMA issue;
//   warps 2-9  the softmax, in two groups of four consecutive warps (which cover
//              the four TMEM lane quarters); group g owns the query rows
//              g * G/2 .., and the thread on TMEM lane r owns key row r of S and
//              dimension r of O.  Row maxima and sums over the 128 key rows are
//              butterflies over the lanes (rows_reduce) and then over the four
//              warps through shared memory.
// Work split, append, window, pages, split-K partials and merge: as in the
// narrow tensor-core kernel (ftd_decode_gqa_tc.cuh).
#pragma once

#include "ftd_decode_gqa_tc.cuh"

namespace ftd {
namespace wide {

constexpr int NS = 2;                       // K slots of the ring (32 KB each)
// V slots (32 KB each): three where the 32-row block's Q and weight buffers leave room,
// since the P.V MMAs wait on V copies, which a slot frees only after its P.V MMAs
constexpr int nsv(int G) { return G == 32 ? 3 : 2; }
constexpr int kMaxNsv = 3;
constexpr int SH = 2;                       // softmax groups (G / 2 query rows per thread)
constexpr int kThreads = 64 + 128 * SH;     // producer and MMA warps, then the softmax warps
// Running reference of a query row before its first visible score: finite, so that
// s - m needs no test for "no reference yet" (a visible score always passes it by
// more than 2^8, and a masked one gives exp2(-inf) = 0).
constexpr float kMInit = -1e30f;

template <int G>
struct Layout {
    static constexpr int QS = 2 * (2 * G) * 128;     // Qs: 2 k-blocks (64 dims) of 2G rows (hi, lo) x 128 B
    static constexpr int PS = (2 * G / 64) * tc::KB; // Ps: 64-column atoms of 128 key rows x 128 B
    static constexpr int P_LO = (G / 64) * tc::KB + (G % 64) * 2;  // byte offset of the lo weights (column G)
    static constexpr int NSV = nsv(G);
    static constexpr int OFF_V = NS * 2 * tc::KB;                // the V ring after the K ring
    static constexpr int OFF_QS = OFF_V + NSV * 2 * tc::KB;
    static constexpr int OFF_P = OFF_QS + QS;
    static constexpr int OFF_RED = OFF_P + PS;
    // per warp of a group, per row: max and sum; then the merge's per-row state (running
    // max and sum, and the factors of one step: old partials, piece a, piece b)
    static constexpr int RED_BYTES = 4 * G * 4 * 2 + 5 * G * 4;
    static constexpr int OFF_MISC = OFF_RED + round_up(RED_BYTES, 128);
    static constexpr int MISC_BYTES = 256;
    static constexpr int OFF_PREFIX = OFF_MISC + MISC_BYTES;
    static constexpr bool HAVE_VP = OFF_PREFIX + round_up((3 * kMaxBatch + 2) * 4, 128) + 1024 <= 232448;
    // weight of a segment boundary in the static split, in tiles: a piece's end (the next
    // piece's q, the partial or the merge, the block's rows) costs about five tiles with
    // 64-row blocks and one with 32-row blocks (measured with the current issue order:
    // boundary weights 3, 4, 5, 6 gave 46.6 / 44.9 / 44.1 / 44.2 us on the multi-query step;
    // 0, 1, 2, 3 gave 117.7 / 117.1 / 121.7 / 117.9 us on the 70B-shaped step with 4 new tokens)
    static constexpr int ALPHA = HAVE_VP ? (G == 64 ? 5 : 1) : 0;
    static constexpr int PREFIX_BYTES = ((HAVE_VP ? 3 : 2) * kMaxBatch + 2) * 4;
    static constexpr int SMEM = OFF_PREFIX + round_up(PREFIX_BYTES, 128) + 1024;
    // TMEM: two S buffers (columns 0 and G), then O.  One P.V MMA per 16 key rows takes the hi
    // and lo weights together (N = 2G) into two O
    // halves (columns 2G and 3G, summed when O is read), so each V operand is read from shared
    // memory once and a V slot is free sooner (70B-shaped step with 4 new tokens 117.2 -> 104.5
    // us, multi-query step 47.5 -> 45.8 us)
    static constexpr bool PVC = true;
    static constexpr int TMEM_COLS = (PVC ? 4 : 3) * G <= 128 ? 128 : 256;
    // split-K partial of a piece: m and l of the G rows, then O as G rows of D floats
    static constexpr int OOFF = round_up(2 * G, 4);
    static constexpr int SLOT = OOFF + G * tc::D;
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(G == 32 || G == 64, "query rows per kv head block");
};

// barriers (count 1 each): the K and V halves of a stage fill and empty separately,
// K after the score MMA, V after the P.V MMA, so the next tiles' K copies run ahead
enum : int { kFullK = 0, kEmptyK = NS, kFullV = 2 * NS, kEmptyV = 2 * NS + kMaxNsv, kSFull = 2 * NS + 2 * kMaxNsv,
             kPFull = kSFull + 2, kOFull = kSFull + 3, kOFree = kSFull + 4, kQReady = kSFull + 5, kDrain = kSFull + 6,
             kSFree = kSFull + 7, kNumBarsW = kSFull + 9 };

// Whether the phase of the given parity of the barrier has completed, without waiting.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
static_assert(kNumBarsW * 8 + 16 <= 256, "misc area");

// 2^x (PTX ex2.approx.ftz: relative error about 2^-22, results below 2^-126 flush to 0)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// NV consecutive TMEM columns of this thread's lane (the wait inside the same asm,
// so no use of the values can be placed before it)
template <int NV>
__device__ __forceinline__ void tmem_ld_rows(uint32_t taddr, float (&v)[NV]);

template <>
__device__ __forceinline__ void tmem_ld_rows<8>(uint32_t taddr, float (&v)[8]) {
    uint32_t u[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(u[i]);
}

template <>
__device__ __forceinline__ void tmem_ld_rows<16>(uint32_t taddr, float (&v)[16]) {
    uint32_t u[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(u[i]);
}

template <>
__device__ __forceinline__ void tmem_ld_rows<32>(uint32_t taddr, float (&v)[32]) {
    uint32_t u[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]), "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(u[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Butterfly over the 32 lanes of a warp holding NV values each (NV = 16 or 32):
// lane L ends with op over all lanes of value L % NV.  Each halving step sends the
// half of the values that the partner lane keeps (NV - 1 exchanges, not 5 NV).
template <int NV, typename Op>
__device__ __forceinline__ float rows_reduce(float (&v)[NV], int lane, Op op) {
#pragma unroll
    for (int h = NV / 2; h >= 1; h >>= 1) {
        const bool up = (lane & h) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = up ? v[i] : v[i + h];
            const float keep = up ? v[i + h] : v[i];
            v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, h));
        }
    }
    float x = v[0];
#pragma unroll
    for (int b = NV; b < 32; b <<= 1) x = op(x, __shfl_xor_sync(0xffffffffu, x, b));
    return x;
}

// a, b as a hi pair (16-bit, nearest) and a lo pair (the rounded remainders),
// element a in the low half of each word
template <typename CT>
__device__ __forceinline__ void split_pair(float a, float b, uint32_t& hi, uint32_t& lo) {
    if constexpr (std::is_same_v<CT, __nv_bfloat16>) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        const float2 hf = __bfloat1622float2(h);
        const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
        memcpy(&hi, &h, 4);
        memcpy(&lo, &l, 4);
    } else {
        const __half2 h = __floats2half2_rn(a, b);
        const float2 hf = __half22float2(h);
        const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
        memcpy(&hi, &h, 4);
        memcpy(&lo, &l, 4);
    }
}

// Byte offset of the 16-byte chunk holding columns e .. e + 7 (e a multiple of 8) of
// key row r in the MN-major weight layout: 64-column atoms of 128 rows x 128 B,
// chunk c of row r at chunk c ^ (r % 8) of the row.
__device__ __forceinline__ uint32_t p_chunk(int e, int r) {
    return static_cast<uint32_t>((e >> 6) * tc::KB + r * 128 + ((((e & 63) >> 3) ^ (r & 7)) << 4));
}

// one q element in the step's qkv type
template <typename T>
__device__ __forceinline__ float ld_as(const void* p, size_t i) {
    if constexpr (std::is_same_v<T, float>) return __ldg(static_cast<const float*>(p) + i);
    else if constexpr (std::is_same_v<T, __half>) return __half2float(static_cast<const __half*>(p)[i]);
    else return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

// The query rows of a block as 16-byte chunks of 8 dimensions: chunk c is row c / 16,
// dimensions 8 (c % 16) .., and softmax thread st owns chunks st + 256 i.  The raw bits
// as loaded (16 bytes of 16-bit values, 32 of fp32) are converted when written to Qs,
// whose K-major rows take them as 16-byte chunks too.
template <typename T, int G>
struct QRaw {
    static constexpr int N = G * 16 / 256;
    static constexpr int W = sizeof(T) == 4 ? 2 : 1;
    uint4 q[N][W], b[N][W];
};

// q (and bias) of piece c's block.  Rows past the block read its last row (zeroed when
// written); without a bias the q chunk stands in.  16-byte loads when q and the bias
// are 16-byte aligned, else element loads (the API asks only for natural alignment).
template <typename T, int G, bool MQ>
__device__ __forceinline__ void fetch_q(const DecodeParams& p, const Cursor& c, int st, QRaw<T, G>& x) {
    constexpr int D = tc::D, W = QRaw<T, G>::W, EB = sizeof(T);
    const int kvh = c.seg / p.nhb, hb = c.seg % p.nhb, QB = p.qblk;
    const bool has_bias = p.bias != nullptr;
    const bool vec = ((reinterpret_cast<uintptr_t>(p.q) | reinterpret_cast<uintptr_t>(p.bias)) & 15u) == 0;
#pragma unroll
    for (int i = 0; i < QRaw<T, G>::N; ++i) {
        const int ci = st + 256 * i, j = min(ci >> 4, QB - 1), d0 = (ci & 15) * 8;
        size_t qrow;
        int h;
        if constexpr (MQ) {
            const int tj = q_token(p, hb * QB + j);
            h = kvh * p.group + (hb * QB + j - tj * p.group);
            qrow = (static_cast<size_t>(c.b) * p.nq + tj) * p.Hq + h;
        } else {
            h = kvh * p.group + hb * QB + j;
            qrow = static_cast<size_t>(c.b) * p.Hq + h;
        }
        const unsigned char* qa = static_cast<const unsigned char*>(p.q) + (qrow * D + d0) * EB;
        const unsigned char* ba =
            has_bias ? static_cast<const unsigned char*>(p.bias) + (static_cast<size_t>(h) * D + d0) * EB : qa;
        if (vec) {
#pragma unroll
            for (int w = 0; w < W; ++w) {
                x.q[i][w] = __ldg(reinterpret_cast<const uint4*>(qa) + w);
                x.b[i][w] = __ldg(reinterpret_cast<const uint4*>(ba) + w);
            }
        } else {
            uint32_t wq[4 * W], wb[4 * W];
#pragma unroll
            for (int e = 0; e < 4 * W; ++e) {
                if constexpr (EB == 4) {
                    wq[e] = __ldg(reinterpret_cast<const uint32_t*>(qa) + e);
                    wb[e] = __ldg(reinterpret_cast<const uint32_t*>(ba) + e);
                } else {
                    const unsigned short* q16 = reinterpret_cast<const unsigned short*>(qa);
                    const unsigned short* b16 = reinterpret_cast<const unsigned short*>(ba);
                    wq[e] = static_cast<uint32_t>(__ldg(q16 + 2 * e)) | (static_cast<uint32_t>(__ldg(q16 + 2 * e + 1)) << 16);
                    wb[e] = static_cast<uint32_t>(__ldg(b16 + 2 * e)) | (static_cast<uint32_t>(__ldg(b16 + 2 * e + 1)) << 16);
                }
            }
#pragma unroll
            for (int w = 0; w < W; ++w) {
                x.q[i][w] = make_uint4(wq[4 * w], wq[4 * w + 1], wq[4 * w + 2], wq[4 * w + 3]);
                x.b[i][w] = make_uint4(wb[4 * w], wb[4 * w + 1], wb[4 * w + 2], wb[4 * w + 3]);
            }
        }
    }
}

// element e (0..7) of a raw chunk as float
template <typename T>
__device__ __forceinline__ float raw_elem(const uint4* w, int e) {
    auto word = [](const uint4& u, int i) { return i == 0 ? u.x : i == 1 ? u.y : i == 2 ? u.z : u.w; };
    if constexpr (sizeof(T) == 4) {
        return __uint_as_float(word(w[e >> 2], e & 3));
    } else {
        const uint32_t wd = word(w[0], e >> 1);
        const unsigned short h = static_cast<unsigned short>((e & 1) ? wd >> 16 : wd & 0xffffu);
        if constexpr (std::is_same_v<T, __half>) return __half2float(__ushort_as_half(h));
        else return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
}

// (q + bias) * qscale of the fetched chunks as hi / lo rows j and G + j of the K-major Qs
template <typename CT, typename T, int G>
__device__ __forceinline__ void put_q(unsigned char* Qs, const QRaw<T, G>& x, const DecodeParams& p, int st) {
    const bool has_bias = p.bias != nullptr;
#pragma unroll
    for (int i = 0; i < QRaw<T, G>::N; ++i) {
        const int ci = st + 256 * i, j = ci >> 4, d0 = (ci & 15) * 8;
        const bool live = j < p.qblk;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float qv = raw_elem<T>(x.q[i], e);
            const float bv = raw_elem<T>(x.b[i], e);
            v[e] = live ? (qv + (has_bias ? bv : 0.f)) * p.qscale : 0.f;
        }
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_pair<CT>(v[2 * e], v[2 * e + 1], hi[e], lo[e]);
        *reinterpret_cast<uint4*>(Qs + tc::sw128_offset(j, d0, 2 * G)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(Qs + tc::sw128_offset(G + j, d0, 2 * G)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// Calls f with a value of the step's qkv type (float, __half or __nv_bfloat16).
template <typename F>
__device__ __forceinline__ void with_qkv_type(int dt, F&& f) {
    if (dt == kF32) f(0.f);
    else if (dt == kF16) f(__half{});
    else f(__nv_bfloat16{});
}

// The q of the block of piece c into Qs (the caller publishes it).  With check, the
// lengths are read again (lengths_changed) while the q loads are in flight, and q is
// written only when they are unchanged; returns whether they changed.  Out of line:
// it runs once per piece, and one copy serves every call site.
template <typename CT, int G, bool MQ>
static __device__ __noinline__ bool stage_q_fn(const DecodeParams& p, const Cursor c, int st, unsigned char* Qs,
                                               const int* Ls, bool check) {
    bool changed = false;
    with_qkv_type(p.qkv_dtype, [&](auto tag) {
        using T = decltype(tag);
        QRaw<T, G> x;
        fetch_q<T, G, MQ>(p, c, st, x);
        // the first piece's q loads go out before the producer's first copies (named barrier 3)
        if (check) asm volatile("bar.arrive 3, %0;" ::"r"(wide::kThreads - 32) : "memory");
        if (check) changed = lengths_changed(p, Ls, threadIdx.x & 31);
        if (!changed) put_q<CT, T, G>(Qs, x, p, st);
    });
    return changed;
}


// The append of a segment's last tile, by the issuing warp: the new tokens' K and V
// rows (rows L - t0 .. of the staged K and V slots, and of the cache when the block is
// the kv head's first) and zeros in the staged V rows past the end.  Out of line: it
// runs once per segment.
template <typename CT>
static __device__ __noinline__ void append_rows(const DecodeParams& p, unsigned char* kst, unsigned char* vst, int b,
                                                int seg, int tile, int L, int lane) {
    constexpr int TM = tc::TM, D = tc::D, KB = tc::KB;
    const int t0 = (window_start(L, p.window) / TM + tile) * TM;
    const int n_total = min(TM, L + p.nq - t0);
    const int kvh = seg / p.nhb, hb = seg % p.nhb;
    const int nz = (TM - n_total) * 8;
    for (int c = lane; c < 2 * nz; c += 32) {
        const int box = c / nz, rem = c - box * nz;
        const int r = n_total + (rem >> 3);
        *reinterpret_cast<uint4*>(vst + box * KB + r * 128 + (rem & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int nr = max(0, L - t0); nr < n_total; ++nr) {
        const int tok = t0 + nr - L, pos = t0 + nr;
        const bool isv = lane >= 16;
        const int d0 = (lane & 15) * 8;
        const void* src = isv ? p.v_new : p.k_new;
        const size_t si = ((static_cast<size_t>(b) * p.nq + tok) * p.Hkv + kvh) * D + d0;
        const size_t bi = static_cast<size_t>(p.Hq + (isv ? p.Hkv : 0) + kvh) * D + d0;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float x0 = ld_qkv(src, p.qkv_dtype, si + 2 * e);
            float x1 = ld_qkv(src, p.qkv_dtype, si + 2 * e + 1);
            if (p.bias) {
                x0 += ld_qkv(p.bias, p.qkv_dtype, bi + 2 * e);
                x1 += ld_qkv(p.bias, p.qkv_dtype, bi + 2 * e + 1);
            }
            const CT y0 = tc::to_ct<CT>(x0), y1 = tc::to_ct<CT>(x1);
            uint16_t u0, u1;
            memcpy(&u0, &y0, 2);
            memcpy(&u1, &y1, 2);
            w[e] = static_cast<uint32_t>(u0) | (static_cast<uint32_t>(u1) << 16);
        }
        const uint4 wv = make_uint4(w[0], w[1], w[2], w[3]);
        unsigned char* srow = (isv ? vst : kst) + (d0 >> 6) * KB + nr * 128 + ((((d0 & 63) >> 3) ^ (nr & 7)) << 4);
        *reinterpret_cast<uint4*>(srow) = wv;
        if (hb == 0) {
            const long long rowg = cache_row(p, b, kvh, pos, page_of(p, b, pos));
            if (rowg >= 0) *reinterpret_cast<uint4*>((isv ? p.v_cache : p.k_cache) + (rowg * D + d0) * 2) = wv;
        }
    }
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float* v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                 "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
                 : "memory");
}

}  // namespace wide

template <typename CT, int G, bool MQ>
__global__ void __launch_bounds__(wide::kThreads, 1)
    decode_wide_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                          const DecodeParams p) {
    using LY = wide::Layout<G>;
    constexpr int TM = tc::TM, D = tc::D, NS = wide::NS, KB = tc::KB;
    constexpr int SH = wide::SH;
    constexpr int SMX = 128 * SH;
    constexpr bool BF = std::is_same_v<CT, __nv_bfloat16>;
    constexpr unsigned FULL = 0xffffffffu;
    using namespace wide;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    unsigned char* stages = smem;
    unsigned char* Qs = smem + LY::OFF_QS;
    unsigned char* Ps = smem + LY::OFF_P;
    float* red_max = reinterpret_cast<float*>(smem + LY::OFF_RED);
    float* red_sum = red_max + 4 * G;
    float* mrg = red_sum + 4 * G;  // merge: [0] running max, [G] running sum, [2G] old, [3G] a, [4G] b factors
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::OFF_MISC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + LY::OFF_MISC + kNumBarsW * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + LY::OFF_MISC + kNumBarsW * 8 + 4);
    int* bcast = reinterpret_cast<int*>(smem + LY::OFF_MISC + kNumBarsW * 8 + 8);
    int* rv = reinterpret_cast<int*>(smem + LY::OFF_MISC + kNumBarsW * 8 + 12);
    int* P = reinterpret_cast<int*>(smem + LY::OFF_PREFIX);
    int* Ls = P + (kMaxBatch + 1);
    int* VP = LY::HAVE_VP ? Ls + kMaxBatch : P;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    auto bar = [&](int i) { return smem_addr(&bars[i]); };

    if (tid == 0) {
        for (int i = 0; i < kNumBarsW; ++i) mbar_init(bar(i), 1);
        *abort_flag = 0;
        *rv = 0;
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(LY::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // single-token steps with several blocks per kv head run them as passes (see PassSplit)
    constexpr bool kPasses = !MQ;
    const int np = kPasses ? p.nhb : 1;
    const int spp = kPasses ? p.Hkv : p.Hkv * p.nhb;
    bool ovf = false;
    if (warp == 0) ovf = build_prefix(p, TM, spp, LY::ALPHA, P, VP, Ls, lane);
    fence_mbar_init();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const long long W = gridDim.x;
    const int wid = blockIdx.x;
    const PassSplit<LY::ALPHA> split{P, VP, p.B, spp, np, static_cast<int>(W)};
    int t_begin = split.begin(wid);
    int n_my = split.begin(wid + 1) - t_begin;
    if (n_my > 0 && tid == 0 && !p.block_table) {
        Cursor c = locate_pass(t_begin, P, p.B, spp, np);
        for (int k = 0; k < min(NS, n_my); ++k) {
            const int L = Ls[c.b];
            const int t0 = (window_start(L, p.window) / TM + c.tile) * TM;
            const int n_cache = min(TM, max(0, L - t0));
            if (n_cache > 0) {
                const size_t rb = static_cast<size_t>(cache_row(p, c.b, c.seg / p.nhb, t0, 0));
                bulk_prefetch_l2(p.k_cache + rb * D * 2, static_cast<uint32_t>(n_cache) * D * 2);
                bulk_prefetch_l2(p.v_cache + rb * D * 2, static_cast<uint32_t>(n_cache) * D * 2);
            }
            if (k + 1 < min(NS, n_my)) advance_pass(c, P, p.B, spp, np);
        }
    }
    grid_dep_wait();    // inputs, caches and outputs may be in use by the previous launch
    grid_dep_launch();  // the next step may take SMs as this grid's blocks finish
    constexpr int GH = G / SH;    // query rows per softmax thread
    const int c0 = ((warp - 2) >> 2) * GH, r = (warp & 3) * 32 + lane, st = tid - 64;
    const bool leader = warp == 2 && lane == 0;
    // q of the block's piece at cursor c into Qs (the softmax warps), then QReady for the
    // issuer, which waits for it before the piece's first score MMA
    auto publish_q = [&]() {
        fence_proxy_async_smem();
        tc::named_bar_sync(1, SMX);
        if (leader) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(kQReady)) : "memory");
    };
    auto stage_q = [&](const Cursor& c) {
        wide::stage_q_fn<CT, G, MQ>(p, c, st, Qs, Ls, false);
        publish_q();
    };
    // the softmax warps fetch the first piece's q (as planned) while the lengths are checked
    bool changed;
    if (warp >= 2 && n_my > 0) {
        changed = wide::stage_q_fn<CT, G, MQ>(p, locate_pass(t_begin, P, p.B, spp, np), st, Qs, Ls, true);
        if (!changed) publish_q();
    } else {
        changed = lengths_changed(p, Ls, lane);
        // the producer issues its first copies once the softmax warps' q loads are out
        if (warp == 0 && n_my > 0) tc::named_bar_sync(3, wide::kThreads - 32);
    }
    if (changed) {
        // (rare) the lengths changed after this block read them: re-plan, as in the narrow kernel
        const int pr = replan(p, TM, spp, LY::ALPHA, P, VP, Ls, rv);
        const bool ok = pr >= 0;
        ovf = pr > 0;
        t_begin = split.begin(wid);
        n_my = ok ? split.begin(wid + 1) - t_begin : 0;
        if (!ok) *abort_flag = 1;
        if (warp >= 2 && n_my > 0) stage_q(locate_pass(t_begin, P, p.B, spp, np));
    }
    if (ovf && warp == 0 && lane == 0 && blockIdx.x == 0) atomicOr(p.err, kErrSeqOverflow);

    for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
        if (P[b + 1] == P[b]) zero_outputs(p, static_cast<size_t>(b) * p.nq * p.Hq * D, p.nq * p.Hq * D);
    }

    const bool withhold0 = p.stall && blockIdx.x == 0;  // test hook: block 0 never issues the K half of tile 0
    int prod_kk = 0, prod_kv = 0;  // producer: K and V halves it got to (issued or withheld)
    if (n_my > 0) {
        if (warp == 0) {
            // ------------------------------------------------ TMA producer
            // Two rings: K(k) may be copied once the score MMA of tile k - NS is done, V(k)
            // once the P.V MMA of tile k - NSV is.  One thread polls both (test_wait, no
            // blocking) and issues whichever copy has a free slot; a wait that makes no
            // progress for the pipeline limit aborts as the other roles' waits do.
            if (lane == 0) {
                Cursor ck = locate_pass(t_begin, P, p.B, spp, np), cv = ck;
                PageCursor pk, pv;
                const uint64_t l2pol = l2_stream_policy();
                // first cache row of the tile at cursor c (row 0 for a bad page, which is flagged)
                auto tile_row = [&](const Cursor& c, PageCursor& pc) -> int {
                    const int t0 = (window_start(Ls[c.b], p.window) / TM + c.tile) * TM;
                    long long rb = cache_row(p, c.b, c.seg / p.nhb, t0, pc.page(p, c.b, t0));
                    if (rb < 0) {
                        atomicOr(p.err, kErrBadPage);
                        rb = 0;
                    }
                    return static_cast<int>(rb);
                };
                constexpr int NSV = LY::NSV;
                int kk = 0, kv = 0;
                if (withhold0) {
                    if (n_my > 1) advance_pass(ck, P, p.B, spp, np);
                    kk = 1;
                }
                long long idle0 = clock64();
                while (kk < n_my || kv < n_my) {
                    bool did = false;
                    if (kk < n_my) {
                        const int s = kk % NS;
                        if (kk < NS || wide::mbar_test(bar(kEmptyK + s), ((kk / NS) - 1) & 1)) {
                            const int row0 = tile_row(ck, pk);
                            const uint32_t st = smem_addr(stages + s * 2 * KB);
                            mbar_arrive_expect_tx(bar(kFullK + s), 2 * KB);
                            tc::tma_load_2d(st, &tmk, 0, row0, bar(kFullK + s), l2pol);
                            tc::tma_load_2d(st + KB, &tmk, 64, row0, bar(kFullK + s), l2pol);
                            if (kk + 1 < n_my) advance_pass(ck, P, p.B, spp, np);
                            ++kk;
                            did = true;
                        }
                    }
                    if (kv < n_my) {
                        const int s = kv % NSV;
                        if (kv < NSV || wide::mbar_test(bar(kEmptyV + s), ((kv / NSV) - 1) & 1)) {
                            const int row0 = tile_row(cv, pv);
                            const uint32_t st = smem_addr(stages + LY::OFF_V + s * 2 * KB);
                            mbar_arrive_expect_tx(bar(kFullV + s), 2 * KB);
                            tc::tma_load_2d(st, &tmv, 0, row0, bar(kFullV + s), l2pol);
                            tc::tma_load_2d(st + KB, &tmv, 64, row0, bar(kFullV + s), l2pol);
                            if (kv + 1 < n_my) advance_pass(cv, P, p.B, spp, np);
                            ++kv;
                            did = true;
                        }
                    }
                    if (did) {
                        idle0 = clock64();
                    } else {
                        if (*abort_flag) break;
                        if (clock64() - idle0 > p.wait_cycles) {
                            atomicOr(p.err, kErrTimeout);
                            *abort_flag = 1;
                            break;
                        }
                    }
                }
                prod_kk = kk;
                prod_kv = kv;
            }
        } else if (warp == 1) {
            // ------------------------------------------- append + MMA issue
            // The score MMAs and the P.V MMAs are two streams, each in tile order, issued as
            // their inputs become ready rather than alternately (the 70B-shaped step with 4 new
            // tokens: 123.7 -> 117.1 us).  The score MMA of tile k needs its K tile, the piece's
            // q (on a piece's first tile) and S buffer k & 1 free (the softmax is done with tile
            // k - 2); the P.V of tile j needs its weights and its V tile, and on a piece's first
            // tile the previous piece's O read.  So a late V copy no longer holds back the next
            // score MMA, and with it the K ring.  The warp tests the barriers (test_wait, no
            // blocking) and issues whichever stream is ready; a loop that makes no progress for
            // the pipeline limit aborts as the other roles' waits do.
            Cursor cu = locate_pass(t_begin, P, p.B, spp, np);  // the tile of the next score MMA
            const uint32_t id_s = tc::instr_desc(BF, TM, G, false);
            const uint32_t id_o = tc::instr_desc(BF, D, LY::PVC ? 2 * G : G, true, true);
            const uint64_t dk0 = tc::smem_desc_sw128(smem_addr(stages), 16, 1024);
            const uint64_t dv0 = tc::smem_desc_sw128(smem_addr(stages) + LY::OFF_V, tc::kVLbo, tc::kVSbo);
            constexpr int NSV = LY::NSV;
            const uint64_t dq0 = tc::smem_desc_sw128(smem_addr(Qs), 16, 1024);
            // the weights, MN-major: 64-column atoms of 128 key rows (16 KB apart), 8-row groups 1 KB apart
            const uint64_t dp0 = tc::smem_desc_sw128(smem_addr(Ps), KB, 1024);
            int qcount = 0, opieces = 0;
            int ks = 0, kp = 0;   // next score MMA, next P.V
            uint32_t firsts = 0;  // bit k % 32: the P.V of tile k is the first of its piece
            long long idle0 = clock64();
            while (kp < n_my) {
                bool did = false;
                // 64-row blocks give the P.V MMAs the first turn, 32-row blocks the score MMAs
                // (multi-query step 45.8 -> 44.6 us; the 70B-shaped step with 4 new tokens kept
                // the score MMAs first: 117.1 against 118.4 us)
                if (G == 64 && kp < ks) {
                    // P.V of tile kp: into O, accumulating after the piece's first tile
                    const bool first = (firsts >> (kp & 31)) & 1u;
                    bool r = wide::mbar_test(bar(kPFull), kp & 1);
                    if (r) r = wide::mbar_test(bar(kFullV + kp % NSV), (kp / NSV) & 1);
                    if (r && first && opieces > 0) r = wide::mbar_test(bar(kOFree), (opieces - 1) & 1);
                    if (__all_sync(FULL, r)) {
                        if (first) ++opieces;
                        if (lane == 0) {
                            tc::tc_fence_after();
                            const uint64_t va = dv0 + static_cast<uint32_t>((kp % NSV) * (2 * KB >> 4));
#pragma unroll
                            for (int kq = 0; kq < TM / 16; ++kq) {
                                const uint64_t a = va + (kq * 2048 >> 4);
                                const uint64_t bh = dp0 + (kq * 2048 >> 4);  // key rows 16 kq .. (hi, then lo at column G)
                                tc::mma_f16(tmem + 2 * G, a, bh, id_o, !first || kq > 0);
                                if constexpr (!LY::PVC) tc::mma_f16(tmem + 2 * G, a, bh + (LY::P_LO >> 4), id_o, true);
                            }
                            tc::mma_commit(bar(kOFull));
                            tc::mma_commit(bar(kEmptyV + kp % NSV));
                        }
                        __syncwarp();
                        ++kp;
                        did = true;
                    }
                }
                if (ks < n_my) {
                    const bool new_piece = (ks == 0) || (cu.tile == 0);
                    bool has_new = cu.tile == cu.nt - 1;
                    if constexpr (MQ)
                        has_new = Ls[cu.b] < (window_start(Ls[cu.b], p.window) / TM + cu.tile + 1) * TM;
                    const bool patch_v = has_new || (cu.tile == 0 && p.window > 0);  // the V tile is written here
                    const int s = ks % NS;
                    // every lane tests (and so acquires) the barriers: the warp writes the
                    // appended rows into the landed tiles
                    bool r = wide::mbar_test(bar(kFullK + s), (ks / NS) & 1);
                    if (r && patch_v) r = wide::mbar_test(bar(kFullV + ks % NSV), (ks / NSV) & 1);
                    if (r && new_piece) r = wide::mbar_test(bar(kQReady), qcount & 1);
                    if (r && ks >= 2) r = wide::mbar_test(bar(kSFree + (ks & 1)), ((ks >> 1) - 1) & 1);
                    if (__all_sync(FULL, r)) {
                        tc::tc_fence_after();
                        if (cu.tile == 0 && p.window > 0) {
                            // rows of the first tile before the window start get weight 0; zero
                            // their staged V so stale or non-finite history cannot reach O
                            const int nlo = window_start(Ls[cu.b], p.window) % TM;
                            unsigned char* vst = stages + LY::OFF_V + (ks % NSV) * 2 * KB;
                            for (int c = lane; c < 2 * nlo * 8; c += 32) {
                                const int box = c / (nlo * 8), rem = c - box * nlo * 8;
                                *reinterpret_cast<uint4*>(vst + box * KB + (rem >> 3) * 128 + (rem & 7) * 16) =
                                    make_uint4(0u, 0u, 0u, 0u);
                            }
                            if (nlo > 0) fence_proxy_async_smem();
                            __syncwarp();
                        }
                        if (has_new) {
                            wide::append_rows<CT>(p, stages + s * 2 * KB, stages + LY::OFF_V + (ks % NSV) * 2 * KB, cu.b,
                                                  cu.seg, cu.tile, Ls[cu.b], lane);
                            fence_proxy_async_smem();
                            __syncwarp();
                        }
                        if (lane == 0) {
                            tc::tc_fence_after();
                            const uint64_t ka = dk0 + static_cast<uint32_t>(s * (2 * KB >> 4));
#pragma unroll
                            for (int kq = 0; kq < D / 16; ++kq) {
                                const uint64_t a = ka + (((kq >> 2) * KB + (kq & 3) * 32) >> 4);
                                const uint64_t bh = dq0 + (((kq >> 2) * (2 * G * 128) + (kq & 3) * 32) >> 4);
                                tc::mma_f16(tmem + (ks & 1) * G, a, bh, id_s, kq > 0);
                                tc::mma_f16(tmem + (ks & 1) * G, a, bh + (G * 128 >> 4), id_s, true);  // the lo rows
                            }
                            tc::mma_commit(bar(kSFull + (ks & 1)));
                            tc::mma_commit(bar(kEmptyK + s));  // the K tile is read
                        }
                        __syncwarp();
                        if (new_piece) {
                            ++qcount;
                            firsts |= 1u << (ks & 31);
                        } else {
                            firsts &= ~(1u << (ks & 31));
                        }
                        if (++ks < n_my) advance_pass(cu, P, p.B, spp, np);
                        did = true;
                    }
                }
                if (G != 64 && kp < ks) {
                    // P.V of tile kp: into O, accumulating after the piece's first tile
                    const bool first = (firsts >> (kp & 31)) & 1u;
                    bool r = wide::mbar_test(bar(kPFull), kp & 1);
                    if (r) r = wide::mbar_test(bar(kFullV + kp % NSV), (kp / NSV) & 1);
                    if (r && first && opieces > 0) r = wide::mbar_test(bar(kOFree), (opieces - 1) & 1);
                    if (__all_sync(FULL, r)) {
                        if (first) ++opieces;
                        if (lane == 0) {
                            tc::tc_fence_after();
                            const uint64_t va = dv0 + static_cast<uint32_t>((kp % NSV) * (2 * KB >> 4));
#pragma unroll
                            for (int kq = 0; kq < TM / 16; ++kq) {
                                const uint64_t a = va + (kq * 2048 >> 4);
                                const uint64_t bh = dp0 + (kq * 2048 >> 4);  // key rows 16 kq .. (hi, then lo at column G)
                                tc::mma_f16(tmem + 2 * G, a, bh, id_o, !first || kq > 0);
                                if constexpr (!LY::PVC) tc::mma_f16(tmem + 2 * G, a, bh + (LY::P_LO >> 4), id_o, true);
                            }
                            tc::mma_commit(bar(kOFull));
                            tc::mma_commit(bar(kEmptyV + kp % NSV));
                        }
                        __syncwarp();
                        ++kp;
                        did = true;
                    }
                }
                if (did) {
                    idle0 = clock64();
                } else {
                    if (*abort_flag) break;
                    if (clock64() - idle0 > p.wait_cycles) {
                        if (lane == 0) atomicOr(p.err, kErrTimeout);
                        *abort_flag = 1;
                        break;
                    }
                }
            }
            // one last commit: it completes once every MMA issued above has (the drain after an abort)
            if (lane == 0) tc::mma_commit(bar(kDrain));
            __syncwarp();
        } else {
            // ------------------------------------------------ softmax and output
            const int q4 = warp & 3;  // the TMEM lane quarter of the warp
            const int QB = p.qblk;
            const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
            Cursor cu = locate_pass(t_begin, P, p.B, spp, np);
            // token of owned query row jj of head block hb (0 unless several new tokens per step)
            auto tok_of = [&](int hb, int jj) -> int {
                if constexpr (MQ) return c0 + jj < QB ? q_token(p, hb * QB + c0 + jj) : 0;
                return 0;
            };
            auto orow = [&](int b, int kvh, int qi) -> size_t {
                if constexpr (MQ) return q_row(p, b, kvh, qi);
                return static_cast<size_t>(b) * p.Hq + kvh * p.group + qi;
            };
            // the owned rows' TMEM columns from column col: S buffer (k & 1) * G, O at 2G (and 3G)
            auto ld_rows = [&](uint32_t col, float (&v)[GH]) { wide::tmem_ld_rows<GH>(tmem + lane_base + col + c0, v); };
            // weights of owned rows jj0 .. jj0 + 7 for key row r: hi at column c0 + jj0, lo at G + c0 + jj0
            auto put_p8 = [&](int jj0, const float* pv) {
                uint32_t h[4], lo[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) wide::split_pair<CT>(pv[2 * i], pv[2 * i + 1], h[i], lo[i]);
                *reinterpret_cast<uint4*>(Ps + wide::p_chunk(c0 + jj0, r)) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4*>(Ps + wide::p_chunk(G + c0 + jj0, r)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            };
            int ocount = 0;  // P.V MMAs waited for (one O accumulator, one phase each)
            auto wait_o = [&]() -> bool {
                const bool okw = tc::wait_or_abort(bar(kOFull), ocount & 1, p.err, abort_flag, p.wait_cycles);
                ++ocount;
                if (tc::bar_any(2, SMX, !okw)) return false;
                tc::tc_fence_after();
                return true;
            };
            auto fmax_op = [](float a, float b) { return fmaxf(a, b); };
            auto add_op = [](float a, float b) { return a + b; };
            bool ok = true;
            int k = 0;
            // one piece (a run of consecutive tiles of one segment) per iteration
            while (ok && k < n_my) {
                const int piece_first = cu.tile;
                const int ntl = min(cu.nt - cu.tile, n_my - k);  // tiles of the piece in this block
                const bool seg_end = piece_first + ntl == cu.nt;  // the piece ends its segment
                const int L = Ls[cu.b];
                const int kvh = cu.seg / p.nhb, hb = cu.seg % p.nhb;
                const int tb = window_start(L, p.window) / TM;
                float m[GH], l[GH];  // running references and sums of the owned rows
#pragma unroll
                for (int jj = 0; jj < GH; ++jj) {
                    m[jj] = wide::kMInit;
                    l[jj] = 0.f;
                }
                for (int i = 0; i < ntl; ++i, ++k) {
                    const int t0 = (tb + piece_first + i) * TM;
                    // ---- scores of this tile ----
                    const bool oks =
                        tc::wait_or_abort(bar(kSFull + (k & 1)), (k >> 1) & 1, p.err, abort_flag, p.wait_cycles);
                    if (tc::bar_any(2, SMX, !oks)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    __syncwarp();
                    // key rows [lo0, hi0) of the tile are visible to query token 0 (token t: shifted by t)
                    const int hi0 = L + 1 - t0, lo0 = p.window > 0 ? L + 1 - p.window - t0 : -(1 << 30);
                    const bool full = hi0 >= TM && lo0 + (MQ ? p.nq - 1 : 0) <= 0;  // no masked key row
                    auto visible = [&](int jj) {
                        const int tj = tok_of(hb, jj);
                        return r >= lo0 + tj && r < hi0 + tj;
                    };
                    const uint32_t scol = static_cast<uint32_t>((k & 1) * G);
                    float pq[GH];  // weights against the current references, kept until the vote
                    ld_rows(scol, pq);
                    if (!full) {
#pragma unroll
                        for (int jj = 0; jj < GH; ++jj)
                            if (!visible(jj)) pq[jj] = -INFINITY;
                    }
                    float dmax = -INFINITY;
#pragma unroll
                    for (int jj = 0; jj < GH; ++jj) {
                        const float d = pq[jj] - m[jj];
                        dmax = fmaxf(dmax, d);
                        pq[jj] = wide::ex2(d);
                    }
                    const bool need = dmax > tc::kRescaleLog2;  // always on a piece's first tile
                    // the single P buffer and O: the P.V of the previous tile of this piece must be done
                    const bool chained = i > 0;
                    if (chained && !wait_o()) {
                        ok = false;
                        break;
                    }
                    if (!need) {
#pragma unroll
                        for (int jj0 = 0; jj0 < GH; jj0 += 8) put_p8(jj0, pq + jj0);
                    }
                    fence_proxy_async_smem();
                    tc::tc_fence_before();
                    if (!tc::bar_any(1, SMX, need)) {
#pragma unroll
                        for (int jj = 0; jj < GH; ++jj) l[jj] += pq[jj];
                    } else {
                        // some row's reference moves: per-row maximum over the group's 128 key rows
                        // (the scores are read from TMEM again rather than kept in registers)
                        {
                            float sc[GH];
                            ld_rows(scol, sc);
                            if (!full) {
#pragma unroll
                                for (int jj = 0; jj < GH; ++jj)
                                    if (!visible(jj)) sc[jj] = -INFINITY;
                            }
                            const float v = wide::rows_reduce<GH>(sc, lane, fmax_op);
                            if (lane < GH) red_max[q4 * G + c0 + lane] = v;
                        }
                        tc::named_bar_sync(1, SMX);
#pragma unroll
                        for (int j8 = 0; j8 < GH; j8 += 8) {
                            float sc[8], alpha[8];
                            wide::tmem_ld_rows<8>(tmem + lane_base + scol + c0 + j8, sc);
#pragma unroll
                            for (int i8 = 0; i8 < 8; ++i8) {
                                const int jj = j8 + i8, j = c0 + jj;
                                if (!full && !visible(jj)) sc[i8] = -INFINITY;
                                const float tmax = fmaxf(fmaxf(red_max[j], red_max[G + j]),
                                                         fmaxf(red_max[2 * G + j], red_max[3 * G + j]));
                                const float mnew = fmaxf(m[jj], tmax);
                                alpha[i8] = wide::ex2(m[jj] - mnew);
                                pq[jj] = wide::ex2(sc[i8] - mnew);
                                l[jj] = l[jj] * alpha[i8] + pq[jj];
                                m[jj] = mnew;
                            }
                            put_p8(j8, pq + j8);
                            if (chained) {
                                // rescale this piece's O (these rows' columns, dimension r)
#pragma unroll
                                for (int h = 0; h < (LY::PVC ? 2 : 1); ++h) {  // both O halves
                                    float o8[8];
                                    const uint32_t oc = tmem + lane_base + (2 + h) * G + c0 + j8;
                                    wide::tmem_ld_rows<8>(oc, o8);
#pragma unroll
                                    for (int i8 = 0; i8 < 8; ++i8) o8[i8] *= alpha[i8];
                                    wide::tmem_st8(oc, o8);
                                }
                            }
                        }
                        if (chained) wide::tmem_st_wait();
                        fence_proxy_async_smem();
                        tc::tc_fence_before();
                        tc::named_bar_sync(1, SMX);
                    }
                    if (leader) {
                        // the weights are in place and S buffer k & 1 is read
                        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(kPFull)) : "memory");
                        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(kSFree + (k & 1))) : "memory");
                    }
                    if (i + 1 < ntl) advance_pass(cu, P, p.B, spp, np);
                }
                if (!ok) break;
                // On a segment's last tile the next piece's query goes to Qs now: its scores
                // are consumed, and the issuer waits for it before the next score MMA.
                Cursor nx = cu;
                if (k < n_my) advance_pass(nx, P, p.B, spp, np);
                if (seg_end && k < n_my) stage_q(nx);
                // ---- end of the piece: O after its last P.V ----
                // O goes once through shared memory as rows x D floats (the weights buffer is
                // free once the piece's last P.V is done); the partial, the merge and the
                // block's rows then run as short loops of coalesced 16-byte accesses
                if (!wait_o()) break;
                float* ostg = reinterpret_cast<float*>(Ps);
                {
                    float o[GH];
                    ld_rows(2 * G, o);
                    if constexpr (LY::PVC) {
                        float o2[GH];
                        ld_rows(3 * G, o2);
#pragma unroll
                        for (int jj = 0; jj < GH; ++jj) o[jj] += o2[jj];
                    }
                    tc::tc_fence_before();
#pragma unroll
                    for (int jj = 0; jj < GH; ++jj) ostg[(c0 + jj) * D + r] = o[jj];
                }
                {
                    const float v = wide::rows_reduce<GH>(l, lane, add_op);
                    if (lane < GH) red_sum[q4 * G + c0 + lane] = v;
                }
                if (r == 0) {
#pragma unroll
                    for (int jj = 0; jj < GH; ++jj) mrg[c0 + jj] = m[jj];  // the piece's references
                }
                tc::named_bar_sync(1, SMX);
                // O is read: the next piece's first P.V may overwrite it
                if (leader) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(kOFree)) : "memory");
                if (st < G) mrg[G + st] = red_sum[st] + red_sum[G + st] + red_sum[2 * G + st] + red_sum[3 * G + st];
                tc::named_bar_sync(1, SMX);
                const int ss = kPasses ? kvh : cu.seg, sh_ = kPasses ? hb : 0;
                const int segg = seg_ordinal(p.B, spp, cu.b, ss, sh_);
                constexpr int NV4 = G * D / 4 / SMX;  // 16-byte pieces of O per thread
                float4* o4 = reinterpret_cast<float4*>(ostg);
                bool fin = piece_first == 0 && seg_end;  // the piece is its whole segment
                bool merged = false;
                if (!fin) {
                    // the partial: m and l of the rows, then O as rows x D
                    float* slot = p.ws + static_cast<size_t>(segg + wid) * LY::SLOT;
                    if (st < G) {
                        slot[st] = mrg[st];
                        slot[G + st] = mrg[G + st];
                    }
#pragma unroll
                    for (int u = 0; u < NV4; ++u)
                        reinterpret_cast<float4*>(slot + LY::OOFF)[st + u * SMX] = o4[st + u * SMX];
                    tc::named_bar_sync(1, SMX);
                    if (leader) {
                        const uint32_t prev = arrive_acq_rel(&p.counters[segg], static_cast<uint32_t>(ntl));
                        bcast[0] = (prev + ntl == static_cast<uint32_t>(cu.nt)) ? 1 : 0;
                    }
                    tc::named_bar_sync(1, SMX);
                    fin = merged = bcast[0] != 0;
                }
                if (merged) {
                    // the last piece to arrive merges the others into its O in shared memory,
                    // two at a time with all their loads in flight; thread st < G keeps row
                    // st's running max and sum and publishes the step's factors
                    const int wf = split.worker_at(cu.b, ss, sh_, cu.nt, 0);
                    const int wl = split.worker_at(cu.b, ss, sh_, cu.nt, cu.nt - 1);
                    int w = wf;
#pragma unroll 1
                    for (;;) {
                        int wa = -1, wb = -1;
                        for (; w <= wl && wb < 0; ++w) {
                            if (w == wid || !split.has_piece(w, wf, wl)) continue;
                            if (wa < 0) wa = w;
                            else wb = w;
                        }
                        if (wa < 0) break;
                        const bool hasb = wb >= 0;
                        const float* sa = p.ws + static_cast<size_t>(segg + wa) * LY::SLOT;
                        const float* sb = p.ws + static_cast<size_t>(segg + (hasb ? wb : wa)) * LY::SLOT;
                        float4 va[NV4], vb[NV4];
#pragma unroll
                        for (int u = 0; u < NV4; ++u) {
                            va[u] = __ldcg(reinterpret_cast<const float4*>(sa + LY::OOFF) + st + u * SMX);
                            vb[u] = hasb ? __ldcg(reinterpret_cast<const float4*>(sb + LY::OOFF) + st + u * SMX)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                        if (st < G) {
                            const float ma = __ldcg(sa + st), la = __ldcg(sa + G + st);
                            const float mb = __ldcg(sb + st), lb = __ldcg(sb + G + st);
                            const float m0 = mrg[st];
                            const float mn = fmaxf(m0, hasb ? fmaxf(ma, mb) : ma);  // finite: every m >= kMInit
                            const float f0 = wide::ex2(m0 - mn), fa = wide::ex2(ma - mn);
                            const float fb = hasb ? wide::ex2(mb - mn) : 0.f;
                            mrg[st] = mn;
                            mrg[G + st] = mrg[G + st] * f0 + la * fa + lb * fb;
                            mrg[2 * G + st] = f0;
                            mrg[3 * G + st] = fa;
                            mrg[4 * G + st] = fb;
                        }
                        tc::named_bar_sync(1, SMX);
#pragma unroll
                        for (int u = 0; u < NV4; ++u) {
                            const int idx = st + u * SMX, j = idx / (D / 4);
                            const float f0 = mrg[2 * G + j], fa = mrg[3 * G + j], fb = mrg[4 * G + j];
                            float4 x = o4[idx];
                            x.x = x.x * f0 + va[u].x * fa + vb[u].x * fb;
                            x.y = x.y * f0 + va[u].y * fa + vb[u].y * fb;
                            x.z = x.z * f0 + va[u].z * fa + vb[u].z * fb;
                            x.w = x.w * f0 + va[u].w * fa + vb[u].w * fb;
                            o4[idx] = x;
                        }
                        tc::named_bar_sync(1, SMX);
                    }
                }
                if (fin) {
                    // the block's rows: O / l, one 16-byte store per 4 dimensions
#pragma unroll 1
                    for (int idx = st; idx < QB * (D / 4); idx += SMX) {
                        const int j = idx / (D / 4), d0 = (idx % (D / 4)) * 4;
                        const float lj = mrg[G + j];
                        const float4 x = o4[idx];
                        store_out4(p, orow(cu.b, kvh, hb * QB + j) * D + d0, x.x / lj, x.y / lj, x.z / lj, x.w / lj);
                    }
                    if (merged && leader) p.counters[segg] = 0u;
                }
                // the staging buffer and the row state are free for the next piece
                tc::named_bar_sync(1, SMX);
                cu = nx;
            }
        }
    }

    __syncwarp();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (*abort_flag && n_my > 0) {
        // a bounded wait ran out: wait (long drain limit) for the copies and MMAs in flight
        if (warp == 0 && lane == 0) {
            tc_drain_copies(bar(kFullK), NS, prod_kk, withhold0, p.err);
            tc_drain_copies(bar(kFullV), LY::NSV, prod_kv, false, p.err);
        }
        if (warp == 1 && lane == 0) mbar_wait_bounded(bar(kDrain), 0u, p.err, kDrainLimitCycles);
    }
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(LY::TMEM_COLS));
    }
}

template <typename CT, int G, bool MQ>
TcKernelInfo wide_kernel_info() {
    using LY = wide::Layout<G>;
    return TcKernelInfo{reinterpret_cast<const void*>(&decode_wide_tc_kernel<CT, G, MQ>), LY::SMEM, LY::SLOT, G,
                        wide::kThreads};
}

TcKernelInfo select_wide(bool bf16, int G, bool multi_token);

}  // namespace ftd
