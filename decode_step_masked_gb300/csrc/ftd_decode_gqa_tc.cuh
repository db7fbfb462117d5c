// ftd_decode_gqa_tc.cuh -- decode step for grouped-query caches on the
// 5th-generation tensor cores (tcgen05 + TMEM, sm_103a).
//
// With g = Hq / Hkv query heads sharing a kv head, every cached K/V element
// feeds g multiply-adds for the scores and g for P.V.  At g = 8 that is
// 8 flop per byte of bf16 cache, more than the CUDA cores can issue at HBM
// speed, so here the two contractions of a 128-row tile run on the tensor
// cores as real dense products ("10 tricks", pptc.cn, section 3.4: the query
// heads of one group share K and V):
//
//   S^T [128 rows x 2G] = K_tile [128 x D]   . Qs^T [D x 2G]     (A, B K-major)
//   O^T [D x 2G]        = V_tile^T [D x 128] . Ps^T [128 x 2G]   (A MN-major)
//
// Qs holds the G query heads twice: a bf16 (or fp16) high part and the
// rounding remainder as a low part, and Ps likewise for the softmax weights,
// so each product keeps about 16 mantissa bits of the fp32 operand; the
// accumulators are fp32 in TMEM and hi + lo are summed when read back.
//
// Roles (one persistent CTA per SM; 256, 384 or 640 threads for blocks of
// 4, 8 or 16 query columns, 640 for INT8 caches):
//   warp 0  bulk tensor copies (TMA, 128B swizzle) of K and V tiles into a
//           3-stage ring (INT8: raw codes and scales into a 2-stage ring);
//   warp 1  TMEM allocation, the append and the tcgen05.mma issue: its lanes
//           wait for every staged tile in order; in the last tile of a segment
//           they write k' = k_new + b_k (and v') rounded to the cache type into
//           the cache and into the staged tile and zero the staged V rows past
//           the sequence end (so 0 * garbage never reaches the product), then
//           lane 0 issues the MMAs;
//   warps 2-3 and 12-19 (INT8 only) the append of quantised rows and the
//           conversion of the codes to fp16: K straight into TMEM (warps 12-19,
//           two per TMEM lane quarter; the score MMA reads its A operand there),
//           V into the V halves of two operand stages;
//   warps 4.. the online softmax in groups of four warps that split the query
//           columns: thread i of a group owns row i of S and dimension i of O;
//           they build Qs, read S from TMEM, keep the running max / sum per
//           head, write Ps, rescale-and-add O, and at the end of a piece write
//           the output or a split-K partial, merged by the last piece exactly as
//           in the CUDA-core kernel.
// Work split: the same balanced contiguous ranges of a global tile space as
// ftd_decode_splitk.cuh, with 128-row tiles and one CTA per worker.
#pragma once

#include <cuda.h>

#include "ftd_decode_splitk.cuh"

namespace ftd {
namespace tc {

constexpr int TM = 128;   // rows per tile (the MMA M of the score product)
constexpr int D = 128;    // head dimension (the MMA M of the P.V product)
constexpr int NS = 3;     // K/V stages
constexpr int KB = 16384; // one 64-column box of 128 rows (bytes)
constexpr int STAGE = 4 * KB;  // K (2 boxes) + V (2 boxes)

// The softmax is the per-tile critical path.  Groups of four warps split the
// query columns so that each thread handles at most four: two groups for 8
// columns, four for 16.  Warps 0-3 copy and issue MMAs, warps 4.. run the softmax.
constexpr int softmax_groups(int G) { return G >= 16 ? 4 : (G >= 8 ? 2 : 1); }

// Weight of a segment boundary in the static split (in 128-row tiles; see WeightedSplit).
constexpr int kAlpha = 1;

// Margin (log2 units) by which a score may pass a column's running reference
// before the softmax moves the reference: weights then stay below 2^8, well
// inside the range of the hi / lo operand pair and of the fp32 accumulators.
constexpr float kRescaleLog2 = 8.f;
// INT8 caches add eight warps (12-19) to the two (2-3) that convert codes to fp16
// (measured: 2 warps 178 us, 6 warps 112 us, 10 warps 103 us on the 70B shape).
constexpr int converter_threads(bool i8) { return i8 ? 320 : 0; }
constexpr int threads_for(int G, bool i8 = false) { return 128 + 128 * softmax_groups(G) + (i8 ? 256 : 0); }

// INT8 caches: a raw stage holds a tile's codes (128 rows x 128 B for K, then for
// V, with the 128-byte swizzle: 16-byte chunk c of row r at chunk c ^ (r % 8)) and
// its 128 K and 128 V scales.
constexpr int STAGE8 = 2 * TM * D + 2 * TM * 4;

template <int G, bool I8 = false>
struct Layout {
    static constexpr int N = 2 * G;                // hi and lo parts
    static constexpr int QS = 2 * N * 128;         // Qs / Ps: 2 k-blocks of N rows x 128 B
    // operand stages the MMAs read: the TMA ring itself (fp16 / bf16), or, for INT8, two
    // stages whose V half the converting warps widen from two raw stages of codes (the K
    // operand goes to TMEM).  Measured on the INT8 70B step: V-only stages of 32 KB with
    // 2 / 3 / 4 raw stages ran 94.7 / 93.8 / 94.0 us, these 64 KB stages with 2 raw stages
    // 92.6 us, so the stage geometry stays that of the fp16 ring.
    static constexpr int NB = I8 ? 2 : NS;
    static constexpr int NR = 2;                                            // INT8 raw stages
    static constexpr int SSTR = STAGE;                                      // operand stage stride
    static constexpr int VOFF = 2 * KB;                                     // the V half in a stage
    static constexpr int OFF_STAGE = 0;
    static constexpr int OFF_S8 = NB * SSTR;                                 // raw INT8 stages
    // [4][K | V][TM] scales, slot k % 4: the softmax of tile k reads its slot until
    // it publishes P, and the slot is rewritten for tile k + 4 only after the score
    // MMAs of tile k + 2, which follow the P.V issue of tile k
    static constexpr int OFF_SC = OFF_S8 + (I8 ? NR * round_up(STAGE8, 1024) : 0);
    static constexpr int OFF_QS = OFF_SC + (I8 ? 4 * 2 * TM * 4 : 0);
    static constexpr int OFF_P = OFF_QS + round_up(QS, 1024);
    static constexpr int OFF_RED = OFF_P + 2 * round_up(QS, 1024);
    static constexpr int RED_BYTES = 4 * G * 4 * 2;  // per warp, per head: max and sum
    static constexpr int OFF_MISC = OFF_RED + round_up(RED_BYTES, 128);
    static constexpr int MISC_BYTES = 256;           // barriers, TMEM base, flags
    static constexpr int OFF_PREFIX = OFF_MISC + MISC_BYTES;
    // P, Ls and, where shared memory has room, the weighted prefix VP (else the split is unweighted)
    static constexpr bool HAVE_VP = OFF_PREFIX + round_up((3 * kMaxBatch + 2) * 4, 128) + 1024 <= 232448;
    static constexpr int ALPHA = HAVE_VP ? kAlpha : 0;
    static constexpr int PREFIX_BYTES = ((HAVE_VP ? 3 : 2) * kMaxBatch + 2) * 4;
    static constexpr int SMEM = OFF_PREFIX + round_up(PREFIX_BYTES, 128) + 1024;  // + alignment slack
    // S (2 x N columns) and O (2 x N); INT8 adds the score MMAs' K operand, widened from
    // the codes straight into TMEM: two buffers of 64 columns (128 fp16 values per row) at KT
    static constexpr int KT = 64;
    static constexpr int TMEM_COLS = I8 ? 256 : ((4 * N <= 32) ? 32 : (4 * N <= 64 ? 64 : 128));
    static_assert(!I8 || 4 * N <= KT, "INT8: S and O below the K operand buffers");
    static constexpr int OOFF = round_up(2 * G, 4);
    static constexpr int SLOT = OOFF + G * D;
    static_assert(SMEM <= 232448, "shared memory budget");
};

// ------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version of tcgen05
    d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
    return d;
}

// kind::f16 instruction descriptor: fp32 accumulate, A/B bf16 (or fp16), M x N.
__device__ __forceinline__ uint32_t instr_desc(bool bf16, int M, int N, bool a_mn_major, bool b_mn_major = false) {
    uint32_t d = 0;
    d |= 1u << 4;                                  // D: f32
    d |= (bf16 ? 1u : 0u) << 7;                    // A type
    d |= (bf16 ? 1u : 0u) << 10;                   // B type
    d |= (a_mn_major ? 1u : 0u) << 15;             // A major-ness
    d |= (b_mn_major ? 1u : 0u) << 16;             // B major-ness
    d |= static_cast<uint32_t>(N >> 3) << 17;
    d |= static_cast<uint32_t>(M >> 4) << 24;
    return d;
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc ? 1 : 0));
}

// The same with the A operand in TMEM (row m on lane m, elements k and k + 1 in the low and
// high halves of column k / 2; checked on the GPU against a CPU product before use).
__device__ __forceinline__ void mma_f16_ta(uint32_t tmem_d, uint32_t a_tmem, uint64_t b, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc ? 1 : 0));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

template <int NC>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&v)[NC]);

template <>
__device__ __forceinline__ void tmem_ld<4>(uint32_t taddr, float (&v)[4]) {
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

template <>
__device__ __forceinline__ void tmem_ld<8>(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, float (&v)[32]) {
    float a[16], b[16];
    tmem_ld<16>(taddr, a);
    tmem_ld<16>(taddr + 16, b);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        v[i] = a[i];
        v[16 + i] = b[i];
    }
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                            uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Byte offset of element (row r, column k) in a K-major operand with 128-byte
// swizzle made of 64-column blocks of `rows` rows: 16-byte chunk c of row r
// sits at chunk c ^ (r % 8) of that row.
__device__ __forceinline__ uint32_t sw128_offset(int r, int k, int rows) {
    const int blk = k >> 6, c = (k & 63) >> 3, e = k & 7;
    return static_cast<uint32_t>(blk * rows * 128 + r * 128 + ((c ^ (r & 7)) << 4) + e * 2);
}

// Operand layout of the MN-major V tile (A of the P.V product): two 64-column
// boxes of 128 rows; the stride between boxes (16 KB) and between 8-row groups
// (1 KB) go into the descriptor's leading / stride byte offsets.
constexpr uint32_t kVLbo = KB;
constexpr uint32_t kVSbo = 1024;

// Barrier-wide OR of a predicate over `n` threads (named barrier `id`).
__device__ __forceinline__ bool bar_any(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// Bounded pipeline wait (`limit` SM cycles) that also gives up as soon as
// another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, uint32_t* err, volatile int* abort_flag,
                                              long long limit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) {
            atomicOr(err, kErrTimeout);
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

template <typename CT>
__device__ __forceinline__ CT to_ct(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 to_ct<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half to_ct<__half>(float x) { return __float2half_rn(x); }
template <typename CT>
__device__ __forceinline__ float from_ct(CT x);
template <>
__device__ __forceinline__ float from_ct<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <>
__device__ __forceinline__ float from_ct<__half>(__half x) { return __half2float(x); }

// Two int8 codes (bytes sel of w, each already offset by 128 through w ^ 0x80808080)
// as an fp16 pair: the offset byte becomes the low mantissa bits under the exponent
// of 1024, so the half is 1024 + 128 + code exactly, and 1152 is subtracted exactly.
__device__ __forceinline__ uint32_t codes_to_h2(uint32_t wo, uint32_t sel) {
    const uint32_t h = __byte_perm(wo, 0x64646464u, sel);
    __half2 v;
    memcpy(&v, &h, 4);
    v = __hsub2(v, __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
    uint32_t r;
    memcpy(&r, &v, 4);
    return r;
}

}  // namespace tc

// ------------------------------------------------- tile space in passes
// The tensor-core kernel can order its tile space as np passes of spp segments per
// slot: a pass runs over the slots b, then the segments, then the tiles.  With one
// pass per block of query rows of a kv head (spp = Hkv), the passes are alike:
// with W workers and np dividing W, worker w and worker w + W / np stream the same
// K/V tiles at the same time and the later passes find them in L2.  P and VP hold
// the prefixes of one pass; Cursor::seg = s * np + h for segment s of pass h, which
// is the kernel's kvh * nhb + hb in both orders.
__device__ __forceinline__ Cursor locate_pass(int t, const int* P, int B, int spp, int np) {
    const int h = np > 1 ? t / P[B] : 0;  // called only for t < np * P[B]
    t -= h * P[B];
    int lo = 0, hi = B - 1;  // largest b with P[b] <= t; then P[b] <= t < P[b + 1]
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    Cursor cu;
    cu.b = lo;
    cu.nt = (P[lo + 1] - P[lo]) / spp;
    const int rem = t - P[lo];
    const int sg = rem / cu.nt;
    cu.seg = sg * np + h;
    cu.tile = rem - sg * cu.nt;
    return cu;
}

// next tile; called only while one is left
__device__ __forceinline__ void advance_pass(Cursor& cu, const int* P, int B, int spp, int np) {
    if (++cu.tile < cu.nt) return;
    cu.tile = 0;
    cu.seg += np;
    if (cu.seg < spp * np) return;
    cu.seg -= spp * np;  // segment 0 of the same pass ...
    do {
        if (++cu.b == B) {  // ... or of the next pass
            cu.b = 0;
            ++cu.seg;
        }
    } while (P[cu.b + 1] == P[cu.b]);
    cu.nt = (P[cu.b + 1] - P[cu.b]) / spp;
}

// Ordinal of segment s of slot b in pass h, in tile order.  A piece (segment
// ordinal o, worker w) keeps its partial in slot o + w: along the tile order each
// step to the next piece raises o or w or both, so no two pieces share a slot.
__device__ __forceinline__ int seg_ordinal(int B, int spp, int b, int s, int h) {
    return (h * B + b) * spp + s;
}

// Static split of the tile space in passes over W workers, weighted as in
// WeightedSplit: tile i of segment s of slot b in pass h sits at weighted position
// h V1 + VP[b] + s (nt + ALPHA) + i, V1 = VP[B] the weighted length of a pass, and
// worker w takes the tiles whose position lies in [ceil(w V / W), ceil((w+1) V / W)),
// V = np V1.
template <int ALPHA>
struct PassSplit {
    const int* P;
    const int* VP;
    int B, spp, np, W;

    __device__ long long V() const { return static_cast<long long>(np) * VP[B]; }

    // first tile of worker w (the whole space for w >= W)
    __device__ int begin(long long w) const {
        const int V1 = VP[B];
        if (w <= 0 || V1 == 0) return 0;
        if (w >= W) return np * P[B];
        const long long vt = (w * V() + W - 1) / W;
        const int h = np > 1 ? static_cast<int>(vt / V1) : 0;  // np when vt = V: the end of the space
        const long long v1 = vt - static_cast<long long>(h) * V1;
        int lo = 0, hi = B - 1;  // largest b with VP[b] <= v1
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (VP[mid] <= v1) lo = mid;
            else hi = mid - 1;
        }
        if (VP[lo + 1] <= v1) return h * P[B] + P[lo + 1];
        const int nt = (P[lo + 1] - P[lo]) / spp;
        const long long o = v1 - VP[lo];
        const long long sg = o / (nt + ALPHA);
        const long long r = o - sg * (nt + ALPHA);
        return h * P[B] + P[lo] + static_cast<int>(sg * nt + (r < nt ? r : nt));
    }

    // worker holding tile i of segment s of slot b in pass h (nt tiles)
    __device__ int worker_at(int b, int s, int h, int nt, int i) const {
        const long long v = static_cast<long long>(h) * VP[B] + VP[b] + static_cast<long long>(s) * (nt + ALPHA) + i;
        const long long vv = V();
        if (vv * W < (1ll << 32))  // the product fits 32 bits: a cheaper division
            return static_cast<int>(static_cast<uint32_t>(v * W) / static_cast<uint32_t>(vv));
        return static_cast<int>(v * W / vv);
    }

    // whether worker w, between the holders wf and wl of a segment's first and last
    // tiles, holds tiles of it: always when V >= W (every weighted range is non-empty)
    __device__ bool has_piece(int w, int wf, int wl) const {
        return V() >= W || w == wf || w == wl || begin(w) < begin(w + 1);
    }
};

// Barrier slots in the misc area.
// For INT8 caches kBarFull / kBarEmpty guard the K halves of the converted
// operand stages, kBarFullV / kBarEmptyV their V halves, kBarFull8 / kBarEmpty8
// the raw stages, and kBarScale the four scale slots.
// kBarDrain takes the MMA issuer's last commit, which completes once every MMA it issued has.
enum : int { kBarFull = 0, kBarEmpty = 3, kBarSFull = 6, kBarPFull = 8, kBarOFull = 10, kBarQReady = 12,
             kBarFull8 = 13, kBarEmpty8 = 15, kBarFullV = 17, kBarEmptyV = 19, kBarScale = 21, kBarDrain = 25,
             kNumBars = 26 };
// after the barriers: the TMEM base, the abort flag, the merge broadcast and the re-planning counter
static_assert(kNumBars * 8 + 16 <= 256, "misc area");

// After an abort (a cold path, kept out of line like replan so it leaves the code
// of the streaming loops as it is): wait (long drain limit) for the producer's copies still in flight,
// the last `stages` tiles before tile k_end (a withheld tile 0 excepted), on the full
// barriers full0 + kk % stages, phase (kk / stages) & 1.
static __device__ __noinline__ void tc_drain_copies(uint32_t full0, int stages, int k_end, bool withheld0, uint32_t* err) {
    for (int kk = max(0, k_end - stages); kk < k_end; ++kk)
        if (!(withheld0 && kk == 0))
            mbar_wait_bounded(full0 + 8u * static_cast<uint32_t>(kk % stages), static_cast<uint32_t>((kk / stages) & 1),
                              err, kDrainLimitCycles);
}

// MQ: several new tokens per slot (q_len > 1), so the columns of S carry
// their own causal limits; without it every column shares one row range.
template <typename CT, int G, bool MQ>
__global__ void __launch_bounds__(tc::threads_for(G, std::is_same_v<CT, int8_t>), 1)
    decode_gqa_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                         const DecodeParams p) {
    // INT8 caches: the MMAs run on fp16 copies of the codes (exact), and the
    // per-row scales multiply the scores and are folded into the weights.
    constexpr bool I8 = std::is_same_v<CT, int8_t>;
    using MT = std::conditional_t<I8, __half, CT>;  // operand type of the MMAs
    using LY = tc::Layout<G, I8>;
    constexpr int N = LY::N, TM = tc::TM, D = tc::D, NS = tc::NS, KB = tc::KB, NB = LY::NB;
    constexpr int EBC = I8 ? 1 : 2;  // bytes per cache element
    constexpr int SH = tc::softmax_groups(G);  // softmax warp groups, splitting the query columns
    constexpr int GH = G / SH;                  // query columns per softmax thread
    constexpr int SMX = 128 * SH;               // softmax threads
    constexpr int PSZ = round_up(LY::QS, 1024);
    constexpr bool BF = std::is_same_v<MT, __nv_bfloat16>;
    constexpr unsigned FULL = 0xffffffffu;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    unsigned char* stages = smem + LY::OFF_STAGE;
    unsigned char* stages8 = smem + LY::OFF_S8;                  // INT8: raw stages
    float* scl = reinterpret_cast<float*>(smem + LY::OFF_SC);   // INT8: [4][K | V][TM] scales
    unsigned char* Qs = smem + LY::OFF_QS;
    unsigned char* Ps = smem + LY::OFF_P;
    float* red_max = reinterpret_cast<float*>(smem + LY::OFF_RED);
    float* red_sum = red_max + 4 * G;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LY::OFF_MISC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + LY::OFF_MISC + kNumBars * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + LY::OFF_MISC + kNumBars * 8 + 4);
    int* bcast = reinterpret_cast<int*>(smem + LY::OFF_MISC + kNumBars * 8 + 8);
    int* rv = reinterpret_cast<int*>(smem + LY::OFF_MISC + kNumBars * 8 + 12);  // re-planning meeting counter
    int* P = reinterpret_cast<int*>(smem + LY::OFF_PREFIX);
    int* Ls = P + (kMaxBatch + 1);
    int* VP = LY::HAVE_VP ? Ls + kMaxBatch : P;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    auto bar = [&](int i) { return smem_addr(&bars[i]); };

    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) mbar_init(bar(i), 1);
        *abort_flag = 0;
        *rv = 0;
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(LY::TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // Single-token steps with blocks of 16 query rows (a kv head shared by 32 or more
    // query heads) run the head blocks of a kv head as passes (np = nhb).  Elsewhere
    // they stay side by side in one pass: with several new tokens per step that keeps
    // the kernel's register budget, and blocks of 8 rows rarely come more than one
    // to a kv head.
    constexpr bool kPasses = !MQ && G >= 16;
    const int np = kPasses ? p.nhb : 1;
    const int spp = kPasses ? p.Hkv : p.Hkv * p.nhb;
    bool ovf = false;
    if (warp == 0) ovf = build_prefix(p, TM, spp, LY::ALPHA, P, VP, Ls, lane);
    fence_mbar_init();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // The split depends only on the lengths, so it runs before the wait on the
    // previous launch, and a block that starts while the previous step drains
    // warms L2 with its first tiles (contiguous fp16 / bf16 caches; the INT8
    // variant measured faster without it, back to back and after a GEMM).  After
    // the wait the lengths are checked again (lengths_changed).  Reads of the
    // caches and writes of shared outputs come after the wait.
    const long long W = gridDim.x;
    const int wid = blockIdx.x;
    const PassSplit<LY::ALPHA> split{P, VP, p.B, spp, np, static_cast<int>(W)};
    int t_begin = split.begin(wid);
    int n_my = split.begin(wid + 1) - t_begin;
    if (!I8 && n_my > 0 && tid == 0 && !p.block_table) {
        Cursor c = locate_pass(t_begin, P, p.B, spp, np);
        for (int k = 0; k < min(NS, n_my); ++k) {
            const int L = Ls[c.b];
            const int t0 = (window_start(L, p.window) / TM + c.tile) * TM;
            const int n_cache = min(TM, max(0, L - t0));
            if (n_cache > 0) {
                const size_t rb = static_cast<size_t>(cache_row(p, c.b, c.seg / p.nhb, t0, 0));
                bulk_prefetch_l2(p.k_cache + rb * D * EBC, static_cast<uint32_t>(n_cache) * D * EBC);
                bulk_prefetch_l2(p.v_cache + rb * D * EBC, static_cast<uint32_t>(n_cache) * D * EBC);
            }
            if (k + 1 < min(NS, n_my)) advance_pass(c, P, p.B, spp, np);
        }
    }
    grid_dep_wait();    // inputs, caches and outputs may be in use by the previous launch
    grid_dep_launch();  // the next step may take SMs as this grid's blocks finish
    if (lengths_changed(p, Ls, lane)) {
        // (rare) the lengths changed after this block read them: the warps meet, warp 0
        // rebuilds the split from the lengths now visible, they meet again.  If the
        // warps disagree (the lengths changed while the step ran) the meeting gives up:
        // the warp then skips its role, and the others' bounded waits run out.
        const int r = replan(p, TM, spp, LY::ALPHA, P, VP, Ls, rv);
        const bool ok = r >= 0;
        ovf = r > 0;
        t_begin = split.begin(wid);
        n_my = ok ? split.begin(wid + 1) - t_begin : 0;
        if (!ok) *abort_flag = 1;
    }
    if (ovf && warp == 0 && lane == 0 && blockIdx.x == 0) atomicOr(p.err, kErrSeqOverflow);

    for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
        if (P[b + 1] == P[b]) {
            zero_outputs(p, static_cast<size_t>(b) * p.nq * p.Hq * D, p.nq * p.Hq * D);
        }
    }

    // Test hook (DecodeParams::stall): block 0 never issues its first tile, so the
    // bounded waits of its consumers run out and the abort path runs.
    const bool withhold0 = p.stall && blockIdx.x == 0;
    int prod_k = 0;  // producer (warp 0, lane 0): tiles it got to (issued or withheld)
    if (n_my > 0) {
        if (warp == 0) {
            // ------------------------------------------------ TMA producer
            if (lane == 0) {
                Cursor cu = locate_pass(t_begin, P, p.B, spp, np);
                PageCursor pages;
                const uint64_t l2pol = l2_stream_policy();
                int k = 0;
                if (withhold0) {  // tile 0 is never issued
                    if (n_my > 1) advance_pass(cu, P, p.B, spp, np);
                    k = 1;
                }
                for (; k < n_my; ++k) {
                    const int s = k % NS;
                    // the tile's address first: a block-table load then overlaps the wait for a free stage
                    const int kvh = cu.seg / p.nhb;
                    const int t0 = (window_start(Ls[cu.b], p.window) / TM + cu.tile) * TM;
                    long long rb = cache_row(p, cu.b, kvh, t0, pages.page(p, cu.b, t0));
                    if (rb < 0) {  // bad page: flag it and read row 0 instead (the slot's output is undefined)
                        atomicOr(p.err, kErrBadPage);
                        rb = 0;
                    }
                    const int row0 = static_cast<int>(rb);
                    if constexpr (I8) {
                        // raw stage: K and V codes (one 128 x 128 B box each) and the scales
                        // of the rows before the new tokens
                        const int s8 = k & 1;
                        if (k >= 2 && !tc::wait_or_abort(bar(kBarEmpty8 + s8), ((k >> 1) - 1) & 1, p.err, abort_flag,
                                                         p.wait_cycles))
                            break;
                        const int n_cache = min(TM, max(0, Ls[cu.b] - t0));
                        const uint32_t sb = static_cast<uint32_t>((n_cache * 4 + 15) & ~15);
                        unsigned char* st8 = stages8 + s8 * round_up(tc::STAGE8, 1024);
                        const uint32_t fb = bar(kBarFull8 + s8);
                        mbar_arrive_expect_tx(fb, 2 * TM * D + 2 * sb);
                        tc::tma_load_2d(smem_addr(st8), &tmk, 0, row0, fb, l2pol);
                        tc::tma_load_2d(smem_addr(st8 + TM * D), &tmv, 0, row0, fb, l2pol);
                        if (sb) {
                            bulk_g2s_hint(smem_addr(st8 + 2 * TM * D), p.k_scales + rb, sb, fb, l2pol);
                            bulk_g2s_hint(smem_addr(st8 + 2 * TM * D + TM * 4), p.v_scales + rb, sb, fb, l2pol);
                        }
                    } else {
                        if (k >= NS && !tc::wait_or_abort(bar(kBarEmpty + s), ((k / NS) - 1) & 1, p.err, abort_flag,
                                                          p.wait_cycles))
                            break;
                        const uint32_t st = smem_addr(stages + s * tc::STAGE);
                        mbar_arrive_expect_tx(bar(kBarFull + s), tc::STAGE);
                        tc::tma_load_2d(st, &tmk, 0, row0, bar(kBarFull + s), l2pol);
                        tc::tma_load_2d(st + KB, &tmk, 64, row0, bar(kBarFull + s), l2pol);
                        tc::tma_load_2d(st + 2 * KB, &tmv, 0, row0, bar(kBarFull + s), l2pol);
                        tc::tma_load_2d(st + 3 * KB, &tmv, 64, row0, bar(kBarFull + s), l2pol);
                    }
                    if (k + 1 < n_my) advance_pass(cu, P, p.B, spp, np);
                }
                prod_k = k;
            }
        } else if (warp == 1) {
            // ------------------------------------------- append + MMA issue
            // All 32 lanes walk every stage phase in order (a waiter that skipped
            // phases could be fooled by the parity of an older one); the lanes
            // patch the last tile of a segment together, lane 0 issues the MMAs.
            Cursor cu = locate_pass(t_begin, P, p.B, spp, np);
            const uint32_t id_s = tc::instr_desc(BF, TM, N, false);
            const uint32_t id_o = tc::instr_desc(BF, D, N, true);
            int qcount = 0;
            bool ok = true;
            // Operand descriptors of stage 0 and of the first Q / P buffers.  An offset
            // of x bytes is x / 16 added to the 14-bit start-address field (shared
            // addresses stay below 256 KB, so the field never carries), which keeps
            // the issuing thread's chain per MMA to an add and the MMA itself.
            const uint64_t dk0 = tc::smem_desc_sw128(smem_addr(stages), 16, 1024);
            const uint64_t dv0 = tc::smem_desc_sw128(smem_addr(stages) + LY::VOFF, tc::kVLbo, tc::kVSbo);
            const uint64_t dq0 = tc::smem_desc_sw128(smem_addr(Qs), 16, 1024);
            const uint64_t dp0 = tc::smem_desc_sw128(smem_addr(Ps), 16, 1024);
            auto issue_pv = [&](int kk) -> bool {
                bool w = tc::wait_or_abort(bar(kBarPFull + (kk & 1)), (kk >> 1) & 1, p.err, abort_flag, p.wait_cycles);
                if constexpr (I8) w = w && tc::wait_or_abort(bar(kBarFullV + kk % NB), (kk / NB) & 1, p.err, abort_flag, p.wait_cycles);
                if (__any_sync(FULL, !w)) return false;
                if (lane == 0) {
                    tc::tc_fence_after();
                    const uint64_t va = dv0 + static_cast<uint32_t>((kk % NB) * (LY::SSTR >> 4));
                    const uint64_t pa = dp0 + static_cast<uint32_t>((kk & 1) * (PSZ >> 4));
#pragma unroll
                    for (int ks = 0; ks < TM / 16; ++ks) {
                        const uint64_t a = va + (ks * 2048 >> 4);
                        const uint64_t bd = pa + (((ks >> 2) * (N * 128) + (ks & 3) * 32) >> 4);
                        tc::mma_f16(tmem + 2 * N + (kk & 1) * N, a, bd, id_o, ks > 0);
                    }
                    tc::mma_commit(bar(kBarOFull + (kk & 1)));
                    tc::mma_commit(bar((I8 ? kBarEmptyV : kBarEmpty) + kk % NB));
                }
                __syncwarp();
                return true;
            };
            for (int k = 0; k < n_my; ++k) {
                const int s = k % NB;
                const bool new_piece = (k == 0) || (cu.tile == 0);
                if (k > 0 && new_piece && !issue_pv(k - 1)) { ok = false; break; }
                const bool wf = tc::wait_or_abort(bar(kBarFull + s), (k / NB) & 1, p.err, abort_flag, p.wait_cycles);
                if (__any_sync(FULL, !wf)) { ok = false; break; }
                // (INT8: the converting warps append, and the weights of rows outside
                // the window or past the end are zero, so no staged row needs zeroing)
                if (!I8 && cu.tile == 0 && p.window > 0) {
                    // rows of the first tile before the window start get weight 0; zero
                    // their staged V so stale or non-finite history cannot reach O
                    const int nlo = window_start(Ls[cu.b], p.window) % TM;
                    unsigned char* st = stages + s * tc::STAGE;
                    for (int c = lane; c < 2 * nlo * 8; c += 32) {
                        const int box = c / (nlo * 8), rem = c - box * nlo * 8;
                        *reinterpret_cast<uint4*>(st + 2 * KB + box * KB + (rem >> 3) * 128 + (rem & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    if (nlo > 0) fence_proxy_async_smem();
                    __syncwarp();
                }
                // a single new token sits in the last tile; several may start a tile earlier
                bool has_new = cu.tile == cu.nt - 1;
                if constexpr (MQ)
                    has_new = Ls[cu.b] < (window_start(Ls[cu.b], p.window) / TM + cu.tile + 1) * TM;
                if (!I8 && has_new) {
                    // ---- append the new tokens (rows L - t0 ..) and zero staged V rows past the end ----
                    const int L = Ls[cu.b];
                    const int t0 = (window_start(L, p.window) / TM + cu.tile) * TM;
                    const int n_total = min(TM, L + p.nq - t0);  // rows holding data
                    const int kvh = cu.seg / p.nhb, hb = cu.seg % p.nhb;
                    unsigned char* st = stages + s * tc::STAGE;
                    const int nz = (TM - n_total) * 8;
                    for (int c = lane; c < 2 * nz; c += 32) {
                        const int box = c / nz, rem = c - box * nz;
                        const int r = n_total + (rem >> 3);
                        *reinterpret_cast<uint4*>(st + 2 * KB + box * KB + r * 128 + (rem & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    for (int nr = max(0, L - t0); nr < n_total; ++nr) {
                        const int tok = t0 + nr - L, pos = t0 + nr;
                        const bool isv = lane >= 16;  // lanes 0-15: K row, 16-31: V row, 8 elements each
                        const int d0 = (lane & 15) * 8;
                        const void* src = isv ? p.v_new : p.k_new;
                        const size_t si = ((static_cast<size_t>(cu.b) * p.nq + tok) * p.Hkv + kvh) * D + d0;
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
                            const MT y0 = tc::to_ct<MT>(x0), y1 = tc::to_ct<MT>(x1);
                            uint16_t u0, u1;
                            memcpy(&u0, &y0, 2);
                            memcpy(&u1, &y1, 2);
                            w[e] = static_cast<uint32_t>(u0) | (static_cast<uint32_t>(u1) << 16);
                        }
                        const uint4 wv = make_uint4(w[0], w[1], w[2], w[3]);
                        unsigned char* srow = st + (isv ? 2 * KB : 0) + (d0 >> 6) * KB + nr * 128 +
                                              ((((d0 & 63) >> 3) ^ (nr & 7)) << 4);
                        *reinterpret_cast<uint4*>(srow) = wv;
                        if (hb == 0) {
                            const long long rowg = cache_row(p, cu.b, kvh, pos, page_of(p, cu.b, pos));
                            if (rowg >= 0)
                                *reinterpret_cast<uint4*>((isv ? p.v_cache : p.k_cache) + (rowg * D + d0) * 2) = wv;
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                if (new_piece) {
                    const bool wq = tc::wait_or_abort(bar(kBarQReady), qcount & 1, p.err, abort_flag, p.wait_cycles);
                    if (__any_sync(FULL, !wq)) { ok = false; break; }
                    ++qcount;
                }
                if (lane == 0) {
                    tc::tc_fence_after();
                    const uint64_t ka = dk0 + static_cast<uint32_t>(s * (tc::STAGE >> 4));
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint64_t bd = dq0 + (((ks >> 2) * (N * 128) + (ks & 3) * 32) >> 4);
                        if constexpr (I8) {
                            // K in TMEM buffer s: 16 elements of each row = 8 columns per MMA
                            tc::mma_f16_ta(tmem + (k & 1) * N, tmem + LY::KT * (1 + s) + ks * 8, bd, id_s, ks > 0);
                        } else {
                            const uint64_t a = ka + (((ks >> 2) * KB + (ks & 3) * 32) >> 4);
                            tc::mma_f16(tmem + (k & 1) * N, a, bd, id_s, ks > 0);
                        }
                    }
                    tc::mma_commit(bar(kBarSFull + (k & 1)));
                    if constexpr (I8) tc::mma_commit(bar(kBarEmpty + s));  // the K half is read
                }
                __syncwarp();
                if (k > 0 && !new_piece && !issue_pv(k - 1)) { ok = false; break; }
                if (k + 1 < n_my) advance_pass(cu, P, p.B, spp, np);
            }
            if (ok) issue_pv(n_my - 1);
            // one last commit: it completes once every MMA issued above has (the drain after an abort)
            if (lane == 0) tc::mma_commit(bar(kBarDrain));
            __syncwarp();
        } else if (I8 && ((warp >= 2 && warp < 4) || warp >= 4 + 4 * SH)) {
            // ------------------------------------- INT8: append and fp16 conversion
            // Warps 2-3 and 12-19 take the raw stages in order.  In a tile holding
            // new tokens warp 2 quantises the K rows and warp 3 the V rows (cache
            // codes and scales, and the staged copies).  Then all 320 threads convert
            // the codes into the fp16 operand layout of the MMAs (128-byte swizzle, as
            // TMA writes it for fp16 caches), copy the scales beside it, publish the
            // operand stage and free the raw stage.
            constexpr int NCV = tc::converter_threads(I8);
            const int ct = warp < 4 ? tid - 64 : tid - (128 + SMX) + 64;  // 0 .. NCV - 1
            const bool isv = warp == 3;
            Cursor cu = locate_pass(t_begin, P, p.B, spp, np);
            for (int k = 0; k < n_my; ++k) {
                const int s8 = k & 1, sb = k % NB;
                const bool okf = tc::wait_or_abort(bar(kBarFull8 + s8), (k >> 1) & 1, p.err, abort_flag, p.wait_cycles);
                if (tc::bar_any(3, NCV, !okf)) break;
                unsigned char* st8 = stages8 + s8 * round_up(tc::STAGE8, 1024);
                float* ssc = reinterpret_cast<float*>(st8 + 2 * TM * D);  // [K | V][TM]
                const int L = Ls[cu.b];
                const int t0 = (window_start(L, p.window) / TM + cu.tile) * TM;
                bool has_new = cu.tile == cu.nt - 1;
                if constexpr (MQ) has_new = L < t0 + TM;
                if (has_new && warp < 4) {  // warp 2 appends K rows, warp 3 V rows
                    const int kvh = cu.seg / p.nhb, hb = cu.seg % p.nhb;
                    const int n_total = min(TM, L + p.nq - t0);
                    for (int nr = max(0, L - t0); nr < n_total; ++nr) {
                        const int tok = t0 + nr - L, pos = t0 + nr;
                        const void* src = isv ? p.v_new : p.k_new;
                        const size_t si = ((static_cast<size_t>(cu.b) * p.nq + tok) * p.Hkv + kvh) * D + lane * 4;
                        const size_t bi = static_cast<size_t>(p.Hq + (isv ? p.Hkv : 0) + kvh) * D + lane * 4;
                        float x[4];
                        float amax = 0.f;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            x[e] = ld_qkv(src, p.qkv_dtype, si + e);
                            if (p.bias) x[e] += ld_qkv(p.bias, p.qkv_dtype, bi + e);  // one binary32 add
                            amax = fmaxf(amax, fabsf(x[e]));
                        }
                        amax = warp_max(amax);
                        const float qs = amax == 0.f ? 1.f : __fdiv_rn(amax, 127.f);
                        uint32_t w = 0u;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            int code = 0;
                            if (amax != 0.f) code = max(-127, min(127, __float2int_rn(__fdiv_rn(x[e], qs))));
                            w |= (static_cast<uint32_t>(code) & 0xffu) << (8 * e);
                        }
                        *reinterpret_cast<uint32_t*>(st8 + (isv ? TM * D : 0) + nr * D +
                                                     ((((lane >> 2) ^ (nr & 7)) << 4) | ((lane & 3) << 2))) = w;
                        if (lane == 0) ssc[(isv ? TM : 0) + nr] = qs;
                        const long long rowL = cache_row(p, cu.b, kvh, pos, page_of(p, cu.b, pos));
                        if (rowL >= 0 && hb == 0) {  // the first head block writes the cache
                            *reinterpret_cast<uint32_t*>((isv ? p.v_cache : p.k_cache) + rowL * D + lane * 4) = w;
                            if (lane == 0) (isv ? p.v_scales : p.k_scales)[rowL] = qs;
                        }
                    }
                }
                // V codes to the fp16 operand stage sb once the P.V MMAs of tile k - NB have
                // read it.  Each thread converts 16-code chunks (row r, chunk j), rows fastest
                // across the threads: with both layouts swizzled, the eight rows a
                // quarter-warp touches fall in distinct banks.
                unsigned char* dst = stages + sb * LY::SSTR;
                // (Not unrolled: with four roles' loops sharing each SM sub-partition's
                // instruction cache, the unrolled copy stalled on instruction fetch and
                // cost 30 % of the step.)
                auto convert = [&](int v) {
#pragma unroll 1
                    for (int i = ct; i < TM * (D / 16); i += NCV) {
                        const int r = i % TM, j = i / TM;
                        const uint4 u =
                            *reinterpret_cast<const uint4*>(st8 + v * TM * D + r * D + ((j ^ (r & 7)) << 4));
                        const uint32_t a0 = u.x ^ 0x80808080u, a1 = u.y ^ 0x80808080u;
                        const uint32_t a2 = u.z ^ 0x80808080u, a3 = u.w ^ 0x80808080u;
                        const uint4 h0 = make_uint4(tc::codes_to_h2(a0, 0x4140), tc::codes_to_h2(a0, 0x4342),
                                                    tc::codes_to_h2(a1, 0x4140), tc::codes_to_h2(a1, 0x4342));
                        const uint4 h1 = make_uint4(tc::codes_to_h2(a2, 0x4140), tc::codes_to_h2(a2, 0x4342),
                                                    tc::codes_to_h2(a3, 0x4140), tc::codes_to_h2(a3, 0x4342));
                        // fp16 columns 16 j .. 16 j + 15: box j / 4, 16-byte chunks 2 (j % 4) and +1
                        unsigned char* row = dst + LY::VOFF + (j >> 2) * KB + r * 128;
                        const int c16 = 2 * (j & 3);
                        *reinterpret_cast<uint4*>(row + ((c16 ^ (r & 7)) << 4)) = h0;
                        *reinterpret_cast<uint4*>(row + (((c16 + 1) ^ (r & 7)) << 4)) = h1;
                    }
                };
                bool oke = true;
                if (k >= NB) oke = tc::wait_or_abort(bar(kBarEmpty + sb), ((k / NB) - 1) & 1, p.err, abort_flag, p.wait_cycles);
                // (the barrier also makes the appended rows visible to both warps)
                if (tc::bar_any(3, NCV, !oke)) break;
                if (warp >= 4) {
                    // K straight into TMEM buffer sb, the score MMAs' A operand: warps 12-19,
                    // two per TMEM lane quarter, each widening half of its 32 rows' dimensions
                    tc::tc_fence_after();
                    const int h = (warp - (4 + 4 * SH)) >> 2, rr = (warp & 3) * 32 + lane;
                    uint32_t wk[32];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int j = 4 * h + jj;
                        const uint4 u = *reinterpret_cast<const uint4*>(st8 + rr * D + ((j ^ (rr & 7)) << 4));
                        const uint32_t a0 = u.x ^ 0x80808080u, a1 = u.y ^ 0x80808080u;
                        const uint32_t a2 = u.z ^ 0x80808080u, a3 = u.w ^ 0x80808080u;
                        wk[8 * jj + 0] = tc::codes_to_h2(a0, 0x4140);
                        wk[8 * jj + 1] = tc::codes_to_h2(a0, 0x4342);
                        wk[8 * jj + 2] = tc::codes_to_h2(a1, 0x4140);
                        wk[8 * jj + 3] = tc::codes_to_h2(a1, 0x4342);
                        wk[8 * jj + 4] = tc::codes_to_h2(a2, 0x4140);
                        wk[8 * jj + 5] = tc::codes_to_h2(a2, 0x4342);
                        wk[8 * jj + 6] = tc::codes_to_h2(a3, 0x4140);
                        wk[8 * jj + 7] = tc::codes_to_h2(a3, 0x4342);
                    }
                    const uint32_t ta = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + LY::KT * (1 + sb) + 32 * h;
                    tc::tmem_st16(ta, wk);
                    tc::tmem_st16(ta + 16, wk + 16);
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    tc::tc_fence_before();
                }
                for (int i = ct; i < 2 * TM; i += NCV) scl[(k & 3) * 2 * TM + i] = ssc[i];  // K and V scales
                fence_proxy_async_smem();  // the MMAs read the stage through the async proxy
                tc::named_bar_sync(3, NCV);
                if (ct == 0) {
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(kBarFull + sb)) : "memory");
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(kBarScale + (k & 3))) : "memory");
                }
                if (k >= NB) oke = tc::wait_or_abort(bar(kBarEmptyV + sb), ((k / NB) - 1) & 1, p.err, abort_flag, p.wait_cycles);
                if (tc::bar_any(3, NCV, !oke)) break;
                convert(1);
                fence_proxy_async_smem();
                tc::named_bar_sync(3, NCV);
                if (ct == 0) {
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(kBarFullV + sb)) : "memory");
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(kBarEmpty8 + s8)) : "memory");
                }
                if (k + 1 < n_my) advance_pass(cu, P, p.B, spp, np);
            }
        } else if (warp >= 4 && warp < 4 + 4 * SH) {
            // ------------------------------------------------ softmax and output
            // SH groups of four warps; group ch owns query columns [ch * GH, (ch + 1) * GH)
            // and thread r of a group owns row r of S (TMEM lane r) and dimension r of O.
            const int sw = warp - 4;
            const int ch = sw >> 2, q4 = sw & 3;
            const int r = (tid - 128) & 127;
            const int c0 = ch * GH;
            const bool leader = ch == 0 && r == 0;  // the thread that arrives on the count-1 barriers
            const int QB = p.qblk;  // real query rows of a block; columns QB .. G-1 carry a zero query
            const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
            Cursor cu = locate_pass(t_begin, P, p.B, spp, np);
            float m[GH], l[GH], o[GH], al[GH];
            int tk[GH];  // token of each owned query column (0 unless several new tokens per step)
            // output row of query row qi of a kv head
            auto orow = [&](int b, int kvh, int qi) -> size_t {
                if constexpr (MQ) return q_row(p, b, kvh, qi);
                return static_cast<size_t>(b) * p.Hq + kvh * p.group + qi;
            };
            // the owned columns of a hi / lo pair of N-column TMEM blocks starting at col
            auto ld_cols = [&](uint32_t col, float (&hi)[GH], float (&lo)[GH]) {
                tc::tmem_ld<GH>(tmem + lane_base + col + c0, hi);
                tc::tmem_ld<GH>(tmem + lane_base + col + G + c0, lo);
            };
            bool pending = false;
            int piece_first = cu.tile;
            auto acc_o = [&](int kk) -> bool {
                const bool okw = tc::wait_or_abort(bar(kBarOFull + (kk & 1)), (kk >> 1) & 1, p.err, abort_flag, p.wait_cycles);
                if (tc::bar_any(2, SMX, !okw)) return false;
                tc::tc_fence_after();
                __syncwarp();
                float oh[GH], ol[GH];
                ld_cols(2 * N + (kk & 1) * N, oh, ol);
#pragma unroll
                for (int j = 0; j < GH; ++j) o[j] = al[j] * o[j] + (oh[j] + ol[j]);
                return true;
            };
            // The scaled query of the owned columns of piece c (dimension r), with the
            // token of each column; columns QB .. G-1 of a padded block get zero.
            float qn[GH];
            int tkn[GH];
            auto load_q = [&](const Cursor& c) {
                const int kvh = c.seg / p.nhb, hb = c.seg % p.nhb;
#pragma unroll
                for (int jj = 0; jj < GH; ++jj) {
                    const int j = c0 + jj;
                    // q row of column j; several tokens per step interleave tokens and heads
                    size_t qrow;
                    int h;
                    if constexpr (MQ) {
                        tkn[jj] = j < QB ? q_token(p, hb * QB + j) : 0;
                        h = kvh * p.group + (hb * QB + j - tkn[jj] * p.group);
                        qrow = (static_cast<size_t>(c.b) * p.nq + tkn[jj]) * p.Hq + h;
                    } else {
                        tkn[jj] = 0;
                        h = kvh * p.group + hb * QB + j;
                        qrow = static_cast<size_t>(c.b) * p.Hq + h;
                    }
                    float x = 0.f;
                    if (j < QB) {
                        x = ld_qkv(p.q, p.qkv_dtype, qrow * D + r);
                        if (p.bias) x += ld_qkv(p.bias, p.qkv_dtype, static_cast<size_t>(h) * D + r);
                        x *= p.qscale;
                    }
                    qn[jj] = x;
                }
            };
            // Q operand (hi / lo) into shared memory, published to the MMA issuer
            auto store_q = [&]() {
#pragma unroll
                for (int jj = 0; jj < GH; ++jj) {
                    const MT hi = tc::to_ct<MT>(qn[jj]);
                    const MT lo = tc::to_ct<MT>(qn[jj] - tc::from_ct<MT>(hi));
                    *reinterpret_cast<MT*>(Qs + tc::sw128_offset(c0 + jj, r, N)) = hi;
                    *reinterpret_cast<MT*>(Qs + tc::sw128_offset(G + c0 + jj, r, N)) = lo;
                }
                fence_proxy_async_smem();
                tc::named_bar_sync(1, SMX);
                if (leader) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(kBarQReady)) : "memory");
            };
            bool q_staged = false;  // the next piece's Q is already in shared memory
            for (int k = 0; k < n_my; ++k) {
                const bool new_piece = (k == 0) || (cu.tile == 0);
                const bool last = cu.tile == cu.nt - 1;
                const int L = Ls[cu.b];
                const int pos0 = window_start(L, p.window);
                const int t0 = (pos0 / TM + cu.tile) * TM;
                const int kvh = cu.seg / p.nhb, hb = cu.seg % p.nhb;
                if (new_piece) {
                    piece_first = cu.tile;
                    if (!q_staged) {
                        load_q(cu);
                        store_q();
                    }
                    q_staged = false;
#pragma unroll
                    for (int jj = 0; jj < GH; ++jj) {
                        tk[jj] = tkn[jj];
                        m[jj] = -INFINITY;
                        l[jj] = 0.f;
                        o[jj] = 0.f;
                    }
                }
                // On a piece's last tile the next piece's query is loaded now and staged
                // as soon as this tile's scores are consumed (the issuer waits for it
                // before the next score MMA, so the single Q buffer is free), ahead of the
                // output or merge of this piece.
                const bool stage_next = last && k + 1 < n_my;
                if (stage_next) {
                    Cursor nx = cu;
                    advance_pass(nx, P, p.B, spp, np);
                    load_q(nx);
                }
                // ---- scores of this tile ----
                bool oks = tc::wait_or_abort(bar(kBarSFull + (k & 1)), (k >> 1) & 1, p.err, abort_flag, p.wait_cycles);
                // INT8: the scales of the tile come from the converting warps; waiting on
                // their publication orders those writes before the reads.  (Slot k % 4 is
                // published again for tile k + 4 only after this softmax has issued P(k).)
                if constexpr (I8) oks = oks && tc::wait_or_abort(bar(kBarScale + (k & 3)), (k >> 2) & 1, p.err, abort_flag, p.wait_cycles);
                if (tc::bar_any(2, SMX, !oks)) break;
                tc::tc_fence_after();
                __syncwarp();
                float sh[GH], sl_[GH];
                ld_cols((k & 1) * N, sh, sl_);
                // column j sees rows [lo0 + tk[j], hi0 + tk[j]): positions up to L + tk[j], from
                // its own window start on
                const int hi0 = L + 1 - t0, lo0 = p.window > 0 ? L + 1 - p.window - t0 : -(1 << 30);
                const bool valid0 = r >= lo0 && r < hi0;  // the rows every column sees (single token)
                float sc[GH];
                float vf[GH];  // INT8: the row's V scale, folded into the weight (0 for rows not seen)
                bool need = false;  // a visible score above the column's reference by more than the margin
                float ksr = 1.f, vsr = 1.f;
                if constexpr (I8) {
                    ksr = scl[(k & 3) * 2 * TM + r];
                    vsr = scl[(k & 3) * 2 * TM + TM + r];
                }
#pragma unroll
                for (int jj = 0; jj < GH; ++jj) {
                    const bool valid = MQ ? (r >= lo0 + tk[jj] && r < hi0 + tk[jj]) : valid0;
                    sc[jj] = valid ? (I8 ? (sh[jj] + sl_[jj]) * ksr : sh[jj] + sl_[jj]) : -INFINITY;
                    vf[jj] = valid ? vsr : 0.f;
                    need |= sc[jj] > m[jj] + tc::kRescaleLog2;  // always when m = -inf and the score is visible
                }
                float alpha[GH];
                unsigned char* pb = Ps + (k & 1) * PSZ;
                auto put_p = [&](int jj, float pj) {
                    const MT hi = tc::to_ct<MT>(pj);
                    const MT lo = tc::to_ct<MT>(pj - tc::from_ct<MT>(hi));
                    *reinterpret_cast<MT*>(pb + tc::sw128_offset(c0 + jj, r, N)) = hi;
                    *reinterpret_cast<MT*>(pb + tc::sw128_offset(G + c0 + jj, r, N)) = lo;
                };
                // Optimistic pass: the weights are taken against the running reference m,
                // which is valid (any reference is) as long as they stay below 2^margin.
                // One barrier then both publishes P and takes the vote; only when some
                // thread saw a larger score do the columns move to the tile's maximum.
                float pq[GH];
                if (!need) {
#pragma unroll
                    for (int jj = 0; jj < GH; ++jj) {
                        // a column with no visible row yet keeps m = -inf; 0 stands in as the reference
                        pq[jj] = exp2f(sc[jj] - (m[jj] == -INFINITY ? 0.f : m[jj]));
                        put_p(jj, I8 ? pq[jj] * vf[jj] : pq[jj]);
                    }
                }
                fence_proxy_async_smem();
                tc::tc_fence_before();
                if (!tc::bar_any(1, SMX, need)) {
#pragma unroll
                    for (int jj = 0; jj < GH; ++jj) {
                        alpha[jj] = 1.f;
                        l[jj] += pq[jj];
                    }
                } else {
#pragma unroll
                    for (int jj = 0; jj < GH; ++jj) {
                        float v = sc[jj];
#pragma unroll
                        for (int mm = 16; mm >= 1; mm >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, mm));
                        if (lane == 0) red_max[q4 * G + c0 + jj] = v;
                    }
                    tc::named_bar_sync(1, SMX);
#pragma unroll
                    for (int jj = 0; jj < GH; ++jj) {
                        const int j = c0 + jj;
                        const float tmax = fmaxf(fmaxf(red_max[j], red_max[G + j]), fmaxf(red_max[2 * G + j], red_max[3 * G + j]));
                        const float mnew = fmaxf(m[jj], tmax);
                        float pj;
                        if constexpr (MQ) {
                            const float mref = mnew == -INFINITY ? 0.f : mnew;
                            alpha[jj] = exp2f(m[jj] - mref);
                            pj = exp2f(sc[jj] - mref);
                        } else {
                            alpha[jj] = exp2f(m[jj] - mnew);
                            pj = valid0 ? exp2f(sc[jj] - mnew) : 0.f;
                        }
                        l[jj] = l[jj] * alpha[jj] + pj;
                        m[jj] = mnew;
                        put_p(jj, I8 ? pj * vf[jj] : pj);
                    }
                    fence_proxy_async_smem();
                    tc::tc_fence_before();
                    tc::named_bar_sync(1, SMX);
                }
                if (leader) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(kBarPFull + (k & 1))) : "memory");
                if (stage_next) {
                    store_q();
                    q_staged = true;
                }
                if (pending && !acc_o(k - 1)) break;
#pragma unroll
                for (int jj = 0; jj < GH; ++jj) al[jj] = alpha[jj];
                pending = true;

                if (last || k == n_my - 1) {
                    if (!acc_o(k)) break;
                    pending = false;
                    // ---- end of a piece ----
#pragma unroll
                    for (int jj = 0; jj < GH; ++jj) {
                        float v = l[jj];
#pragma unroll
                        for (int mm = 16; mm >= 1; mm >>= 1) v += __shfl_xor_sync(FULL, v, mm);
                        if (lane == 0) red_sum[q4 * G + c0 + jj] = v;
                    }
                    tc::named_bar_sync(1, SMX);
                    float lt[GH];
#pragma unroll
                    for (int jj = 0; jj < GH; ++jj) {
                        const int j = c0 + jj;
                        lt[jj] = red_sum[j] + red_sum[G + j] + red_sum[2 * G + j] + red_sum[3 * G + j];
                    }
                    // segment s of pass h in the tile order: (kvh, hb) in passes, (seg, 0) in one pass
                    const int ss = kPasses ? kvh : cu.seg, sh_ = kPasses ? hb : 0;
                    const int segg = seg_ordinal(p.B, spp, cu.b, ss, sh_);
                    if (piece_first == 0 && last) {
#pragma unroll
                        for (int jj = 0; jj < GH; ++jj)
                            if (c0 + jj < QB)
                                store_out1(p, orow(cu.b, kvh, hb * QB + c0 + jj) * D + r, o[jj] / lt[jj]);
                    } else {
                        float* slot = p.ws + static_cast<size_t>(segg + wid) * LY::SLOT;
                        if (r == 0) {
#pragma unroll
                            for (int jj = 0; jj < GH; ++jj) {
                                slot[c0 + jj] = m[jj];
                                slot[G + c0 + jj] = lt[jj];
                            }
                        }
#pragma unroll
                        for (int jj = 0; jj < GH; ++jj) slot[LY::OOFF + (c0 + jj) * D + r] = o[jj];
                        // the barrier orders the softmax threads' partial stores before the leader's release
                        tc::named_bar_sync(1, SMX);
                        const uint32_t piece_tiles = static_cast<uint32_t>(cu.tile - piece_first + 1);
                        if (leader) {
                            const uint32_t prev = arrive_acq_rel(&p.counters[segg], piece_tiles);
                            bcast[0] = (prev + piece_tiles == static_cast<uint32_t>(cu.nt)) ? 1 : 0;
                        }
                        // and the leader's acquire before every thread's merge reads
                        tc::named_bar_sync(1, SMX);
                        if (bcast[0]) {
                            const int wf = split.worker_at(cu.b, ss, sh_, cu.nt, 0);
                            const int wl = split.worker_at(cu.b, ss, sh_, cu.nt, cu.nt - 1);
                            // one pass over the pieces with a running log-sum-exp; all loads
                            // of a piece are independent, so each piece costs one L2 round trip
                            float Mx[GH], Ls_[GH], Ac[GH];
#pragma unroll
                            for (int jj = 0; jj < GH; ++jj) {
                                Mx[jj] = -INFINITY;
                                Ls_[jj] = 0.f;
                                Ac[jj] = 0.f;
                            }
                            for (int w = wf; w <= wl; ++w) {
                                if (!split.has_piece(w, wf, wl)) continue;
                                const float* sl = p.ws + static_cast<size_t>(segg + w) * LY::SLOT;
                                float mw[GH], lw[GH], ow[GH];
#pragma unroll
                                for (int jj = 0; jj < GH; ++jj) {
                                    mw[jj] = __ldcg(sl + c0 + jj);
                                    lw[jj] = __ldcg(sl + G + c0 + jj);
                                    ow[jj] = __ldcg(sl + LY::OOFF + (c0 + jj) * D + r);
                                }
#pragma unroll
                                for (int jj = 0; jj < GH; ++jj) {
                                    const float mn = fmaxf(Mx[jj], mw[jj]);
                                    const float mref = (MQ && mn == -INFINITY) ? 0.f : mn;
                                    const float a = exp2f(Mx[jj] - mref), bb = exp2f(mw[jj] - mref);
                                    Ls_[jj] = Ls_[jj] * a + lw[jj] * bb;
                                    Ac[jj] = Ac[jj] * a + ow[jj] * bb;
                                    Mx[jj] = mn;
                                }
                            }
#pragma unroll
                            for (int jj = 0; jj < GH; ++jj)
                                if (c0 + jj < QB)
                                    store_out1(p, orow(cu.b, kvh, hb * QB + c0 + jj) * D + r,
                                               Ac[jj] / Ls_[jj]);
                            if (leader) p.counters[segg] = 0u;
                        }
                        tc::named_bar_sync(1, SMX);
                    }
                }
                if (k + 1 < n_my) advance_pass(cu, P, p.B, spp, np);
            }
        }
    }

    __syncwarp();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (*abort_flag && n_my > 0) {
        // Some role gave up (a bounded wait ran out).  Every role has left its loop, so
        // nothing waits on the pipeline any more; before TMEM is freed and the block
        // exits, wait for what is still in flight: the producer's copies, and the MMAs,
        // through the issuer's last commit.
        if (warp == 0 && lane == 0)
            tc_drain_copies(I8 ? bar(kBarFull8) : bar(kBarFull), I8 ? 2 : NS, prod_k, withhold0, p.err);
        if (warp == 1 && lane == 0) mbar_wait_bounded(bar(kBarDrain), 0u, p.err, kDrainLimitCycles);
    }
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(LY::TMEM_COLS));
    }
}

// ---------------------------------------------------------- host selection
struct TcKernelInfo {
    const void* fn;
    int smem;
    int slot_floats;
    int G;
    int threads;  // threads per CTA (tc::threads_for)
};

template <typename CT, int G, bool MQ>
TcKernelInfo tc_kernel_info() {
    using LY = tc::Layout<G, std::is_same_v<CT, int8_t>>;
    return TcKernelInfo{reinterpret_cast<const void*>(&decode_gqa_tc_kernel<CT, G, MQ>), LY::SMEM, LY::SLOT, G,
                        tc::threads_for(G, std::is_same_v<CT, int8_t>)};
}

TcKernelInfo select_tc(bool bf16, int G, bool multi_token);
TcKernelInfo select_tc_i8(bool multi_token);

}  // namespace ftd
