// ftd_decode_splitk.cuh -- one decode step of masked multi-head attention as a
// single persistent kernel on CUDA cores (sm_103a).
//
// What one launch computes (see include/ftd.h for the full contract):
//   fused QKV bias add, append of the new K/V row at position L_b, scores of
//   the current token against positions 0..L_b, a numerically stable softmax
//   and the weighted sum of V -- the decode path of the FasterTransformer
//   masked multi-head attention kernel ("FasterTransformer source reading",
//   lmnt.cn, section 4.1; lpnh.cn section 2.1: q.K, softmax and x V fused so
//   no score tensor reaches HBM).
//
// Work decomposition (split-K over the cache length):
//   A "segment" is one (slot b, kv head, block of G query heads).  Segment
//   (b, .) owns ceil((L_b + 1) / T) tiles of T cache rows.  All tiles of all
//   segments form one global index space, ordered slot-major.  Every warp of
//   the grid is an independent worker that takes an equal contiguous range of
//   that space (static, balanced to one tile), so ragged batches cannot leave
//   SMs idle.  A worker streams its tiles through a private ring of shared
//   memory stages filled by the bulk-copy engine (cp.async.bulk, one copy per
//   K tile and per V tile, completing on an mbarrier), keeps the running max,
//   sum and output of an online softmax in registers ("10 tricks",
//   pptc.cn, section 2.2), and at the end of each piece of a segment either
//   writes the final output (the piece is the whole segment) or a partial
//   (max, sum, o) to the workspace, in slot (segment index + worker index),
//   which is unique because both indices only grow along the tile space.
//   Each piece adds its tile count to the segment's counter; the piece that
//   completes the count merges the partials by log-sum-exp and resets the
//   counter, so the whole step is one launch with no inter-block waiting.
//
// Lane layout inside a warp: half-warp hr = lane / 16 takes the even or odd
// rows of a tile, lane c = lane % 16 owns head dimensions [c*EPL, (c+1)*EPL).
// q.k partial sums are reduced across the 16 lanes with a reduce-scatter
// (log2(16) shuffle rounds that halve the live values each round).
#pragma once

#include <cmath>
#include <type_traits>

#include "ftd_common.cuh"

namespace ftd {

template <typename CT>
struct CacheTraits;
template <>
struct CacheTraits<float> { static constexpr int EB = 4; static constexpr bool I8 = false; };
template <>
struct CacheTraits<__half> { static constexpr int EB = 2; static constexpr bool I8 = false; };
template <>
struct CacheTraits<__nv_bfloat16> { static constexpr int EB = 2; static constexpr bool I8 = false; };
template <>
struct CacheTraits<int8_t> { static constexpr int EB = 1; static constexpr bool I8 = true; };

constexpr int cmin(int a, int b) { return a < b ? a : b; }
constexpr int cmax(int a, int b) { return a > b ? a : b; }
constexpr int round_up(int a, int b) { return (a + b - 1) / b * b; }

template <typename CT, int D, int G>
struct Tiling {
    static constexpr int EB = CacheTraits<CT>::EB;
    static constexpr bool I8 = CacheTraits<CT>::I8;
    static constexpr int ROW = D * EB;                         // bytes per cache row
    static constexpr int T = cmax(8, cmin(32, 4096 / ROW));    // rows per tile (4 KB K tiles)
    static constexpr int R = T / 2;                            // rows per half-warp
    static constexpr int EPL = D / 16;                         // elements per lane
    static constexpr int TILE = T * ROW;
    static constexpr int SCL = I8 ? T * 4 : 0;                 // per-row scales of one tile
    static constexpr int STAGE = 2 * TILE + 2 * SCL;
    // Workers per CTA.  The INT8 tile loop issues more instructions per byte than
    // 8 warps can hide, so INT8 with small query blocks runs 12 workers of 2
    // stages each: the same bytes in flight per SM, 1.5x the warps to issue from
    // (and at most 170 registers a thread, which those instantiations fit).
    static constexpr int WARPS = (I8 && G <= 2) ? 12 : kWarps;
    static constexpr int SPW = WARPS > 8 ? 2 : cmax(2, cmin(4, 26624 / STAGE));  // ring stages per warp
    static constexpr int RB = cmax(1, cmin(R, 16 / G));        // rows per reduce-scatter batch
    static constexpr int SCRATCH = 2 * G * T * 4;              // scores + probabilities
    static constexpr int WARP_BYTES = round_up(SPW * STAGE + SCRATCH + SPW * 8, 128);
    // Static split weights: a segment boundary inside a worker's range costs it a partial,
    // an arrival, the append and the next segment's q (and often the merge), so each
    // segment start counts ALPHA extra tiles and a worker that crosses one gets fewer.
    // The weighted prefix needs one more [B + 1] array; where shared memory has no room
    // for it, ALPHA is 0 and the plain tile prefix serves.
    static constexpr bool HAVE_VP =
        round_up((3 * kMaxBatch + 2) * 4, 128) + WARPS * WARP_BYTES <= 232448;
    static constexpr int ALPHA = HAVE_VP ? (I8 ? 1 : 4) : 0;  // measured: 7B/13B best at 4, INT8 at 1
    static constexpr int PREFIX_BYTES = round_up(((HAVE_VP ? 3 : 2) * kMaxBatch + 2) * 4, 128);
    static constexpr int SMEM = PREFIX_BYTES + WARPS * WARP_BYTES;
    static constexpr int OOFF = round_up(2 * G, 4);            // o offset in a partial slot
    static constexpr int SLOT = OOFF + G * D;                  // floats per partial slot
    static_assert(D % 16 == 0 && (EPL == 4 || EPL == 8), "head_dim 64 or 128");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(G * RB <= 16 && R % RB == 0, "reduce-scatter batch");
    static_assert(((HAVE_VP ? 3 : 2) * kMaxBatch + 3) * 4 <= PREFIX_BYTES, "room for the re-planning counter");
};

// ------------------------------------------------ shared-memory row access
template <typename CT, int N>
__device__ __forceinline__ void ld_cvt(const unsigned char* p, float (&f)[N]) {
    if constexpr (std::is_same_v<CT, __nv_bfloat16>) {
        // bfloat16 -> binary32 is exact: the pattern becomes the upper half
        uint32_t w[N / 2];
        if constexpr (N == 8) {
            const uint4 u = *reinterpret_cast<const uint4*>(p);
            w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
        } else {
            const uint2 u = *reinterpret_cast<const uint2*>(p);
            w[0] = u.x; w[1] = u.y;
        }
#pragma unroll
        for (int k = 0; k < N / 2; ++k) {
            f[2 * k] = __uint_as_float(w[k] << 16);
            f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    } else if constexpr (std::is_same_v<CT, __half>) {
        uint32_t w[N / 2];
        if constexpr (N == 8) {
            const uint4 u = *reinterpret_cast<const uint4*>(p);
            w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
        } else {
            const uint2 u = *reinterpret_cast<const uint2*>(p);
            w[0] = u.x; w[1] = u.y;
        }
#pragma unroll
        for (int k = 0; k < N / 2; ++k) {
            __half2 h2;
            memcpy(&h2, &w[k], 4);
            const float2 ff = __half22float2(h2);
            f[2 * k] = ff.x;
            f[2 * k + 1] = ff.y;
        }
    } else if constexpr (std::is_same_v<CT, float>) {
#pragma unroll
        for (int k = 0; k < N / 4; ++k) {
            const float4 u = reinterpret_cast<const float4*>(p)[k];
            f[4 * k] = u.x; f[4 * k + 1] = u.y; f[4 * k + 2] = u.z; f[4 * k + 3] = u.w;
        }
    } else {  // int8 codes
        // Integer to float without the int-to-float unit: flipping the sign bit
        // turns code c into the unsigned byte c + 128; placed as the low
        // mantissa byte under the exponent of 2^23 (0x4B000000) it forms the
        // binary32 value 2^23 + c + 128 exactly, and subtracting 2^23 + 128
        // (also exact) leaves c.  One byte permute and one add per element.
        uint32_t w[N / 4];
        if constexpr (N == 8) {
            const uint2 u = *reinterpret_cast<const uint2*>(p);
            w[0] = u.x ^ 0x80808080u; w[1] = u.y ^ 0x80808080u;
        } else {
            w[0] = *reinterpret_cast<const uint32_t*>(p) ^ 0x80808080u;
        }
#pragma unroll
        for (int k = 0; k < N; ++k)
            f[k] = __uint_as_float(__byte_perm(w[k / 4], 0x4B000000u, 0x7540u + (k % 4))) - 8388736.0f;
    }
}

// Round N binary32 values to the cache type (nearest even) and store them.
template <typename CT, int N>
__device__ __forceinline__ void cvt_st(unsigned char* p, const float (&x)[N]) {
    if constexpr (std::is_same_v<CT, float>) {
#pragma unroll
        for (int k = 0; k < N / 4; ++k)
            reinterpret_cast<float4*>(p)[k] = make_float4(x[4 * k], x[4 * k + 1], x[4 * k + 2], x[4 * k + 3]);
    } else {
        uint32_t w[N / 2];
#pragma unroll
        for (int k = 0; k < N / 2; ++k) {
            uint16_t lo, hi;
            if constexpr (std::is_same_v<CT, __half>) {
                lo = __half_as_ushort(__float2half_rn(x[2 * k]));
                hi = __half_as_ushort(__float2half_rn(x[2 * k + 1]));
            } else {
                lo = __bfloat16_as_ushort(__float2bfloat16_rn(x[2 * k]));
                hi = __bfloat16_as_ushort(__float2bfloat16_rn(x[2 * k + 1]));
            }
            w[k] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
        }
        if constexpr (N == 8) *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
        else *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
    }
}

// ------------------------------------------------------- reduce-scatter
// Sum N values over the 16 lanes of a half-warp.  Each halving round sends
// half of the live values to the partner lane and keeps the other half, so
// after log2(N) rounds every lane holds one fully reduced value, whose index
// is returned in idx; remaining rounds are plain butterflies.
template <int N, int MASK, typename V = float>
struct ReduceScatter {
    static __device__ __forceinline__ void run(V* v, int c, int& idx) {
        if constexpr (MASK == 0) {
            return;
        } else if constexpr (N > 1) {
            const bool up = (c & MASK) != 0;
#pragma unroll
            for (int k = 0; k < N / 2; ++k) {
                const V send = up ? v[k] : v[k + N / 2];
                const V keep = up ? v[k + N / 2] : v[k];
                v[k] = keep + __shfl_xor_sync(0xffffffffu, send, MASK);
            }
            if (up) idx += N / 2;
            ReduceScatter<N / 2, MASK / 2, V>::run(v, c, idx);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], MASK);
            ReduceScatter<1, MASK / 2, V>::run(v, c, idx);
        }
    }
};

// ---------------------------------------------------------- tile cursor
struct Cursor {
    int b, seg, tile, nt;
};

__device__ __forceinline__ Cursor locate(int t, const int* P, int B, int segs) {
    int lo = 0, hi = B - 1;  // largest b with P[b] <= t; then P[b] <= t < P[b + 1]
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (P[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    Cursor cu;
    cu.b = lo;
    cu.nt = (P[lo + 1] - P[lo]) / segs;
    const int rem = t - P[lo];
    cu.seg = rem / cu.nt;
    cu.tile = rem - cu.seg * cu.nt;
    return cu;
}

__device__ __forceinline__ void advance(Cursor& cu, const int* P, int segs) {
    if (++cu.tile < cu.nt) return;
    cu.tile = 0;
    if (++cu.seg < segs) return;
    cu.seg = 0;
    do {
        ++cu.b;
    } while (P[cu.b + 1] == P[cu.b]);
    cu.nt = (P[cu.b + 1] - P[cu.b]) / segs;
}

// Tiles per slot and their prefixes, computed by one warp: P[b] counts the tiles
// of the slots before b (segments of T rows, from the tile holding the window start
// to the tile of position L + nq - 1, times segs), VP[b] the same plus ALPHA per
// segment, Ls[b] the cached length (-1 for slots without work).  Returns, in every
// lane, whether some slot has L + nq > Lmax (the caller raises the overflow flag).
__device__ __forceinline__ bool build_prefix(const DecodeParams& p, int T, int segs, int alpha, int* P, int* VP,
                                             int* Ls, int lane) {
    constexpr unsigned FULL = 0xffffffffu;
    int carry = 0, vcarry = 0;
    bool ovf = false;
    for (int base = 0; base < p.B; base += 32) {
        const int b = base + lane;
        const int L = b < p.B ? __ldcg(p.seq_lens + b) : -1;  // L2: may run before the wait on the previous launch
        const bool valid = L >= 0 && L <= p.Lmax - p.nq;
        ovf |= (b < p.B) && (L > p.Lmax - p.nq);
        int v = valid ? ((L + p.nq - 1) / T + 1 - window_start(L, p.window) / T) * segs : 0;
        int vw = v + (valid ? alpha * segs : 0);
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const int y = __shfl_up_sync(FULL, v, m);
            const int yw = __shfl_up_sync(FULL, vw, m);
            if (lane >= m) {
                v += y;
                vw += yw;
            }
        }
        if (b < p.B) {
            P[b + 1] = carry + v;
            VP[b + 1] = vcarry + vw;
            Ls[b] = valid ? L : -1;
        }
        carry += __shfl_sync(FULL, v, 31);
        vcarry += __shfl_sync(FULL, vw, 31);
    }
    if (lane == 0) {
        P[0] = 0;
        VP[0] = 0;
    }
    return __any_sync(FULL, ovf);
}

// Whether the lengths differ from the ones the split was built from (Ls).  The
// split is built from lengths read before grid_dep_wait, so that a block placed
// while the previous launch drains can warm L2 with its first tiles; but a
// preceding kernel's writes are guaranteed visible only after the wait (a kernel
// that allows an early start, or that has ended without its writes landing yet,
// may still be writing seq_lens).  So after the wait every warp reads all the
// lengths again, through L2, and votes.  All warps read the same final values,
// so they reach the same answer without waiting for one another.
__device__ __forceinline__ bool lengths_changed(const DecodeParams& p, const int* Ls, int lane) {
    bool changed = false;
    for (int b = lane; b < p.B; b += 32) {
        const int L = __ldcg(p.seq_lens + b);
        changed |= ((L >= 0 && L <= p.Lmax - p.nq) ? L : -1) != Ls[b];
    }
    return __any_sync(0xffffffffu, changed);
}

// Bounded meeting of the block's nwarps warps on the re-planning path: lane 0 of
// each warp adds 1 to the shared counter *ctr and waits until it reaches target.
// Shared-memory writes a warp made before the call are visible to every warp after
// it.  Returns false, with the timeout bit raised, when some warp has not come
// within `limit` cycles: that happens only if the warps disagreed about the
// lengths (they changed while the step ran), and it must not hang the block.
__device__ __forceinline__ bool warp_rendezvous(int* ctr, int target, long long limit, uint32_t* err, int lane) {
    __syncwarp();
    bool ok = true;
    if (lane == 0) {
        __threadfence_block();
        atomicAdd(ctr, 1);
        const long long t0 = clock64();
        while (*static_cast<volatile int*>(ctr) < target) {
            if (clock64() - t0 > limit) {
                atomicOr(err, kErrTimeout);
                ok = false;
                break;
            }
        }
        __threadfence_block();
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok;
}

// Re-planning after the lengths changed (lengths_changed), by every warp of the
// block: the warps meet (bounded), warp 0 rebuilds the prefixes from the lengths
// now visible, they meet again.  Returns -1 when a meeting gave up (the warps
// disagreed), else whether some slot overflows (meaningful in warp 0).  The
// tensor-core kernel calls it out of line, which keeps its streaming loops' code
// as it was; the CUDA-core kernel measured faster with the same steps inline.
static __device__ __noinline__ int replan(const DecodeParams& p, int T, int segs, int alpha, int* P, int* VP, int* Ls,
                                          int* rv) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = static_cast<int>(blockDim.x) / 32;
    if (!warp_rendezvous(rv, nw, p.wait_cycles, p.err, lane)) return -1;
    bool ovf = false;
    if (warp == 0) ovf = build_prefix(p, T, segs, alpha, P, VP, Ls, lane);
    if (!warp_rendezvous(rv, 2 * nw, p.wait_cycles, p.err, lane)) return -1;
    return ovf ? 1 : 0;
}

// Static split of the tile space over W workers, weighted: a segment boundary inside
// a worker's range costs it a partial, an arrival, the append and the next segment's
// q (and often the merge), so tile i of segment s of slot b sits at weighted position
// VP[b] + s (nt + ALPHA) + i, and worker w takes the tiles whose position lies in
// [ceil(w V / W), ceil((w+1) V / W)), V the weighted length.  A worker that crosses a
// boundary therefore gets about ALPHA fewer tiles.  ALPHA = 0 is the plain equal split.
// P and VP live in shared memory; their totals are read from there when needed.
template <int ALPHA>
struct WeightedSplit {
    const int* P;
    const int* VP;
    int B, segs, W;

    __device__ long long U() const { return P[B]; }
    __device__ long long V() const { return VP[B]; }

    // first tile of worker w (U for w >= W)
    __device__ int begin(long long w) const {
        if (w <= 0) return 0;
        if (w >= W) return P[B];
        const long long vt = (w * V() + W - 1) / W;
        int lo = 0, hi = B - 1;  // largest b with VP[b] <= vt
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (VP[mid] <= vt) lo = mid;
            else hi = mid - 1;
        }
        if (VP[lo + 1] <= vt) return P[lo + 1];
        const int nt = (P[lo + 1] - P[lo]) / segs;
        const long long o = vt - VP[lo];
        const long long sg = o / (nt + ALPHA);
        const long long r = o - sg * (nt + ALPHA);
        return P[lo] + static_cast<int>(sg * nt + (r < nt ? r : nt));
    }

    // worker holding tile i of segment seg (nt tiles) of slot b
    __device__ int worker_at(int b, int seg, int nt, int i) const {
        const long long v = VP[b] + static_cast<long long>(seg) * (nt + ALPHA) + i;
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

// ================================================================ kernel
template <typename CT, int D, int G>
__global__ void __launch_bounds__(Tiling<CT, D, G>::WARPS * 32, 1) decode_splitk_kernel(const DecodeParams p) {
    using TL = Tiling<CT, D, G>;
    constexpr int T = TL::T, R = TL::R, EPL = TL::EPL, ROW = TL::ROW, SPW = TL::SPW, RB = TL::RB;
    constexpr int TILE = TL::TILE, SCL = TL::SCL, STAGE = TL::STAGE, EB = TL::EB;
    constexpr bool I8 = TL::I8;
    // INT8 blocks of <= 2 query rows on 32-row tiles: P.V on dp4a with integer weights
    constexpr bool IPV = I8 && G <= 2 && T == 32;
    constexpr unsigned FULL = 0xffffffffu;

    extern __shared__ __align__(128) unsigned char smem[];
    int* P = reinterpret_cast<int*>(smem);  // [B + 1] tile prefix over slots
    int* Ls = P + (kMaxBatch + 1);          // [B] cached length, -1 when the slot has no work
    int* VP = TL::HAVE_VP ? Ls + kMaxBatch : P;  // [B + 1] weighted prefix: tiles + ALPHA per segment
    int* rv = P + (TL::HAVE_VP ? 3 : 2) * kMaxBatch + 2;  // re-planning meeting counter (prefix slack)

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int hr = lane >> 4, c = lane & 15;
    unsigned char* wbase = smem + TL::PREFIX_BYTES + warp * TL::WARP_BYTES;
    float* sc = reinterpret_cast<float*>(wbase + SPW * STAGE);  // [G][T] scores
    float* pb = sc + G * T;                                     // [G][T] weights
    uint64_t* bars = reinterpret_cast<uint64_t*>(wbase + SPW * STAGE + TL::SCRATCH);
    const int segs = p.Hkv * p.nhb;

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < SPW; ++s) mbar_init(smem_addr(&bars[s]), 1);
    }
    if (threadIdx.x == 0) *rv = 0;
    // The split depends only on the lengths, so it is computed before waiting on
    // the previous launch: a block that starts while the previous step drains
    // then warms L2 with its first tiles (contiguous caches) instead of idling:
    // each warp's first tile, or, for INT8 caches, as many tiles as it has stages
    // (measured after a GEMM and back to back: deeper prefetches of the fp16/bf16
    // tiles queue ahead of the first demand copies and lengthen the step's start).
    // After the wait the lengths are checked again (lengths_changed).  Everything
    // that reads the caches' contents or writes memory comes after the wait.
    bool ovf = false;
    if (warp == 0) ovf = build_prefix(p, T, segs, TL::ALPHA, P, VP, Ls, lane);
    fence_mbar_init();
    __syncthreads();

    const long long W = static_cast<long long>(gridDim.x) * TL::WARPS;
    const int wid = blockIdx.x * TL::WARPS + warp;
    const WeightedSplit<TL::ALPHA> split{P, VP, p.B, segs, static_cast<int>(W)};
    int t_begin = split.begin(wid);
    int n_my = split.begin(wid + 1) - t_begin;
    if (n_my > 0 && lane == 0 && !p.block_table) {
        Cursor c = locate(t_begin, P, p.B, segs);
        constexpr int NPF = I8 ? SPW : 1;  // tiles prefetched per warp
        for (int k = 0; k < min(NPF, n_my); ++k) {
            const int L = Ls[c.b];
            const int t0 = (window_start(L, p.window) / T + c.tile) * T;
            const int n_cache = min(T, max(0, L - t0));
            if (n_cache > 0) {
                const size_t rb = static_cast<size_t>(cache_row(p, c.b, c.seg / p.nhb, t0, 0));
                bulk_prefetch_l2(p.k_cache + rb * ROW, static_cast<uint32_t>(n_cache) * ROW);
                bulk_prefetch_l2(p.v_cache + rb * ROW, static_cast<uint32_t>(n_cache) * ROW);
            }
            if (k + 1 < min(NPF, n_my)) advance(c, P, segs);
        }
    }
    grid_dep_wait();    // inputs, caches and outputs may be in use by the previous launch
    grid_dep_launch();  // the next step may take SMs as this grid's blocks finish
    if (lengths_changed(p, Ls, lane)) {
        // (rare) the lengths changed after this block read them: the warps meet, warp 0
        // rebuilds the split from the lengths now visible, they meet again
        if (!warp_rendezvous(rv, TL::WARPS, p.wait_cycles, p.err, lane)) return;
        if (warp == 0) ovf = build_prefix(p, T, segs, TL::ALPHA, P, VP, Ls, lane);
        if (!warp_rendezvous(rv, 2 * TL::WARPS, p.wait_cycles, p.err, lane)) return;
        t_begin = split.begin(wid);
        n_my = split.begin(wid + 1) - t_begin;
    }
    if (ovf && warp == 0 && lane == 0 && blockIdx.x == 0) atomicOr(p.err, kErrSeqOverflow);

    // Slots without work (inactive or overflowing) get a zero output.
    for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
        if (P[b + 1] == P[b]) {
            zero_outputs(p, static_cast<size_t>(b) * p.nq * p.Hq * D, p.nq * p.Hq * D);
        }
    }
    if (n_my <= 0) return;

    // ---- bulk copies of one tile (lane 0 only) ----
    // Paged caches: the page of the tile comes from the block table; the entry
    // of the current page is kept and the next page's entry is loaded early.
    PageCursor pages;
    const uint64_t l2pol = l2_stream_policy();
    // Test hook (DecodeParams::stall): worker 0 never issues its first tile, so its
    // bounded wait runs out and the abort path runs.
    const bool stall_me = p.stall && wid == 0;
    auto issue = [&](int s, const Cursor& cu) {
        const int L = Ls[cu.b];
        const int t0 = (window_start(L, p.window) / T + cu.tile) * T;
        const int n_cache = min(T, max(0, L - t0));  // rows before the new tokens come from the cache
        const int kvh = cu.seg / p.nhb;
        const long long rb = cache_row(p, cu.b, kvh, t0, pages.page(p, cu.b, t0));
        if (rb < 0) atomicOr(p.err, kErrBadPage);
        const size_t rowbase = rb < 0 ? 0 : static_cast<size_t>(rb);
        const uint32_t kb = rb < 0 ? 0u : static_cast<uint32_t>(n_cache) * ROW;
        const uint32_t sb = (I8 && rb >= 0) ? static_cast<uint32_t>((n_cache * 4 + 15) & ~15) : 0u;
        unsigned char* st = wbase + s * STAGE;
        const uint32_t bar = smem_addr(&bars[s]);
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, 2 * kb + 2 * sb);
        if (kb) {
            bulk_g2s_hint(smem_addr(st), p.k_cache + rowbase * ROW, kb, bar, l2pol);
            bulk_g2s_hint(smem_addr(st + TILE), p.v_cache + rowbase * ROW, kb, bar, l2pol);
        }
        if constexpr (I8) {
            if (sb) {
                bulk_g2s_hint(smem_addr(st + 2 * TILE), p.k_scales + rowbase, sb, bar, l2pol);
                bulk_g2s_hint(smem_addr(st + 2 * TILE + SCL), p.v_scales + rowbase, sb, bar, l2pol);
            }
        }
    };

    // When the copy cursor enters a segment, pull that segment's q rows and new
    // K/V rows into L1: the compute cursor reaches them SPW tiles later and then
    // finds them on chip instead of stalling on a global round trip mid-stream.
    // (The issue-bound INT8 instantiation does better without the extra work.)
    const int qeb = p.qkv_dtype == kF32 ? 4 : 2;
    auto prefetch_segment = [&](const Cursor& cu) {
        const int kvh = cu.seg / p.nhb, hb = cu.seg % p.nhb;
        const int lines = D * qeb / 128;  // 128-byte lines per row
        const int nlines = (G + 2 * p.nq) * lines;
        for (int i = lane; i < nlines; i += 32) {
            const int row = i / lines, part = i - row * lines;
            const unsigned char* base;
            if (row < G) {
                base = static_cast<const unsigned char*>(p.q) + q_row(p, cu.b, kvh, hb * G + row) * D * qeb;
            } else {
                const int tok = (row - G) % p.nq;
                const void* src = row < G + p.nq ? p.k_new : p.v_new;
                base = static_cast<const unsigned char*>(src) +
                       ((static_cast<size_t>(cu.b) * p.nq + tok) * p.Hkv + kvh) * D * qeb;
            }
            asm volatile("prefetch.global.L1 [%0];" ::"l"(base + part * 128));
        }
    };

    Cursor ci = locate(t_begin, P, p.B, segs);
    Cursor cc = ci;
    if (!I8) prefetch_segment(ci);  // the first segment's new K/V rows are needed at its last tile
    const int npre = min(SPW, n_my);
    for (int k = 0; k < npre; ++k) {
        if (lane == 0 && !(stall_me && k == 0)) issue(k, ci);
        if (k + 1 < n_my) {
            advance(ci, P, segs);
            if (!I8 && ci.tile == 0) prefetch_segment(ci);
        }
    }

    float qr[G][EPL], o[G][EPL], m[G], l[G];
    int tk[G];  // token of each query row (0 unless several new tokens per step)
    // INT8 caches: the scaled query as two int8 levels, q ~ s1 * hi + (s1 / 254) * lo, so
    // q . k runs as dp4a integer dot products with the int8 codes (four products per
    // instruction) and needs no per-byte conversion; relative error about 1.5e-5 of max |q|,
    // the same budget as the tensor-core kernel's hi/lo split.  qsc = s1 / 254.
    uint32_t qh[G][I8 ? EPL / 4 : 1], ql[G][I8 ? EPL / 4 : 1];
    float qsc[G];
    auto begin_segment = [&](const Cursor& cu) {
        const int kvh = cu.seg / p.nhb, hb = cu.seg % p.nhb;
#pragma unroll
        for (int j = 0; j < G; ++j) {
            const size_t qrow = q_row(p, cu.b, kvh, hb * G + j);
            tk[j] = q_token(p, hb * G + j);
            const int h = kvh * p.group + (hb * G + j - tk[j] * p.group);
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                const int d = c * EPL + e;
                float x = ld_qkv(p.q, p.qkv_dtype, qrow * D + d);
                if (p.bias) x += ld_qkv(p.bias, p.qkv_dtype, static_cast<size_t>(h) * D + d);
                qr[j][e] = x * p.qscale;
                o[j][e] = 0.f;
            }
            m[j] = -INFINITY;
            l[j] = 0.f;
            if constexpr (I8) {
                float amax = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(qr[j][e]));
#pragma unroll
                for (int mm = 8; mm >= 1; mm >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, mm));
                const float s1 = amax > 0.f ? amax / 127.f : 1.f;
                const float inv1 = 1.f / s1, inv2 = 254.f / s1;
#pragma unroll
                for (int w = 0; w < EPL / 4; ++w) {
                    uint32_t hw = 0u, lw = 0u;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float x = qr[j][4 * w + k];
                        const int hi = max(-127, min(127, __float2int_rn(x * inv1)));
                        const int lo = max(-127, min(127, __float2int_rn((x - static_cast<float>(hi) * s1) * inv2)));
                        hw |= (static_cast<uint32_t>(hi) & 0xffu) << (8 * k);
                        lw |= (static_cast<uint32_t>(lo) & 0xffu) << (8 * k);
                    }
                    qh[j][w] = hw;
                    ql[j][w] = lw;
                }
                qsc[j] = s1 / 254.f;
            }
        }
    };
    begin_segment(cc);
    int piece_first = cc.tile;

    // Log-sum-exp merge of all partials of segment mc, by the worker whose
    // arrival completed its tile count; then the counter is reset for the next launch.
    auto merge_segment = [&](const Cursor& mc) {
        const int segg = mc.b * segs + mc.seg;
        const int kvh = mc.seg / p.nhb, hb = mc.seg % p.nhb;
        const int wf = split.worker_at(mc.b, mc.seg, mc.nt, 0);
        const int wl = split.worker_at(mc.b, mc.seg, mc.nt, mc.nt - 1);
        auto has_piece = [&](int w) { return split.has_piece(w, wf, wl); };
        // one pass over the pieces with a running log-sum-exp per query row
        constexpr int DL = D / 32;
        float Mx[G], Ls_[G], Ac[G][DL];
#pragma unroll
        for (int j = 0; j < G; ++j) {
            Mx[j] = -INFINITY;
            Ls_[j] = 0.f;
#pragma unroll
            for (int e = 0; e < DL; ++e) Ac[j][e] = 0.f;
        }
        // pieces in batches of NB: the loads of a batch are issued together, so a merge
        // costs one L2 round trip per batch rather than one per piece
        constexpr int NB = G >= 8 ? 1 : 8 / G;
        if constexpr (NB == 1) {  // eight query rows: one piece at a time keeps registers in budget
            for (int w = wf; w <= wl; ++w) {
                if (!has_piece(w)) continue;
                const float* sl = p.ws + static_cast<size_t>(segg + w) * TL::SLOT;
                float mw[G], lw[G], ow[G][DL];
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    mw[j] = __ldcg(sl + j);
                    lw[j] = __ldcg(sl + G + j);
                    const float* ov = sl + TL::OOFF + j * D + lane * DL;
                    if constexpr (DL == 4) {
                        const float4 u = __ldcg(reinterpret_cast<const float4*>(ov));
                        ow[j][0] = u.x; ow[j][1] = u.y; ow[j][2] = u.z; ow[j][3] = u.w;
                    } else {
                        const float2 u = __ldcg(reinterpret_cast<const float2*>(ov));
                        ow[j][0] = u.x; ow[j][1] = u.y;
                    }
                }
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    const float mn = fmaxf(Mx[j], mw[j]);
                    const float mref = mn == -INFINITY ? 0.f : mn;
                    const float a = exp2f(Mx[j] - mref), bb = exp2f(mw[j] - mref);
                    Ls_[j] = Ls_[j] * a + lw[j] * bb;
#pragma unroll
                    for (int e = 0; e < DL; ++e) Ac[j][e] = Ac[j][e] * a + ow[j][e] * bb;
                    Mx[j] = mn;
                }
            }
        } else {
            for (int w0 = wf; w0 <= wl; w0 += NB) {
                float mw[NB][G], lw[NB][G], ow[NB][G][DL];
#pragma unroll
                for (int i = 0; i < NB; ++i) {
                    const int w = w0 + i;
                    const bool ok = w <= wl && has_piece(w);
                    const float* sl = p.ws + static_cast<size_t>(segg + (ok ? w : wf)) * TL::SLOT;
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        mw[i][j] = ok ? __ldcg(sl + j) : -INFINITY;
                        lw[i][j] = ok ? __ldcg(sl + G + j) : 0.f;
                        const float* ov = sl + TL::OOFF + j * D + lane * DL;
                        if constexpr (DL == 4) {
                            float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (ok) u = __ldcg(reinterpret_cast<const float4*>(ov));
                            ow[i][j][0] = u.x; ow[i][j][1] = u.y; ow[i][j][2] = u.z; ow[i][j][3] = u.w;
                        } else {
                            float2 u = make_float2(0.f, 0.f);
                            if (ok) u = __ldcg(reinterpret_cast<const float2*>(ov));
                            ow[i][j][0] = u.x; ow[i][j][1] = u.y;
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < NB; ++i) {
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        // a piece whose tiles a query row could not see yet (or an empty batch
                        // entry) has m = -inf and contributes nothing
                        const float mn = fmaxf(Mx[j], mw[i][j]);
                        const float mref = mn == -INFINITY ? 0.f : mn;
                        const float a = exp2f(Mx[j] - mref), bb = exp2f(mw[i][j] - mref);
                        Ls_[j] = Ls_[j] * a + lw[i][j] * bb;
#pragma unroll
                        for (int e = 0; e < DL; ++e) Ac[j][e] = Ac[j][e] * a + ow[i][j][e] * bb;
                        Mx[j] = mn;
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < G; ++j) {
            const size_t dst = q_row(p, mc.b, kvh, hb * G + j) * D + lane * DL;
            const float inv = 1.f / Ls_[j];
            if constexpr (DL == 4) {
                store_out4(p, dst, Ac[j][0] * inv, Ac[j][1] * inv, Ac[j][2] * inv, Ac[j][3] * inv);
            } else {
#pragma unroll
                for (int e = 0; e < DL; ++e) store_out1(p, dst + e, Ac[j][e] * inv);
            }
        }
        if (lane == 0) p.counters[segg] = 0u;
    };
    // Read lane 0's arrival result; the arrival that completes the count merges.
    auto resolve = [&](uint32_t r0, const Cursor& mc, uint32_t tiles) {
        const uint32_t prev = __shfl_sync(FULL, r0, 0);
        if (prev + tiles == static_cast<uint32_t>(mc.nt)) {
            __syncwarp();  // lane 0's acquire orders every lane's merge reads
            merge_segment(mc);
        }
    };
    bool pend = false;  // a mid-stream arrival whose answer is still to be read
    uint32_t pend_ret = 0, pend_tiles = 0;
    Cursor pend_cu{};

    int k = 0;
    for (; k < n_my; ++k) {
        const int s = k % SPW;
        unsigned char* st = wbase + s * STAGE;
        if (!mbar_wait_bounded(smem_addr(&bars[s]), static_cast<uint32_t>((k / SPW) & 1), p.err, p.wait_cycles))
            break;
        if (pend) {  // the arrival of the piece that ended one tile ago has returned by now
            resolve(pend_ret, pend_cu, pend_tiles);
            pend = false;
        }

        const int L = Ls[cc.b];
        const int pos0 = window_start(L, p.window);  // window start of the first new token
        const int t0 = (pos0 / T + cc.tile) * T;
        const int n_total = min(T, L + p.nq - t0);   // rows holding data (history or new tokens)
        const int r_lo = max(0, pos0 - t0);          // rows before the window start are masked
        const bool last_tile = cc.tile == cc.nt - 1;
        const int kvh = cc.seg / p.nhb, hb = cc.seg % p.nhb;

        // ---- append: rows at positions L .. L + nq - 1 are the new tokens ----
        for (int nr = max(0, L - t0); nr < n_total; ++nr) {
            const int tok = t0 + nr - L;  // token of this row
            const int pos = t0 + nr;
            const bool isv = hr != 0;   // half-warp 0 writes K, half-warp 1 writes V
            const void* src = isv ? p.v_new : p.k_new;
            const size_t si = ((static_cast<size_t>(cc.b) * p.nq + tok) * p.Hkv + kvh) * D + c * EPL;
            const size_t bi = static_cast<size_t>(p.Hq + (isv ? p.Hkv : 0) + kvh) * D + c * EPL;
            float x[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                x[e] = ld_qkv(src, p.qkv_dtype, si + e);
                if (p.bias) x[e] += ld_qkv(p.bias, p.qkv_dtype, bi + e);  // one binary32 add
            }
            const long long rowL = cache_row(p, cc.b, kvh, pos, page_of(p, cc.b, pos));  // cache row of pos
            const bool gok = rowL >= 0 && hb == 0;  // the first head block writes the cache
            unsigned char* srow = st + (isv ? TILE : 0) + nr * ROW + c * EPL * EB;
            unsigned char* grow = (isv ? p.v_cache : p.k_cache) + (gok ? rowL : 0) * ROW + c * EPL * EB;
            if constexpr (I8) {
                float amax = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
                for (int mm = 8; mm >= 1; mm >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, mm));
                const float qs = amax == 0.f ? 1.f : __fdiv_rn(amax, 127.f);
                uint32_t w[EPL / 4];
#pragma unroll
                for (int k4 = 0; k4 < EPL / 4; ++k4) w[k4] = 0u;
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    int code = 0;
                    if (amax != 0.f) code = max(-127, min(127, __float2int_rn(__fdiv_rn(x[e], qs))));
                    w[e / 4] |= (static_cast<uint32_t>(code) & 0xffu) << (8 * (e % 4));
                }
                if constexpr (EPL == 8) {
                    *reinterpret_cast<uint2*>(srow) = make_uint2(w[0], w[1]);
                    if (gok) *reinterpret_cast<uint2*>(grow) = make_uint2(w[0], w[1]);
                } else {
                    *reinterpret_cast<uint32_t*>(srow) = w[0];
                    if (gok) *reinterpret_cast<uint32_t*>(grow) = w[0];
                }
                if (c == 0) {
                    reinterpret_cast<float*>(st + 2 * TILE + (isv ? SCL : 0))[nr] = qs;
                    if (gok) (isv ? p.v_scales : p.k_scales)[rowL] = qs;
                }
            } else {
                cvt_st<CT, EPL>(srow, x);
                if (gok) cvt_st<CT, EPL>(grow, x);
            }
            __syncwarp();
        }

        // ---- scores: q . k for every row, reduced across the 16 lanes ----
        const unsigned char* Kt = st;
        const unsigned char* Vt = st + TILE;
#pragma unroll
        for (int ib = 0; ib < R / RB; ++ib) {
            if constexpr (I8) {
                // integer partial sums 254 * (hi . k) + (lo . k): |value| < 2^31 for D <= 128
                int part[G * RB];
#pragma unroll
                for (int i = 0; i < RB; ++i) {
                    const int row = 2 * (ib * RB + i) + hr;
                    uint32_t kw[EPL / 4];
                    if constexpr (EPL == 8) {
                        const uint2 u = *reinterpret_cast<const uint2*>(Kt + row * ROW + c * EPL);
                        kw[0] = u.x;
                        kw[EPL / 4 - 1] = u.y;
                    } else {
                        kw[0] = *reinterpret_cast<const uint32_t*>(Kt + row * ROW + c * EPL);
                    }
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        int ah = 0, al = 0;
#pragma unroll
                        for (int w = 0; w < EPL / 4; ++w) {
                            ah = __dp4a(static_cast<int>(kw[w]), static_cast<int>(qh[j][w]), ah);
                            al = __dp4a(static_cast<int>(kw[w]), static_cast<int>(ql[j][w]), al);
                        }
                        part[j * RB + i] = ah * 254 + al;
                    }
                }
                int idx = 0;
                ReduceScatter<G * RB, 8, int>::run(part, c, idx);
                const int j = idx / RB, i = idx % RB;
                sc[j * T + 2 * (ib * RB + i) + hr] = static_cast<float>(part[0]) * qsc[j];
            } else {
                float part[G * RB];
#pragma unroll
                for (int i = 0; i < RB; ++i) {
                    const int row = 2 * (ib * RB + i) + hr;
                    float kf[EPL];
                    ld_cvt<CT, EPL>(Kt + row * ROW + c * EPL * EB, kf);
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        float a = 0.f;
#pragma unroll
                        for (int e = 0; e < EPL; ++e) a = fmaf(qr[j][e], kf[e], a);
                        part[j * RB + i] = a;
                    }
                }
                int idx = 0;
                ReduceScatter<G * RB, 8>::run(part, c, idx);
                const int j = idx / RB, i = idx % RB;
                sc[j * T + 2 * (ib * RB + i) + hr] = part[0];
            }
        }
        __syncwarp();

        // ---- online softmax over the tile (log2 domain) ----
        float alpha[G];
        float wsc[G];  // dp4a P.V: the tile's weight scale per query row
        const int r = lane % T;
        // query row j sees rows [lo_j, hi_j) of the tile: positions up to L + tk[j], and from
        // its own window start on
        const int hi0 = L + 1 - t0, lo0 = p.window > 0 ? L + 1 - p.window - t0 : -(1 << 30);
        const bool full = hi0 + tk[0] >= T && lo0 + tk[G - 1] <= 0;  // every query row sees every row
#pragma unroll
        for (int j = 0; j < G; ++j) {
            float sv = -INFINITY;
            if (full || (r >= lo0 + tk[j] && r < hi0 + tk[j])) {
                sv = sc[j * T + r];
                if constexpr (I8) sv *= reinterpret_cast<const float*>(st + 2 * TILE)[r];
            }
            float tmax = sv;
#pragma unroll
            for (int mm = T / 2; mm >= 1; mm >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(FULL, tmax, mm));
            const float mnew = fmaxf(m[j], tmax);
            // a query row with no visible row yet keeps m = -inf; 0 stands in as the reference
            const float mref = (!full && mnew == -INFINITY) ? 0.f : mnew;
            alpha[j] = exp2f(m[j] - mref);
            const float pv = exp2f(sv - mref);
            float tsum = pv;
#pragma unroll
            for (int mm = T / 2; mm >= 1; mm >>= 1) tsum += __shfl_xor_sync(FULL, tsum, mm);
            l[j] = l[j] * alpha[j] + tsum;
            m[j] = mnew;
            if constexpr (IPV) {
                // weights w = p * vscale as three int8 levels of the tile's largest weight,
                // w ~ s1 (h + m / 254 + q / 254^2), byte-packed per group of 4 rows of a half-warp
                const float wgt =
                    (r >= r_lo && r < n_total) ? pv * reinterpret_cast<const float*>(st + 2 * TILE + SCL)[r] : 0.f;
                float wmax = wgt;
#pragma unroll
                for (int mm = 16; mm >= 1; mm >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(FULL, wmax, mm));
                const float s1 = wmax > 0.f ? wmax / 127.f : 1.f;
                const float inv1 = 1.f / s1;
                const int h = __float2int_rn(wgt * inv1);
                const float r1 = wgt - static_cast<float>(h) * s1;
                const int mq = max(-127, min(127, __float2int_rn(r1 * (254.f * inv1))));
                const float r2 = r1 - static_cast<float>(mq) * (s1 * (1.f / 254.f));
                const int lq = max(-127, min(127, __float2int_rn(r2 * (64516.f * inv1))));
                const int rh = r & 1, gi = (r >> 1) >> 2, kk = (r >> 1) & 3;  // half-warp, group, position
                signed char* pq = reinterpret_cast<signed char*>(pb);
#pragma unroll
                for (int lv = 0; lv < 3; ++lv)
                    pq[((((lv * G + j) * 2 + rh) * 4 + gi) * 4) + kk] =
                        static_cast<signed char>(lv == 0 ? h : (lv == 1 ? mq : lq));
                wsc[j] = s1;
            } else if (lane < T) {
                float wgt = pv;
                if constexpr (I8)
                    wgt = (r >= r_lo && r < n_total) ? pv * reinterpret_cast<const float*>(st + 2 * TILE + SCL)[r] : 0.f;
                pb[j * T + r] = wgt;
            }
        }
        __syncwarp();

        // ---- o = alpha * o + sum_rows p * v ----
#pragma unroll
        for (int j = 0; j < G; ++j)
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[j][e] *= alpha[j];
        auto pv_row = [&](int row) {
            float vf[EPL];
            ld_cvt<CT, EPL>(Vt + row * ROW + c * EPL * EB, vf);
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const float pj = pb[j * T + row];
#pragma unroll
                for (int e = 0; e < EPL; ++e) o[j][e] = fmaf(pj, vf[e], o[j][e]);
            }
        };
        if constexpr (IPV) {
            // dp4a P.V: four rows of codes, transposed so each word holds one column's four
            // bytes, times the four rows' packed weights, for each weight level.  Rows with
            // weight 0 (masked or stale) contribute nothing; codes are plain integers.
            int acc[G][EPL][3];
#pragma unroll
            for (int j = 0; j < G; ++j)
#pragma unroll
                for (int e = 0; e < EPL; ++e)
#pragma unroll
                    for (int lv = 0; lv < 3; ++lv) acc[j][e][lv] = 0;
            const int* pw = reinterpret_cast<const int*>(pb);
#pragma unroll
            for (int g = 0; g < R / 4; ++g) {
                uint32_t col[EPL];
#pragma unroll
                for (int half = 0; half < EPL / 4; ++half) {
                    uint32_t a[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        a[k] = *reinterpret_cast<const uint32_t*>(Vt + (2 * (4 * g + k) + hr) * ROW + c * EPL + 4 * half);
                    const uint32_t t0 = __byte_perm(a[0], a[1], 0x5140), t1 = __byte_perm(a[0], a[1], 0x7362);
                    const uint32_t t2 = __byte_perm(a[2], a[3], 0x5140), t3 = __byte_perm(a[2], a[3], 0x7362);
                    col[4 * half + 0] = __byte_perm(t0, t2, 0x5410);
                    col[4 * half + 1] = __byte_perm(t0, t2, 0x7632);
                    col[4 * half + 2] = __byte_perm(t1, t3, 0x5410);
                    col[4 * half + 3] = __byte_perm(t1, t3, 0x7632);
                }
#pragma unroll
                for (int j = 0; j < G; ++j)
#pragma unroll
                    for (int lv = 0; lv < 3; ++lv) {
                        const int wq = pw[((lv * G + j) * 2 + hr) * 4 + g];
#pragma unroll
                        for (int e = 0; e < EPL; ++e) acc[j][e][lv] = __dp4a(static_cast<int>(col[e]), wq, acc[j][e][lv]);
                    }
            }
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const float s2 = wsc[j] * (1.f / 254.f);
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    const float hm = static_cast<float>(acc[j][e][0] * 254 + acc[j][e][1]);
                    o[j][e] = fmaf(s2, hm + static_cast<float>(acc[j][e][2]) * (1.f / 254.f), o[j][e]);
                }
            }
        } else if (r_lo == 0 && n_total == T) {  // whole tile visible: no per-row test
#pragma unroll
            for (int i = 0; i < R; ++i) pv_row(2 * i + hr);
        } else {  // rows outside [r_lo, n_total) hold stale stage data and are skipped
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const int row = 2 * i + hr;
                if (row >= r_lo && row < n_total) pv_row(row);
            }
        }
        __syncwarp();

        // ---- refill this stage with the tile SPW ahead ----
        if (k + SPW < n_my) {
            if (lane == 0) issue(s, ci);
            if (k + SPW + 1 < n_my) {
                advance(ci, P, segs);
                if (!I8 && ci.tile == 0) prefetch_segment(ci);
            }
        }

        // ---- end of a piece: final output, or partial + merge by the last arrival ----
        if (last_tile || k == n_my - 1) {
#pragma unroll
            for (int j = 0; j < G; ++j)
#pragma unroll
                for (int e = 0; e < EPL; ++e) o[j][e] += __shfl_xor_sync(FULL, o[j][e], 16);
            const int segg = cc.b * segs + cc.seg;
            if (piece_first == 0 && last_tile) {
                if (hr == 0) {
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        const float inv = 1.f / l[j];
                        const size_t dst = q_row(p, cc.b, kvh, hb * G + j) * D + c * EPL;
#pragma unroll
                        for (int e4 = 0; e4 < EPL / 4; ++e4)
                            store_out4(p, dst + 4 * e4, o[j][4 * e4] * inv, o[j][4 * e4 + 1] * inv,
                                       o[j][4 * e4 + 2] * inv, o[j][4 * e4 + 3] * inv);
                    }
                }
            } else {
                float* slot = p.ws + static_cast<size_t>(segg + wid) * TL::SLOT;
                if (lane == 0) {
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        slot[j] = m[j];
                        slot[G + j] = l[j];
                    }
                }
                if (hr == 0) {
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        float* dst = slot + TL::OOFF + j * D + c * EPL;
#pragma unroll
                        for (int e4 = 0; e4 < EPL / 4; ++e4)
                            reinterpret_cast<float4*>(dst)[e4] =
                                make_float4(o[j][4 * e4], o[j][4 * e4 + 1], o[j][4 * e4 + 2], o[j][4 * e4 + 3]);
                    }
                }
                __syncwarp();  // every lane's partial stores come before lane 0's release
                // The counter accumulates tiles, not pieces: when U < W some
                // workers own no tile, so the number of pieces is not wf..wl.
                const uint32_t piece_tiles = static_cast<uint32_t>(cc.tile - piece_first + 1);
                uint32_t ret = 0;
                if (lane == 0) ret = arrive_acq_rel(&p.counters[segg], piece_tiles);
                if (k == n_my - 1) {
                    resolve(ret, cc, piece_tiles);
                } else {
                    // the worker streams on; the atomic's answer is read after the next tile
                    pend = true;
                    pend_ret = ret;
                    pend_cu = cc;
                    pend_tiles = piece_tiles;
                }
            }
            if (k + 1 < n_my) {
                advance(cc, P, segs);
                begin_segment(cc);
                piece_first = cc.tile;
            }
        } else {
            advance(cc, P, segs);
        }
    }

    if (k < n_my) {
        // A copy did not arrive in time: the error bit is set.  Wait for the
        // copies this warp still has in flight before leaving (tiles k .. k +
        // SPW - 1 were issued, all but a withheld one), with the long drain
        // limit, so no transfer lands in shared memory after the block has exited.
        const int last_issued = min(n_my, k + SPW) - 1;
        for (int kk = k; kk <= last_issued; ++kk)
            if (!(stall_me && kk == 0))
                mbar_wait_bounded(smem_addr(&bars[kk % SPW]), static_cast<uint32_t>((kk / SPW) & 1), p.err,
                                  kDrainLimitCycles);
    }
}

// ---------------------------------------------------------- host selection
struct KernelInfo {
    const void* fn;
    int smem;
    int T;
    int slot_floats;
    int G;
    int warps;  // workers (warps) per CTA; the launch uses warps * 32 threads
};

template <typename CT, int D, int G>
KernelInfo kernel_info() {
    using TL = Tiling<CT, D, G>;
    return KernelInfo{reinterpret_cast<const void*>(&decode_splitk_kernel<CT, D, G>), TL::SMEM, TL::T, TL::SLOT, G,
                      TL::WARPS};
}

template <typename CT>
KernelInfo select_kernel(int D, int G) {
    if (D == 64) {
        switch (G) {
            case 1: return kernel_info<CT, 64, 1>();
            case 2: return kernel_info<CT, 64, 2>();
            case 4: return kernel_info<CT, 64, 4>();
            case 8: return kernel_info<CT, 64, 8>();
        }
    } else if (D == 128) {
        switch (G) {
            case 1: return kernel_info<CT, 128, 1>();
            case 2: return kernel_info<CT, 128, 2>();
            case 4: return kernel_info<CT, 128, 4>();
            case 8: return kernel_info<CT, 128, 8>();
        }
    }
    return KernelInfo{nullptr, 0, 0, 0, 0};
}

void set_last_error(const char* msg);
void note_launch();

KernelInfo select_f32(int D, int G);
KernelInfo select_f16(int D, int G);
KernelInfo select_bf16(int D, int G);
KernelInfo select_i8(int D, int G);

}  // namespace ftd
