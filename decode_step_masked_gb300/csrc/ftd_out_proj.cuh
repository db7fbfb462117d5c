// ftd_out_proj.cuh -- the output projection that follows the decode step, on
// the 5th-generation tensor cores (tcgen05 + TMEM + TMA, sm_103a).
//
// The fused attention kernels hand their result straight to the next
// projection in half precision ("FasterTransformer practice", lpnh.cn,
// section 2.1).  Here the decode kernels' final stores write each output value
// also as a high and a low half of the projection's operand type (planes Oh, Ol
// laid out like out: [tokens][Hq * D]), and this kernel, launched right after
// them on the same stream, computes for every token t and output feature f
//
//   y[t][f] = sum_k W[f][k] * (Oh[t][k] + Ol[t][k]),   k < K = Hq * D,
//
// with W the caller's [F][K] weight (nn.Linear layout) in the same type, so the
// product keeps about 16 mantissa bits of the fp32 attention output.  The
// product is a skinny GEMM: a decode step has few tokens (the batch), so the
// time is the one read of W from HBM.  W takes the MMA's A side (M = 128 output
// features per tile) and the tokens its N side:
//
//   Y^T [128 x 2 NTB] = W_tile [128 x 64] . [Oh; Ol]^T [64 x 2 NTB]   per unit,
//
// accumulated over the K chunks of a tile in TMEM.  Units (token block, feature
// tile, K chunk of 64) are ordered K-fastest and split into equal contiguous
// ranges over one persistent CTA per SM; a CTA's units of one tile form a piece,
// whose fp32 partial goes to the workspace, and the piece whose arrival completes
// the tile's K chunks sums the partials and writes y (as the decode kernels
// merge their split-K partials).  W tiles are independent of the decode step,
// so the first stages' W copies are issued before griddepcontrol.wait and
// overlap the decode kernel's last blocks; the O copies follow the wait.
//
// Roles (192 threads): warp 0 TMA producer, warp 1 TMEM allocation and MMA
// issue, warps 2-5 the epilogue (warp w reads TMEM lanes 32 (w % 4) ..).
#pragma once

#include <cuda.h>

#include "ftd_decode_gqa_tc.cuh"

namespace ftd {
namespace op {

constexpr int MT = 128;                  // output features per tile (MMA M)
constexpr int KCH = 64;                  // K elements per unit: one 128-byte swizzled row
constexpr int WBYTES = MT * KCH * 2;     // one W tile of a unit (16 KB)
constexpr int kMaxStages = 8;
constexpr int kStageBudget = 196608;     // shared memory for the stage ring
constexpr int kMaxNtb = 128;             // tokens per block, a multiple of 16 (N = 2 NTB <= 256)
constexpr int kThreads = 192;

// stage = W tile, then the Oh and Ol boxes of NTB rows each; as many stages as fit the
// budget, at most 8 (eight 16 KB W tiles in flight per SM keep HBM busy)
__host__ __device__ constexpr int stage_bytes(int ntb) { return WBYTES + 2 * ntb * 128; }
__host__ __device__ constexpr int stages_for(int ntb) {
    return kStageBudget / stage_bytes(ntb) < kMaxStages ? kStageBudget / stage_bytes(ntb) : kMaxStages;
}
__host__ __device__ constexpr int smem_bytes(int ntb) { return stages_for(ntb) * stage_bytes(ntb) + 1024 + 1024; }

enum : int { kFull = 0, kEmpty = kMaxStages, kAccFull = 2 * kMaxStages, kAccEmpty = 2 * kMaxStages + 2,
             kDrain = 2 * kMaxStages + 4, kNumBarsP = 2 * kMaxStages + 5 };

}  // namespace op

struct ProjParams {
    void* y;              // [tokens][F], out dtype
    float* ws;            // partial slots [tiles + grid][NTB][128]
    uint32_t* counters;   // one arrival counter (K chunks) per tile (token block, feature tile), zero between launches
    uint32_t* err;        // sticky error word (shared with the decode step)
    int tokens;           // B * q_len
    int ntb;              // tokens per block: a multiple of 16, <= 128
    int nblk;             // token blocks
    int mtiles;           // F / 128
    int kch;              // K / 64
    int out_dtype;        // kF32 / kF16 / kBF16
    long long wait_cycles;
};

template <bool BF>
__global__ void __launch_bounds__(op::kThreads, 1)
    out_proj_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmh,
                    const __grid_constant__ CUtensorMap tml, const ProjParams pp) {
    using namespace op;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
    const int NTB = pp.ntb, N = 2 * NTB;
    const int SB = stage_bytes(NTB);
    const int NSTAGE = stages_for(NTB);
    unsigned char* misc = smem + NSTAGE * SB;
    uint64_t* bars = reinterpret_cast<uint64_t*>(misc);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + kNumBarsP * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + kNumBarsP * 8 + 4);
    int* bcast = reinterpret_cast<int*>(misc + kNumBarsP * 8 + 8);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    auto bar = [&](int i) { return smem_addr(&bars[i]); };
    const uint32_t tcols = N * 2 <= 32 ? 32 : (N * 2 <= 64 ? 64 : (N * 2 <= 128 ? 128 : (N * 2 <= 256 ? 256 : 512)));

    if (tid == 0) {
        for (int i = 0; i < kNumBarsP; ++i) mbar_init(bar(i), 1);
        *abort_flag = 0;
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(tcols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    fence_mbar_init();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // this CTA's units [u0, u1) of U = blocks x tiles x chunks, K chunk fastest
    const long long U = static_cast<long long>(pp.nblk) * pp.mtiles * pp.kch;
    const long long G = gridDim.x;
    auto begin_of = [&](long long c) { return static_cast<long long>(c * U / G); };
    const long long u0 = begin_of(blockIdx.x), u1 = begin_of(blockIdx.x + 1);
    const int n_my = static_cast<int>(u1 - u0);
    // CTA holding unit u: the largest c with begin_of(c) <= u
    auto cta_of = [&](long long u) { return static_cast<int>(((u + 1) * G + U - 1) / U - 1); };

    const uint64_t l2pol = l2_stream_policy();  // W is read once
    const uint64_t l2keep = l2_keep_policy();   // the planes are read by every feature tile
    // Unit cursors (tile j = block * mtiles + feature tile, K chunk kc), advanced one unit
    // at a time so the loops need no 64-bit division: the next W copy and the next O copy.
    struct UnitCursor {
        int j, kc;
    };
    const UnitCursor first{static_cast<int>(u0 / pp.kch), static_cast<int>(u0 % pp.kch)};
    auto next_unit = [&](UnitCursor& c) {
        if (++c.kc == pp.kch) {
            c.kc = 0;
            ++c.j;
        }
    };
    UnitCursor cw = first, co = first;
    // W rows of tile j, K chunk kc: the box at (kc * 64, feature tile * 128)
    auto issue_w = [&](int k) {
        const int s = k % NSTAGE;
        const uint32_t st = smem_addr(smem + s * SB);
        mbar_arrive_expect_tx(bar(kFull + s), static_cast<uint32_t>(SB));
        tc::tma_load_2d(st, &tmw, cw.kc * KCH, (cw.j % pp.mtiles) * MT, bar(kFull + s), l2pol);
        next_unit(cw);
    };
    auto issue_o = [&](int k) {
        const int s = k % NSTAGE;
        const uint32_t st = smem_addr(smem + s * SB);
        const int row = (co.j / pp.mtiles) * NTB;
        tc::tma_load_2d(st + WBYTES, &tmh, co.kc * KCH, row, bar(kFull + s), l2keep);
        tc::tma_load_2d(st + WBYTES + NTB * 128, &tml, co.kc * KCH, row, bar(kFull + s), l2keep);
        next_unit(co);
    };
    const int npre = n_my < NSTAGE ? n_my : NSTAGE;
    if (tid == 0)
        for (int k = 0; k < npre; ++k) issue_w(k);  // W does not depend on the decode step

    grid_dep_wait();    // the planes Oh / Ol are written by the decode kernel just before
    grid_dep_launch();  // the next launch (the next decode step) may take SMs as blocks finish

    int prod_k = 0;
    if (n_my > 0) {
        if (warp == 0) {
            // ------------------------------------------------ TMA producer
            if (lane == 0) {
                int k = 0;
                for (; k < npre; ++k) issue_o(k);
                for (; k < n_my; ++k) {
                    const int s = k % NSTAGE;
                    if (!tc::wait_or_abort(bar(kEmpty + s), ((k / NSTAGE) - 1) & 1, pp.err, abort_flag, pp.wait_cycles))
                        break;
                    issue_w(k);
                    issue_o(k);
                }
                prod_k = k;
            }
        } else if (warp == 1) {
            // ------------------------------------------------ MMA issue
            const uint32_t idesc = tc::instr_desc(BF, MT, N, false);
            const uint64_t da0 = tc::smem_desc_sw128(smem_addr(smem), 16, 1024);
            const uint64_t db0 = tc::smem_desc_sw128(smem_addr(smem + WBYTES), 16, 1024);
            int buf = 0, pieces = 0;
            int kc = first.kc;  // K chunk of unit k
            for (int k = 0; k < n_my; ++k, kc = kc + 1 == pp.kch ? 0 : kc + 1) {
                const bool first = k == 0 || kc == 0;  // a new piece starts
                if (first && k > 0) {
                    if (lane == 0) tc::mma_commit(bar(kAccFull + buf));  // the finished piece's sums
                    __syncwarp();
                    buf ^= 1;
                }
                if (first) {
                    // the epilogue has read this accumulator's previous piece (two pieces ago)
                    const bool ok = pieces < 2 || tc::wait_or_abort(bar(kAccEmpty + buf), ((pieces - 2) >> 1) & 1,
                                                                     pp.err, abort_flag, pp.wait_cycles);
                    if (__any_sync(0xffffffffu, !ok)) break;
                    ++pieces;
                }
                const int s = k % NSTAGE;
                const bool okf = tc::wait_or_abort(bar(kFull + s), (k / NSTAGE) & 1, pp.err, abort_flag, pp.wait_cycles);
                if (__any_sync(0xffffffffu, !okf)) break;
                if (lane == 0) {
                    tc::tc_fence_after();
                    const uint32_t off = static_cast<uint32_t>((s * SB) >> 4);
#pragma unroll
                    for (int ks = 0; ks < KCH / 16; ++ks)
                        tc::mma_f16(tmem + buf * N, da0 + off + ks * 2, db0 + off + ks * 2, idesc, !first || ks > 0);
                    tc::mma_commit(bar(kEmpty + s));
                }
                __syncwarp();
                if (k == n_my - 1) {
                    if (lane == 0) tc::mma_commit(bar(kAccFull + buf));
                    __syncwarp();
                }
            }
            // one last commit: it completes once every MMA issued above has (the drain after an abort)
            if (lane == 0) tc::mma_commit(bar(kDrain));
            __syncwarp();
        } else {
            // ------------------------------------------------ epilogue (warps 2-5)
            // thread r owns feature row r of the tile: TMEM lane r
            const int q4 = warp & 3;
            const int r = q4 * 32 + lane;
            const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
            const bool leader = warp == 2 && lane == 0;
            int buf = 0, pc = 0;
            long long u = u0;
            while (u < u1) {
                const int j = static_cast<int>(u / pp.kch);
                const long long ue = (static_cast<long long>(j) + 1) * pp.kch < u1 ? (static_cast<long long>(j) + 1) * pp.kch : u1;
                const uint32_t nch = static_cast<uint32_t>(ue - u);
                const bool whole = nch == static_cast<uint32_t>(pp.kch);
                const int blk = j / pp.mtiles, mt = j % pp.mtiles;
                const int nt = min(NTB, pp.tokens - blk * NTB);  // tokens of this block
                const bool ok = tc::wait_or_abort(bar(kAccFull + buf), (pc >> 1) & 1, pp.err, abort_flag, pp.wait_cycles);
                if (tc::bar_any(4, 128, !ok)) break;
                tc::tc_fence_after();
                float* slot = pp.ws + static_cast<size_t>(j + blockIdx.x) * NTB * MT;
                const size_t ybase = static_cast<size_t>(blk) * NTB * (static_cast<size_t>(pp.mtiles) * MT) +
                                     static_cast<size_t>(mt) * MT + r;
                const size_t F = static_cast<size_t>(pp.mtiles) * MT;
                for (int c0 = 0; c0 < NTB; c0 += 16) {
                    float hi[16], lo[16];
                    tc::tmem_ld<16>(tmem + lane_base + buf * N + c0, hi);
                    tc::tmem_ld<16>(tmem + lane_base + buf * N + NTB + c0, lo);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int t = c0 + i;
                        if (t < nt) {
                            const float v = hi[i] + lo[i];
                            if (whole) st_out1(pp.y, ybase + static_cast<size_t>(t) * F, v, pp.out_dtype);
                            else slot[t * MT + r] = v;
                        }
                    }
                }
                // the accumulator is free for the piece after next
                tc::tc_fence_before();
                tc::named_bar_sync(4, 128);
                if (leader) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar(kAccEmpty + buf)) : "memory");
                if (!whole) {
                    // the partial is stored (the barrier above ordered every thread's stores);
                    // the arrival that completes the tile's K chunks sums the pieces
                    if (leader) {
                        const uint32_t prev = arrive_acq_rel(&pp.counters[j], nch);
                        bcast[0] = (prev + nch == static_cast<uint32_t>(pp.kch)) ? 1 : 0;
                    }
                    tc::named_bar_sync(4, 128);
                    if (bcast[0]) {
                        const long long ua = static_cast<long long>(j) * pp.kch;
                        const int cf = cta_of(ua), cl = cta_of(ua + pp.kch - 1);
                        // 32 tokens at a time: per piece, 32 independent loads in flight, so the
                        // merge costs one L2 round trip per piece and chunk of tokens
                        for (int t0 = 0; t0 < nt; t0 += 32) {
                            float acc[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) acc[i] = 0.f;
                            for (int c = cf; c <= cl; ++c) {
                                // with fewer units than CTAs some CTAs hold none, and no piece
                                if (U < G && begin_of(c) == begin_of(c + 1)) continue;
                                const float* sp = pp.ws + (static_cast<size_t>(j + c) * NTB + t0) * MT + r;
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    if (t0 + i < nt) acc[i] += __ldcg(sp + i * MT);
                            }
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (t0 + i < nt) st_out1(pp.y, ybase + static_cast<size_t>(t0 + i) * F, acc[i], pp.out_dtype);
                        }
                        if (leader) pp.counters[j] = 0u;
                    }
                    tc::named_bar_sync(4, 128);
                }
                buf ^= 1;
                ++pc;
                u = ue;
            }
        }
    }

    __syncwarp();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (*abort_flag && n_my > 0) {
        // a bounded wait ran out: before TMEM is freed and the block exits, wait (long
        // drain limit) for the copies of the last stages issued and for the MMAs
        if (warp == 0 && lane == 0) {
            // (the producer issues the O half of every pre-issued stage right after the wait,
            // so prod_k >= npre and these are all the copies that can be in flight)
            for (int kk = max(0, prod_k - NSTAGE); kk < prod_k; ++kk)
                mbar_wait_bounded(bar(kFull + kk % NSTAGE), static_cast<uint32_t>((kk / NSTAGE) & 1), pp.err,
                                  kDrainLimitCycles);
        }
        if (warp == 1 && lane == 0) mbar_wait_bounded(bar(kDrain), 0u, pp.err, kDrainLimitCycles);
    }
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tcols));
    }
}

struct ProjKernelInfo {
    const void* fn;
};

ProjKernelInfo select_proj(bool bf16);

}  // namespace ftd
