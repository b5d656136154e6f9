// fwd_kernel.cuh -- the fused MaxSim forward kernel on the sm_103a tensor cores.
//
// "FLASH-MAXSIM: IO-Aware Fused Kernels for Late-Interaction Retrieval"
// (arXiv 2605.29517) §4.1, Alg. 2: stream document tiles, form the
// similarity sub-tile on chip, fold it into a running row maximum (§4.1.1,
// masking positions outside the document to -inf before the reduction), and
// write one scalar per (query, document) pair; padding-free packed documents
// per §4.3.2; INT8 x INT8 per §4.3.1 (one scale per tensor, or one per
// token).
//
// GB300 design (differs from the pages' one-program-per-pair scheme):
//  * One CTA owns 1, 2 or 4 M-tiles of 128 padded query rows resident in
//    shared memory, and streams a token-balanced contiguous range of
//    documents through a TMA pipeline, so every document row is read from
//    HBM once for all those queries (further row groups re-read it from L2).
//    With 1 or 2 M-tiles two CTAs share an SM, each with half of TMEM and of
//    shared memory; at 2 M-tiles the single document stage may be streamed
//    one K-block half at a time so the next tile's first half loads while
//    the last MMAs of the current one run.
//  * tcgen05.mma (M=128, N=128 tokens, K=16, FP32 accumulate) writes
//    similarity tiles into TMEM accumulator slots of 128 columns (4 per SM),
//    which the MMA fills while the epilogue drains the others.
//  * Epilogue warps (one warp-set of 4 per M-tile, one thread per query row;
//    a single 16-bit M-tile gets two sets, each folding half of every tile's
//    columns, their per-document results merged through shared memory)
//    read TMEM with tcgen05.ld and fold each 32-column chunk into the row's
//    running (max, argmax) with a balanced comparison tree (ties keep the
//    lowest token), splitting chunks at document boundaries; at a document's
//    end the warp writes the argmax row and reduces the maxima over query
//    tokens with a fixed shuffle tree.  Queries longer than 32 tokens leave
//    one partial per 32-token chunk, summed in chunk order by a second pass.
//  * INT8: a converter warp-set widens each int8 tile to FP16 in shared
//    memory (exact: |x| <= 127) for the same FP16 MMA; every product and
//    partial sum is an integer below 2^24, so the FP32 accumulator holds the
//    exact int32 dot product, and sums over query tokens run in int64.  With
//    one scale per token the epilogue multiplies each exact dot product by
//    its document token's scale (FP32) before the row maximum and the
//    maximum by the query token's scale, and sums in FP32.
#pragma once

#include "internal.cuh"
#include "sm103.cuh"
#include "fwd_epilogue.cuh"

#include <cuda_fp16.h>

namespace maxsim {
namespace {

using namespace ptx;

constexpr int kKBlockBytes = 128 * 128;        // 128 rows x 64 16-bit elements, 128B-swizzled
constexpr int kTileBytes = 2 * kKBlockBytes;   // 128 rows x 128 16-bit elements
constexpr int kI8TileBytes = 128 * 128;        // 128 rows x 128 int8
constexpr int kMaxSlots = 4;                   // TMEM accumulator slots (4 x 128 columns: all of TMEM)

constexpr int kMaxStages = 4;

struct SharedCtl {
    // per-token INT8: one 16-column scale slot per epilogue warp (broadcast reads)
    alignas(16) float scale_buf[16][16];
    uint64_t q_full;
    uint64_t d_full[kMaxStages];    // FP16 D stage ready for the MMA
    uint64_t d_empty[kMaxStages];   // FP16 D stage consumed by the MMA
    uint64_t i_full[kMaxStages];    // INT8 staging tile landed
    uint64_t i_empty[kMaxStages];   // INT8 staging tile converted
    uint64_t t_full[kMaxSlots];
    uint64_t t_empty[kMaxSlots];
    uint64_t mma_done;
    uint32_t tmem_base;
    int32_t abort;
    int32_t b_begin, b_end;
    int32_t t_begin, t_end;
};

template <int NMT, bool INT8>
struct Cfg {
    // One or two M-tiles: two CTAs share an SM, each with half of TMEM and of
    // shared memory, so twice the epilogue warps with valid rows run per SM.
    // One M-tile: 2 slots (double-buffered), 2 document stages (INT8: one FP16
    // stage, two INT8 staging tiles, two converter warps); 16-bit: two
    // epilogue warps per TMEM lane quarter, each folding half of every
    // tile's columns (kPaired), merged per document through shared memory.
    // Two M-tiles (16-bit only): one slot per M-tile, one document stage,
    // single-buffered TMEM reads (five warps per scheduler leave 96
    // registers).
    static constexpr int kCtasPerSm = (NMT == 1 || (NMT == 2 && !INT8)) ? 2 : 1;
    static constexpr bool kPaired = NMT == 1 && !INT8;
    static constexpr int kEpiWarps = 4 * NMT * (kPaired ? 2 : 1);
    static constexpr int kSlots = kCtasPerSm == 2 ? 2 : 4;
    static constexpr int kTmemCols = kSlots * kSlotCols;
    static constexpr int kStages = INT8 ? (NMT == 4 ? 2 : (NMT == 1 ? 1 : 3)) : (NMT == 4 ? 3 : (NMT == 1 ? 2 : 1));
    static constexpr int kI8Stages = INT8 ? (NMT == 2 ? 4 : 2) : 0;
    static constexpr int kConvWarps = INT8 ? (NMT == 2 ? 4 : 2) : 0;
    static constexpr bool kDoubleBuffer = INT8 && NMT <= 2;
    // A single 16-bit stage may be filled and consumed one K-block (64 of the
    // 128 dimensions) at a time (chosen per launch): the next tile's first
    // half loads while the MMAs of the second half run.
    static constexpr bool kKSplit = !INT8 && kStages == 1;
    static constexpr int kFirstEpiWarp = 2 + kConvWarps;
    static constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps);
    static constexpr int kQBytes = NMT * kTileBytes;
    static constexpr int kDBytes = kStages * kTileBytes;
    static constexpr int kIBytes = kI8Stages * kI8TileBytes;
    static constexpr int kPairBytes = kPaired ? 4 * (int)sizeof(PairBuf) : 0;
    static constexpr int kSmem = 1024 + kQBytes + kDBytes + kIBytes + (int)sizeof(SharedCtl) + kPairBytes;
    static_assert(kStages >= 1 && kStages <= kMaxStages, "barrier arrays hold kMaxStages stages");
    static_assert(kI8Stages <= kMaxStages, "barrier arrays hold kMaxStages stages");
    static_assert(kSmem <= 232448, "exceeds the 227 KB shared-memory limit per CTA");
    static_assert(kSlots <= kMaxSlots && kSlots % NMT == 0, "slots hold whole row groups");
    // A paired warp may wait at a meeting while it still holds tile j's slot,
    // and its partner may need tile j + 1 to reach the same meeting: tile
    // j + 1 must go to another slot, or the two wait on each other.
    static_assert(!kPaired || kSlots / NMT >= 2, "paired epilogue warps need two slots per M-tile");
    // at most kCtasPerSm CTAs fit an SM's 228 KB, so their TMEM never exceeds 512 columns
    static_assert(kCtasPerSm == 1 || 3 * (kSmem + 1024) > 233472, "a third CTA could oversubscribe TMEM");
};

// int8 x4 -> fp16 x4 exactly: (x ^ 0x80) in the low byte of 1024.0 gives
// 1024 + x + 128; subtracting 1152 leaves x.
__device__ __forceinline__ uint2 widen_i8x4(uint32_t w) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t lo = __byte_perm(u, 0x64646464u, 0x4140);
    const uint32_t hi = __byte_perm(u, 0x64646464u, 0x4342);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    __half2 l = __hsub2(*reinterpret_cast<const __half2 *>(&lo), bias);
    __half2 h = __hsub2(*reinterpret_cast<const __half2 *>(&hi), bias);
    return make_uint2(*reinterpret_cast<uint32_t *>(&l), *reinterpret_cast<uint32_t *>(&h));
}

template <int NMT, bool ARGMAX, bool INT8, bool SCALE>
__global__ void __launch_bounds__(Cfg<NMT, INT8>::kThreads, Cfg<NMT, INT8>::kCtasPerSm)
maxsim_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmD,
                  const FwdParams p) {
    using C = Cfg<NMT, INT8>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem;
    uint8_t *sD = smem + C::kQBytes;
    uint8_t *sI = sD + C::kDBytes;
    SharedCtl *ctl = reinterpret_cast<SharedCtl *>(sI + C::kIBytes);
    PairBuf *pairs = reinterpret_cast<PairBuf *>(ctl + 1);   // kPaired: one per TMEM lane quarter
    volatile int32_t *abort_flag = &ctl->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = blockIdx.x % p.groups;
    const int part = blockIdx.x / p.groups;
    const int64_t rows_total = static_cast<int64_t>(p.n_q) * p.lq_pad;
    const int row0 = g * NMT * 128;
    const int64_t mt_left = (rows_total - row0 + 127) / 128;
    const int n_mt = mt_left < NMT ? static_cast<int>(mt_left) : NMT;

    if (threadIdx.x == 0) {
        mbar_init(&ctl->q_full, 1);
        for (int s = 0; s < kMaxStages; ++s) {
            mbar_init(&ctl->d_full[s], INT8 ? 32 * C::kConvWarps : 1);
            mbar_init(&ctl->d_empty[s], 1);
            mbar_init(&ctl->i_full[s], 1);
            mbar_init(&ctl->i_empty[s], INT8 ? 32 * C::kConvWarps : 1);
        }
        for (int s = 0; s < C::kSlots; ++s) {
            mbar_init(&ctl->t_full[s], 1);
            mbar_init(&ctl->t_empty[s], 4 * (C::kPaired ? 2 : 1));
        }
        if constexpr (C::kPaired)
            for (int k = 0; k < 4; ++k) mbar_init(&pairs[k].bar, 2);
        mbar_init(&ctl->mma_done, 1);
        fence_mbar_init();
        ctl->abort = 0;
        // token-balanced contiguous document range of this part (the token
        // count is read from the offsets: the tensor map may extend past it)
        const int64_t T = p.cu_seqlens[p.n_docs];
        const int64_t lo = T * part / p.parts;
        const int64_t hi = T * (part + 1) / p.parts;
        const int bb = lower_bound_cu(p.cu_seqlens, p.n_docs, lo);
        const int be = (part == p.parts - 1) ? p.n_docs : lower_bound_cu(p.cu_seqlens, p.n_docs, hi);
        ctl->b_begin = bb;
        ctl->b_end = max(bb, be);
        ctl->t_begin = p.cu_seqlens[bb];
        ctl->t_end = p.cu_seqlens[max(bb, be)];
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = ctl->tmem_base;
    const int b_begin = ctl->b_begin, b_end = ctl->b_end;
    const int t_begin = ctl->t_begin, t_end = ctl->t_end;
    const int n_tiles = (t_end - t_begin + kBlockN - 1) / kBlockN;
    const bool run_pipeline = n_tiles > 0 && n_mt > 0;
    const bool ksplit = C::kKSplit && p.ksplit != 0;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0 && run_pipeline) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmD);
            mbar_arrive_expect_tx(&ctl->q_full, n_mt * 8 * 4096);
            for (int c = 0; c < 4 * n_mt; ++c) {
                const int rho0 = row0 + 32 * c;
                const int qq = rho0 / p.lq_pad;
                const int i0 = rho0 - qq * p.lq_pad;
                uint8_t *dst = sQ + (c >> 2) * kTileBytes + (c & 3) * 4096;
                tma_load_3d(dst, &tmQ, &ctl->q_full, 0, i0, qq);
                tma_load_3d(dst + kKBlockBytes, &tmQ, &ctl->q_full, 64, i0, qq);
            }
            // K-split: a ring of two half-stages (one K-block each), load u =
            // 2 * tile + K-block
            const int kS = INT8 ? C::kI8Stages : (ksplit ? 2 : C::kStages);
            const int n_loads = ksplit ? 2 * n_tiles : n_tiles;
            int issued = 0;
            for (int j = 0; j < n_loads; ++j) {
                const int s = j % kS;
                const uint32_t ph = (j / kS) & 1;
                const int row = t_begin + (ksplit ? j >> 1 : j) * kBlockN;
                if (ksplit) {
                    if (!mbar_wait(&ctl->d_empty[s], ph ^ 1, abort_flag, p.status, kStatusTimeoutProducer)) break;
                    mbar_arrive_expect_tx(&ctl->d_full[s], kKBlockBytes);
                    tma_load_2d(sD + s * kKBlockBytes, &tmD, &ctl->d_full[s], 64 * s, row);
                } else if (INT8) {
                    if (!mbar_wait(&ctl->i_empty[s], ph ^ 1, abort_flag, p.status, kStatusTimeoutProducer)) break;
                    mbar_arrive_expect_tx(&ctl->i_full[s], kI8TileBytes);
                    tma_load_2d(sI + s * kI8TileBytes, &tmD, &ctl->i_full[s], 0, row);
                } else {
                    if (!mbar_wait(&ctl->d_empty[s], ph ^ 1, abort_flag, p.status, kStatusTimeoutProducer)) break;
                    mbar_arrive_expect_tx(&ctl->d_full[s], kTileBytes);
                    tma_load_2d(sD + s * kTileBytes, &tmD, &ctl->d_full[s], 0, row);
                    tma_load_2d(sD + s * kTileBytes + kKBlockBytes, &tmD, &ctl->d_full[s], 64, row);
                }
                issued = j + 1;
            }
            // no TMA copy may still be landing when the CTA exits
            mbar_wait(&ctl->q_full, 0, nullptr, p.status, kStatusTimeoutDrain);
            for (int j = max(0, issued - kS); j < issued; ++j)
                mbar_wait(INT8 ? &ctl->i_full[j % kS] : &ctl->d_full[j % kS], (j / kS) & 1, nullptr,
                          p.status, kStatusTimeoutDrain);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0 && run_pipeline) {
            bool ok = mbar_wait(&ctl->q_full, 0, abort_flag, p.status, kStatusTimeoutMma);
            tc_fence_after();
            // Descriptors advance by adding (byte offset >> 4) to the start
            // address field; every operand lies below 256 KB of shared memory,
            // so the 14-bit field never carries.
            const uint64_t a_desc0 = desc_sw128_kmajor(smem_u32(sQ));
            const uint64_t b_desc0 = desc_sw128_kmajor(smem_u32(sD));
            if (ksplit) {
                // per tile, M-tile by M-tile: K-block 0 then K-block 1 into
                // its slot (K in order, the slot handed to the epilogue as
                // early as before); the K-block-0 half-stage is released
                // after the last M-tile's K-block 0, so the next tile's first
                // half loads while the last K-block-1 MMAs run
                for (int j = 0; ok && j < n_tiles; ++j) {
                    if (!mbar_wait(&ctl->d_full[0], j & 1, abort_flag, p.status, kStatusTimeoutMma)) break;
                    tc_fence_after();
                    for (int mt = 0; mt < n_mt; ++mt) {
                        const int slot = mt + NMT * (j % (C::kSlots / NMT));
                        const uint32_t use = j / (C::kSlots / NMT);
                        if (!mbar_wait(&ctl->t_empty[slot], (use & 1) ^ 1, abort_flag, p.status, kStatusTimeoutMma)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t a_desc = a_desc0 + static_cast<uint64_t>((mt * kTileBytes) >> 4);
                        const uint32_t d_tmem = tmem_base + slot * kSlotCols;
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4) {
                            const uint64_t koff = static_cast<uint64_t>((k4 * 32) >> 4);
                            mma_f16_ss(d_tmem, a_desc + koff, b_desc0 + koff, p.idesc, k4 > 0 ? 1u : 0u);
                        }
                        if (mt == n_mt - 1) mma_commit(&ctl->d_empty[0]);
                        if (mt == 0) {
                            if (!mbar_wait(&ctl->d_full[1], j & 1, abort_flag, p.status, kStatusTimeoutMma)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4) {
                            const uint64_t koff = static_cast<uint64_t>((kKBlockBytes + k4 * 32) >> 4);
                            mma_f16_ss(d_tmem, a_desc + koff, b_desc0 + koff, p.idesc, 1u);
                        }
                        mma_commit(&ctl->t_full[slot]);
                    }
                    if (ok) mma_commit(&ctl->d_empty[1]);
                }
            } else
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int s = j % C::kStages;
                if (!mbar_wait(&ctl->d_full[s], (j / C::kStages) & 1, abort_flag, p.status, kStatusTimeoutMma)) break;
                tc_fence_after();
                const uint64_t b_desc = b_desc0 + static_cast<uint64_t>((s * kTileBytes) >> 4);
                for (int mt = 0; mt < n_mt; ++mt) {
                    const int slot = mt + NMT * (j % (C::kSlots / NMT));
                    const uint32_t use = j / (C::kSlots / NMT);
                    if (!mbar_wait(&ctl->t_empty[slot], (use & 1) ^ 1, abort_flag, p.status, kStatusTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_desc = a_desc0 + static_cast<uint64_t>((mt * kTileBytes) >> 4);
                    const uint32_t d_tmem = tmem_base + slot * kSlotCols;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t koff = static_cast<uint64_t>(((kk >> 2) * kKBlockBytes + (kk & 3) * 32) >> 4);
                        mma_f16_ss(d_tmem, a_desc + koff, b_desc + koff, p.idesc, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&ctl->t_full[slot]);
                }
                mma_commit(&ctl->d_empty[s]);
            }
            // every MMA has finished before TMEM is released
            mma_commit(&ctl->mma_done);
            mbar_wait(&ctl->mma_done, 0, nullptr, p.status, kStatusTimeoutDrain);
        }
        __syncwarp();
    } else if (warp < C::kFirstEpiWarp) {
        // ------------------------------------------------ INT8 -> FP16 widening
        const int t0 = threadIdx.x - 64;  // first row of the tile this thread widens
        if constexpr (INT8) if (run_pipeline) {
            for (int j = 0; j < n_tiles; ++j) {
                const int si = j % C::kI8Stages;
                const int sd = j % C::kStages;
                if (!mbar_wait(&ctl->i_full[si], (j / C::kI8Stages) & 1, abort_flag, p.status, kStatusTimeoutProducer)) break;
                if (!mbar_wait(&ctl->d_empty[sd], ((j / C::kStages) & 1) ^ 1, abort_flag, p.status, kStatusTimeoutProducer)) break;
#pragma unroll 1
                for (int t = t0; t < 128; t += 32 * C::kConvWarps) {
                const uint8_t *src = sI + si * kI8TileBytes + t * 128;
                uint8_t *dst = sD + sd * kTileBytes + t * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    // 16 int8 at logical chunk c (128B-swizzled by the TMA)
                    const uint4 w = *reinterpret_cast<const uint4 *>(src + ((c ^ (t & 7)) << 4));
                    const uint2 e0 = widen_i8x4(w.x), e1 = widen_i8x4(w.y);
                    const uint2 e2 = widen_i8x4(w.z), e3 = widen_i8x4(w.w);
                    // 16 halves = logical 16-byte chunks 2(c%4), 2(c%4)+1 of K-block c/4
                    uint8_t *kb = dst + (c >> 2) * kKBlockBytes;
                    const int c16 = 2 * (c & 3);
                    *reinterpret_cast<uint4 *>(kb + ((c16 ^ (t & 7)) << 4)) = make_uint4(e0.x, e0.y, e1.x, e1.y);
                    *reinterpret_cast<uint4 *>(kb + (((c16 + 1) ^ (t & 7)) << 4)) = make_uint4(e2.x, e2.y, e3.x, e3.y);
                }
                }
                fence_proxy_async_smem();   // generic-proxy writes -> visible to the tensor core
                mbar_arrive(&ctl->i_empty[si]);
                mbar_arrive(&ctl->d_full[sd]);
            }
        }
    } else {
        // ------------------------------------------------ epilogue
        const int e = warp - C::kFirstEpiWarp;
        const int mt = C::kPaired ? 0 : e >> 2;
        const int half = C::kPaired ? e >> 2 : 0;   // kPaired: which half of each tile's columns
        const int qd = warp & 3;  // TMEM lane quarter this warp may access
        if (mt < n_mt) {
            epilogue_warp<ARGMAX, INT8 && !SCALE, SCALE, C::kDoubleBuffer, C::kPaired>(
                p, row0 + mt * 128 + qd * 32, rows_total, tmem_base, qd, b_begin, b_end, t_begin, t_end,
                n_tiles, ctl->t_full, ctl->scale_buf[warp - C::kFirstEpiWarp],
                [&](int j) { return make_int2(mt + NMT * (j % (C::kSlots / NMT)), j / (C::kSlots / NMT)); },
                [&](int slot) { mbar_arrive(&ctl->t_empty[slot]); }, abort_flag,
                C::kPaired ? pairs + qd : nullptr, half);
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, C::kTmemCols);
}

}  // namespace
}  // namespace maxsim
