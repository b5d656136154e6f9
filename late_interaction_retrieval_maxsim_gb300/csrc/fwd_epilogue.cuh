// fwd_epilogue.cuh -- the epilogue shared by the fused MaxSim forward
// kernels: fold TMEM accumulator tiles into running row maxima (and their
// lowest argmax), split at document boundaries, and reduce over query tokens
// at each document's end.
//
// "FLASH-MAXSIM: IO-Aware Fused Kernels for Late-Interaction Retrieval"
// (arXiv 2605.29517) §4.1.1 (online-max recurrence, masking to -inf before
// the reduction), §4.1 (query-chunk decomposition of the sum), §4.3.2
// (documents packed with cu_seqlens).
#pragma once

#include "internal.cuh"
#include "sm103.cuh"

#include <cuda_fp16.h>

namespace maxsim {
namespace {

using namespace ptx;

constexpr int kBlockN = 128;    // document tokens per tile (MMA N)
constexpr int kSlotCols = 128;  // TMEM columns per accumulator slot

// Two epilogue warps on one TMEM lane quarter, each folding half of every
// tile's columns for the same 32 query rows, hand their per-document
// partial (maximum, lowest argmax) to each other through this buffer: each
// writes the partials of the documents it closes, both meet at `bar`
// (arrival count 2) once kPairDocs are buffered, and the documents are
// merged and written out by the two warps in turn; a second meeting frees
// the buffer.
constexpr int kPairDocs = 4;    // documents buffered between meetings
struct PairBuf {
    uint64_t bar;
    int32_t doc_lo[kPairDocs], doc_hi[kPairDocs];
    float m[2][kPairDocs][32];
    int32_t a[2][kPairDocs][32];
};

__device__ __forceinline__ int lower_bound_cu(const int32_t *cu, int n, int64_t key) {
    // first index in [0, n] with cu[index] >= key (cu[n] is the token total)
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (static_cast<int64_t>(cu[mid]) >= key) hi = mid; else lo = mid + 1;
    }
    return lo;
}

// Column k of a 32-column chunk of the accumulator; with MASKED, columns
// outside [lo, hi) read as -inf so they can never be selected (the masking
// of §4.1.1, applied before the reduction).
template <bool MASKED>
__device__ __forceinline__ float col(const uint32_t (&r)[32], int k, int lo, int hi) {
    const float x = __uint_as_float(r[k]);
    if (MASKED) return (k >= lo && k < hi) ? x : -INFINITY;
    return x;
}

// Maximum of a chunk with 3-input max instructions (16 per 32 columns).
template <bool MASKED>
__device__ __forceinline__ float chunk_max(const uint32_t (&r)[32], int lo, int hi) {
    float y[11];
#pragma unroll
    for (int k = 0; k < 10; ++k)
        y[k] = fmax3(col<MASKED>(r, 3 * k, lo, hi), col<MASKED>(r, 3 * k + 1, lo, hi),
                     col<MASKED>(r, 3 * k + 2, lo, hi));
    y[10] = fmaxf(col<MASKED>(r, 30, lo, hi), col<MASKED>(r, 31, lo, hi));
    const float z0 = fmax3(y[0], y[1], y[2]);
    const float z1 = fmax3(y[3], y[4], y[5]);
    const float z2 = fmax3(y[6], y[7], y[8]);
    return fmax3(fmax3(z0, z1, z2), y[9], y[10]);
}

// True when the one-instruction indicator below is exact for maximum cm:
// every finite value below cm then lies at least 2^-100 below it.  The
// closest float below cm is half an ulp of cm away when cm is a power of
// two (2^-101 for cm = 2^-77), so the bound is 2^-76, not 2^-77.
__device__ __forceinline__ bool fast_indicator_ok(float cm) {
    const float x = fabsf(cm);
    return x >= 0x1p-76f && x < 0x1p27f;
}

// The 32-bit mask from its two 16-bit halves, each held as the float
// 2^23 + half (so its low 16 mantissa bits are the half): one byte permute.
__device__ __forceinline__ uint32_t mask_from_halves(float lo, float hi) {
    return __byte_perm(__float_as_uint(lo), __float_as_uint(hi), 0x5410);
}

// Bit k set when column k holds a value below cm, clear when it equals cm
// (columns above cm, which only occur outside a segment, come out clear and
// must be masked by the caller).
//
// Each column's indicator is an exact 0.0 / 1.0 computed on the FMA pipe
// (the ALU pipe that compares and selects use issues at half rate): with
// S = 2^100 and C = cm * S (exact), fma.sat(value, -S, C) = sat(S * (cm -
// value)) is 0 when value == cm and 1 when value < cm, because a nonzero
// cm - value is at least half an ulp of cm (the gap below a power of two),
// >= 2^-100 when |cm| >= 2^-76, and C stays finite when |cm| < 2^27
// (`fast`).  Otherwise two saturating
// multiplies of (cm - value) by 2^127 and 2^23 reach 1 for every nonzero
// finite difference.  Indicators are packed into the mask 8 at a time (sums
// of distinct powers of two below 2^16 are exact in FP32).
__device__ __forceinline__ uint32_t below_mask32(const uint32_t (&r)[32], float cm, bool fast) {
    // acc[g] accumulates columns (16g + j, 16g + 8 + j), j = 0..7, with weight 2^j
    // in its x / y lane: two indicators per packed FMA.  The x lanes start at
    // 2^23, so each combined 16-bit half is read straight out of a float's
    // mantissa (2^23 + n, n < 2^16, is exact).
    float2 acc[2] = {make_float2(0x1p23f, 0.f), make_float2(0x1p23f, 0.f)};
    if (fast) {
        const float S = 0x1p100f;
        const float C = cm * S;
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float w = static_cast<float>(1u << j);
                const float2 ind = make_float2(fma_sat(__uint_as_float(r[16 * g + j]), -S, C),
                                               fma_sat(__uint_as_float(r[16 * g + 8 + j]), -S, C));
                acc[g] = fma2(ind, make_float2(w, w), acc[g]);
            }
    } else {
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float w = static_cast<float>(1u << j);
                const float t0 = cm - __uint_as_float(r[16 * g + j]);
                const float t1 = cm - __uint_as_float(r[16 * g + 8 + j]);
                const float2 ind = make_float2(mul_sat(mul_sat(t0, 0x1p127f), 0x1p23f),
                                               mul_sat(mul_sat(t1, 0x1p127f), 0x1p23f));
                acc[g] = fma2(ind, make_float2(w, w), acc[g]);
            }
    }
    // bits 0-7 / 8-15 of each half from the x / y lanes
    return mask_from_halves(fmaf(acc[0].y, 256.f, acc[0].x), fmaf(acc[1].y, 256.f, acc[1].x));
}

// Bits lo .. hi-1 set (0 <= lo < hi <= 32).
__device__ __forceinline__ uint32_t bit_range(int lo, int hi) {
    const uint32_t upto_hi = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
    return upto_hi & ~((1u << lo) - 1u);
}

// Fold columns [lo, hi) of a chunk starting at global column c0 into the
// running row maximum m (and, with ARGMAX, its lowest index a).  Later
// chunks replace the running winner only when strictly greater, so ties keep
// the lowest column.  Must be called by the whole warp.
template <bool ARGMAX, bool MASKED>
__device__ __forceinline__ void fold_chunk(const uint32_t (&r)[32], int c0, int lo, int hi, float &m, int &a) {
    const float cm = chunk_max<MASKED>(r, lo, hi);
    if (!ARGMAX) {
        m = fmaxf(m, cm);
        return;
    }
    const bool up = cm > m;
    if (__any_sync(0xffffffffu, up)) {
        const bool fast = __all_sync(0xffffffffu, !up || fast_indicator_ok(cm));
        uint32_t mask = below_mask32(r, cm, fast);
        if (MASKED) mask |= ~bit_range(lo, hi);
        if (up) {
            m = cm;
            a = c0 + __ffs(~mask) - 1;
        }
    }
}

template <int B>
__device__ __forceinline__ float max8(const uint32_t (&r)[32]) {
    auto f = [&](int k) { return __uint_as_float(r[B + k]); };
    return fmax3(fmax3(f(0), f(1), f(2)), fmax3(f(3), f(4), f(5)), fmaxf(f(6), f(7)));
}

// Columns B .. B+7 split at o (0 <= o < 8, warp-uniform): maxima of
// [B, B+o) and [B+o, B+8), -inf for an empty side.
template <int B>
__device__ __forceinline__ void split8(const uint32_t (&r)[32], int o, float &below, float &above) {
    float x[8], y[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float v = __uint_as_float(r[B + k]);
        x[k] = k < o ? v : -INFINITY;
        y[k] = k < o ? -INFINITY : v;
    }
    below = fmax3(fmax3(x[0], x[1], x[2]), fmax3(x[3], x[4], x[5]), fmaxf(x[6], x[7]));
    above = fmax3(fmax3(y[0], y[1], y[2]), fmax3(y[3], y[4], y[5]), fmaxf(y[6], y[7]));
}

// Maxima of columns [0, p) and [p, 32) for a document boundary at p = 8G + o
// (1 <= p <= 31): eight-column group maxima, with only group G, the one
// holding the boundary, masked column by column.
template <int G>
__device__ __forceinline__ void split_max32(const uint32_t (&r)[32], int o, float &left, float &right) {
    float lo, hi;
    split8<8 * G>(r, o, lo, hi);
    if constexpr (G == 0) {
        left = lo;
        right = fmax3(hi, max8<8>(r), fmaxf(max8<16>(r), max8<24>(r)));
    } else if constexpr (G == 1) {
        left = fmaxf(max8<0>(r), lo);
        right = fmax3(hi, max8<16>(r), max8<24>(r));
    } else if constexpr (G == 2) {
        left = fmax3(max8<0>(r), max8<8>(r), lo);
        right = fmaxf(hi, max8<24>(r));
    } else {
        left = fmax3(max8<0>(r), max8<8>(r), fmaxf(max8<16>(r), lo));
        right = hi;
    }
}

// below_mask32 against two maxima at once: bit k set when column k holds a
// value below its own segment's maximum -- tl for k < 8G + o, tr from there
// on -- so one pass serves the ending document's search and the next one's.
// Only the eight columns of group G choose their target at run time.
template <int G>
__device__ __forceinline__ uint32_t below_mask32_split(const uint32_t (&r)[32], int o, float tl, float tr,
                                                       bool fast) {
    auto left_of = [&](int k) -> bool {
        if (k < 8 * G) return true;
        if (k >= 8 * G + 8) return false;
        return k - 8 * G < o;
    };
    // x lanes start at 2^23 (see below_mask32)
    float2 acc[2] = {make_float2(0x1p23f, 0.f), make_float2(0x1p23f, 0.f)};
    if (fast) {
        const float S = 0x1p100f;
        const float Cl = tl * S, Cr = tr * S;
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int k0 = 16 * g + j, k1 = 16 * g + 8 + j;
                const float w = static_cast<float>(1u << j);
                const float2 ind = make_float2(fma_sat(__uint_as_float(r[k0]), -S, left_of(k0) ? Cl : Cr),
                                               fma_sat(__uint_as_float(r[k1]), -S, left_of(k1) ? Cl : Cr));
                acc[g] = fma2(ind, make_float2(w, w), acc[g]);
            }
    } else {
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int k0 = 16 * g + j, k1 = 16 * g + 8 + j;
                const float w = static_cast<float>(1u << j);
                const float t0 = (left_of(k0) ? tl : tr) - __uint_as_float(r[k0]);
                const float t1 = (left_of(k1) ? tl : tr) - __uint_as_float(r[k1]);
                const float2 ind = make_float2(mul_sat(mul_sat(t0, 0x1p127f), 0x1p23f),
                                               mul_sat(mul_sat(t1, 0x1p127f), 0x1p23f));
                acc[g] = fma2(ind, make_float2(w, w), acc[g]);
            }
    }
    return mask_from_halves(fmaf(acc[0].y, 256.f, acc[0].x), fmaf(acc[1].y, 256.f, acc[1].x));
}

// A chunk in which the current document ends at column p = 8G + o and the
// next one covers the rest: [0, p) is folded into (m, a); the next
// document's running state starts as (m_next, a_next) from [p, 32).
template <bool ARGMAX, int G>
__device__ __forceinline__ void fold_split_g(const uint32_t (&r)[32], int c0, int o, float &m, int &a,
                                             float &m_next, int &a_next) {
    float left, right;
    split_max32<G>(r, o, left, right);
    m_next = right;
    if (!ARGMAX) {
        m = fmaxf(m, left);
        return;
    }
    const int p = 8 * G + o;
    const uint32_t low = (1u << p) - 1u;
    const bool fast = __all_sync(0xffffffffu, fast_indicator_ok(right) && fast_indicator_ok(left));
    const uint32_t mask = below_mask32_split<G>(r, o, left, right, fast);
    a_next = c0 + __ffs(~(mask | low)) - 1;
    if (left > m) {
        m = left;
        a = c0 + __ffs(~(mask | ~low)) - 1;
    }
}

template <bool ARGMAX>
__device__ __forceinline__ void fold_split(const uint32_t (&r)[32], int c0, int p, float &m, int &a,
                                           float &m_next, int &a_next) {
    const int o = p & 7;
    switch (p >> 3) {
        case 0: fold_split_g<ARGMAX, 0>(r, c0, o, m, a, m_next, a_next); break;
        case 1: fold_split_g<ARGMAX, 1>(r, c0, o, m, a, m_next, a_next); break;
        case 2: fold_split_g<ARGMAX, 2>(r, c0, o, m, a, m_next, a_next); break;
        default: fold_split_g<ARGMAX, 3>(r, c0, o, m, a, m_next, a_next); break;
    }
}

// One epilogue warp owns 32 consecutive padded query rows (rho_warp ..
// rho_warp+31) of an accumulator tile that lives in TMEM lane quarter qd.
// For every document tile j it waits t_full[slot_of(j).x] (phase
// slot_of(j).y), reads the 128 columns 32 at a time, hands the slot back
// with release(slot) once the last chunk is in registers, and folds the
// chunks into the running maxima; at each document end it writes the argmax
// row and the (partial) score.  DB double-buffers the TMEM reads.  INT8 sums
// the (integer) maxima in int64; SCALE multiplies each column by its
// document token's scale before the maximum and the row maximum by the
// query token's scale, then sums in FP32.  PAIRED: this warp folds only the
// chunks 2 half, 2 half + 1 of every tile and hands each document's partial
// to `pair`; both warps close the same documents in the same order, so every
// kPairDocs-th close (and the last) is a meeting point where the buffered
// documents are merged and written out (the maxima are exact and ties go to
// the lower column either way, so the outputs are the same bits as one
// warp's).  Per-tile meetings measured slower: one query 321 vs 330 us.
template <bool ARGMAX, bool INT8, bool SCALE, bool DB, bool PAIRED, typename SlotOf, typename Release>
__device__ __forceinline__ void epilogue_warp(const FwdParams &p, int rho_warp, int64_t rows_total,
                                              uint32_t tmem_base, int qd, int b_begin, int b_end,
                                              int t_begin, int t_end, int n_tiles, uint64_t *t_full,
                                              float *scale_slot, SlotOf slot_of, Release release,
                                              volatile int32_t *abort_flag, PairBuf *pair, int half) {
    static_assert(!PAIRED || (!DB && !SCALE && !INT8), "pairs split 16-bit single-buffered epilogues");
    const int lane = threadIdx.x & 31;
    const bool warp_rows = rho_warp < rows_total;
    const int rho = rho_warp + lane;
    const int q = rho / p.lq_pad;
    const int i = rho - q * p.lq_pad;
    const bool row_valid = q < p.n_q && i < p.lq_max;
    const int qlen = (q < p.n_q) ? p.q_lens[q] : 0;
    const bool active = row_valid && i < qlen;
    const uint32_t lane_base = static_cast<uint32_t>(qd * 32) << 16;
    [[maybe_unused]] const float q_scale = (SCALE && active) ? p.q_tok_scale[q * p.lq_max + i] : 0.0f;

    // SCALE: lane l holds the scale of column c0 + l of the next chunk (0
    // past this CTA's tokens); every column of the row is multiplied by its
    // scale.  The warp passes the scales through its 16-float shared slot,
    // half a chunk at a time, and every lane reads them back as broadcasts.
    auto chunk_scale = [&](int c0) -> float {
        return (SCALE && c0 + lane < t_end) ? __ldg(p.d_tok_scale + c0 + lane) : 0.0f;
    };
    auto apply_scale = [&](uint32_t (&r)[32], float s) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            __syncwarp();
            if ((lane >> 4) == h) scale_slot[lane & 15] = s;
            __syncwarp();
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const float4 v = reinterpret_cast<const float4 *>(scale_slot)[k4];
                const int k = 16 * h + 4 * k4;
                // two IEEE products per instruction (the same roundings as scalar ones)
                const float2 lo = mul2(make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])),
                                       make_float2(v.x, v.y));
                const float2 hi = mul2(make_float2(__uint_as_float(r[k + 2]), __uint_as_float(r[k + 3])),
                                       make_float2(v.z, v.w));
                r[k] = __float_as_uint(lo.x);
                r[k + 1] = __float_as_uint(lo.y);
                r[k + 2] = __float_as_uint(hi.x);
                r[k + 3] = __float_as_uint(hi.y);
            }
        }
    };

    // Upcoming document boundaries: lane l holds cu[cu_base + l]; one
    // coalesced load serves 32 documents, read back by shuffles.
    int cu_base = b_begin + 1;
    int cu_val = (cu_base + lane <= b_end) ? p.cu_seqlens[cu_base + lane] : INT32_MAX;
    auto boundary = [&](int idx) -> int {  // cu[idx], idx warp-uniform in (b_begin, b_end]
        if (idx >= cu_base + 32) {
            cu_base = idx;
            cu_val = (cu_base + lane <= b_end) ? p.cu_seqlens[cu_base + lane] : INT32_MAX;
        }
        return __shfl_sync(0xffffffffu, cu_val, idx - cu_base);
    };

    float m = -INFINITY;
    int a = -1;
    int b = b_begin;
    int doc_lo = t_begin;
    int doc_hi = (b < b_end) ? boundary(b + 1) : INT32_MAX;
    bool aborted = false;

    // Document bb with row maximum mm (argmax aa, a column index) for this
    // warp's rows: argmax row, then the sum of row maxima over the query's
    // tokens (fixed shuffle tree).
    auto emit = [&](int bb, float mm, int aa, int lo, int hi) {
        if (ARGMAX && row_valid)
            p.argmax[(static_cast<int64_t>(q) * p.ld_out + bb) * p.lq_max + i] =
                (active && aa >= 0) ? aa - lo : -1;
        if (INT8) {
            const bool empty_doc = hi == lo;
            long long c = (active && !empty_doc) ? static_cast<long long>(mm) : 0ll;
            if (p.lq_pad <= 32) {
                for (int off = 1; off < p.lq_pad; off <<= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
                if (i == 0 && q < p.n_q) {
                    const bool neg_inf = empty_doc && qlen > 0;
                    const int64_t idx = static_cast<int64_t>(q) * p.ld_out + bb;
                    if (p.raw_scores) p.raw_scores[idx] = neg_inf ? INT64_MIN : c;
                    p.scores[idx] = neg_inf ? -INFINITY
                                            : static_cast<float>(static_cast<double>(c) * p.int8_scale);
                }
            } else {
                for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
                if (lane == 0 && q < p.n_q)
                    p.ipartials[(static_cast<int64_t>(i >> 5) * p.n_q + q) * p.n_docs + bb] = c;
            }
        } else {
            float c = active ? mm : 0.0f;
            if (SCALE && active && mm != -INFINITY) c = mm * q_scale;
            if (p.lq_pad == 32) {
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
                if (lane == 0 && q < p.n_q) p.scores[static_cast<int64_t>(q) * p.ld_out + bb] = c;
            } else if (p.lq_pad < 32) {
                for (int off = 1; off < p.lq_pad; off <<= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
                if (i == 0 && q < p.n_q) p.scores[static_cast<int64_t>(q) * p.ld_out + bb] = c;
            } else {
                for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
                if (lane == 0 && q < p.n_q)
                    p.partials[(static_cast<int64_t>(i >> 5) * p.n_q + q) * p.n_docs + bb] = c;
            }
        }
    };

    // PAIRED: the documents closed since the last meeting (the first is
    // buf_b), and the parity of the next meeting at pair->bar.
    [[maybe_unused]] int n_buf = 0, buf_b = b_begin;
    [[maybe_unused]] uint32_t pair_phase = 0;
    // Meet the partner (both have closed the same documents), merge and
    // write out documents d = half, half + 2, ..., meet again.
    [[maybe_unused]] auto flush = [&]() {
        if (n_buf == 0 || aborted) return;
        __syncwarp();
        if (lane == 0) mbar_arrive(&pair->bar);
        if (!mbar_wait(&pair->bar, pair_phase, abort_flag, p.status, kStatusTimeoutEpilogue)) {
            aborted = true;
            return;
        }
        pair_phase ^= 1u;
        for (int d = half; d < n_buf; d += 2) {
            const float m0 = pair->m[0][d][lane], m1 = pair->m[1][d][lane];
            const int a0 = pair->a[0][d][lane], a1 = pair->a[1][d][lane];
            emit(buf_b + d, fmaxf(m0, m1), m0 > m1 ? a0 : (m1 > m0 ? a1 : min(a0, a1)), pair->doc_lo[d],
                 pair->doc_hi[d]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&pair->bar);
        if (!mbar_wait(&pair->bar, pair_phase, abort_flag, p.status, kStatusTimeoutEpilogue)) {
            aborted = true;
            return;
        }
        pair_phase ^= 1u;
        buf_b += n_buf;
        n_buf = 0;
    };

    // End of document b for this warp's rows: write it out (PAIRED: hand
    // this warp's partial to the pair buffer), then move to document b + 1.
    auto finalize = [&]() {
        if constexpr (PAIRED) {
            if (!aborted) {
                pair->m[half][n_buf][lane] = m;
                pair->a[half][n_buf][lane] = a;
                if (half == 0 && lane == 0) {
                    pair->doc_lo[n_buf] = doc_lo;
                    pair->doc_hi[n_buf] = doc_hi;
                }
                ++n_buf;
            }
        } else {
            emit(b, m, a, doc_lo, doc_hi);
        }
        m = -INFINITY;
        a = -1;
        ++b;
        doc_lo = doc_hi;
        doc_hi = (b < b_end) ? boundary(b + 1) : INT32_MAX;
        if constexpr (PAIRED)
            if (n_buf == kPairDocs) flush();
    };

    // Columns c0 .. c0+31 of the current tile: split at document ends.
    auto process = [&](const uint32_t (&r)[32], int c0) {
        if (c0 >= t_end) return;                 // past the last document of this CTA
        while (doc_hi <= c0) finalize();         // documents ending at the chunk start (or empty)
        if (doc_hi >= c0 + 32) {                 // the whole chunk lies in the current document
            fold_chunk<ARGMAX, false>(r, c0, 0, 32, m, a);
            return;
        }
        if (c0 + 32 <= t_end && b + 1 < b_end && boundary(b + 2) >= c0 + 32) {
            // exactly one document boundary inside the chunk
            float m_next;
            int a_next = -1;
            fold_split<ARGMAX>(r, c0, doc_hi - c0, m, a, m_next, a_next);
            finalize();
            m = m_next;
            a = a_next;
            return;
        }
        // several boundaries, or the end of this CTA's documents
        const int cend = min(c0 + 32, t_end);
        int c = c0;
        while (c < cend) {
            if (doc_hi <= c) {
                finalize();
                continue;
            }
            const int seg_end = min(doc_hi, cend);
            if (c == c0 && seg_end == c0 + 32) fold_chunk<ARGMAX, false>(r, c0, 0, 32, m, a);
            else fold_chunk<ARGMAX, true>(r, c0, c - c0, seg_end - c0, m, a);
            c = seg_end;
        }
    };

    uint32_t ra[32];
    [[maybe_unused]] uint32_t rb[32];
    [[maybe_unused]] float sc_cur[4] = {0.f, 0.f, 0.f, 0.f}, sc_nxt[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (SCALE && !DB)
        if (warp_rows)
#pragma unroll
            for (int kc = 0; kc < 4; ++kc) sc_nxt[kc] = chunk_scale(t_begin + 32 * kc);
    for (int j = 0; j < n_tiles; ++j) {
        const int2 su = slot_of(j);
        const int slot = su.x;
        const uint32_t use = static_cast<uint32_t>(su.y);
        if (!mbar_wait(&t_full[slot], use & 1, abort_flag, p.status, kStatusTimeoutEpilogue)) {
            aborted = true;
            break;
        }
        tc_fence_after();
        if (!warp_rows) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release(slot);
            continue;
        }
        const uint32_t tb = tmem_base + lane_base + slot * kSlotCols;
        const int tile0 = t_begin + j * kBlockN;
        if constexpr (DB) {
            // four 32-column chunks, the next one loading while one is folded
            [[maybe_unused]] float sa = chunk_scale(tile0), sb = 0.0f;
            __syncwarp();
            tmem_ld32_async(tb, ra);
            tmem_wait_ld(ra);
            if constexpr (SCALE) apply_scale(ra, sa);
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                if constexpr (SCALE) sb = chunk_scale(tile0 + 64 * h + 32);
                __syncwarp();
                tmem_ld32_async(tb + 64 * h + 32, rb);
                process(ra, tile0 + 64 * h);
                if constexpr (SCALE) if (h == 0) sa = chunk_scale(tile0 + 64);
                __syncwarp();
                tmem_wait_ld(rb);
                if (h == 0) {
                    tmem_ld32_async(tb + 64, ra);
                } else {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) release(slot);
                }
                if constexpr (SCALE) apply_scale(rb, sb);
                process(rb, tile0 + 64 * h + 32);
                if (h == 0) {
                    __syncwarp();
                    tmem_wait_ld(ra);
                    if constexpr (SCALE) apply_scale(ra, sa);
                }
            }
        } else {
            // SCALE: this tile's column scales were loaded one tile ahead (lane
            // l holds column 32 kc + l of chunk kc); load the next tile's now
            if constexpr (SCALE) {
#pragma unroll
                for (int kc = 0; kc < 4; ++kc) {
                    sc_cur[kc] = sc_nxt[kc];
                    sc_nxt[kc] = chunk_scale(tile0 + kBlockN + 32 * kc);
                }
            }
            // registers are scarce with 18-20 warps per SM: one chunk at a time
            constexpr int kc_n = PAIRED ? 2 : 4;
            const int kc_lo = PAIRED ? 2 * half : 0;
#pragma unroll 1
            for (int kc = kc_lo; kc < kc_lo + kc_n; ++kc) {
                [[maybe_unused]] float sc = 0.0f;
                if constexpr (SCALE) sc = kc == 0 ? sc_cur[0] : kc == 1 ? sc_cur[1] : kc == 2 ? sc_cur[2] : sc_cur[3];
                __syncwarp();
                tmem_ld32_async(tb + 32 * kc, ra);
                tmem_wait_ld(ra);
                if (kc == kc_lo + kc_n - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) release(slot);
                }
                if constexpr (SCALE) apply_scale(ra, sc);
                process(ra, tile0 + 32 * kc);
            }
            if constexpr (PAIRED)
                if (aborted) break;
        }
    }
    if (!aborted && warp_rows) {
        while (b < b_end && !aborted) finalize();
        if constexpr (PAIRED) flush();
    }
}

}  // namespace
}  // namespace maxsim
