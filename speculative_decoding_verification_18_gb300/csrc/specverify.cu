// specverify: batched speculative-decoding verify on GB300 (sm_103a).
//
// The one-call entry points run ONE kernel, sv_verify_kernel: a thread-block
// cluster of G CTAs per sequence (distributed shared memory, hardware cluster
// barriers; no global-memory handshakes) does the whole verify of that
// sequence:
//
//  1. Row statistics ("Speculative Decoding" (ch15, LLM serving from scratch),
//     §"Why the result is exactly the target model": the target's logits in,
//     p = softmax(l/T)): every CTA streams its vocabulary slice of the rows
//     with 16-byte coalesced loads and keeps an online max / sum-of-exponentials
//     (one ex2 per element) and the first index of the maximum.  Rows are
//     taken in waves: all k+1 at once when the batch is too small to fill the
//     GPU, one at a time (stopping at the first rejection, so later rows are
//     never read) when other sequences keep the HBM busy.  Warp shuffles,
//     shared memory and DSMEM merge the partials; every CTA then holds the same
//     row statistics.
//  2. The accept scan ("Decodificação especulativa explicada: rascunhe barato,
//     verifique numa passada", §"A regra de amostragem por rejeição": accept x
//     with probability min(1, p(x)/q(x)), stop at the first rejection; greedy:
//     accept while x == argmax p), computed redundantly by every CTA.
//  3. The draw (same section, rules 2 and 3: the residual norm(max(0, p - q))
//     at a rejection, p itself for the bonus; the categorical draw is the first
//     j with C_j > u * C_{V-1}, the right-sided search of §"Amostragem
//     especulativa em numpy, com prova").  The decision row's exponentials are
//     recomputed in float-float (~48 bits), the normaliser summed to ~2^-47,
//     and the weights turned into 60-bit fixed-point integers per 8-element
//     chunk, so every prefix sum is exact and order-independent; a DSMEM scan
//     over the cluster finds the CTA, a block scan the chunk, and one thread
//     the token.
//
// The two-stage entry points (spec_verify_rows / spec_verify_finish) run the
// same work as two kernels with the per-row statistics in the workspace:
// sv_rows_kernel (one CTA or cluster per row) and sv_finish_greedy_kernel /
// sv_finish_sample_kernel (one cluster per sequence), sharing the device code
// above.
//
// Nothing here allocates memory, synchronises the host, or waits on another
// CTA outside hardware cluster barriers.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <mutex>
#include <new>

#include "../../include/specverify.h"
#include "../../include/specverify_debug.h"
#include "ff.cuh"

namespace cg = cooperative_groups;

namespace sv {

// ------------------------------------------------------------------ workspace

constexpr uint32_t kMagic = 0x53564632u;  // "SVF2"
constexpr int kMaxK = 64;
constexpr int kMaxV = 1 << 21;

struct alignas(16) Header {
    uint32_t magic;
    uint32_t B, k, V, mode;
    // Layout of the row records the greedy row stream left: 0 for one record per
    // row; else the flat stream's CTA count, and the rows' length in 16-byte
    // vectors (the records then hold per-CTA partial keys).
    uint32_t flat_ctas, flat_vpr, flat_per, flat_rem;
    uint32_t pad[55];
};
static_assert(sizeof(Header) == 256, "header size");

// One record per logits row.
struct alignas(16) RowRec {
    float mraw;       // max_j l_j (raw logits); NaN for a row the scan never reached
    float S;          // sum_j exp((l_j - mraw)/T)  (sampled mode)
    double px;        // p(x) (sampled, rows < k)
    float lx;         // l[x]
    float qx;         // q[x]
    int32_t argmax;   // lowest index of the maximum raw logit
    uint32_t flags;   // kRow* bits
};
static_assert(sizeof(RowRec) == 32, "row record size");

constexpr uint32_t kRowBad = 1u, kRowTokenBad = 2u, kRowQBad = 4u, kRowSkipped = 8u;

// The record of a row that was never (or only partly) read.
__device__ __forceinline__ RowRec skipped_record() {
    RowRec rec;
    rec.mraw = NAN;
    rec.S = NAN;
    rec.px = NAN;
    rec.lx = NAN;
    rec.qx = NAN;
    rec.argmax = -1;
    rec.flags = kRowSkipped;
    return rec;
}

// Layout: header | B*(k+1) row records | B per-sequence status words | B
// per-sequence stop rows (the row-skipping path) | a 16-byte counter and B
// entries of the list of draws left to the precise kernel (large batches).
__host__ __device__ inline size_t ws_rows_offset() { return sizeof(Header); }
__host__ __device__ inline size_t ws_seq_offset(long long B, int k) {
    return sizeof(Header) + (size_t)B * (k + 1) * sizeof(RowRec);
}
__host__ __device__ inline size_t ws_stop_offset(long long B, int k) {
    return ws_seq_offset(B, k) + (size_t)B * sizeof(uint32_t);
}
__host__ __device__ inline size_t ws_plist_offset(long long B, int k) {
    return (ws_stop_offset(B, k) + (size_t)B * sizeof(uint32_t) + 15) & ~(size_t)15;
}
// The split draws' region follows, 16-byte aligned (its size depends on V:
// split_ws_bytes, defined with the split draw).
__host__ __device__ inline size_t ws_split_offset(long long B, int k) {
    return (ws_plist_offset(B, k) + 16 + (size_t)B * sizeof(uint32_t) + 15) & ~(size_t)15;
}
__host__ __device__ size_t split_ws_bytes(long long B, int V);
// Then the split row-skipping stream's region: per row an arrival counter, up
// to 8 partial statistics of 16 bytes and a 16-byte record of its gathers.
__host__ __device__ inline size_t ws_rowsplit_offset(long long B, int k, int V) {
    return (ws_split_offset(B, k) + split_ws_bytes(B, V) + 15) & ~(size_t)15;
}
__host__ __device__ inline size_t rowsplit_bytes(long long B, int k) {
    const size_t R = (size_t)B * (k + 1);
    return ((R * 4 + 15) & ~(size_t)15) + R * 8 * 16 + R * 16;
}
__host__ __device__ inline size_t ws_bytes_for(long long B, int k, int V) {
    size_t b = ws_rowsplit_offset(B, k, V) + rowsplit_bytes(B, k);
    return (b + 255) & ~(size_t)255;
}
// Without the split region (every path but the split draw).
__host__ __device__ inline size_t ws_base_bytes(long long B, int k) {
    return (ws_split_offset(B, k) + 255) & ~(size_t)255;
}

// ------------------------------------------------------------------ small helpers

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float fmax_nan(float a, float b) {
    float y;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
    return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <typename DT> struct Elt;
template <> struct Elt<__nv_bfloat16> {
    static constexpr int kVec = 8;  // elements per 16-byte vector
    __device__ static __forceinline__ float load1(const __nv_bfloat16* p) {
        return __bfloat162float(*p);
    }
    __device__ static __forceinline__ void unpack(const uint4& v, float* f) {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
        f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
        f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    }
};
template <> struct Elt<float> {
    static constexpr int kVec = 4;
    __device__ static __forceinline__ float load1(const float* p) { return *p; }
    __device__ static __forceinline__ void unpack(const uint4& v, float* f) {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
};

// Read-only 16-byte load that does not allocate in L1 (the stream is read once).
__device__ __forceinline__ uint4 ld_stream16(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ------------------------------------------------------------------ online softmax partials

// Running max m (raw logits), sum s of 2^((l - m) c), index of the first maximum,
// and a NaN flag (greedy mode, which forms no sum that would carry the NaN).
struct Partial {
    float m, s;
    int idx;
    int nan;
};

__device__ __forceinline__ Partial empty_partial() { return Partial{-INFINITY, 0.0f, -1, 0}; }

template <bool SAMPLED>
__device__ __forceinline__ void merge(Partial& a, const Partial& b, float c) {
    float mn = fmaxf(a.m, b.m);
    if (SAMPLED) {
        float fa = (a.m == mn) ? 1.0f : ex2_approx((a.m - mn) * c);
        float fb = (b.m == mn) ? 1.0f : ex2_approx((b.m - mn) * c);
        a.s = a.s * fa + b.s * fb;
    }
    if (b.m > a.m || (b.m == a.m && (unsigned)b.idx < (unsigned)a.idx)) a.idx = b.idx;
    a.m = mn;
    a.nan |= b.nan;
}

template <bool SAMPLED>
__device__ __forceinline__ Partial warp_merge(Partial p, float c) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        Partial o;
        o.m = __shfl_xor_sync(0xffffffffu, p.m, off);
        o.s = __shfl_xor_sync(0xffffffffu, p.s, off);
        o.idx = __shfl_xor_sync(0xffffffffu, p.idx, off);
        o.nan = __shfl_xor_sync(0xffffffffu, p.nan, off);
        merge<SAMPLED>(p, o, c);
    }
    return p;
}

// One thread's share of a vocabulary slice of one row: vectors [vb, ve) of the
// row's aligned body handled by threads tg = 0..ng-1 (stride ng), plus the
// unaligned head (if `head_here`) and tail (if `tail_here`) as scalars.
// With POLL: every batch also reads *poll, and once it holds a value below
// `poll_row` the thread sets `aborted` and stops reading (its partial is then
// meaningless; the caller discards the row).
// Early rejection on the row-skipping stream: every batch each thread
// publishes its running statistics as one 64-bit shared word, and every
// second batch warp 0 merges them and, when the row's test must fail whatever
// the rest of the row holds, lowers the stop row at once, so that rows after
// it in its sequence stop being read sooner.
struct EarlyRej {
    unsigned long long* tpub;  // [nt] each thread's (max, sum) so far (shared)
    int nt;
    float lx, uq;              // thread 0's l(x) and u q(x)
    uint32_t* stop;
    uint32_t row;
    int* fired;                // shared: the stop row was lowered
};
// The initial word: max -inf, sum 0 (a partial of no element).
constexpr unsigned long long kEmptyPub = 0x00000000FF800000ull;

// One batch's share of the early rejection (called by every lane of every
// warp; the loop around it is warp-uniform, t its batch number).  Each word is
// a valid partial of its thread's elements so far, so any mix of old and new
// words bounds the row from below.  Sampled: warp 0 forms Z = sum over the
// threads of s_t 2^((m_t - l(x)) c), a lower bound of sum_j 2^((l_j - l(x)) c)
// over the whole row, so p(x) <= 1/Z; when u q(x) Z >= 1 + 2^-10 the row's own
// test at the end (u < p/q unless p >= q, in rounded arithmetic whose errors
// are far below that margin) rejects for sure.  Greedy: a thread's max above
// l(x) means the argmax is not x.
template <bool SAMPLED>
__device__ __forceinline__ void early_check(EarlyRej& er, const Partial& p, float c, int tg,
                                            int t) {
    volatile unsigned long long* pub = er.tpub;
    pub[tg] = ((unsigned long long)__float_as_uint(p.s) << 32) | __float_as_uint(p.m);
    if ((t & 1) == 0 || tg >= 32) return;
    // warp 0: the merge, every second batch
    const float lx = __shfl_sync(0xffffffffu, er.lx, 0), uq = __shfl_sync(0xffffffffu, er.uq, 0);
    float z = SAMPLED ? 0.0f : -INFINITY;
    for (int j = tg; j < er.nt; j += 32) {
        const unsigned long long v = pub[j];
        const float m = __uint_as_float((uint32_t)v), sw = __uint_as_float((uint32_t)(v >> 32));
        if (SAMPLED) {
            if (sw > 0.0f) z = __fadd_rn(z, __fmul_rn(sw, ex2_approx(__fmul_rn(__fsub_rn(m, lx), c))));
        } else {
            z = fmaxf(z, m);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, z, off);
        z = SAMPLED ? __fadd_rn(z, o) : fmaxf(z, o);
    }
    const bool rej = SAMPLED ? __fmul_rn(uq, z) >= 1.0009765625f : z > lx;
    if (tg == 0 && rej && !*er.fired) {
        atomicMin(er.stop, er.row);
        *er.fired = 1;
    }
}

template <typename DT, bool SAMPLED, int U, bool POLL = false>
__device__ __forceinline__ Partial stream_slice(const DT* __restrict__ rowp, int V, long long vb,
                                                long long ve, int head, long long tail0,
                                                bool head_here, bool tail_here, int tg, int ng,
                                                float c, const uint32_t* poll = nullptr,
                                                uint32_t poll_row = 0, bool* aborted = nullptr,
                                                EarlyRej* er = nullptr) {
    using E = Elt<DT>;
    constexpr int VW = E::kVec;
    Partial p = empty_partial();
    int best_vec = 0;  // p.idx names the first element of a vector to resolve at the end
    auto scalar = [&](long long j) {
        float v = E::load1(rowp + j);
        if (!SAMPLED) p.nan |= (v != v);
        if (v > p.m) {
            if (SAMPLED) p.s *= ex2_approx((p.m - v) * c);
            p.m = v;
            p.idx = (int)j;
            best_vec = 0;
        }
        if (SAMPLED) p.s += ex2_approx((v - p.m) * c);
    };
    auto vector = [&](const uint4& raw, long long j0) {
        float f[VW];
        E::unpack(raw, f);
        float vmax = f[0];
#pragma unroll
        for (int e = 1; e < VW; ++e) vmax = SAMPLED ? fmaxf(vmax, f[e]) : fmax_nan(vmax, f[e]);
        if (!SAMPLED) p.nan |= (vmax != vmax);
        if (vmax > p.m) {
            if (SAMPLED) p.s *= ex2_approx((p.m - vmax) * c);
            p.m = vmax;
            p.idx = (int)j0;
            best_vec = 1;
        }
        if (SAMPLED) {
            float acc = 0.0f;
#pragma unroll
            for (int e = 0; e < VW; ++e) acc += ex2_approx((f[e] - p.m) * c);
            p.s += acc;
        }
    };
    if (head_here)
        for (long long j = tg; j < head; j += ng) scalar(j);
    const uint4* vp = reinterpret_cast<const uint4*>(rowp + head);
    // Batches of U vectors per thread, the loads of a batch issued together (the
    // last batch predicated), so a thread with up to U*n vectors waits for n
    // round trips.
    // Polling: the batches are counted per warp (the warp's first lane's
    // count; lanes past the end have their loads predicated off) and the
    // abandon decision is the warp's, so every lane takes every batch's
    // shuffles (the early rejection's warp merge) together.
    const long long step = (long long)U * ng;
    const long long vend = POLL ? vb + (tg & ~31) + ((ve - vb - (tg & ~31) + step - 1) / step) * step
                                : ve;
    int bt = 0;  // batch number
    for (long long v = vb + tg; POLL ? (v - tg + (tg & ~31) < vend) : (v < ve); v += step, ++bt) {
        uint4 buf[U];
        uint32_t st = 0xFFFFFFFFu;
        if (POLL) st = *reinterpret_cast<const volatile uint32_t*>(poll);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v + (long long)u * ng < ve) buf[u] = ld_stream16(vp + v + (long long)u * ng);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v + (long long)u * ng < ve) vector(buf[u], head + (v + (long long)u * ng) * VW);
        if (POLL && er) early_check<SAMPLED>(*er, p, c, tg, bt);
        if (POLL && __any_sync(0xffffffffu, st < poll_row)) {
            *aborted = true;
            break;
        }
    }
    if (tail_here)
        for (long long j = tail0 + tg; j < V; j += ng) scalar(j);
    if (best_vec) {  // first element equal to the maximum inside its vector
        float f[VW];
        E::unpack(*reinterpret_cast<const uint4*>(rowp + p.idx), f);
        int e = 0;
        while (e < VW - 1 && !(f[e] == p.m)) ++e;
        p.idx += e;
    }
    return p;
}

// Aligned body of a row: `head` unaligned leading elements, `nvec` 16-byte
// vectors, scalars from `tail0`.
template <typename DT>
__device__ __forceinline__ void row_layout(const DT* rowp, int V, int& head, long long& nvec,
                                           long long& tail0) {
    const uintptr_t addr = reinterpret_cast<uintptr_t>(rowp);
    head = (int)(((16 - (addr & 15)) & 15) / sizeof(DT));
    if (head > V) head = V;
    nvec = (V - head) / Elt<DT>::kVec;
    tail0 = head + nvec * Elt<DT>::kVec;
}

// kRowBad when the merged statistics show a NaN, a +inf, or an all -inf row.
template <bool SAMPLED>
__device__ __forceinline__ uint32_t row_flags(const Partial& p) {
    bool bad = !(p.m > -INFINITY) || p.m == INFINITY || p.nan;
    if (SAMPLED) bad = bad || !(p.s > 0.0f) || !(p.s < INFINITY);
    return bad ? kRowBad : 0u;
}

// ------------------------------------------------------------------ draw phase

constexpr int kThreads = 512;       // threads per CTA of the per-sequence kernels
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 8;           // contiguous elements per draw work item
constexpr int kSliceMax = 163840;   // largest slice of a row one CTA draws from

// Error model of the fast fp32 draw.  ex2.approx.ftz.f32 is taken to be within
// kEx2RelErr of 2^a (relative) on [-126, 0]: a test measures its worst case
// exhaustively over every float of that range (on GB300: 1.715e-7, 2^-22.48)
// and requires it to be at most this value, so the bound holds for every input
// the draw can see on this GPU (inputs below -126 give 0 and are counted as 0).
constexpr float kEx2RelErr = 1.75e-7f;
// Relative error of one element's y.  The exponent's parts are all recovered:
// l - m exactly (TwoSum), the rounding of a = (l - m) c_hi exactly (an FMA),
// and the low part of c = log2(e)/T; their sum t (at most 3 2^-24 |a|, so below
// 2^-15 for |a| < 126; below that y is 0) corrects ex2(a) to first order,
// y = ex2(a) (1 + t ln2).  What is left: ex2 itself, the one rounding of that
// FMA, and terms below 2^-33 (the second order of t ln2, the roundings inside
// t, c's float-float residual), covered by the extra 2^-28.
constexpr float kFastEy = kEx2RelErr + 1.0625f * 5.96046448e-08f;
// Classes of a residual's elements, decided during the one pass with the row
// stream's normaliser S_row in place of the pass's own S (which is checked
// afterwards to lie within 2^-13 of S_row): p > q for sure when
// y / (S_row (1 + 2^-12)) > q, p < q for sure when y / (S_row (1 - 2^-12)) < q
// (the margin exceeds 2^-13, the relative errors of y and of S, and the few
// roundings of the scaled reciprocals and the product).  An element in between
// is left out of the weights and its exact weight, at most kUndecided q
// (2^-12 + 2^-13 + those errors, about 3.8e-4), goes into the error bound.
constexpr float kClassHi = 1.0f + 1.0f / 4096.0f, kClassLo = 1.0f - 1.0f / 4096.0f;
constexpr double kRowSigma = 1.0 / 8192.0;
constexpr float kUndecided = 3.9e-4f;

// The fast draw's certificate, in units of 2^-62 of p (the linear form C's
// units).  An edge of the chosen bin with the positive mass P_b and the q mass
// Q_b before it (P_a, Q_a after it) is kept at more than
//   kP ((1 - u) P_b + u P_a) + kQ ((1 - u) Q_b + u Q_a)
//   + e_S 1.004 (|u Q_tot - Q_b| + 1 + the bin's width) + max(u, 1 - u) D
//   (+ without EXACT, 2 kQ' (P_c + Q_c) for the edge's chunk) + 2
// from u C_tot; the derivation is at fast_bound.
struct FastCert {
    float kP, kQ;               // per unit of P and of Q: the elements' own errors
    float eS;                   // the normaliser's relative error
    float D;                    // undecided weights, float-float sums, truncations
    long long Pt;               // P_tot (units)
    unsigned long long Qt, uQ;  // Q_tot and floor(u Q_tot) (units)
};

template <typename DT>
__device__ __forceinline__ void load_chunk(const DT* __restrict__ rowp, long long j0, int V,
                                           bool aligned, float* f) {
    if (aligned && j0 + kChunk <= V) {
        if constexpr (sizeof(DT) == 2) {
            uint4 v = *reinterpret_cast<const uint4*>(rowp + j0);
            Elt<__nv_bfloat16>::unpack(v, f);
        } else {
            uint4 v0 = *reinterpret_cast<const uint4*>(rowp + j0);
            uint4 v1 = *reinterpret_cast<const uint4*>(rowp + j0 + 4);
            Elt<float>::unpack(v0, f);
            Elt<float>::unpack(v1, f + 4);
        }
    } else {
#pragma unroll
        for (int e = 0; e < kChunk; ++e)
            f[e] = (j0 + e < V) ? Elt<DT>::load1(rowp + j0 + e) : -INFINITY;
    }
}

__device__ __forceinline__ void load_q_chunk(const float* __restrict__ qrow, long long j0, int V,
                                             bool aligned, float* f) {
    if (aligned && j0 + kChunk <= V) {
        float4 a = *reinterpret_cast<const float4*>(qrow + j0);
        float4 b = *reinterpret_cast<const float4*>(qrow + j0 + 4);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    } else {
#pragma unroll
        for (int e = 0; e < kChunk; ++e) f[e] = (j0 + e < V) ? qrow[j0 + e] : 0.0f;
    }
}

// Weight of one element for the precise draw: p = e/S (bonus) or max(0, p - q)
// (residual), branch-free.
__device__ __forceinline__ ff draw_weight(ff e, ff inv, float qv, bool residual) {
    ff p = ff_mul(e, inv);
    if (!residual) return p;  // uniform across the CTA
    ff s = two_sum(p.hi, -qv);
    ff w = fast_two_sum(s.hi, __fadd_rn(s.lo, p.lo));
    const bool pos = w.hi > 0.0f;
    const bool big = w.hi > 1.0f;  // only reachable with a negative q entry
    return ff{pos ? (big ? 1.0f : w.hi) : 0.0f, (pos && !big) ? w.lo : 0.0f};
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ ff warp_sum_ff(ff v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        ff o{__shfl_xor_sync(0xffffffffu, v.hi, off), __shfl_xor_sync(0xffffffffu, v.lo, off)};
        v = ff_add(v, o);
    }
    return v;
}

// floor(u * C) for u in [0, 1) given as a float, C < 2^64, exactly.
__device__ __forceinline__ unsigned long long scale_floor(float u, unsigned long long C) {
    uint32_t bits = __float_as_uint(u);
    int ex = (int)((bits >> 23) & 0xFF);
    unsigned long long mant = bits & 0x7FFFFF;
    if (ex == 0) ex = 1;
    else mant |= 0x800000;
    if (mant == 0) return 0ull;
    int sh = 150 - ex;  // u = mant * 2^-sh, sh >= 24 for u < 1
    unsigned long long lo = mant * C;
    unsigned long long hi = __umul64hi(mant, C);
    if (sh >= 128) return 0ull;
    if (sh >= 64) return hi >> (sh - 64);
    return (lo >> sh) | (hi << (64 - sh));
}

// Shared memory of the draw besides its dynamic arrays.  Values exchanged
// between the CTAs of a cluster are pushed: each CTA writes its total into slot
// [rank] of every CTA of the cluster (DSMEM stores), then one cluster barrier;
// afterwards every CTA reads only its own copies, in the same order, so every
// CTA computes the same totals, and no CTA touches another's shared memory
// after the last barrier it passes.  Every slot array is written once per draw.
constexpr int kMaxG = 16;
// Per-thread sums of the fast pass.
struct FastTotals {
    ff S;                        // y of the elements that are not positive
    unsigned long long Y, Q;     // fixed-point sums of the positive elements' y and q
    float Aq;                    // q of the undecided elements
    float qmin;                  // the smallest q (negative: the precise pass decides)
};
static_assert(sizeof(FastTotals) == 32, "fast totals");
struct DrawShared {
    ff red_ff[kWarps];
    float red_f[kWarps];
    unsigned long long red_u[kWarps];
    unsigned long long woff[kWarps];
    ff xS[2][kMaxG];                  // normaliser totals: fast, precise
    float xA[kMaxG];                  // sum of e * |a| totals (fast)
    unsigned long long xW[3][kMaxG];  // weight totals: fast, precise, fallback round
    float xD[kMaxG];                  // error-bound totals (fast)
    int xC[kMaxG];                    // certificate flags (fast)
    ff S_tot;
    float A_tot;
    unsigned long long prefix, total, mytot;
    unsigned long long before;  // find_block's result
    float D_tot;
    int blk;
    int cert, cert_all;
    int token;
    // the fast pass
    FastTotals red_t[kWarps];
    FastTotals xT[kMaxG];             // each rank's sums
    unsigned long long f_M, f_tau;    // floor(2^(123 - EY) / S), floor(u C_tot)
    unsigned long long f_Y, f_Q;      // this rank's starting point (sums of the ranks before)
    unsigned long long f_bY, f_bQ;    // the owner's block's starting point
    FastCert f_c;                     // the certificate's parts
    int f_ok, f_owner;
};

__device__ const Exp2Table g_exp2_table = make_exp2_table();

// Cluster barrier, or a CTA barrier for a cluster of one.
__device__ __forceinline__ void xsync(cg::cluster_group& cluster, int G) {
    if (G > 1) cluster.sync();
    else __syncthreads();
}

// Cluster sum of a float-float value (and, with `xa`, of one float into
// sh.A_tot): a block reduction, the CTA total pushed to slot [rank] of every
// CTA of the cluster, then each CTA adds the G totals in one fixed order.
__device__ __forceinline__ ff cluster_sum_ff(cg::cluster_group& cluster, DrawShared& sh,
                                             ff* xslot, ff v, int rank, int G,
                                             float* xa = nullptr, float va = 0.0f) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum_ff(ff_normalize(v));
    if (xa) va = warp_sum(va);
    if (lane == 0) {
        sh.red_ff[warp] = v;
        sh.red_f[warp] = va;
    }
    __syncthreads();
    if (warp == 0) {
        ff w = lane < kWarps ? sh.red_ff[lane] : ff{0.0f, 0.0f};
        float f = (xa && lane < kWarps) ? sh.red_f[lane] : 0.0f;
        w = warp_sum_ff(w);
        w = ff{__shfl_sync(0xffffffffu, w.hi, 0), __shfl_sync(0xffffffffu, w.lo, 0)};
        if (xa) f = __shfl_sync(0xffffffffu, warp_sum(f), 0);
        if (lane < G) {
            *cluster.map_shared_rank(&xslot[rank], lane) = w;
            if (xa) *cluster.map_shared_rank(&xa[rank], lane) = f;
        }
    }
    xsync(cluster, G);
    if (warp == 0) {
        ff w = lane < G ? xslot[lane] : ff{0.0f, 0.0f};
        float f = (xa && lane < G) ? xa[lane] : 0.0f;
        w = warp_sum_ff(w);
        if (xa) f = warp_sum(f);
        if (lane == 0) {
            sh.S_tot = w;
            sh.A_tot = f;
        }
    }
    __syncthreads();
    return sh.S_tot;
}

// Cluster prefix of the chunk-weight totals: a block reduction (and of one
// float), the CTA totals pushed to slot [rank] of every CTA; then this rank's
// exclusive prefix, its own total and the grand total (sh.prefix, sh.mytot,
// sh.total) and the float's cluster sum (sh.D_tot).  `xw` is the slot array of
// this round; `xd` may be null.
__device__ __forceinline__ void cluster_prefix(cg::cluster_group& cluster, DrawShared& sh,
                                               unsigned long long* xw, float* xd,
                                               unsigned long long t, float d, int rank, int G) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    t = warp_sum(t);
    d = warp_sum(d);
    if (lane == 0) {
        sh.red_u[warp] = t;
        sh.red_f[warp] = d;
    }
    __syncthreads();
    if (warp == 0) {
        unsigned long long w = lane < kWarps ? sh.red_u[lane] : 0ull;
        float f = lane < kWarps ? sh.red_f[lane] : 0.0f;
        w = __shfl_sync(0xffffffffu, warp_sum(w), 0);
        f = __shfl_sync(0xffffffffu, warp_sum(f), 0);
        if (lane < G) {
            *cluster.map_shared_rank(&xw[rank], lane) = w;
            if (xd) *cluster.map_shared_rank(&xd[rank], lane) = f;
        }
    }
    xsync(cluster, G);
    if (warp == 0) {
        const unsigned long long v = lane < G ? xw[lane] : 0ull;  // lane r: rank r's total
        float f = (xd && lane < G) ? xd[lane] : 0.0f;
        unsigned long long incl = v;  // inclusive prefix over ranks
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            unsigned long long o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        f = warp_sum(f);
        const unsigned long long tot = __shfl_sync(0xffffffffu, incl, 31);
        const unsigned long long pre = __shfl_sync(0xffffffffu, incl - v, rank);
        const unsigned long long mine = __shfl_sync(0xffffffffu, v, rank);
        if (lane == 0) {
            sh.prefix = pre;
            sh.total = tot;
            sh.mytot = mine;
            sh.D_tot = f;
        }
    }
    __syncthreads();
}

// ---- work layout of a draw
//
// The CTA of rank r owns chunks [c0, c0 + mych) of the row (nch chunks of 8
// elements split evenly over the G ranks).  Thread t takes chunks t, t + kThreads,
// ...; a warp's 32 lanes thus cover 32 consecutive chunks per iteration, a
// "block" of 256 elements whose fixed-point weight total the warp keeps in
// bsum[block].  Locating the drawn token needs only the block totals: the
// owning block is recomputed by one warp, the owning chunk by one lane.
constexpr int kBlockChunks = 32;

template <typename DT>
struct DrawCtx {
    const DT* rowp;
    const float* qrow;
    int V;
    bool residual;
    float m, c;     // row max (raw logit), log2(e)/T in float (its high part)
    float clo;      // low part of log2(e)/T
    ff c2;          // log2(e)/T in float-float
    float u;
    long long c0;
    int mych, nblk;
    bool al_l, al_q;
    int rank, G;
    unsigned long long* bsum;  // block sums (the fast pass: Y then Q per 64 elements)
    ff* ecache;                // [mych * 8] precise exponentials, or null
    float* thi;                // [kExpTable] each; loaded by the precise pass
    float* tlo;
    float s_row;               // the row stream's fp32 normaliser (relative to m)
    ff* pY;                    // [mych] one-read precise pass: chunk sums, or null
    ff* pQ;                    // [mych]
    unsigned char* pamb;       // [mych]
};

template <typename DT>
__device__ __forceinline__ void load_l(const DrawCtx<DT>& d, int ci, float* f) {
    load_chunk<DT>(d.rowp, (d.c0 + ci) * kChunk, d.V, d.al_l, f);
}
template <typename DT>
__device__ __forceinline__ void load_q(const DrawCtx<DT>& d, int ci, bool use, float* f) {
    if (use) {
        load_q_chunk(d.qrow, (d.c0 + ci) * kChunk, d.V, d.al_q, f);
    } else {
#pragma unroll
        for (int e = 0; e < kChunk; ++e) f[e] = 0.0f;
    }
}

// Raw bits of one chunk, so that a thread can hold several chunks in flight in
// few registers: 8 logits (one or two 16-byte vectors) or 8 q values.  Elements
// past V read as -inf (logits) or 0 (q), the fill of the scalar loads.
template <typename DT> struct RawL;
template <> struct RawL<__nv_bfloat16> { uint4 v[1]; };
template <> struct RawL<float> { uint4 v[2]; };
struct RawQ { uint4 v[2]; };

template <typename DT>
__device__ __forceinline__ void raw_load_l(const DrawCtx<DT>& d, int ci, RawL<DT>& r) {
    const long long j0 = (d.c0 + ci) * kChunk;
    constexpr int NV = (int)(sizeof(RawL<DT>) / 16);
    if (d.al_l && j0 + kChunk <= d.V) {
#pragma unroll
        for (int w = 0; w < NV; ++w) r.v[w] = ld_stream16(reinterpret_cast<const uint4*>(d.rowp + j0) + w);
    } else {
        float f[kChunk];
        load_chunk<DT>(d.rowp, j0, d.V, d.al_l, f);
        if constexpr (sizeof(DT) == 2) {  // back to bf16 bits (exact: they came from bf16)
            uint32_t h[kChunk];
#pragma unroll
            for (int e = 0; e < kChunk; ++e) h[e] = __float_as_uint(f[e]) >> 16;
            r.v[0] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                                h[6] | (h[7] << 16));
        } else {
            r.v[0] = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                                __float_as_uint(f[2]), __float_as_uint(f[3]));
            r.v[1] = make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]),
                                __float_as_uint(f[6]), __float_as_uint(f[7]));
        }
    }
}
template <typename DT>
__device__ __forceinline__ void raw_unpack(const RawL<DT>& r, float* f) {
    if constexpr (sizeof(DT) == 2) {
        Elt<__nv_bfloat16>::unpack(r.v[0], f);
    } else {
        Elt<float>::unpack(r.v[0], f);
        Elt<float>::unpack(r.v[1], f + 4);
    }
}
template <typename DT>
__device__ __forceinline__ void raw_load_q(const DrawCtx<DT>& d, int ci, RawQ& r) {
    const long long j0 = (d.c0 + ci) * kChunk;
    if (d.al_q && j0 + kChunk <= d.V) {
        r.v[0] = ld_stream16(reinterpret_cast<const uint4*>(d.qrow + j0));
        r.v[1] = ld_stream16(reinterpret_cast<const uint4*>(d.qrow + j0) + 1);
    } else {
        float f[kChunk];
        load_q_chunk(d.qrow, j0, d.V, d.al_q, f);
        r.v[0] = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                            __float_as_uint(f[3]));
        r.v[1] = make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]),
                            __float_as_uint(f[7]));
    }
}
__device__ __forceinline__ void raw_unpack_q(const RawQ& r, float* f) {
    Elt<float>::unpack(r.v[0], f);
    Elt<float>::unpack(r.v[1], f + 4);
}

// Inside the CTA: the block holding `want` (0 <= want < the CTA's total) and
// the total of the blocks before it.  Every thread returns the same values.
__device__ __forceinline__ void find_block(DrawShared& sh, const unsigned long long* bsum,
                                           int nblk, unsigned long long want, int* blk,
                                           unsigned long long* before) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = (nblk + kThreads - 1) / kThreads;
    const int cb = min(nblk, tid * L), ce = min(nblk, cb + L);
    if (tid == 0) {  // replaced by the one thread whose range holds `want`
        sh.blk = 0;
        sh.before = 0;
    }
    unsigned long long mine = 0;
    for (int i = cb; i < ce; ++i) mine += bsum[i];
    unsigned long long incl = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        unsigned long long o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) sh.red_u[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        unsigned long long wv = lane < kWarps ? sh.red_u[lane] : 0ull;
        unsigned long long wi = wv;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            unsigned long long o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        if (lane < kWarps) sh.woff[lane] = wi - wv;  // exclusive warp offsets
    }
    __syncthreads();
    const unsigned long long excl = sh.woff[warp] + incl - mine;
    if (mine > 0 && excl <= want && want - excl < mine) {  // exactly one thread
        unsigned long long run = excl;
        int i = cb;
        for (; i < ce - 1; ++i) {
            if (want - run < bsum[i]) break;
            run += bsum[i];
        }
        sh.blk = i;
        sh.before = run;
    }
    __syncthreads();
    *blk = min(max(sh.blk, 0), max(nblk - 1, 0));
    *before = sh.before;
}

// Inside warp 0: lane values v (chunk weights of a block, in chunk order); the
// lane whose chunk holds `want` (relative to the block) returns true with the
// weight before its chunk.
__device__ __forceinline__ bool find_lane(unsigned long long v, unsigned long long want,
                                          unsigned long long* before) {
    const int lane = threadIdx.x & 31;
    unsigned long long incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        unsigned long long o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    const unsigned long long excl = incl - v;
    *before = excl;
    return v > 0 && excl <= want && want - excl < v;
}

// ---- fast pass: one read, fp32 exponentials, fixed-point sums, error bound
//
// One pass over the CTA's slice of the decision row (and of its q row) forms,
// per element, y = 2^((l - m) log2(e)/T) in fp32 and decides whether p = y/S
// exceeds q (the classes above).  The weight max(0, p - q) is then the linear
// form p - q over the positive elements, so the cumulative weight up to any
// point is Y/S - Q, Y and Q the sums of y and of q over the positive elements
// before it.  Each lane sums the positive y and q of its chunk of 8 elements
// and turns the two sums into fixed point (Y in units 2^-EY, Q in units 2^-62):
// EXACT, in element order in float-float (error ~2^-44); otherwise pairwise in
// fp32 (three roundings, counted in the error bound), which is about half the
// work per element.  From there on everything is exact integer arithmetic:
// the sums per block of 8 chunks (64 elements), per CTA and per cluster, and
// the cumulative weight C = floor(Y M / 2^61) - Q (units 2^-62 of p) with
// M = floor(2^(123 - EY) / S).  The normaliser S is Y plus the other elements'
// y (summed pairwise per chunk, in float-float across chunks).  One cluster
// exchange gives every CTA the totals and its starting point; the owning CTA
// finds the block from its block sums in shared memory, and the block's 8
// lanes the element, recomputing only those 64 elements with the pass's own
// arithmetic, so that the lanes' and elements' boundaries inside the block
// agree exactly with the block sums.  No step uses FP64 (slow on this GPU) or
// 64-bit float-to-integer conversions.

// The fixed-point scale 2^EY of y: EY = 61 - e with S_row < 2^e, so that Y stays
// below 2^62 (S is within 2^-9 of S_row for any valid row).
__device__ __forceinline__ int fast_ey(float s_row) {
    int e = 0;
    (void)frexpf(s_row, &e);
    return max(0, min(61, 61 - e));
}

constexpr int kFastGroup = 8;  // lanes (chunks of 8 elements) per block of the fast pass

struct FastScale {
    float m, chi;       // row max (raw logit); log2(e)/T rounded to float
    float cll, chl;     // (log2(e)/T - chi) ln2 and chi ln2, for the correction
    float ih, il;       // 1 / (S_row (1 + 2^-12)), 1 / (S_row (1 - 2^-12)) (residual draws)
    int ey;             // EY
};

__device__ __forceinline__ FastScale make_fast_scale(float m, ff c2, float s_row, bool res) {
    FastScale f;
    f.m = m;
    f.chi = c2.hi;
    f.cll = __fmul_rn(c2.lo, 0.693147181f);
    f.chl = __fmul_rn(c2.hi, 0.693147181f);
    f.ih = res ? __frcp_rn(__fmul_rn(s_row, kClassHi)) : 0.0f;
    f.il = res ? __frcp_rn(__fmul_rn(s_row, kClassLo)) : 0.0f;
    f.ey = fast_ey(s_row);
    return f;
}

// acc += v in float-float (TwoSum into the high part, its error into lo).
__device__ __forceinline__ void ff_acc1(ff& acc, float v) {
    const ff s = two_sum(acc.hi, v);
    acc.hi = s.hi;
    acc.lo = __fadd_rn(acc.lo, s.lo);
}

// Pairwise sum of 8 floats (three rounding levels).
__device__ __forceinline__ float sum8(const float* v) {
    return __fadd_rn(__fadd_rn(__fadd_rn(v[0], v[1]), __fadd_rn(v[2], v[3])),
                     __fadd_rn(__fadd_rn(v[4], v[5]), __fadd_rn(v[6], v[7])));
}

// The pairwise prefix of 8 floats up to element e (the nodes of sum8's tree
// left of e, then e's own partial nodes): monotone in e, and for e = 7 equal to
// sum8 exactly.
__device__ __forceinline__ float prefix8(const float* v, int e) {
    const float n01 = __fadd_rn(v[0], v[1]), n45 = __fadd_rn(v[4], v[5]);
    const float n03 = __fadd_rn(n01, __fadd_rn(v[2], v[3]));
    float left, part;
    if (e < 4) {
        left = 0.0f;
        part = e == 0 ? v[0] : e == 1 ? n01 : e == 2 ? __fadd_rn(n01, v[2]) : n03;
        return part;
    }
    left = n03;
    part = e == 4 ? v[4] : e == 5 ? n45 : e == 6 ? __fadd_rn(n45, v[6])
                                               : __fadd_rn(n45, __fadd_rn(v[6], v[7]));
    return __fadd_rn(left, part);
}

// The fixed-point value of a non-negative float-float v = hi + lo (|lo| small):
// floor(hi 2^s) plus or minus floor(|lo| 2^s).
__device__ __forceinline__ unsigned long long ff_fixed(ff v, int s) {
    const unsigned long long h = fix_pow2(v.hi, s);
    const unsigned long long l = fix_pow2(fabsf(v.lo), s);
    return v.lo < 0.0f ? h - l : h + l;
}

// y of one element: d = l - m exact; a = d c_hi rounded; t = (the product's
// rounding + d c_lo + d_lo c_hi) ln2; y = ex2(a) (1 + t).  Every float
// operation is explicitly rounded, so the pass and the owner's search compute
// identical values.  l = -inf gives a NaN t and y = max(NaN, 0) = 0.
__device__ __forceinline__ float fast_y(float l, const FastScale& f) {
    const ff d = two_sum(l, -f.m);
    const float a = __fmul_rn(d.hi, f.chi);
    const float r = __fmaf_rn(d.hi, f.chi, -a);  // exact
    float t = __fmaf_rn(d.hi, f.cll, __fmul_rn(d.lo, f.chl));
    t = __fmaf_rn(r, 0.693147181f, t);
    const float y0 = ex2_approx(a);
    return fmaxf(__fmaf_rn(y0, t, y0), 0.0f);
}

// Pairwise tree of 8 values fed in index order: ((v0+v1)+(v2+v3)) + ((v4+v5)+(v6+v7)),
// folded as the values arrive (sum8's order, few live registers).
struct Tree8 {
    float a, p, h;  // the pending value, the pending pair, the first half
    template <int E>
    __device__ __forceinline__ void add(float v) {
        if (E % 2 == 0) {
            a = v;
        } else if (E == 1 || E == 5) {
            p = __fadd_rn(a, v);
        } else if (E == 3) {
            h = __fadd_rn(p, __fadd_rn(a, v));
        } else {  // E == 7
            h = __fadd_rn(h, __fadd_rn(p, __fadd_rn(a, v)));
        }
    }
};

// Element E of a chunk of the fast pass: y, and (residual draws) its class:
// positive when y / (S_row (1 + 2^-12)) > q, zero when y / (S_row (1 - 2^-12))
// < q, undecided otherwise (its q goes to aq, for the bound).  The positive
// elements' y and q go to the chunk's sums (EXACT: in element order in
// float-float, else the pairwise trees), the others' y to tr.
template <int E, bool RES, bool EXACT>
__device__ __forceinline__ void fast_chunk_elem(const float* l, const float* q, const FastScale& f,
                                                ff& Y, ff& Q, Tree8& ty, Tree8& tq, Tree8& tr,
                                                float& aq, uint32_t& qor, float* yp, float* qp) {
    const float y = fast_y(l[E], f);
    bool pos = true;
    if (RES) {
        pos = __fmul_rn(y, f.ih) > q[E];
        const bool und = !pos && !(__fmul_rn(y, f.il) < q[E]);
        aq = und ? __fadd_rn(aq, q[E]) : aq;
        qor |= __float_as_uint(q[E]);  // the sign bits: a negative q
    }
    const float yv = pos ? y : 0.0f, qv = (RES && pos) ? q[E] : 0.0f;
    if (yp) {
        yp[E] = yv;
        qp[E] = qv;
    }
    if (EXACT) {
        ff_acc1(Y, yv);
        if (RES) ff_acc1(Q, qv);
    } else {
        ty.add<E>(yv);
        if (RES) tq.add<E>(qv);
    }
    tr.add<E>(__fsub_rn(y, yv));  // the other elements' y (exact: yv is y or 0)
}

// One chunk (8 elements, logits l and q) of the fast pass: the fixed-point
// sums of the positive elements' y and q (cy, cq), the other elements' y
// summed pairwise (returned), the undecided elements' q into aq; qmin becomes
// -1 when a q of the chunk has its sign bit set (a negative q, caught by the
// caller; -0 too, conservatively); with `yp`, yp and qp receive each element's
// y and q when it is positive, else 0.  A NaN q is undecided (its bound is NaN,
// so the draw goes to the precise pass, which weighs it 0).
template <bool RES, bool EXACT>
__device__ __forceinline__ float fast_chunk(const float* l, const float* q, const FastScale& f,
                                            unsigned long long& cy, unsigned long long& cq,
                                            float& aq, float& qmin, float* yp, float* qp) {
    ff Y{0.0f, 0.0f}, Q{0.0f, 0.0f};
    Tree8 ty{}, tq{}, tr{};
    uint32_t qor = 0u;
    fast_chunk_elem<0, RES, EXACT>(l, q, f, Y, Q, ty, tq, tr, aq, qor, yp, qp);
    fast_chunk_elem<1, RES, EXACT>(l, q, f, Y, Q, ty, tq, tr, aq, qor, yp, qp);
    fast_chunk_elem<2, RES, EXACT>(l, q, f, Y, Q, ty, tq, tr, aq, qor, yp, qp);
    fast_chunk_elem<3, RES, EXACT>(l, q, f, Y, Q, ty, tq, tr, aq, qor, yp, qp);
    fast_chunk_elem<4, RES, EXACT>(l, q, f, Y, Q, ty, tq, tr, aq, qor, yp, qp);
    fast_chunk_elem<5, RES, EXACT>(l, q, f, Y, Q, ty, tq, tr, aq, qor, yp, qp);
    fast_chunk_elem<6, RES, EXACT>(l, q, f, Y, Q, ty, tq, tr, aq, qor, yp, qp);
    fast_chunk_elem<7, RES, EXACT>(l, q, f, Y, Q, ty, tq, tr, aq, qor, yp, qp);
    if (RES && (qor >> 31)) qmin = -1.0f;
    if (EXACT) {
        cy = ff_fixed(ff_normalize(Y), f.ey);
        cq = RES ? ff_fixed(ff_normalize(Q), 62) : 0ull;
    } else {
        cy = fix_pow2(ty.h, f.ey);
        cq = RES ? fix_pow2(tq.h, 62) : 0ull;
    }
    return tr.h;
}

// The fixed-point sums of the first e + 1 elements of a chunk, in the
// arithmetic of fast_chunk (for e = 7 its cy and cq exactly).
template <bool RES, bool EXACT>
__device__ __forceinline__ void fast_prefix(const float* yp, const float* qp, int e,
                                            const FastScale& f, unsigned long long& py,
                                            unsigned long long& pq) {
    if (EXACT) {
        ff Y{0.0f, 0.0f}, Q{0.0f, 0.0f};
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
            if (j > e) break;
            ff_acc1(Y, yp[j]);
            if (RES) ff_acc1(Q, qp[j]);
        }
        py = ff_fixed(ff_normalize(Y), f.ey);
        pq = RES ? ff_fixed(ff_normalize(Q), 62) : 0ull;
    } else {
        py = fix_pow2(prefix8(yp, e), f.ey);
        pq = RES ? fix_pow2(prefix8(qp, e), 62) : 0ull;
    }
}

// A 64-bit unsigned integer as float-float (each 32-bit half converted; the
// low half's rounding is 2^-24 of it).
__device__ __forceinline__ ff u64_to_ff(unsigned long long v) {
    const float hi = __fmul_rn(__uint2float_rn((uint32_t)(v >> 32)), 4294967296.0f);
    const float lo = __uint2float_rn((uint32_t)v);
    return ff_normalize(two_sum(hi, lo));
}

__device__ __forceinline__ FastTotals warp_fast_totals(FastTotals t) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const ff so{__shfl_xor_sync(0xffffffffu, t.S.hi, off),
                    __shfl_xor_sync(0xffffffffu, t.S.lo, off)};
        t.S = ff_add(t.S, so);
        t.Y += __shfl_xor_sync(0xffffffffu, t.Y, off);
        t.Q += __shfl_xor_sync(0xffffffffu, t.Q, off);
        t.Aq += __shfl_xor_sync(0xffffffffu, t.Aq, off);
        t.qmin = fminf(t.qmin, __shfl_xor_sync(0xffffffffu, t.qmin, off));
    }
    return t;
}

// C = floor(Y M / 2^61) - Q (Y M < 2^125 for Y within S 2^EY).
__device__ __forceinline__ long long fast_cval(unsigned long long Y, unsigned long long Q,
                                               unsigned long long M) {
    const unsigned long long lo = Y * M, hi = __umul64hi(Y, M);
    return (long long)((hi << 3) | (lo >> 61)) - (long long)Q;
}

// The sum of v over lanes [g*8, g*8 + 8) of the warp (every lane of the group
// ends with it).
__device__ __forceinline__ unsigned long long group_sum_u64(unsigned long long v) {
#pragma unroll
    for (int off = 1; off < kFastGroup; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ FastTotals zero_totals() {
    return FastTotals{ff{0.0f, 0.0f}, 0ull, 0ull, 0.0f, 0.0f};
}

__device__ __forceinline__ FastTotals add_fast_totals(FastTotals t, const FastTotals& x) {
    t.S = ff_add(t.S, x.S);
    t.Y += x.Y;
    t.Q += x.Q;
    t.Aq = __fadd_rn(t.Aq, x.Aq);
    t.qmin = fminf(t.qmin, x.qmin);
    return t;
}

// The fast pass over the CTA's slice of the decision row (and of its q row):
// this thread's sums.  Each warp takes 32 consecutive chunks (a chunk per lane,
// four blocks of 8 chunks), two such rounds in flight.  With BLOCKS the fixed-
// point sums of each block, {Y, Q}, go to d.bsum[2 blk], d.bsum[2 blk + 1]
// (shared or global memory, 16-byte aligned).
template <typename DT, bool RES, bool EXACT, bool BLOCKS>
__device__ __forceinline__ FastTotals fast_pass(const DrawCtx<DT>& d, const FastScale& f) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = lane / kFastGroup, gl = lane % kFastGroup;
    const int fnb = (d.mych + kFastGroup - 1) / kFastGroup;  // blocks of this CTA's slice
    FastTotals t = zero_totals();
    constexpr int UB = 1;  // (two in flight spill at 64 registers; 32 warps per SM cover it)
    for (int base0 = warp * 32; base0 < d.mych; base0 += UB * kThreads) {
        RawQ rq[UB];
        RawL<DT> rl[UB];
#pragma unroll
        for (int u = 0; u < UB; ++u) {
            const int ci = base0 + u * kThreads + lane;
            if (ci < d.mych) {
                if (RES) raw_load_q(d, ci, rq[u]);
                raw_load_l(d, ci, rl[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < UB; ++u) {
            const int base = base0 + u * kThreads;
            if (base >= d.mych) break;  // uniform across the warp
            unsigned long long cy = 0ull, cq = 0ull;
            if (base + lane < d.mych) {
                float l[kChunk], q[kChunk] = {};
                raw_unpack(rl[u], l);
                if (RES) raw_unpack_q(rq[u], q);
                const float rest =
                    fast_chunk<RES, EXACT>(l, q, f, cy, cq, t.Aq, t.qmin, nullptr, nullptr);
                ff_acc1(t.S, rest);
            }
            t.Y += cy;
            t.Q += cq;
            if (BLOCKS) {
                const unsigned long long by = group_sum_u64(cy);
                const unsigned long long bq = RES ? group_sum_u64(cq) : 0ull;
                const int blk = (base + grp * kFastGroup) / kFastGroup;
                if (gl == 0 && blk < fnb)
                    reinterpret_cast<ulonglong2*>(d.bsum)[blk] = make_ulonglong2(by, bq);
            }
        }
    }
    return t;
}

// The CTA's totals of the fast pass, left in *out (shared memory) for every
// thread after the barrier at the end.
__device__ __forceinline__ void cta_fast_totals(DrawShared& sh, FastTotals t, FastTotals* out) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    t = warp_fast_totals(t);
    if (lane == 0) sh.red_t[warp] = t;
    __syncthreads();
    if (warp == 0) {
        FastTotals c = lane < kWarps ? sh.red_t[lane] : zero_totals();
        c = warp_fast_totals(c);
        if (lane == 0) *out = c;
    }
    __syncthreads();
}

// The normaliser, the check against S_row, M = floor(2^(123 - EY) / S), C_tot,
// tau = floor(u C_tot) and the certificate's parts from a row's totals.
//
// Error bound.  Each positive element's p_fast = y/S carries its own error
// eta_j <= kFastEy (ex2 and the correction's FMA) and the normaliser's common
// eta_S <= e_S (kFastEy, and without EXACT the roundings of the pairwise chunk
// sums, 3 2^-24); p_fast = p (1 + eta_j) / (1 + eta_S).  The error of
// u C_tot - C_b at a bin edge b is, element by element, (u - 1) times the
// errors before the edge plus u times those after it.  So the elements' own
// errors contribute at most kFastEy ((1 - u) P_b + u P_a), with P_b and P_a the
// positive mass before and after the edge; without EXACT each chunk sum's
// three roundings (3 2^-24 of its y and of its q) split the same way, except
// in the edge's own chunk, whose prefix is not a part of the chunk's sum: its
// roundings are counted twice in full.  The normaliser's common factor
// contributes eta_S (u P_tot - P_b) = eta_S (u Q_tot - Q_b + (u C_tot - C_b)),
// at most e_S (|u Q_tot - Q_b| + the bin's width).  The undecided elements'
// weights (at most kUndecided q each, wherever they lie) contribute at most
// max(u, 1 - u) times their sum, as do the float-float sums (2^-44), M (2^-44)
// and the fixed-point truncations (2^20 + 2 per chunk + 64 units in all).  All
// are bounds of sums of positive terms computed in float: inflated by 1.004
// for their own roundings.  The token is kept when u C_tot lies more than its
// edge's bound (plus 2 units) inside both edges of its bin.
struct FastBound {
    unsigned long long M, tau;
    FastCert c;
    float S;  // the normaliser (high part)
    bool ok;
};
template <bool EXACT>
__device__ __forceinline__ FastBound fast_bound(const FastTotals& tot, float s_row, float u,
                                                int ey, long long nch) {
    FastBound fb;
    const unsigned long long Yall = tot.Y, Qall = tot.Q;
    const float pw = __int_as_float((127 - ey) << 23);  // 2^-EY
    const ff Yf = u64_to_ff(Yall);
    const ff S = ff_normalize(ff_add(ff{__fmul_rn(Yf.hi, pw), __fmul_rn(Yf.lo, pw)}, tot.S));
    fb.S = S.hi;
    bool ok = tot.qmin >= 0.0f && S.hi > 0.0f &&
              fabsf(__fsub_rn(S.hi, s_row)) <= S.hi * (float)kRowSigma;
    // M = floor(2^(123 - EY) / S): below 2^63 once S is within 2^-13 of S_row
    fb.M = ok ? ff_fixed(ff_recip(S), 123 - ey) : 0ull;
    const long long Ctot = ok ? fast_cval(Yall, Qall, fb.M) : 0ll;
    ok = ok && Ctot > 0;
    fb.tau = ok ? scale_floor(u, (unsigned long long)Ctot) : 0ull;
    fb.ok = ok;
    constexpr float u24 = 5.96046448e-08f;
    const float invS = __frcp_rn(S.hi);
    const float Ppos = __fmul_rn(__fmul_rn(Yf.hi, pw), invS);
    fb.c.eS = kFastEy + 3.0f * u24 * (EXACT ? fmaxf(0.0f, 1.0f - Ppos) : 1.0f);
    fb.c.kP = (kFastEy + (EXACT ? 0.0f : 3.0f * u24)) * 1.004f;
    fb.c.kQ = (EXACT ? 0.0f : 3.0f * u24) * 1.004f;
    fb.c.D = kUndecided * tot.Aq * 1.004f * 4.611686018427388e18f + 1048576.0f +
             2.0f * (float)nch + 64.0f;
    fb.c.Pt = ok ? fast_cval(Yall, 0ull, fb.M) : 0ll;
    fb.c.Qt = Qall;
    fb.c.uQ = ok ? scale_floor(u, Qall) : 0ull;
    return fb;
}

// The bound at one edge of the chosen bin (units), given the fixed-point sums
// (Yb, Qb) through the edge, the bin's width and (without EXACT) the positive
// and q mass of the edge's chunk (Pc + Qc, units).
__device__ __forceinline__ long long fast_edge_bound(const FastCert& c, unsigned long long M,
                                                     float u, unsigned long long Yb,
                                                     unsigned long long Qb, long long width,
                                                     float chunk_mass) {
    const long long Pb = fast_cval(Yb, 0ull, M);
    const float w1 = __fsub_rn(1.0f, u);
    const float pb = (float)Pb, pa = (float)max(c.Pt - Pb, 0ll);
    const float qb = (float)Qb, qa = (float)(c.Qt > Qb ? c.Qt - Qb : 0ull);
    const float dq = (float)(c.uQ > Qb ? c.uQ - Qb : Qb - c.uQ);
    float dp = c.kP * (w1 * pb + u * pa) + c.kQ * (w1 * qb + u * qa + 2.0f * chunk_mass);
    dp += c.eS * 1.004f * (dq + 1.0f + (float)width);
    dp += fmaxf(u, w1) * c.D + 2.0f;
    return (long long)fminf(dp, 4.0e18f) + 1ll;
}

// Block sums {Y, Q} of a slice: from shared memory, or (GLOBAL) written to the
// workspace by other CTAs of this launch, read past L1.
template <bool GLOBAL>
__device__ __forceinline__ ulonglong2 load_block(const unsigned long long* bsum, int i) {
    const ulonglong2* p = reinterpret_cast<const ulonglong2*>(bsum) + i;
    if (GLOBAL) return __ldcg(p);
    return *p;
}

// The owner CTA's search: given M, tau, D, e_S and the starting point (Y0, Q0)
// of its slice, find the block from the slice's block sums (d.bsum), then the
// chunk and the element, and certify it.  Every thread of the CTA calls it;
// sh.token and sh.cert hold the result after the last barrier.
template <typename DT, bool RES, bool EXACT, bool GLOBAL>
__device__ __forceinline__ void fast_search(DrawShared& sh, const DrawCtx<DT>& d,
                                            const FastScale& f, unsigned long long M,
                                            unsigned long long tau, unsigned long long Y0,
                                            unsigned long long Q0, const FastCert& c) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int fnb = (d.mych + kFastGroup - 1) / kFastGroup;
    // The block: each thread sums a contiguous range of block sums; a block
    // scan of (Y, Q) gives each range's start; the first range whose end
    // passes tau holds the block.
    const int L = (fnb + kThreads - 1) / kThreads;
    const int cb = min(fnb, tid * L), ce = min(fnb, cb + L);
    unsigned long long my = 0ull, mq = 0ull;
    for (int i = cb; i < ce; ++i) {
        const ulonglong2 v = load_block<GLOBAL>(d.bsum, i);
        my += v.x;
        mq += v.y;
    }
    unsigned long long iy = my, iq = mq;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long yo = __shfl_up_sync(0xffffffffu, iy, off);
        const unsigned long long qo = __shfl_up_sync(0xffffffffu, iq, off);
        if (lane >= off) {
            iy += yo;
            iq += qo;
        }
    }
    if (lane == 31) {
        sh.red_u[warp] = iy;
        sh.woff[warp] = iq;
    }
    if (tid == 0) {
        sh.token = -1;
        sh.cert = 0;
    }
    __syncthreads();
    unsigned long long wy = 0ull, wq = 0ull;  // totals of the warps before this one
    for (int w = 0; w < warp; ++w) {
        wy += sh.red_u[w];
        wq += sh.woff[w];
    }
    const unsigned long long sy0 = Y0 + wy + iy - my, sq0 = Q0 + wq + iq - mq;
    const bool past = ce > cb && fast_cval(sy0 + my, sq0 + mq, M) > (long long)tau;
    const unsigned bw = __ballot_sync(0xffffffffu, past);
    if (lane == 0) sh.red_f[warp] = bw ? (float)(__ffs(bw) - 1) : -1.0f;
    __syncthreads();
    int first = -1;  // the first thread (by index) whose range passes tau
    for (int w = 0; w < kWarps && first < 0; ++w)
        if (sh.red_f[w] >= 0.0f) first = w * 32 + (int)sh.red_f[w];
    if (tid == first) {
        unsigned long long ry = sy0, rq = sq0;
        int i = cb;
        for (; i < ce - 1; ++i) {
            const ulonglong2 v = load_block<GLOBAL>(d.bsum, i);
            if (fast_cval(ry + v.x, rq + v.y, M) > (long long)tau) break;
            ry += v.x;
            rq += v.y;
        }
        sh.blk = i;
        sh.f_bY = ry;
        sh.f_bQ = rq;
    }
    __syncthreads();
    if (first >= 0 && warp == 0) {  // (first < 0 is not reachable: the slice's end passes tau)
        // The chunk: lanes 0..7 take the block's chunks in the pass's
        // arithmetic (the same fixed-point values as the block sums); the
        // first lane whose end passes tau holds it.
        const int ci = sh.blk * kFastGroup + (lane & (kFastGroup - 1));
        float l[kChunk], q[kChunk] = {}, yp[kChunk] = {}, qp[kChunk] = {};
        unsigned long long cy = 0ull, cq = 0ull;
        const bool have = lane < kFastGroup && ci < d.mych;
        if (have) {
            RawL<DT> rl;
            raw_load_l(d, ci, rl);
            raw_unpack(rl, l);
            if (RES) {
                RawQ rq;
                raw_load_q(d, ci, rq);
                raw_unpack_q(rq, q);
            }
            float a1 = 0.0f, a2 = 0.0f;
            (void)fast_chunk<RES, EXACT>(l, q, f, cy, cq, a1, a2, yp, qp);
        }
        unsigned long long iy2 = cy, iq2 = cq;
#pragma unroll
        for (int off = 1; off < kFastGroup; off <<= 1) {
            const unsigned long long yo = __shfl_up_sync(0xffffffffu, iy2, off);
            const unsigned long long qo = __shfl_up_sync(0xffffffffu, iq2, off);
            if (lane >= off) {
                iy2 += yo;
                iq2 += qo;
            }
        }
        const unsigned long long ly = sh.f_bY + iy2 - cy, lq = sh.f_bQ + iq2 - cq;
        const bool lp = have && fast_cval(ly + cy, lq + cq, M) > (long long)tau;
        const unsigned bl = __ballot_sync(0xffffffffu, lp);
        const int oc = bl ? __ffs(bl) - 1 : 0;  // the chunk's lane
        // The element: lane e < 8 takes element e of that chunk (its y and q
        // and the chunk's start shuffled from the chunk's lane) and forms the
        // cumulative weight through e; the first positive e past tau is it.
        float ype[kChunk], qpe[kChunk];
#pragma unroll
        for (int e = 0; e < kChunk; ++e) {
            ype[e] = __shfl_sync(0xffffffffu, yp[e], oc);
            qpe[e] = __shfl_sync(0xffffffffu, qp[e], oc);
        }
        const unsigned long long cly = __shfl_sync(0xffffffffu, ly, oc);
        const unsigned long long clq = __shfl_sync(0xffffffffu, lq, oc);
        const int e = lane & (kChunk - 1);
        float mine = ype[0];  // ype[e] without indexing a register array at run time
#pragma unroll
        for (int j = 1; j < kChunk; ++j) mine = j == e ? ype[j] : mine;
        unsigned long long py, pq;
        fast_prefix<RES, EXACT>(ype, qpe, e, f, py, pq);
        const long long h = fast_cval(cly + py, clq + pq, M);
        const bool ep = bl && lane < kChunk && mine > 0.0f && h > (long long)tau;
        const unsigned be = __ballot_sync(0xffffffffu, ep);
        // lo: the cumulative weight before the element (the last positive
        // element before it, or the chunk's start)
        const bool before = lane < kChunk && mine > 0.0f && h <= (long long)tau;
        const unsigned bb = __ballot_sync(0xffffffffu, before) & (be ? ((1u << (__ffs(be) - 1)) - 1u) : 0u);
        const int te = be ? __ffs(be) - 1 : -1;
        const int tl = te >= 0 ? te : 0, bl0 = bb ? 31 - __clz(bb) : 0;
        const long long hi = __shfl_sync(0xffffffffu, h, tl);
        const long long hb = __shfl_sync(0xffffffffu, h, bl0);
        // the sums through each edge, and the edge chunk's sums
        const unsigned long long yhi = __shfl_sync(0xffffffffu, cly + py, tl);
        const unsigned long long qhi = __shfl_sync(0xffffffffu, clq + pq, tl);
        const unsigned long long ylb = __shfl_sync(0xffffffffu, cly + py, bl0);
        const unsigned long long qlb = __shfl_sync(0xffffffffu, clq + pq, bl0);
        const unsigned long long ccy = __shfl_sync(0xffffffffu, cy, oc);
        const unsigned long long ccq = __shfl_sync(0xffffffffu, cq, oc);
        if (lane == 0 && te >= 0) {
            const long long lo = bb ? hb : fast_cval(cly, clq, M);
            const float cm = EXACT ? 0.0f : (float)(fast_cval(ccy, 0ull, M) + (long long)ccq);
            const long long Dlo = fast_edge_bound(c, M, d.u, bb ? ylb : cly, bb ? qlb : clq,
                                                  hi - lo, cm);
            const long long Dhi = fast_edge_bound(c, M, d.u, yhi, qhi, hi - lo, cm);
            sh.cert = ((long long)tau - lo >= Dlo && hi - (long long)tau > Dhi) ? 1 : 0;
            sh.token = (int)((d.c0 + sh.blk * kFastGroup + oc) * kChunk + te);
        }
    }
    __syncthreads();
}

// The fast draw by the G CTAs of a cluster (RES: the residual max(0, p - q),
// else p).  Returns true (in every thread of every CTA) when the token is
// certified: u C lies far enough inside the chosen bin that the exact draw
// picks the same one (the bound of fast_bound).  The owner CTA then holds the
// token in sh.token.
template <typename DT, bool RES, bool EXACT>
__device__ bool draw_fast(cg::cluster_group& cluster, DrawShared& sh, const DrawCtx<DT>& d) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        sh.token = -1;
        sh.cert = 0;
    }
    const FastScale f = make_fast_scale(d.m, d.c2, d.s_row, RES);
    const FastTotals t = fast_pass<DT, RES, EXACT, true>(d, f);
    // The CTA's totals, pushed to slot [rank] of every CTA of the cluster.
    cta_fast_totals(sh, t, &sh.red_t[0]);
    if (warp == 0 && lane < d.G) *cluster.map_shared_rank(&sh.xT[d.rank], lane) = sh.red_t[0];
    xsync(cluster, d.G);

    // Every CTA, from the same slots in the same order: the totals, the bound,
    // the owning rank and this rank's starting point.  Float, float-float and
    // integer arithmetic only.
    if (warp == 0) {
        // Every lane adds the G slots in rank order (no shuffles: a lone warp's
        // shuffles right after the barrier measured several microseconds here).
        FastTotals tot = zero_totals();
        unsigned long long ybef = 0ull, qbef = 0ull, yend = 0ull, qend = 0ull;
        for (int r = 0; r < d.G; ++r) {
            const FastTotals x = sh.xT[r];
            if (r == d.rank) {
                ybef = tot.Y;
                qbef = tot.Q;
            }
            tot = add_fast_totals(tot, x);
            if (r == lane) {  // lane r: the sums up to and including rank r
                yend = tot.Y;
                qend = tot.Q;
            }
        }
        const FastBound fb =
            fast_bound<EXACT>(tot, d.s_row, d.u, f.ey, ((long long)d.V + kChunk - 1) / kChunk);
        const bool past = lane < d.G && fb.ok && fast_cval(yend, qend, fb.M) > (long long)fb.tau;
        const unsigned ballot = __ballot_sync(0xffffffffu, past);
        const int owner = ballot ? __ffs(ballot) - 1 : -1;
        if (lane == 0) {
            sh.f_ok = fb.ok && owner >= 0;
            sh.f_owner = owner;
            sh.f_M = fb.M;
            sh.f_tau = fb.tau;
            sh.f_Y = ybef;
            sh.f_Q = qbef;
            sh.f_c = fb.c;
        }
    }
    __syncthreads();
    if (!sh.f_ok) return false;  // uniform across the cluster

    int cert = 1;
    if (d.rank == sh.f_owner) {  // uniform across the CTA
        fast_search<DT, RES, EXACT, false>(sh, d, f, sh.f_M, sh.f_tau, sh.f_Y, sh.f_Q, sh.f_c);
        cert = sh.cert;
    }
    if (d.G > 1) {
        if (tid < d.G) *cluster.map_shared_rank(&sh.xC[d.rank], tid) = cert;
        xsync(cluster, d.G);
        if (warp == 0) {
            int ok = lane < d.G ? sh.xC[lane] : 1;
            ok = __all_sync(0xffffffffu, ok);
            if (lane == 0) sh.cert_all = ok;
        }
        __syncthreads();
        return sh.cert_all != 0;
    }
    return cert != 0;
}

// ---- precise pass: float-float exponentials, exact integer prefix sums

// Fixed-point value of chunk ci for the precise draw: the float-float sum of its
// eight weights, quantised.  Element-level cumulative values inside the chunk
// are quantisations of the partial sums in the same order, so the last one
// equals the chunk value.  With `token` set, the first element (0..7) whose
// cumulative value exceeds `want` is stored there.  The exponentials come from
// the cache (`e_cached`) or are recomputed from the logits l; with `wstore`
// the weights are stored there (over the cached exponentials they came from).
template <typename DT, bool RES, bool ECACHED, bool WSTORE>
__device__ __forceinline__ unsigned long long precise_chunk(const DrawCtx<DT>& d, int ci,
                                                            const float* l, const float* q,
                                                            ff inv, unsigned long long want,
                                                            int* token) {
    ff acc{0.0f, 0.0f};
    ff* wstore = WSTORE ? d.ecache + (size_t)ci * kChunk : nullptr;
#pragma unroll
    for (int e = 0; e < kChunk; ++e) {
        const ff ev = ECACHED ? d.ecache[(size_t)ci * kChunk + e]
                              : exp_rel(l[e], d.m, d.c2, d.thi, d.tlo);
        const ff w = draw_weight(ev, inv, RES ? q[e] : 0.0f, RES);
        if (WSTORE) wstore[e] = w;
        ff_accumulate(acc, w);
        if (token && *token < 0 && w.hi > 0.0f && to_fixed(ff_normalize(acc)) > want) *token = e;
    }
    return to_fixed(ff_normalize(acc));
}

// One round of the precise pass B over the CTA's slice: chunk values into the
// block totals; returns this thread's share of the CTA total.
template <typename DT, bool RES, bool ECACHED, bool WSTORE>
__device__ __forceinline__ unsigned long long precise_pass_b(const DrawCtx<DT>& d, ff inv) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long tacc = 0;
    float nq[kChunk] = {}, nl[kChunk] = {};
    int ci = warp * kBlockChunks + lane;
    if (ci < d.mych) {
        load_q(d, ci, RES, nq);
        if (!ECACHED) load_l(d, ci, nl);
    }
    for (int base = warp * kBlockChunks; base < d.mych; base += kThreads) {
        ci = base + lane;
        float q[kChunk], l[kChunk];
#pragma unroll
        for (int e = 0; e < kChunk; ++e) {
            q[e] = nq[e];
            l[e] = nl[e];
        }
        if (ci + kThreads < d.mych) {
            load_q(d, ci + kThreads, RES, nq);
            if (!ECACHED) load_l(d, ci + kThreads, nl);
        }
        const unsigned long long W =
            ci < d.mych ? precise_chunk<DT, RES, ECACHED, WSTORE>(d, ci, l, q, inv, 0ull, nullptr)
                        : 0ull;
        const unsigned long long bw = warp_sum(W);
        if (lane == 0) {
            d.bsum[base / kBlockChunks] = bw;
            tacc += bw;
        }
    }
    return tacc;
}

// The same value (and token search) from stored weights.
__device__ __forceinline__ unsigned long long stored_chunk(const ff* w, unsigned long long want,
                                                           int* token) {
    ff acc{0.0f, 0.0f};
#pragma unroll
    for (int e = 0; e < kChunk; ++e) {
        const ff we = w[e];
        ff_accumulate(acc, we);
        if (token && *token < 0 && we.hi > 0.0f && to_fixed(ff_normalize(acc)) > want) *token = e;
    }
    return to_fixed(ff_normalize(acc));
}

// Precise pass A over the CTA's slice: this thread's float-float share of
// S = sum_j exp((l_j - m)/T), the exponentials kept in the cache when ECACHE.
template <typename DT, bool ECACHE>
__device__ __forceinline__ ff precise_pass_a(const DrawCtx<DT>& d) {
    const int tid = threadIdx.x;
    ff acc{0.0f, 0.0f};
    float nf[kChunk] = {};
    if (tid < d.mych) load_l(d, tid, nf);
    for (int ci = tid; ci < d.mych; ci += kThreads) {
        float f[kChunk];
#pragma unroll
        for (int e = 0; e < kChunk; ++e) f[e] = nf[e];
        if (ci + kThreads < d.mych) load_l(d, ci + kThreads, nf);
#pragma unroll
        for (int e = 0; e < kChunk; ++e) {
            const ff ev = exp_rel(f[e], d.m, d.c2, d.thi, d.tlo);
            if (ECACHE) d.ecache[(size_t)ci * kChunk + e] = ev;
            ff_accumulate(acc, ev);
        }
    }
    return acc;
}

// The precise draw on one row by the G CTAs of a cluster.  The owner CTA holds
// the token in sh.token; `degenerate` is set in all threads.
template <typename DT>
__device__ void draw_precise(cg::cluster_group& cluster, DrawShared& sh, const DrawCtx<DT>& d,
                             bool& degenerate) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < kExpTable; i += kThreads) {
        d.thi[i] = g_exp2_table.hi[i];
        d.tlo[i] = g_exp2_table.lo[i];
    }
    __syncthreads();

    // Pass A: e_j = exp((l_j - m)/T) and the normaliser S = sum_j e_j.
    const ff acc = d.ecache ? precise_pass_a<DT, true>(d) : precise_pass_a<DT, false>(d);
    const ff inv = ff_recip(cluster_sum_ff(cluster, sh, sh.xS[1], acc, d.rank, d.G));

    // Pass B: chunk values, block totals, cluster prefix; a second round draws
    // from p when the residual has no mass.
    bool use_res = d.residual;
    degenerate = false;
    unsigned long long prefix = 0, total = 0, mytot = 0;
    for (int round = 0; round < 2; ++round) {
        // The first round reads the cached exponentials and leaves the weights
        // in their place; a second round recomputes the exponentials.
        unsigned long long tacc;
        if (round == 0 && d.ecache)
            tacc = use_res ? precise_pass_b<DT, true, true, true>(d, inv)
                           : precise_pass_b<DT, false, true, true>(d, inv);
        else if (d.ecache)
            tacc = precise_pass_b<DT, false, false, true>(d, inv);  // round 1: from p
        else
            tacc = use_res ? precise_pass_b<DT, true, false, false>(d, inv)
                           : precise_pass_b<DT, false, false, false>(d, inv);
        cluster_prefix(cluster, sh, sh.xW[1 + round], nullptr, tacc, 0.0f, d.rank, d.G);
        prefix = sh.prefix;
        total = sh.total;
        mytot = sh.mytot;
        if (total > 0 || !use_res) break;
        use_res = false;  // zero residual mass: draw from p (counted)
        degenerate = true;
    }

    const unsigned long long tau = scale_floor(d.u, total);
    const bool owner = mytot > 0 && prefix <= tau && tau - prefix < mytot;
    if (owner) {  // uniform across the CTA
        const unsigned long long want = tau - prefix;
        int blk;
        unsigned long long bbefore;
        find_block(sh, d.bsum, d.nblk, want, &blk, &bbefore);
        if (warp == 0) {
            const int ci = blk * kBlockChunks + lane;
            float l[kChunk] = {}, q[kChunk] = {};
            const ff* wc = d.ecache ? d.ecache + (size_t)ci * kChunk : nullptr;
            unsigned long long W = 0;
            if (ci < d.mych) {
                if (wc) {
                    W = stored_chunk(wc, 0ull, nullptr);
                } else {
                    load_l(d, ci, l);
                    load_q(d, ci, use_res, q);
                    W = use_res ? precise_chunk<DT, true, false, false>(d, ci, l, q, inv, 0ull, nullptr)
                                : precise_chunk<DT, false, false, false>(d, ci, l, q, inv, 0ull,
                                                                          nullptr);
                }
            }
            const unsigned long long wb = want - bbefore;
            unsigned long long cb;
            if (find_lane(W, wb, &cb)) {
                int tok = -1;
                if (wc)
                    stored_chunk(wc, wb - cb, &tok);
                else if (use_res)
                    precise_chunk<DT, true, false, false>(d, ci, l, q, inv, wb - cb, &tok);
                else
                    precise_chunk<DT, false, false, false>(d, ci, l, q, inv, wb - cb, &tok);
                if (tok >= 0) sh.token = (int)((d.c0 + ci) * kChunk + tok);
            }
        }
    }
}

// ---- precise pass in one read
//
// The weight of element j is p_j = e_j / S (bonus draw) or max(0, e_j / S - q_j)
// (residual), with e_j = exp((l_j - m)/T) in float-float.  Whether e_j / S
// exceeds q_j is settled for almost every element by the row stream's fp32
// normaliser: with it within 2^-12 of S (checked), e_j.hi / S_row above
// q_j (1 + 2^-10) means a positive weight and below q_j (1 - 2^-10) a zero one.
// A chunk whose elements are all settled has the weight Y_c / S - Q_c, with Y_c
// and Q_c the float-float sums of e_j and q_j over its positive elements, so a
// single pass over the logits and q forms S and every (Y_c, Q_c) at once; a
// chunk with an unsettled element is recomputed element by element once S is
// known.  Inside a chunk the cumulative weights are the same linear form of the
// partial sums, accumulated in the same order, so the last equals the chunk's.

constexpr float kP1Hi = 1.0f + 1.0f / 1024.0f, kP1Lo = 1.0f - 1.0f / 1024.0f;

// y * inv - q for float-float y, inv, q (the difference of two non-negative
// values), clamped at zero.
__device__ __forceinline__ ff p1_linear(ff y, ff inv, ff q) {
    const ff a = ff_mul(ff_normalize(y), inv);
    const ff qn = ff_normalize(q);
    const ff s = two_sum(a.hi, -qn.hi);
    const ff w = fast_two_sum(s.hi, __fadd_rn(s.lo, __fsub_rn(a.lo, qn.lo)));
    return w.hi > 0.0f ? w : ff{0.0f, 0.0f};
}

// One chunk's pass: the exponentials into S, and into (Y, Q) those of settled
// positive elements; `amb` when an element is not settled.  With `want` and
// `token` (the search inside a settled chunk), also the first element whose
// cumulative weight exceeds `want`.
template <typename DT, bool RES>
__device__ __forceinline__ void p1_chunk(const DrawCtx<DT>& d, const float* l, const float* q,
                                         float inv_row, ff& S, ff& Y, ff& Q, bool& amb,
                                         ff inv = ff{0.0f, 0.0f}, unsigned long long want = 0ull,
                                         int* token = nullptr) {
#pragma unroll
    for (int e = 0; e < kChunk; ++e) {
        const ff ev = exp_rel(l[e], d.m, d.c2, d.thi, d.tlo);
        ff_accumulate(S, ev);
        bool pos = true;
        if (RES) {
            const float ph = __fmul_rn(ev.hi, inv_row), qe = q[e];
            pos = qe >= 0.0f && ph > __fmul_rn(qe, kP1Hi);
            const bool zero = qe >= 0.0f && (ev.hi == 0.0f || ph < __fmul_rn(qe, kP1Lo));
            amb |= !pos && !zero;
            if (pos) ff_accumulate(Q, ff{qe, 0.0f});
        }
        if (pos) ff_accumulate(Y, ev);
        if (token && *token < 0 && pos && ev.hi > 0.0f &&
            to_fixed(ff_normalize(p1_linear(Y, inv, Q))) > want)
            *token = e;
    }
}

// Fixed-point weight of chunk ci from the table (or, for an unsettled chunk,
// recomputed element by element as the two-pass precise draw does).
template <typename DT, bool RES>
__device__ __forceinline__ unsigned long long p1_value(const DrawCtx<DT>& d, int ci, ff inv) {
    if (RES && d.pamb[ci]) {
        float l[kChunk], q[kChunk];
        load_l(d, ci, l);
        load_q(d, ci, true, q);
        return precise_chunk<DT, true, false, false>(d, ci, l, q, inv, 0ull, nullptr);
    }
    return to_fixed(ff_normalize(p1_linear(d.pY[ci], inv, d.pQ[ci])));
}

// The precise draw in one read of the slices (the chunk table must fit:
// d.pY).  Returns false, in every thread of every CTA, when it cannot decide:
// the row stream's normaliser is more than 2^-12 from S, or the residual has no
// mass; the caller then runs the two-pass draw.
template <typename DT, bool RES>
__device__ bool draw_precise_1p(cg::cluster_group& cluster, DrawShared& sh, const DrawCtx<DT>& d) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < kExpTable; i += kThreads) {
        d.thi[i] = g_exp2_table.hi[i];
        d.tlo[i] = g_exp2_table.lo[i];
    }
    __syncthreads();
    const float inv_row = RES ? __frcp_rn(d.s_row) : 0.0f;
    // The pass: S, and each chunk's (Y, Q) and flag into the table.
    ff accS{0.0f, 0.0f};
    float nl[kChunk] = {}, nq[kChunk] = {};
    if (tid < d.mych) {
        load_l(d, tid, nl);
        load_q(d, tid, RES, nq);
    }
    for (int ci = tid; ci < d.mych; ci += kThreads) {
        float l[kChunk], q[kChunk];
#pragma unroll
        for (int e = 0; e < kChunk; ++e) {
            l[e] = nl[e];
            q[e] = nq[e];
        }
        if (ci + kThreads < d.mych) {
            load_l(d, ci + kThreads, nl);
            load_q(d, ci + kThreads, RES, nq);
        }
        ff Y{0.0f, 0.0f}, Q{0.0f, 0.0f};
        bool amb = false;
        p1_chunk<DT, RES>(d, l, q, inv_row, accS, Y, Q, amb);
        d.pY[ci] = Y;
        d.pQ[ci] = Q;
        d.pamb[ci] = amb ? 1 : 0;
    }
    const ff S = cluster_sum_ff(cluster, sh, sh.xS[1], accS, d.rank, d.G);
    if (RES && !(fabsf(__fsub_rn(S.hi, d.s_row)) <= S.hi * (1.0f / 4096.0f))) return false;
    const ff inv = ff_recip(S);
    // Chunk values into block totals, then the cluster prefix.
    unsigned long long tacc = 0;
    for (int base = warp * kBlockChunks; base < d.mych; base += kThreads) {
        const int ci = base + lane;
        const unsigned long long W = ci < d.mych ? p1_value<DT, RES>(d, ci, inv) : 0ull;
        const unsigned long long bw = warp_sum(W);
        if (lane == 0) {
            d.bsum[base / kBlockChunks] = bw;
            tacc += bw;
        }
    }
    cluster_prefix(cluster, sh, sh.xW[1], nullptr, tacc, 0.0f, d.rank, d.G);
    const unsigned long long prefix = sh.prefix, total = sh.total, mytot = sh.mytot;
    if (total == 0) return false;  // zero residual mass: the two-pass draw handles it
    const unsigned long long tau = scale_floor(d.u, total);
    const bool owner = mytot > 0 && prefix <= tau && tau - prefix < mytot;
    if (owner) {  // uniform across the CTA
        const unsigned long long want = tau - prefix;
        int blk;
        unsigned long long bbefore;
        find_block(sh, d.bsum, d.nblk, want, &blk, &bbefore);
        if (warp == 0) {
            const int ci = blk * kBlockChunks + lane;
            const unsigned long long W = ci < d.mych ? p1_value<DT, RES>(d, ci, inv) : 0ull;
            const unsigned long long wb = want - bbefore;
            unsigned long long cb;
            if (find_lane(W, wb, &cb)) {
                int tok = -1;
                float l[kChunk], q[kChunk] = {};
                load_l(d, ci, l);
                load_q(d, ci, RES, q);
                if (RES && d.pamb[ci]) {
                    precise_chunk<DT, true, false, false>(d, ci, l, q, inv, wb - cb, &tok);
                } else {
                    ff S1{0.0f, 0.0f}, Y{0.0f, 0.0f}, Q{0.0f, 0.0f};
                    bool amb = false;
                    p1_chunk<DT, RES>(d, l, q, inv_row, S1, Y, Q, amb, inv, wb - cb, &tok);
                }
                if (tok >= 0) sh.token = (int)((d.c0 + ci) * kChunk + tok);
            }
        }
    }
    return true;
}

// The precise draw: in one read when the chunk table fits and the row's
// normaliser settles the residual's signs, else in two passes.
template <typename DT>
__device__ void draw_precise_any(cg::cluster_group& cluster, DrawShared& sh,
                                 const DrawCtx<DT>& d, bool& degenerate) {
    degenerate = false;
    if (d.pY) {
        const bool done = d.residual ? draw_precise_1p<DT, true>(cluster, sh, d)
                                     : draw_precise_1p<DT, false>(cluster, sh, d);
        if (done) return;
        if (threadIdx.x == 0) sh.token = -1;
        xsync(cluster, d.G);  // the table's place is the two-pass draw's cache
    }
    draw_precise<DT>(cluster, sh, d, degenerate);
}

// Dynamic shared memory of a draw: block sums, the 2^(i/1024) table, and room
// for the precise pass: its one-read chunk table, or (level 2) a cache of the
// slice's float-float exponentials.
// log2 of a cluster size (a power of two, at most 16): slices are cut with
// shifts, not 64-bit divisions.
__host__ __device__ inline int log2_pow2(int G) {
    int lg = 0;
    while ((1 << lg) < G && lg < 4) ++lg;
    return lg;
}
__host__ __device__ inline long long draw_slice_chunks(int V, int G) {
    const long long nch = ((long long)V + kChunk - 1) / kChunk;
    return (nch + G - 1) >> log2_pow2(G);
}
// Block sums: two 64-bit sums per 64-element block of the fast pass (the
// precise pass's one per 256 elements fits in the same room).
__host__ __device__ inline size_t draw_bsum_bytes(int V, int G) {
    const long long nblk = (draw_slice_chunks(V, G) + 7) / 8;
    return (size_t)nblk * 16;
}
// Dynamic shared memory a draw may use: two 512-thread CTAs of the drawing
// kernels still fit on one SM.
constexpr size_t kDrawSmemBudget = 96 * 1024;
// The one-read precise pass's chunk table: two float-float sums and a flag
// per chunk of the slice.
__host__ __device__ inline size_t precise_table_bytes(int V, int G) {
    const size_t nch = (size_t)draw_slice_chunks(V, G);
    return nch * 2 * sizeof(ff) + ((nch + 15) & ~(size_t)15);
}
__host__ __device__ inline size_t draw_smem_bytes(int V, int G, int level) {
    const size_t slice = (size_t)draw_slice_chunks(V, G) * kChunk;
    const size_t base = draw_bsum_bytes(V, G) + 2 * kExpTable * sizeof(float);
    const size_t cache = level >= 2 ? slice * sizeof(ff) : 0;
    const size_t tab = precise_table_bytes(V, G);
    return base + (tab > cache && base + tab <= kDrawSmemBudget ? tab : cache);
}

template <typename DT>
__device__ __forceinline__ DrawCtx<DT> make_draw_ctx(unsigned char* dyn, int level,
                                                    const DT* rowp, const float* qrow,
                                                    bool residual, int V, float m, float c,
                                                    ff c2, float u, int rank, int G,
                                                    float s_row) {
    DrawCtx<DT> d;
    d.rowp = rowp;
    d.qrow = qrow;
    d.V = V;
    d.residual = residual;
    d.m = m;
    d.c = c2.hi;
    d.clo = c2.lo;
    (void)c;
    d.c2 = c2;
    d.u = u;
    const long long nch = ((long long)V + kChunk - 1) / kChunk;
    const int lg = log2_pow2(G);
    d.c0 = (nch * rank) >> lg;
    d.mych = (int)(((nch * (rank + 1)) >> lg) - d.c0);
    d.nblk = (d.mych + kBlockChunks - 1) / kBlockChunks;
    d.al_l = (reinterpret_cast<uintptr_t>(rowp) & 15) == 0;
    d.al_q = residual && (reinterpret_cast<uintptr_t>(qrow) & 15) == 0;
    d.rank = rank;
    d.G = G;
    const size_t bb = draw_bsum_bytes(V, G);
    d.bsum = reinterpret_cast<unsigned long long*>(dyn);
    d.thi = reinterpret_cast<float*>(dyn + bb);
    d.tlo = d.thi + kExpTable;
    unsigned char* cache = dyn + bb + 2 * kExpTable * sizeof(float);
    d.ecache = level >= 2 ? reinterpret_cast<ff*>(cache) : nullptr;
    // The chunk table of the one-read precise pass shares the cache's place
    // (the fast pass is over when it is written).
    d.s_row = s_row;
    const bool tab = bb + 2 * kExpTable * sizeof(float) + precise_table_bytes(V, G) <=
                     kDrawSmemBudget;
    d.pY = tab ? reinterpret_cast<ff*>(cache) : nullptr;
    d.pQ = tab ? d.pY + d.mych : nullptr;
    d.pamb = tab ? reinterpret_cast<unsigned char*>(d.pQ + d.mych) : nullptr;
    return d;
}

// The draw: the certified fast pass, and the precise pass when the fast one
// cannot certify its bin (or when `force_precise`).  Every CTA calls it; the
// owner CTA's thread 0 writes the token to *token_out.  Sets `degenerate` and
// `fallback` in all threads.  The CTA's slices of the decision row and of the
// q row are read with loads that do not allocate in L1.  With `defer_precise` a draw that
// needs the precise pass returns true at once (in every thread) and writes no
// token: the caller hands it to the precise kernel.
template <typename DT, bool EXACT>
__device__ bool draw(cg::cluster_group& cluster, DrawShared& sh, const DrawCtx<DT>& d,
                     bool force_precise, bool defer_precise, int32_t* token_out,
                     bool& degenerate, bool& fallback) {
    degenerate = false;
    fallback = true;
    const bool certified =
        !force_precise && (d.residual ? draw_fast<DT, true, EXACT>(cluster, sh, d)
                                      : draw_fast<DT, false, EXACT>(cluster, sh, d));
    if (certified) {
        fallback = false;
        if (threadIdx.x == 0 && sh.token >= 0) *token_out = sh.token;
        return false;
    }
    if (defer_precise) return true;
    if (threadIdx.x == 0) sh.token = -1;
    __syncthreads();
    draw_precise_any<DT>(cluster, sh, d, degenerate);
    __syncthreads();
    if (threadIdx.x == 0 && sh.token >= 0) *token_out = sh.token;
    return false;
}

// ------------------------------------------------------------------ the fused kernel

// Optional epilogue of a verify, done by the thread that writes num_accepted[b]:
// kv_len[b] += n + 1 for a valid sequence (the round's committed tokens: the n
// accepted drafts and the drawn one; entries past the first rejection are
// dropped, "Decodificação especulativa explicada", §"O ciclo de rascunho e
// verificação", bookkeeping paragraph), and the counters of sv_spec_stats.
struct Epilogue {
    int32_t* kv_len;               // [B] or null
    unsigned long long* stats;     // sv_spec_stats as 5 counters, or null
};
__device__ __forceinline__ void commit_sequence(const Epilogue& ep, int b, int n, int k) {
    if (n >= 0) {
        if (ep.kv_len) ep.kv_len[b] += n + 1;
        if (ep.stats) {
            atomicAdd(ep.stats + 0, 1ull);
            atomicAdd(ep.stats + 1, (unsigned long long)k);
            atomicAdd(ep.stats + 2, (unsigned long long)n);
            atomicAdd(ep.stats + 3, (unsigned long long)(n + 1));
        }
    } else if (ep.stats) {
        atomicAdd(ep.stats + 4, 1ull);
    }
}

struct VerifyArgs {
    const void* logits;
    const float* q;
    const int32_t* x;
    const float* ua;
    const float* ur;
    Header* hdr;
    RowRec* rows;
    uint32_t* seqstat;
    int32_t* out;
    int32_t* nacc;
    uint32_t* plist_count;  // with plist: draws needing the precise pass are
    uint32_t* plist;        // appended here for sv_precise_kernel (else run here)
    Epilogue ep;
    int B, k, V, G, W;
    int draw_level;     // shared-memory cache level of the draw
    int force_precise;  // test hook: skip the fast draw
    float c;     // log2(e)/T (float, for the row statistics and the fast draw)
    ff c2;       // log2(e)/T in float-float (p(x) and the precise draw)
};

// Outcome of one row's test: accept, reject, the bonus row, or an error bit.
constexpr uint32_t kCodeAccept = 0u, kCodeReject = 1u, kCodeBonus = 2u, kCodeError = 0x100u;

struct FusedShared {
    Partial wpart[kWarps];
    Partial part[2][kWarps];   // this CTA's per-row partials of a wave (read through DSMEM)
    Partial rowstat[kWarps];   // merged statistics of the wave's rows
    float lx[kMaxK], qx[kMaxK], ua[kMaxK];
    int xs[kMaxK];
    uint32_t gfl[kMaxK];
    float px[kWarps];
    uint32_t code[kWarps];
    float ur;
    int n, bits;
};

template <typename DT, bool SAMPLED>
__global__ void __launch_bounds__(kThreads, 2) sv_verify_kernel(VerifyArgs a) {
    using E = Elt<DT>;
    extern __shared__ __align__(16) unsigned char dyn[];
    __shared__ FusedShared fs;
    __shared__ DrawShared ds;

    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.G;
    const int b = blockIdx.x / G;
    const int rank = blockIdx.x % G;  // == cluster rank: clusters are (G,1,1) along x
    const int k = a.k, V = a.V;
    const DT* seq_logits = static_cast<const DT*>(a.logits) + (long long)b * (k + 1) * V;

    if (blockIdx.x == 0 && tid == 0) {
        a.hdr->magic = kMagic;
        a.hdr->B = a.B;
        a.hdr->k = k;
        a.hdr->V = V;
        a.hdr->mode = SAMPLED ? SV_MODE_SAMPLE : SV_MODE_GREEDY;
        a.hdr->flat_ctas = 0;  // one record per row
    }
    // Draft tokens, their logits and q values, and the uniforms of this sequence.
    for (int i = tid; i < k; i += kThreads) {
        const int xi = a.x[(long long)b * k + i];
        fs.xs[i] = xi;
        uint32_t fl = 0;
        float lx = NAN, qx = NAN;
        if (xi < 0 || xi >= V) {
            fl = kRowTokenBad;
        } else {
            lx = E::load1(seq_logits + (long long)i * V + xi);
            if (SAMPLED) {
                qx = a.q[((long long)b * k + i) * V + xi];
                if (!(qx >= 0.0f)) fl = kRowQBad;
            }
        }
        fs.lx[i] = lx;
        fs.qx[i] = qx;
        fs.gfl[i] = fl;
        fs.ua[i] = SAMPLED ? a.ua[(long long)b * k + i] : 0.0f;
    }
    if (tid == 0) {
        fs.n = -1;
        fs.bits = 0;
        if (SAMPLED) fs.ur = a.ur[b];
    }
    __syncthreads();

    // ---- row statistics and the accept scan, wave by wave
    const float c = a.c;
    int buf = 0;
    int last_wave_end = 0, wave_row0 = 0;
    for (int i0 = 0; i0 <= k; i0 += a.W) {
        const int Wc = min(a.W, k + 1 - i0);
        // warps [g0, g1) stream row i0 + w, w = warp * Wc / kWarps
        const int w = warp * Wc / kWarps;
        const int g0 = (w * kWarps + Wc - 1) / Wc, g1 = ((w + 1) * kWarps + Wc - 1) / Wc;
        const int tg = tid - g0 * 32, ng = (g1 - g0) * 32;
        const DT* rowp = seq_logits + (long long)(i0 + w) * V;
        int head;
        long long nvec, tail0;
        row_layout<DT>(rowp, V, head, nvec, tail0);
        const int lgG = log2_pow2(G);
    const long long vb = (nvec * rank) >> lgG, ve = (nvec * (rank + 1)) >> lgG;
        Partial p = stream_slice<DT, SAMPLED, 4>(rowp, V, vb, ve, head, tail0, rank == 0,
                                                 rank == G - 1, tg, ng, c);
        p = warp_merge<SAMPLED>(p, c);
        if (lane == 0) fs.wpart[warp] = p;
        __syncthreads();
        if (tid < Wc) {  // CTA partial of row i0 + tid from its warp group
            const int h0 = (tid * kWarps + Wc - 1) / Wc, h1 = ((tid + 1) * kWarps + Wc - 1) / Wc;
            Partial r = fs.wpart[h0];
            for (int h = h0 + 1; h < h1; ++h) merge<SAMPLED>(r, fs.wpart[h], c);
            fs.part[buf][tid] = r;
        }
        if (G > 1) {
            cluster.sync();
            if (warp < Wc) {  // merge over ranks: lane r holds rank r's partial
                Partial r = lane < G ? *cluster.map_shared_rank(&fs.part[buf][warp], lane)
                                     : empty_partial();
                r = warp_merge<SAMPLED>(r, c);
                if (lane == 0) fs.rowstat[warp] = r;
            }
        } else {
            if (tid < Wc) fs.rowstat[tid] = fs.part[buf][tid];
        }
        __syncthreads();
        if (tid < Wc) {  // each row's test, in parallel (kCode* values)
            const int i = i0 + tid;
            const Partial& r = fs.rowstat[tid];
            uint32_t c;
            if (row_flags<SAMPLED>(r) & kRowBad) {
                c = kCodeError | SV_DEV_BAD_ROW;
            } else if (i == k) {
                c = kCodeBonus;
            } else if (fs.gfl[i] & kRowTokenBad) {
                c = kCodeError | SV_DEV_BAD_TOKEN;
            } else if (SAMPLED) {
                const float u = fs.ua[i];
                if (!(u >= 0.0f && u < 1.0f)) {
                    c = kCodeError | SV_DEV_BAD_UNIFORM;
                } else if (fs.gfl[i] & kRowQBad) {
                    c = kCodeError | SV_DEV_BAD_Q;
                } else {
                    ff ex = exp_rel(fs.lx[i], r.m, a.c2, g_exp2_table.hi, g_exp2_table.lo);
                    const float P = __fdiv_rn(ex.hi, r.s);
                    const float Q = fs.qx[i];
                    fs.px[tid] = P;
                    c = ((P >= Q) || (u < __fdiv_rn(P, Q))) ? kCodeAccept : kCodeReject;
                }
            } else {
                c = fs.xs[i] == r.idx ? kCodeAccept : kCodeReject;
            }
            fs.code[tid] = c;
        }
        __syncthreads();
        if (tid == 0) {  // the scan over this wave's rows: the first row that stops it
            int n = -1, bits = 0;
            for (int ww = 0; ww < Wc; ++ww) {
                const uint32_t c = fs.code[ww];
                if (c == kCodeAccept) continue;
                if (c & kCodeError) bits = (int)(c & ~kCodeError);
                else n = c == kCodeBonus ? k : i0 + ww;
                break;
            }
            fs.n = n;
            fs.bits = bits;
        }
        __syncthreads();
        if (rank == 0 && tid < Wc) {  // row records for the statistics read-back
            const int i = i0 + tid;
            const Partial& r = fs.rowstat[tid];
            RowRec rec;
            rec.mraw = r.m;
            rec.S = SAMPLED ? r.s : 0.0f;
            rec.argmax = r.idx < 0 ? 0 : r.idx;
            uint32_t fl = row_flags<SAMPLED>(r);
            if (i < k) {
                fl |= fs.gfl[i];
                rec.lx = fs.lx[i];
                rec.qx = fs.qx[i];
                // p(x) was formed by the scan only up to the decision row
                rec.px = (SAMPLED && (fs.n < 0 || i <= fs.n)) ? (double)fs.px[tid] : 0.0;
            } else {
                rec.lx = NAN;
                rec.qx = NAN;
                rec.px = NAN;
            }
            rec.flags = fl;
            a.rows[(long long)b * (k + 1) + i] = rec;
        }
        wave_row0 = i0;
        last_wave_end = i0 + Wc;
        buf ^= 1;
        if (fs.n >= 0 || fs.bits) break;
    }
    // Rows past the last wave were never read.
    if (rank == 0)
        for (int i = last_wave_end + tid; i <= k; i += kThreads)
            a.rows[(long long)b * (k + 1) + i] = skipped_record();

    const int n = fs.n;
    const int bits = fs.bits;
    int32_t* o = a.out + (long long)b * (k + 1);
    if (bits || !SAMPLED) {
        if (rank == 0) {
            for (int i = tid; i <= k; i += kThreads)
                o[i] = bits ? -1 : (i < n ? fs.xs[i] : (i == n ? fs.rowstat[n - wave_row0].idx : -1));
            if (tid == 0) {
                a.nacc[b] = bits ? -1 : n;
                a.seqstat[b] = (uint32_t)bits;
                commit_sequence(a.ep, b, bits ? -1 : n, k);
            }
        }
        if (G > 1) cluster.sync();  // partial slots may still be read by other ranks
        return;
    }

    // ---- the draw on row n, then the outputs
    const float u = fs.ur;
    if (!(u >= 0.0f && u < 1.0f)) {  // every CTA sees the same uniform
        if (rank == 0) {
            for (int i = tid; i <= k; i += kThreads) o[i] = -1;
            if (tid == 0) {
                a.nacc[b] = -1;
                a.seqstat[b] = SV_DEV_BAD_UNIFORM;
                commit_sequence(a.ep, b, -1, k);
            }
        }
        if (G > 1) cluster.sync();
        return;
    }
    const DT* drow = seq_logits + (long long)n * V;
    const float* qrow = n < k ? a.q + ((long long)b * k + n) * V : nullptr;
    const float m = fs.rowstat[n - wave_row0].m;
    bool degenerate = false, fallback = false;
    const DrawCtx<DT> dc =
        make_draw_ctx<DT>(dyn, a.draw_level, drow, qrow, n < k, V, m, a.c, a.c2,
                          u, rank, G, fs.rowstat[n - wave_row0].s);
    const bool deferred = draw<DT, true>(cluster, ds, dc, a.force_precise != 0,
                                         a.plist != nullptr, o + n, degenerate, fallback);
    if (rank == 0) {
        for (int i = tid; i <= k; i += kThreads)
            if (i != n) o[i] = i < n ? fs.xs[i] : -1;
        if (tid == 0) {
            a.nacc[b] = n;
            a.seqstat[b] = (degenerate ? SV_DEV_DEGENERATE : 0u) | (fallback ? SV_DEV_PRECISE : 0u);
            commit_sequence(a.ep, b, n, k);
            if (deferred) {
                const uint32_t j = atomicAdd(a.plist_count, 1u);
                if (j < (uint32_t)a.B) a.plist[j] = (uint32_t)b;  // at most B entries
            }
        }
    }
    // No final cluster barrier: the draw's exchanges are pushed before its last
    // barrier, and the row partials were read before its first.
}

// ------------------------------------------------------------------ two-stage kernels

struct RowsArgs {
    const void* logits;
    const float* q;
    const int32_t* x;
    const float* ua;   // u_accept (sampled, with `skip`)
    Header* hdr;
    RowRec* rows;
    uint32_t* stop;    // [B] lowest row known to end its sequence's scan (with `skip`)
    uint32_t* zero;    // nzero words CTA 0 clears (the split draw's counters), or null
    int nzero;
    int B, k, V, G, mode;
    int skip;          // rows in position-major order; rows past a known stop are skipped
    float c;        // log2(e) / T
    ff c2;          // log2(e) / T in float-float (p(x))
};

// One CTA (or a cluster of G CTAs splitting the vocabulary) per row.
//
// With `skip` (only for G == 1) the grid enumerates rows position-major (row 0
// of every sequence, then row 1, ...), each CTA decides its own row's test
// (every test depends on its row alone) and lowers stop[b] to its row index
// when the scan would end there; a CTA whose row lies past stop[b] when it
// starts reads nothing and marks the row skipped.  The scan ends at its first
// stopping row n, and no row at or before n can be skipped (that would need a
// stopping row below n), so the finish kernel reads only rows this kernel
// computed.  stop[] must hold 0xFFFFFFFF when the grid starts.
// At most 64 registers per thread: 2048 threads' worth of CTAs per SM stay
// resident (2 CTAs of 512 threads; 1 of 1024 threads).
// The record of row `row` (sequence b, position i) from its merged statistics
// p and its gathers (token xi, l(x), q(x), u_accept); on the row-skipping
// stream also the row's test, and the sequence's stop row lowered when the
// scan would end here.
template <bool SAMPLED>
__device__ __forceinline__ void write_row_record(const RowsArgs& a, const Partial& p, int b, int i,
                                                 long long row, int xi, float lx, float qx,
                                                 float ua) {
    const int k = a.k, V = a.V;
    RowRec rec;
    rec.mraw = p.m;
    rec.S = SAMPLED ? p.s : 0.0f;
    rec.argmax = p.idx < 0 ? 0 : p.idx;
    rec.px = 0.0;
    rec.lx = NAN;
    rec.qx = NAN;
    uint32_t fl = row_flags<SAMPLED>(p);
    bool ends = false;  // the scan stops at this row (sequences with `skip`)
    if (i < k && a.x) {
        if (xi < 0 || xi >= V) {
            fl |= kRowTokenBad;
        } else {
            rec.lx = lx;
            if (SAMPLED) {
                rec.qx = qx;
                if (!(qx >= 0.0f)) fl |= kRowQBad;
                if (!(fl & kRowBad)) {
                    ff ex = exp_rel(lx, p.m, a.c2, g_exp2_table.hi, g_exp2_table.lo);
                    rec.px = (double)__fdiv_rn(ex.hi, p.s);
                }
            }
        }
        if (a.skip) {
            // The same tests, in the same arithmetic, as the finish kernels' scans.
            if (fl & (kRowBad | kRowTokenBad | kRowQBad)) {
                ends = true;
            } else if (SAMPLED) {
                const float P = (float)rec.px, Q = rec.qx;
                ends = !(ua >= 0.0f && ua < 1.0f) || !((P >= Q) || (ua < __fdiv_rn(P, Q)));
            } else {
                ends = xi != rec.argmax;
            }
        }
    } else {
        rec.px = NAN;
    }
    rec.flags = fl;
    a.rows[row] = rec;
    if (ends) atomicMin(a.stop + b, (uint32_t)i);
}

template <typename DT, bool SAMPLED, int NT>
__global__ void __launch_bounds__(NT, 1024 / NT) sv_rows_kernel(RowsArgs a) {
    using E = Elt<DT>;
    constexpr int NW = NT / 32;
    __shared__ Partial wpart[NW];
    __shared__ Partial cta_part;  // read by cluster rank 0 through DSMEM
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.G;
    const long long r0 = blockIdx.x / G;
    const int rank = blockIdx.x % G;
    const int V = a.V, k = a.k;
    const int b = a.skip ? (int)(r0 % a.B) : (int)(r0 / (k + 1));
    const int i = a.skip ? (int)(r0 / a.B) : (int)(r0 % (k + 1));
    const long long row = (long long)b * (k + 1) + i;
    const DT* rowp = static_cast<const DT*>(a.logits) + row * (long long)V;
    // The finish kernel is launched as a programmatic dependent: let it start
    // its launch now; it waits (griddepcontrol.wait) for this grid's results.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (blockIdx.x == 0 && tid == 0) {
        a.hdr->magic = kMagic;
        a.hdr->B = a.B;
        a.hdr->k = k;
        a.hdr->V = V;
        a.hdr->mode = a.mode;
        a.hdr->flat_ctas = 0;
    }
    if (blockIdx.x == 0 && a.zero)  // read by the next launch only (after this grid)
        for (int i0 = tid; i0 < a.nzero; i0 += NT) a.zero[i0] = 0u;
    // Set when the row turns out to lie past the stop row while it is read.
    __shared__ int s_abort;
    __shared__ unsigned long long s_tpub[NT];  // early rejection: threads' statistics
    __shared__ int s_fired;
    if (a.skip) {
        s_tpub[tid] = kEmptyPub;
        if (tid == 0) {
            s_fired = 0;
            s_abort = 0;
        }
    }
    if (a.skip && i > 0) {
        // One thread reads the stop row and the CTA follows its decision (the
        // value may change under concurrent CTAs, so each thread reading it
        // could decide differently).  G == 1: no other CTA shares the row.
        __shared__ int s_skip;
        if (tid == 0) {
            s_skip = *reinterpret_cast<volatile const uint32_t*>(a.stop + b) < (uint32_t)i;
            s_abort = 0;
        }
        __syncthreads();
        if (s_skip) {
            if (tid == 0) a.rows[row] = skipped_record();
            return;
        }
    }
    // The gathers of this row, issued now and used after the stream.
    int xi = -1;
    float lx = NAN, qx = NAN, ua = 0.0f;
    // (no drafted tokens, a.x null: the tree verify's rows, statistics only)
    if (rank == 0 && tid == 0 && i < k && a.x) {
        xi = a.x[(long long)b * k + i];
        if (xi >= 0 && xi < V) {
            lx = E::load1(rowp + xi);
            if (SAMPLED) qx = a.q[((long long)b * k + i) * V + xi];
        }
        if (SAMPLED && a.skip) ua = a.ua[(long long)b * k + i];
    }
    int head;
    long long nvec, tail0;
    row_layout<DT>(rowp, V, head, nvec, tail0);
    const int lgG = log2_pow2(G);
    const long long vb = (nvec * rank) >> lgG, ve = (nvec * (rank + 1)) >> lgG;
    // Eight 16-byte loads in flight per thread: a row slice of up to 8 vectors
    // per thread costs one round trip.  On the row-skipping stream every batch
    // also re-reads stop[b]: a row that falls past the stop row while it is read
    // is abandoned (stop[b] only decreases, so one observation suffices for
    // the whole CTA, whatever the other threads saw).
    const bool poll = a.skip;
    Partial p;
    if (poll) {
        __syncthreads();  // the early rejection's shared words are set
        bool aborted = false;
        EarlyRej er;
        er.tpub = s_tpub;
        er.nt = NT;
        er.lx = lx;
        er.uq = __fmul_rn(ua, qx);
        er.stop = a.stop + b;
        er.row = (uint32_t)i;
        er.fired = &s_fired;
        const bool early = i < k && a.x;  // the bonus row has no test
        p = stream_slice<DT, SAMPLED, 8, true>(rowp, V, vb, ve, head, tail0, true, true, tid, NT,
                                               a.c, a.stop + b, (uint32_t)i, &aborted,
                                               early ? &er : nullptr);
        if (aborted) s_abort = 1;
    } else {
        p = stream_slice<DT, SAMPLED, 8>(rowp, V, vb, ve, head, tail0, rank == 0, rank == G - 1,
                                         tid, NT, a.c);
    }
    p = warp_merge<SAMPLED>(p, a.c);
    if (lane == 0) wpart[warp] = p;
    __syncthreads();
    if (poll && s_abort) {
        if (tid == 0) a.rows[row] = skipped_record();
        return;
    }
    if (warp == 0) {
        Partial w = lane < NW ? wpart[lane] : empty_partial();
        w = warp_merge<SAMPLED>(w, a.c);
        p = w;
        if (lane == 0) cta_part = w;
    }
    if (G > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        if (rank == 0 && warp == 0) {
            Partial w = lane < G ? *cluster.map_shared_rank(&cta_part, lane) : empty_partial();
            p = warp_merge<SAMPLED>(w, a.c);
        }
        cluster.sync();
    }
    if (rank != 0 || tid != 0) return;
    write_row_record<SAMPLED>(a, p, b, i, row, xi, lx, qx, ua);
}

// The row-skipping stream with each row cut into G parts, one CTA each and no
// cluster, so that a row's statistics (and its test) are ready G times sooner
// and fewer rows are read before an earlier row of their sequence has stopped
// the scan.  Each CTA streams its part unless the row lies past its sequence's
// known stop row (checked at the start and with every batch of loads, as the
// one-CTA stream does), leaves its partial statistics in the workspace, and the
// last CTA of the row (an arrival counter, zeroed before the launch) merges the
// G partials in rank order and writes the record and the test.  A row any part
// of which was skipped or abandoned is marked skipped: it lies past the stop.
struct RowPart {
    float m, s;
    int idx;
    uint32_t flags;  // 1: NaN seen; 2: skipped or abandoned
};
struct RowGather {
    int xi;
    float lx, qx, ua;
};
static_assert(sizeof(RowPart) == 16 && sizeof(RowGather) == 16, "row parts");
constexpr int kRowSplitMax = 8;
struct RowSplitArgs {
    RowPart* parts;       // [R * G]
    RowGather* gath;      // [R] written by rank 0
    uint32_t* rowcnt;     // [R] CTAs done per row
};

template <typename DT, bool SAMPLED>
__global__ void __launch_bounds__(512, 2) sv_rows_skip_kernel(RowsArgs a, RowSplitArgs rs) {
    using E = Elt<DT>;
    constexpr int NT = 512, NW = NT / 32;
    __shared__ Partial wpart[NW];
    __shared__ int s_skip, s_abort, s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.G;
    const long long r0 = blockIdx.x / G;
    const int rank = blockIdx.x % G;
    const int V = a.V, k = a.k;
    const int b = (int)(r0 % a.B), i = (int)(r0 / a.B);
    const long long row = (long long)b * (k + 1) + i;
    const DT* rowp = static_cast<const DT*>(a.logits) + row * (long long)V;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (blockIdx.x == 0 && tid == 0) {
        a.hdr->magic = kMagic;
        a.hdr->B = a.B;
        a.hdr->k = k;
        a.hdr->V = V;
        a.hdr->mode = a.mode;
        a.hdr->flat_ctas = 0;
    }
    if (blockIdx.x == 0 && a.zero)  // read by the next launch only (after this grid)
        for (int i0 = tid; i0 < a.nzero; i0 += NT) a.zero[i0] = 0u;
    if (tid == 0) {
        s_skip = i > 0 && *reinterpret_cast<volatile const uint32_t*>(a.stop + b) < (uint32_t)i;
        s_abort = 0;
    }
    __syncthreads();
    Partial p = empty_partial();
    if (!s_skip) {
        int xi = -1;
        float lx = NAN, qx = NAN, ua = 0.0f;
        if (rank == 0 && tid == 0 && i < k && a.x) {
            xi = a.x[(long long)b * k + i];
            if (xi >= 0 && xi < V) {
                lx = E::load1(rowp + xi);
                if (SAMPLED) qx = a.q[((long long)b * k + i) * V + xi];
            }
            if (SAMPLED) ua = a.ua[(long long)b * k + i];
        }
        int head;
        long long nvec, tail0;
        row_layout<DT>(rowp, V, head, nvec, tail0);
        const long long vb = nvec * rank / G, ve = nvec * (rank + 1) / G;
        bool aborted = false;
        if (i > 0)
            p = stream_slice<DT, SAMPLED, 8, true>(rowp, V, vb, ve, head, tail0, rank == 0,
                                                   rank == G - 1, tid, NT, a.c, a.stop + b,
                                                   (uint32_t)i, &aborted);
        else
            p = stream_slice<DT, SAMPLED, 8>(rowp, V, vb, ve, head, tail0, rank == 0,
                                             rank == G - 1, tid, NT, a.c);
        if (aborted) s_abort = 1;
        p = warp_merge<SAMPLED>(p, a.c);
        if (lane == 0) wpart[warp] = p;
        if (rank == 0 && tid == 0 && i < k && a.x) rs.gath[r0] = RowGather{xi, lx, qx, ua};
        __syncthreads();
        if (warp == 0) {
            Partial w = lane < NW ? wpart[lane] : empty_partial();
            p = warp_merge<SAMPLED>(w, a.c);
        }
    }
    if (tid == 0) {
        RowPart part;
        part.m = p.m;
        part.s = p.s;
        part.idx = p.idx;
        part.flags = (p.nan ? 1u : 0u) | ((s_skip || s_abort) ? 2u : 0u);
        rs.parts[r0 * G + rank] = part;
        __threadfence();
        s_last = atomicAdd(rs.rowcnt + r0, 1u) == (uint32_t)(G - 1);
    }
    __syncthreads();
    if (!s_last || tid != 0) return;
    __threadfence();
    // the last part of the row: merge in rank order, then the record and the test
    Partial mp = empty_partial();
    bool skipped = false;
    for (int r = 0; r < G; ++r) {
        const uint4 v = __ldcg(reinterpret_cast<const uint4*>(rs.parts + r0 * G + r));
        Partial q;
        q.m = __uint_as_float(v.x);
        q.s = __uint_as_float(v.y);
        q.idx = (int)v.z;
        q.nan = (v.w & 1u) ? 1 : 0;
        skipped |= (v.w & 2u) != 0;
        merge<SAMPLED>(mp, q, a.c);
    }
    if (skipped) {
        a.rows[row] = skipped_record();
        return;
    }
    int xi = -1;
    float lx = NAN, qx = NAN, ua = 0.0f;
    if (i < k && a.x) {
        const uint4 g = __ldcg(reinterpret_cast<const uint4*>(rs.gath + r0));
        xi = (int)g.x;
        lx = __uint_as_float(g.y);
        qx = __uint_as_float(g.z);
        ua = __uint_as_float(g.w);
    }
    write_row_record<SAMPLED>(a, mp, b, i, row, xi, lx, qx, ua);
}

// ------------------------------------------------------------------ flat greedy stream
//
// Greedy only needs each row's argmax.  When the batch has about as many rows as
// the GPU has resident CTAs, one CTA per row (or a fixed split of each row)
// leaves a partial last wave; the flat stream instead cuts the whole logits
// tensor, seen as one run of 16-byte vectors (rows are whole vectors), into P
// equal ranges, one per resident CTA.  A range meets at most kFlatSlots rows
// and a row at most kFlatSlots ranges.  Each CTA leaves one key per row it
// meets, key = (order-preserving bits of the max) << 32 | (2^32 - 1 - index), so
// that the largest key names the lowest index of the maximum; a NaN anywhere
// gives the all-ones key.  The key of CTA c for row r goes to 64-bit word
// c - c_first(r) of r's record; the finish kernel merges a row's words.

constexpr int kFlatSlots = 4;
constexpr int kFlatThreads = 512;

struct FlatArgs {
    const void* logits;
    RowRec* rows;
    Header* hdr;
    int vpr;       // vectors per row
    int P;         // CTAs
    int per, rem;  // the tensor's R * vpr < 2^31 vectors = P * per + rem
    int B, k, V;
};

// The ranges: the first `rem` hold per + 1 vectors, the others per.  First
// vector of range c, and the range that holds vector x.
__host__ __device__ __forceinline__ int flat_start(int c, int per, int rem) {
    return c * per + min(c, rem);
}
__host__ __device__ __forceinline__ int flat_owner(int x, int per, int rem) {
    const int big = rem * (per + 1);
    return x < big ? x / (per + 1) : rem + (x - big) / per;
}

__device__ __forceinline__ uint32_t ordered_bits(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_ordered_bits(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, off);
        v = o > v ? o : v;
    }
    return v;
}

// NaN-propagating maximum of one 16-byte vector (bf16: pairwise on packed
// halves first).
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
    uint32_t y;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
    return y;
}
template <typename DT>
__device__ __forceinline__ float vec_max(const uint4& v);
template <>
__device__ __forceinline__ float vec_max<__nv_bfloat16>(const uint4& v) {
    const uint32_t w = bf16x2_max_nan(bf16x2_max_nan(v.x, v.y), bf16x2_max_nan(v.z, v.w));
    return fmax_nan(bf16_lo(w), bf16_hi(w));
}
template <>
__device__ __forceinline__ float vec_max<float>(const uint4& v) {
    return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                    fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
}
// A vector of -inf, the padding of a batch past the end of a range.
template <typename DT> struct kFlatPad;
template <> struct kFlatPad<__nv_bfloat16> {
    __device__ static __forceinline__ uint4 vec() {
        return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
    }
};
template <> struct kFlatPad<float> {
    __device__ static __forceinline__ uint4 vec() {
        return make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
    }
};

// The range of a CTA falls into nseg <= kFlatSlots row segments; the 16 warps
// are shared out among them in proportion to their lengths (at least one each),
// so that every warp reads a contiguous part of a single row.
template <typename DT>
__global__ void __launch_bounds__(kFlatThreads, 2) sv_flat_greedy_kernel(FlatArgs a) {
    using E = Elt<DT>;
    constexpr int VW = E::kVec;
    constexpr int U = 10;
    constexpr int NW = kFlatThreads / 32;
    __shared__ unsigned long long s_key[NW];
    __shared__ int s_seg[NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x;
    // Launched as a programmatic dependent of whatever precedes it on the
    // stream: wait for that grid (which may produce the logits, or still read
    // this workspace) before touching memory; then let the finish kernel launch.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (c == 0 && tid == 0) {
        a.hdr->magic = kMagic;
        a.hdr->B = a.B;
        a.hdr->k = a.k;
        a.hdr->V = a.V;
        a.hdr->mode = SV_MODE_GREEDY;
        a.hdr->flat_ctas = (uint32_t)a.P;
        a.hdr->flat_vpr = (uint32_t)a.vpr;
        a.hdr->flat_per = (uint32_t)a.per;
        a.hdr->flat_rem = (uint32_t)a.rem;
    }
    // The range: n vectors from s0; row r0 starts h vectors before it.  Segment
    // i (row r0 + i) covers offsets [e_i, e_i+1) of the range.
    const int s0 = flat_start(c, a.per, a.rem);
    const int n = a.per + (c < a.rem ? 1 : 0);
    const int r0 = s0 / a.vpr;
    const int h = s0 - r0 * a.vpr;
    const int e1 = min(n, a.vpr - h), e2 = min(n, e1 + a.vpr), e3 = min(n, e2 + a.vpr);
    const int nseg = 1 + (e1 < n) + (e2 < n) + (e3 < n);
    // First warp of segment i: i + round((NW - nseg) * e_i / n).
    auto first_warp = [&](int i, int e) {
        return i >= nseg ? NW : i + (2 * (NW - nseg) * e + n) / (2 * n);
    };
    const int w1 = first_warp(1, e1), w2 = first_warp(2, e2), w3 = first_warp(3, e3);
    const int seg = (warp >= w1) + (warp >= w2) + (warp >= w3);
    const int ws = seg == 0 ? 0 : seg == 1 ? w1 : seg == 2 ? w2 : w3;
    const int we = seg == 0 ? w1 : seg == 1 ? w2 : seg == 2 ? w3 : NW;
    const int eb = seg == 0 ? 0 : seg == 1 ? e1 : seg == 2 ? e2 : e3;
    const int ee = seg == 0 ? e1 : seg == 1 ? e2 : seg == 2 ? e3 : n;
    const int len = ee - eb, q = warp - ws, Q = we - ws;
    const int lo = eb + (len * q) / Q, hi = eb + (len * (q + 1)) / Q;
    const uint4* vp = static_cast<const uint4*>(a.logits) + s0;

    float best = 0.0f;  // running maximum, valid once bidx >= 0
    int bidx = -1;      // its element offset from the start of the range
    bool nan = false;
    for (int v = lo + lane; v < hi; v += U * 32) {
        const int last = min(U - 1, (hi - 1 - v) / 32);  // last vector of the batch
        uint4 buf[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            buf[u] = u <= last ? ld_stream16(vp + v + u * 32) : kFlatPad<DT>::vec();
        // The batch maximum (padding is -inf, after every real vector), then
        // the position of its first occurrence only when it beats the running
        // maximum.
        float m = vec_max<DT>(buf[0]);
#pragma unroll
        for (int u = 1; u < U; ++u) m = fmax_nan(m, vec_max<DT>(buf[u]));
        if (m != m) {
            nan = true;
        } else if (bidx < 0 || m > best) {
            int uf = 0;
            uint4 sel = buf[0];
#pragma unroll
            for (int u = U - 1; u >= 0; --u)
                if (vec_max<DT>(buf[u]) == m) {
                    uf = u;
                    sel = buf[u];
                }
            float f[VW];
            E::unpack(sel, f);
            int e = 0;  // the first element equal to the maximum
#pragma unroll
            for (int t = VW - 1; t >= 0; --t)
                if (f[t] == m) e = t;
            best = m;
            bidx = (v + uf * 32) * VW + e;
        }
    }
    unsigned long long kv = 0ull;
    if (nan) {
        kv = ~0ull;
    } else if (bidx >= 0) {
        // index in row r0 + seg; -0 counts as +0 (equal maxima are told apart by
        // index alone)
        const uint32_t idx = (uint32_t)(bidx + (h - seg * a.vpr) * VW);
        kv = ((unsigned long long)ordered_bits(best + 0.0f) << 32) | (0xFFFFFFFFu - idx);
    }
    kv = warp_max_u64(kv);
    if (lane == 0) {
        s_key[warp] = kv;
        s_seg[warp] = seg;
    }
    __syncthreads();
    if (tid < nseg) {
        unsigned long long m = 0ull;
#pragma unroll
        for (int i = 0; i < NW; ++i)
            if (s_seg[i] == tid && s_key[i] > m) m = s_key[i];
        const int r = r0 + tid;
        const int word = c - flat_owner(r * a.vpr, a.per, a.rem);
        reinterpret_cast<unsigned long long*>(a.rows + r)[word] = m;
    }
}

// One warp per sequence: the lanes load the records in parallel, lane 0 scans.
// After the flat stream, the lanes first merge their rows' partial keys into
// row records of their own (the keys stay in the workspace, so running the
// finish twice gives the same result, and the host merges them the same way
// for the row statistics).
__global__ void sv_finish_greedy_kernel(const int32_t* __restrict__ x, const RowRec* __restrict__ rows,
                                        const Header* __restrict__ hdr,
                                        uint32_t* __restrict__ seqstat, int B, int k,
                                        int32_t* __restrict__ out, int32_t* __restrict__ nacc,
                                        Epilogue ep) {
    __shared__ RowRec recs[4][kMaxK + 1];
    __shared__ int xs[4][kMaxK];
    const int wi = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * 4 + wi;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the row records are complete
    // A flat stream launched next waits for this whole grid before it writes.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (b >= B) return;
    RowRec* rr = recs[wi];
    int* xx = xs[wi];
    // The lane's first record and token are loaded before the header, so the
    // three loads are in flight together (none depends on another).
    RowRec rec0{};
    int x0 = 0;
    if (lane <= k) {
        rec0 = rows[(long long)b * (k + 1) + lane];
        if (lane < k) x0 = x[(long long)b * k + lane];
    }
    const uint32_t P = hdr->flat_ctas;
    const int vpr = (int)hdr->flat_vpr, per = (int)hdr->flat_per, rem = (int)hdr->flat_rem;
    const int V = (int)hdr->V;
    for (int i = lane; i <= k; i += 32) {
        const long long r = (long long)b * (k + 1) + i;
        const int xi = i == lane ? x0 : (i < k ? x[(long long)b * k + i] : 0);
        RowRec rec = i == lane ? rec0 : rows[r];
        if (i < k) xx[i] = xi;
        if (P) {
            const int c0 = flat_owner((int)r * vpr, per, rem);
            const int c1 = flat_owner((int)(r + 1) * vpr - 1, per, rem);
            const unsigned long long* w = reinterpret_cast<const unsigned long long*>(&rec);
            unsigned long long key = 0ull;
            for (int c = c0; c <= c1 && c - c0 < kFlatSlots; ++c)
                key = w[c - c0] > key ? w[c - c0] : key;
            const bool nan = key == ~0ull;
            const float m = from_ordered_bits((uint32_t)(key >> 32));
            rec.mraw = nan ? NAN : m;
            rec.S = 0.0f;
            rec.px = i < k ? 0.0 : (double)NAN;
            rec.lx = NAN;
            rec.qx = NAN;
            rec.argmax = nan ? 0 : (int32_t)(0xFFFFFFFFu - (uint32_t)key);
            rec.flags = (nan || !(m > -INFINITY) || m == INFINITY) ? kRowBad : 0u;
            if (i < k && (xi < 0 || xi >= V)) rec.flags |= kRowTokenBad;
            // The keys stay in the workspace (not overwritten by the merged
            // record), so the finish can run again on the same stream output.
        }
        rr[i] = rec;
    }
    __syncwarp();
    if (lane != 0) return;
    int32_t* o = out + (long long)b * (k + 1);
    uint32_t bits = 0;
    int n = k;
    for (int i = 0; i < k; ++i) {
        if (rr[i].flags & (kRowBad | kRowSkipped)) { bits = SV_DEV_BAD_ROW; break; }
        if (rr[i].flags & kRowTokenBad) { bits = SV_DEV_BAD_TOKEN; break; }
        if (xx[i] != rr[i].argmax) { n = i; break; }
    }
    if (!bits && (rr[n].flags & (kRowBad | kRowSkipped))) bits = SV_DEV_BAD_ROW;
    seqstat[b] = bits;
    if (bits) {
        for (int i = 0; i <= k; ++i) o[i] = -1;
        nacc[b] = -1;
        commit_sequence(ep, b, -1, k);
        return;
    }
    for (int i = 0; i < n; ++i) o[i] = xx[i];
    o[n] = rr[n].argmax;
    for (int i = n + 1; i <= k; ++i) o[i] = -1;
    nacc[b] = n;
    commit_sequence(ep, b, n, k);
}

// ------------------------------------------------------------------ tree verification
//
// Several drafted continuations checked at once ("Decodificação especulativa
// explicada", §"A família de rascunhos": Medusa's tree attention; "Speculative
// decoding: el secretario...", §"Tree attention").  A sequence's tree has N
// nodes: node 0 the root, node j >= 1 a drafted token with a parent before it;
// logits row j is the target's distribution after node j.  The walk starts at
// the root.  Greedy: the first child (in index order) whose token is the
// node's argmax is accepted.  Sampled: recursive rejection over the node's
// children, drawn independently from the node's draft distribution q: the
// current distribution r starts as p; child j is accepted iff r(x) >= q(x) or
// u_j < r(x)/q(x); a rejection replaces r by the normalised residual
// max(0, r - q) (by p again, flagged, when that has no mass).  With no child
// accepted the final token is drawn from r.  One child per node is the chain
// rule.  The row stream provides each row's max, normaliser and argmax; this
// kernel (one CTA per sequence) walks the tree, making a pass over a node's
// logits and q rows for each rejected child and for the final draw.

constexpr int kTreeMaxN = kMaxK + 1;

// Dynamic shared memory of the sampled walk: the final draw's block sums, a
// double per 32 chunks of 8 elements.
__host__ __device__ inline size_t tree_bsum_bytes(int V) {
    const long long nch = ((long long)V + kChunk - 1) / kChunk;
    return (size_t)((nch + 31) / 32) * sizeof(double);
}

struct TreeArgs {
    const void* logits;
    const float* q;
    const int32_t* tok;
    const int32_t* par;
    const float* ua;
    const float* ur;
    const Header* hdr;
    RowRec* rows;
    uint32_t* seqstat;
    int32_t* out;
    int32_t* nodes;
    int32_t* nacc;
    int B, N, V;
    ff c2;  // log2(e)/T
};

// A row's record, with the flat stream's partial keys merged when it left them.
__device__ __forceinline__ RowRec row_record(const RowRec* rows, long long r, uint32_t P,
                                             int vpr, int per, int rem) {
    RowRec rec = rows[r];
    if (P) {
        const int c0 = flat_owner((int)r * vpr, per, rem);
        const int c1 = flat_owner((int)(r + 1) * vpr - 1, per, rem);
        const unsigned long long* w = reinterpret_cast<const unsigned long long*>(&rec);
        unsigned long long key = 0ull;
        for (int c = c0; c <= c1 && c - c0 < kFlatSlots; ++c) key = w[c - c0] > key ? w[c - c0] : key;
        const bool nan = key == ~0ull;
        const float m = from_ordered_bits((uint32_t)(key >> 32));
        rec.mraw = nan ? NAN : m;
        rec.S = 0.0f;
        rec.px = NAN;
        rec.lx = NAN;
        rec.qx = NAN;
        rec.argmax = nan ? 0 : (int32_t)(0xFFFFFFFFu - (uint32_t)key);
        rec.flags = (nan || !(m > -INFINITY) || m == INFINITY) ? kRowBad : 0u;
    }
    return rec;
}

// p_v = 2^((l_v - m) c) / S in fp32 (the fast pass's corrected exponential).
__device__ __forceinline__ float tree_p(float l, float m, ff c2, float inv_s) {
    const float d = __fsub_rn(l, m);
    const float a = __fmul_rn(d, c2.hi);
    float err = __fmaf_rn(d, c2.hi, -a);
    err = __fmaf_rn(d, c2.lo, err);
    const float y0 = ex2_approx(a);
    const float y = y0 > 0.0f ? __fmaf_rn(y0, __fmul_rn(err, 0.693147181f), y0) : 0.0f;
    return __fmul_rn(y, inv_s);
}

// r_t(v): p_v through t residual steps r <- max(0, r - q_v) / Z.
__device__ __forceinline__ float tree_r(float p, float qv, const float* invz, int t) {
    float r = p;
    for (int s = 0; s < t; ++s) r = __fmul_rn(fmaxf(__fsub_rn(r, qv), 0.0f), invz[s]);
    return r;
}

template <int NT>
__device__ __forceinline__ double block_sum_d(double v, double* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    double t = 0.0;
    for (int i = 0; i < NT / 32; ++i) t += red[i];
    return t;
}

template <typename DT, bool SAMPLED>
__global__ void __launch_bounds__(SAMPLED ? kThreads : 64)
    sv_tree_kernel(TreeArgs a) {
    using E = Elt<DT>;
    constexpr int NT = SAMPLED ? kThreads : 64;
    __shared__ int s_tok[kTreeMaxN], s_par[kTreeMaxN];
    __shared__ RowRec s_rec[kTreeMaxN];  // greedy: every row's record
    __shared__ float s_invz[kTreeMaxN];  // 1 / Z_t of the current node's residual steps
    __shared__ double s_red[NT / 32];
    __shared__ int s_bits, s_info, s_n, s_cur, s_next, s_nrej, s_token, s_path[kTreeMaxN];
    __shared__ int s_lp[NT / 32];
    __shared__ double s_red2;
    __shared__ float s_cl[kTreeMaxN], s_cq[kTreeMaxN], s_cu[kTreeMaxN];  // children's l(x), q(x), u
    extern __shared__ double tree_bsum[];  // sampled: block sums of the final draw
    const int tid = threadIdx.x;
    const int b = blockIdx.x, N = a.N, V = a.V;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the row records are complete
    for (int i = tid; i < N; i += NT) {
        s_tok[i] = a.tok[(long long)b * N + i];
        s_par[i] = a.par[(long long)b * N + i];
    }
    if (tid == 0) {
        s_bits = 0;
        s_info = 0;
        s_n = 0;
        s_cur = 0;
        s_token = -1;
    }
    __syncthreads();
    if (tid == 0)
        for (int j = 1; j < N; ++j)
            if (s_par[j] < 0 || s_par[j] >= j) s_bits |= SV_DEV_BAD_TREE;
    const DT* seq = static_cast<const DT*>(a.logits) + (long long)b * N * V;
    if (!SAMPLED) {
        // every row's record (merged from the flat stream's keys when needed)
        const uint32_t P = a.hdr->flat_ctas;
        const int vpr = (int)a.hdr->flat_vpr, per = (int)a.hdr->flat_per,
                  rem = (int)a.hdr->flat_rem;
        for (int i = tid; i < N; i += NT) {
            const long long r = (long long)b * N + i;
            s_rec[i] = row_record(a.rows, r, P, vpr, per, rem);
        }
        __syncthreads();
        if (tid == 0 && !s_bits) {
            int cur = 0, n = 0;
            for (;;) {
                if (s_rec[cur].flags & kRowBad) {
                    s_bits |= SV_DEV_BAD_ROW;
                    break;
                }
                const int am = s_rec[cur].argmax;
                int next = -1;
                for (int j = cur + 1; j < N; ++j) {
                    if (s_par[j] != cur) continue;
                    if (s_tok[j] < 0 || s_tok[j] >= V) {
                        s_bits |= SV_DEV_BAD_TOKEN;
                        break;
                    }
                    if (s_tok[j] == am) {
                        next = j;
                        break;
                    }
                }
                if (s_bits) break;
                if (next < 0) {
                    s_token = am;
                    break;
                }
                s_path[n++] = next;
                cur = next;
            }
            s_n = n;
        }
    } else {
        const float* qseq = a.q + (long long)b * N * V;
        for (;;) {
            __syncthreads();
            if (s_bits || s_token >= 0) break;
            const int cur = s_cur;
            const RowRec rec = a.rows[(long long)b * N + cur];
            if (rec.flags & kRowBad) {
                if (tid == 0) s_bits |= SV_DEV_BAD_ROW;
                continue;
            }
            const float m = rec.mraw, inv_s = __frcp_rn(rec.S);
            const DT* lrow = seq + (long long)cur * V;
            const float* qrow = qseq + (long long)cur * V;
            // the rows in chunks of 8 elements (16-byte loads when aligned)
            const bool al_l = (reinterpret_cast<uintptr_t>(lrow) & 15) == 0;
            const bool al_q = (reinterpret_cast<uintptr_t>(qrow) & 15) == 0;
            const int nch = (V + kChunk - 1) / kChunk;
            if (tid == 0) {
                s_nrej = 0;
                s_next = -1;
            }
            // every child's l(x), q(x) and uniform, gathered at once
            for (int j = cur + 1 + tid; j < N; j += NT)
                if (s_par[j] == cur) {
                    const int x = s_tok[j];
                    const bool ok = x >= 0 && x < V;
                    s_cl[j] = ok ? E::load1(lrow + x) : 0.0f;
                    s_cq[j] = ok ? qrow[x] : 0.0f;
                    s_cu[j] = a.ua[(long long)b * N + j];
                }
            __syncthreads();
            // the children in index order
            for (int j = cur + 1; j < N; ++j) {
                if (s_par[j] != cur) continue;  // uniform: shared data
                if (tid == 0) {
                    const int x = s_tok[j];
                    if (x < 0 || x >= V) {
                        s_bits |= SV_DEV_BAD_TOKEN;
                    } else {
                        const float u = s_cu[j], Q = s_cq[j];
                        if (!(u >= 0.0f && u < 1.0f)) s_bits |= SV_DEV_BAD_UNIFORM;
                        else if (!(Q >= 0.0f)) s_bits |= SV_DEV_BAD_Q;
                        else {
                            const float P =
                                tree_r(tree_p(s_cl[j], m, a.c2, inv_s), Q, s_invz, s_nrej);
                            if (P >= Q || u < __fdiv_rn(P, Q)) s_next = j;
                        }
                    }
                }
                __syncthreads();
                if (s_bits || s_next >= 0) break;
                // rejected: Z = sum_v max(0, r(v) - q(v)) over the row, two
                // chunks per thread in flight
                const int t = s_nrej;
                double z = 0.0;
                for (int c0 = tid; c0 < nch; c0 += 2 * NT) {
                    float l[2][kChunk], qv[2][kChunk];
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                        if (c0 + u * NT < nch) {
                            load_chunk<DT>(lrow, (long long)(c0 + u * NT) * kChunk, V, al_l, l[u]);
                            load_q_chunk(qrow, (long long)(c0 + u * NT) * kChunk, V, al_q, qv[u]);
                        }
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        if (c0 + u * NT >= nch) break;
                        float zc = 0.0f;
#pragma unroll
                        for (int e = 0; e < kChunk; ++e) {
                            const float r =
                                tree_r(tree_p(l[u][e], m, a.c2, inv_s), qv[u][e], s_invz, t);
                            zc += fmaxf(__fsub_rn(r, qv[u][e]), 0.0f);
                        }
                        z += (double)zc;
                    }
                }
                z = block_sum_d<NT>(z, s_red);
                if (tid == 0) {
                    if (z > 0.0) {
                        s_invz[t] = (float)(1.0 / z);
                        s_nrej = t + 1;
                    } else {  // zero residual mass: back to p
                        s_nrej = 0;
                        s_info |= SV_DEV_DEGENERATE;
                    }
                }
                __syncthreads();
            }
            if (s_bits) continue;
            if (s_next >= 0) {
                if (tid == 0) {
                    s_path[s_n++] = s_next;
                    s_cur = s_next;
                }
                continue;
            }
            // No child accepted: draw from r with u_resample.  Weights: p, or the
            // last rejection's residual max(0, r - q) (unnormalised).  A pass
            // sums blocks of 32 chunks (a warp, a chunk per lane) into shared
            // memory; the block holding u * C is found from their prefix; its
            // warp reloads it and one lane finds the element.
            const float u = a.ur[b];
            if (!(u >= 0.0f && u < 1.0f)) {
                if (tid == 0) s_bits |= SV_DEV_BAD_UNIFORM;
                continue;
            }
            const int t = s_nrej;
            const int lane = tid & 31, warp = tid >> 5;
            auto weights = [&](int c, float* w) {
                float l[kChunk], qv[kChunk];
                load_chunk<DT>(lrow, (long long)c * kChunk, V, al_l, l);
                if (t > 0) load_q_chunk(qrow, (long long)c * kChunk, V, al_q, qv);
#pragma unroll
                for (int e = 0; e < kChunk; ++e) {
                    const float p = tree_p(l[e], m, a.c2, inv_s);
                    w[e] = t == 0 ? p
                                  : fmaxf(__fsub_rn(tree_r(p, qv[e], s_invz, t - 1), qv[e]), 0.0f);
                }
            };
            auto chunk_sum = [&](const float* w) {
                double cs = 0.0;
#pragma unroll
                for (int e = 0; e < kChunk; ++e) cs += (double)w[e];
                return cs;
            };
            const int nblk = (nch + 31) / 32;
            for (int blk = warp; blk < nblk; blk += NT / 32) {
                const int c = blk * 32 + lane;
                double cs = 0.0;
                if (c < nch) {
                    float w[kChunk];
                    weights(c, w);
                    cs = chunk_sum(w);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) cs += __shfl_xor_sync(0xffffffffu, cs, off);
                if (lane == 0) tree_bsum[blk] = cs;
            }
            __syncthreads();
            // prefix of the block sums: each thread a contiguous share
            const int Lb = (nblk + NT - 1) / NT, b0 = min(nblk, tid * Lb), b1 = min(nblk, b0 + Lb);
            double mine = 0.0;
            for (int i = b0; i < b1; ++i) mine += tree_bsum[i];
            double incl = mine;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const double o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            if (lane == 31) s_red[warp] = incl;
            if (tid == 0) {
                s_next = -1;  // the block holding u * C
                s_token = -1;
            }
            __syncthreads();
            double before = 0.0, total = 0.0;
            for (int i = 0; i < NT / 32; ++i) {
                if (i < warp) before += s_red[i];
                total += s_red[i];
            }
            before += incl - mine;
            const double tau = (double)u * total;
            if (mine > 0.0 && before <= tau && tau < before + mine) {
                double run = before;
                int i = b0;
                for (; i < b1 - 1; ++i) {
                    if (tau < run + tree_bsum[i]) break;
                    run += tree_bsum[i];
                }
                s_next = i;
                s_red2 = run;
            }
            __syncthreads();
            if (warp == 0 && s_next >= 0) {
                const int c = s_next * 32 + lane;
                float w[kChunk] = {};
                double cs = 0.0;
                if (c < nch) {
                    weights(c, w);
                    cs = chunk_sum(w);
                }
                double ci = cs;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const double o = __shfl_up_sync(0xffffffffu, ci, off);
                    if (lane >= off) ci += o;
                }
                const double cb = s_red2 + ci - cs;  // weight before this lane's chunk
                bool mine_c = cs > 0.0 && cb <= tau && tau < cb + cs;
                if (!__any_sync(0xffffffffu, mine_c)) {
                    // the block's own sums rounded differently: the last chunk
                    // starting at or before u * C
                    const unsigned mk = __ballot_sync(0xffffffffu, cs > 0.0 && cb <= tau);
                    mine_c = mk != 0u && lane == 31 - __clz(mk);
                }
                if (mine_c) {
                    double cum = cb;
                    int tok = -1;
#pragma unroll
                    for (int e = 0; e < kChunk; ++e) {
                        cum += (double)w[e];
                        if (tok < 0 && w[e] > 0.0f && cum > tau) tok = c * kChunk + e;
                    }
                    if (tok < 0)  // rounding at the chunk's end: its last positive element
#pragma unroll
                        for (int e = 0; e < kChunk; ++e)
                            if (w[e] > 0.0f) tok = c * kChunk + e;
                    s_token = tok;
                }
            }
            __syncthreads();
            if (s_token < 0) {
                // u * C fell outside every bin (rounding): the last positive bin
                int lp = -1;
                for (int c = tid; c < nch; c += NT) {
                    float w[kChunk];
                    weights(c, w);
#pragma unroll
                    for (int e = 0; e < kChunk; ++e)
                        if (w[e] > 0.0f) lp = max(lp, c * kChunk + e);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, off));
                if (lane == 0) s_lp[warp] = lp;
                __syncthreads();
                if (tid == 0) {
                    int best = -1;
                    for (int i = 0; i < NT / 32; ++i) best = max(best, s_lp[i]);
                    s_token = best < 0 ? 0 : best;
                }
            }
        }
    }
    __syncthreads();
    if (tid != 0) return;
    int32_t* o = a.out + (long long)b * N;
    int32_t* nd = a.nodes + (long long)b * N;
    const uint32_t bits = (uint32_t)s_bits;
    a.seqstat[b] = bits | (uint32_t)s_info;
    if (bits) {
        for (int i = 0; i < N; ++i) {
            o[i] = -1;
            nd[i] = -1;
        }
        a.nacc[b] = -1;
        return;
    }
    const int n = s_n;
    for (int i = 0; i < n; ++i) {
        o[i] = s_tok[s_path[i]];
        nd[i] = s_path[i];
    }
    o[n] = s_token;
    for (int i = n + 1; i < N; ++i) o[i] = -1;
    for (int i = n; i < N; ++i) nd[i] = -1;
    a.nacc[b] = n;
}

struct FinishArgs {
    const void* logits;
    const float* q;
    const int32_t* x;
    const float* ua;
    const float* ur;
    const RowRec* rows;
    uint32_t* seqstat;
    int32_t* out;
    int32_t* nacc;
    uint32_t* plist_count;  // with plist: draws needing the precise pass are
    uint32_t* plist;        // appended here for sv_precise_kernel (else run here)
    Epilogue ep;
    int B, k, V, G;
    int draw_level;
    int force_precise;
    float c;
    ff c2;
};

// EXACT: the fast draw's chunk sums in float-float (small batches, whose
// precise draws run here); else pairwise (large batches, whose precise draws
// go to sv_precise_kernel in one wave, so a few more of them cost little).
// The scan of sequence b over its row records, by every thread of the CTA:
// each row's test in parallel ("Decodificação especulativa explicada",
// §"A regra de amostragem por rejeição": accept x_i when p >= q or u < p/q),
// then the first row that stops the scan.  Leaves the records, the decision
// row n and the error bits (0: a valid sequence) in `sc`.
struct ScanShared {
    RowRec recs[kMaxK + 1];
    float uas[kMaxK];
    uint32_t codes[kMaxK];
    float ur;
    int n, bits;
};
__device__ __forceinline__ void scan_sequence(ScanShared& sc, const RowRec* rows, const float* ua,
                                              const float* ur, int b, int k) {
    const int tid = threadIdx.x;
    for (int i = tid; i <= k; i += blockDim.x) sc.recs[i] = rows[(long long)b * (k + 1) + i];
    for (int i = tid; i < k; i += blockDim.x) sc.uas[i] = ua[(long long)b * k + i];
    if (tid == blockDim.x - 1) sc.ur = ur[b];
    __syncthreads();
    for (int i = tid; i < k; i += blockDim.x) {  // each row's test, in parallel
        const RowRec& r = sc.recs[i];
        const float u = sc.uas[i];
        uint32_t c;
        if (r.flags & (kRowBad | kRowSkipped)) {  // a skipped row is never reached
            c = kCodeError | SV_DEV_BAD_ROW;
        } else if (r.flags & kRowTokenBad) {
            c = kCodeError | SV_DEV_BAD_TOKEN;
        } else if (!(u >= 0.0f && u < 1.0f)) {
            c = kCodeError | SV_DEV_BAD_UNIFORM;
        } else if (r.flags & kRowQBad) {
            c = kCodeError | SV_DEV_BAD_Q;
        } else {
            const float P = (float)r.px, Q = r.qx;
            c = ((P >= Q) || (u < __fdiv_rn(P, Q))) ? kCodeAccept : kCodeReject;
        }
        sc.codes[i] = c;
    }
    __syncthreads();
    if (tid == 0) {  // the first row that stops the scan
        int bits = 0, n = k;
        for (int i = 0; i < k; ++i) {
            const uint32_t c = sc.codes[i];
            if (c == kCodeAccept) continue;
            if (c & kCodeError) bits = (int)(c & ~kCodeError);
            else n = i;
            break;
        }
        if (!bits && (sc.recs[n].flags & (kRowBad | kRowSkipped))) bits = SV_DEV_BAD_ROW;
        if (!bits && !(sc.ur >= 0.0f && sc.ur < 1.0f)) bits = SV_DEV_BAD_UNIFORM;
        sc.n = n;
        sc.bits = bits;
    }
    __syncthreads();
}

template <typename DT, bool EXACT>
__global__ void __launch_bounds__(kThreads, 2) sv_finish_sample_kernel(FinishArgs a) {
    extern __shared__ __align__(16) unsigned char dyn[];
    __shared__ DrawShared ds;
    __shared__ ScanShared sc;
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x;
    const int G = a.G;
    const int b = blockIdx.x / G;
    const int rank = blockIdx.x % G;
    const int k = a.k, V = a.V;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the row records are complete
    scan_sequence(sc, a.rows, a.ua, a.ur, b, k);
    const RowRec* recs = sc.recs;
    const int s_n = sc.n, s_bits = sc.bits;
    const float s_ur = sc.ur;
    const int n = s_n;
    int32_t* o = a.out + (long long)b * (k + 1);
    if (s_bits) {
        if (rank == 0) {
            for (int i = tid; i <= k; i += kThreads) o[i] = -1;
            if (tid == 0) {
                a.nacc[b] = -1;
                a.seqstat[b] = (uint32_t)s_bits;
                commit_sequence(a.ep, b, -1, k);
            }
        }
        return;  // every CTA of the cluster takes this branch together
    }
    const DT* drow = static_cast<const DT*>(a.logits) + ((long long)b * (k + 1) + n) * V;
    const float* qrow = n < k ? a.q + ((long long)b * k + n) * V : nullptr;
    bool degenerate = false, fallback = false;
    const DrawCtx<DT> dc = make_draw_ctx<DT>(dyn, a.draw_level, drow, qrow, n < k,
                                             V, recs[n].mraw, a.c, a.c2, s_ur, rank, G,
                                             recs[n].S);
    const bool deferred = draw<DT, EXACT>(cluster, ds, dc, a.force_precise != 0,
                                          a.plist != nullptr, o + n, degenerate, fallback);
    if (rank == 0) {
        for (int i = tid; i <= k; i += kThreads)
            if (i != n) o[i] = i < n ? a.x[(long long)b * k + i] : -1;
        if (tid == 0) {
            a.nacc[b] = n;
            a.seqstat[b] = (degenerate ? SV_DEV_DEGENERATE : 0u) | (fallback ? SV_DEV_PRECISE : 0u);
            commit_sequence(a.ep, b, n, k);
            if (deferred) {
                const uint32_t j = atomicAdd(a.plist_count, 1u);
                if (j < (uint32_t)a.B) a.plist[j] = (uint32_t)b;  // at most B entries
            }
        }
    }
}

// The precise draws of a large batch, left by sv_finish_sample_kernel in the
// workspace list: persistent clusters of G CTAs (as many as fit at once),
// cluster c taking entries c, c + clusters, ...  Each draw is the precise pass
// of the finish kernel over a slice of V / G elements per CTA.
struct PreciseArgs {
    const void* logits;
    const float* q;
    const float* ur;
    const RowRec* rows;
    const int32_t* nacc;
    const uint32_t* plist_count;
    const uint32_t* plist;
    uint32_t* seqstat;
    int32_t* out;
    int B, k, V, G;
    int draw_level;
    float c;
    ff c2;
};

template <typename DT>
__global__ void __launch_bounds__(kThreads, 2) sv_precise_kernel(PreciseArgs a) {
    extern __shared__ __align__(16) unsigned char dyn[];
    __shared__ DrawShared ds;
    cg::cluster_group cluster = cg::this_cluster();
    const int G = a.G;
    const int tid = threadIdx.x;
    const int rank = blockIdx.x % G, cid = blockIdx.x / G, ncl = gridDim.x / G;
    const int k = a.k, V = a.V;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the list is complete
    const uint32_t cnt = min(*a.plist_count, (uint32_t)a.B);
    for (uint32_t j = cid; j < cnt; j += ncl) {
        const int b = (int)a.plist[j];
        const int n = a.nacc[b];
        const DT* drow = static_cast<const DT*>(a.logits) + ((long long)b * (k + 1) + n) * V;
        const float* qrow = n < k ? a.q + ((long long)b * k + n) * V : nullptr;
        const RowRec& rec = a.rows[(long long)b * (k + 1) + n];
        const DrawCtx<DT> dc = make_draw_ctx<DT>(dyn, a.draw_level, drow, qrow, n < k, V,
                                                 rec.mraw, a.c, a.c2, a.ur[b], rank, G, rec.S);
        if (tid == 0) ds.token = -1;
        __syncthreads();
        bool degenerate = false;
        draw_precise_any<DT>(cluster, ds, dc, degenerate);
        __syncthreads();
        if (tid == 0 && ds.token >= 0) a.out[(long long)b * (k + 1) + n] = ds.token;
        if (rank == 0 && tid == 0 && degenerate)
            a.seqstat[b] = SV_DEV_PRECISE | SV_DEV_DEGENERATE;
        cluster.sync();  // the exchange slots serve the next draw
    }
}

// ------------------------------------------------------------------ split draw
//
// The draw of a sampled verify with each decision row cut into NS slices, one
// CTA per slice and no cluster, so that a batch's draws spread over every SM in
// small, equal pieces.  Every CTA runs its sequence's scan from the row records,
// then the fast pass over its slice, and leaves the slice's sums in the
// workspace.  The CTA that completes a sequence's set (an arrival counter: the
// last to arrive sees NS - 1) finishes the draw: the totals and the bound of
// fast_bound, the owning slice (a prefix over the slices' sums), the owner's
// block (from the block sums every slice leaves in the workspace) and its
// element (that block's 64 elements recomputed in the same arithmetic, so they
// agree with the block sums exactly).  A
// draw the bound cannot certify is listed for the split precise draw, which
// runs in the same fashion in two launches: the float-float normaliser's
// slice sums, then each slice's fixed-point weight total, the last CTA of an
// entry finding the token.  No CTA waits for another: the arrival counter
// only tells the last one that the others' sums are in memory.

// CTAs a fast split draw aims for: one per SM on large batches (whose
// pairwise pass is short), two per SM on small ones (float-float sums).
constexpr int kSplitTargetLarge = 152, kSplitTargetSmall = 304;
constexpr int kSplitMinChunks = 128;    // smallest slice (chunks of 8 elements)
constexpr int kSplitMaxChunks = 1 << 18;  // largest slice (a whole row of the largest V)
constexpr int kSplitMaxSlices = kThreads;

// Slices per sequence of the fast split draw: about kSplitTarget* CTAs in all
// (measured on B = 256, V = 151936: one slice per row 1.5 us faster than two,
// 6 us faster than four), slices of at least kSplitMinChunks chunks, at most
// kSplitMaxSlices.  Returns the slice length in chunks in *sc.
__host__ __device__ inline int split_slices(int B, int V, int* sc) {
    const long long nch = ((long long)V + kChunk - 1) / kChunk;
    const long long target = B < kSplitTargetLarge ? kSplitTargetSmall : kSplitTargetLarge;
    long long ns = (target + (long long)B - 1) / (B > 0 ? B : 1);
    const long long lo = (nch + kSplitMaxChunks - 1) / kSplitMaxChunks;
    const long long hi = (nch + kSplitMinChunks - 1) / kSplitMinChunks;
    if (ns > hi) ns = hi;
    if (ns < lo) ns = lo;
    if (ns > kSplitMaxSlices) ns = kSplitMaxSlices;
    if (ns < 1) ns = 1;
    long long c = (nch + ns - 1) / ns;
    c = (c + kFastGroup - 1) / kFastGroup * kFastGroup;  // whole blocks of 8 chunks
    *sc = (int)c;
    return (int)((nch + c - 1) / c);
}
// The split precise draw's persistent grid (at most this many CTAs; its
// per-CTA item sums are sized for it) and the list of ambiguous elements each
// listed draw can hold.
constexpr int kPreciseGrid = 512;
constexpr int kAmbCap = 32;
struct AmbElem {
    int idx;      // element index in the row
    float q;      // its q
    float ehi, elo;  // its e = exp((l - m)/T) in float-float
};
struct PreciseItem {
    unsigned long long Y, Q;  // the slice's fixed-point sums of the positive elements
    ff S;                     // the slice's float-float sum of e
    unsigned long long pad;
};
static_assert(sizeof(AmbElem) == 16 && sizeof(PreciseItem) == 32, "precise records");

// The split draws' part of the workspace (after the list of precise draws):
// B fast arrival counters (zeroed with the list's counter, which they follow);
// per list entry (B of them) an arrival counter, an ambiguous-element count,
// the classifying normaliser and its margin, and kAmbCap ambiguous elements;
// B * NS slice sums; max(kPreciseGrid, B) precise item sums; and the fast
// pass's block sums, {Y, Q} per 64 elements of each decision row (reused by
// the precise pass for the rows it draws).
constexpr long long kSplitMaxTotal = 16384;          // slices of a launch
constexpr size_t kSplitMaxBlockBytes = 64ull << 20;  // block sums of a launch
__host__ __device__ inline long long split_row_blocks(int V) {
    const long long nch = ((long long)V + kChunk - 1) / kChunk;
    return (nch + kFastGroup - 1) / kFastGroup;
}
__host__ __device__ inline bool split_fits(long long B, int V) {
    int sc = 0;
    return B > 0 && B * split_slices((int)B, V, &sc) <= kSplitMaxTotal &&
           (size_t)B * split_row_blocks(V) * 16 <= kSplitMaxBlockBytes;
}
struct SplitLayout {
    size_t parrive, pambn, pS, pD, amb, srec, items, bsum, end;  // from the region's start
};
__host__ __device__ inline SplitLayout split_layout(long long B, int V) {
    int sc = 0;
    const int ns = split_slices((int)B, V, &sc);
    const size_t nb = (size_t)B;
    SplitLayout L;
    L.parrive = nb * 4;
    L.pambn = L.parrive + nb * 4;
    L.pS = L.pambn + nb * 4;
    L.pD = L.pS + nb * 4;
    L.amb = (L.pD + nb * 4 + 15) & ~(size_t)15;
    L.srec = L.amb + nb * kAmbCap * sizeof(AmbElem);
    L.items = L.srec + nb * ns * sizeof(FastTotals);
    L.bsum = L.items + (size_t)(B > kPreciseGrid ? B : kPreciseGrid) * sizeof(PreciseItem);
    L.end = L.bsum + nb * split_row_blocks(V) * 16;
    return L;
}
__host__ __device__ size_t split_ws_bytes(long long B, int V) {
    return split_fits(B, V) ? split_layout(B, V).end : 0;
}

struct SplitArgs {
    const void* logits;
    const float* q;
    const int32_t* x;
    const float* ua;
    const float* ur;
    const RowRec* rows;
    uint32_t* seqstat;
    int32_t* out;
    int32_t* nacc;
    uint32_t* plist_count;  // the draws for the precise pass (count, entries)
    uint32_t* plist;
    uint32_t* arrive;       // [B] slices done per sequence (zero before the launch)
    uint32_t* parrive;      // [B] per entry of the list (zeroed when it is listed)
    uint32_t* pambn;        // [B] ambiguous elements per entry (zeroed when it is listed)
    float* pS;              // [B] per entry: the fast pass's normaliser S (or S_row)
    float* pD;              // [B] per entry: the classification margin delta
    FastTotals* srec;       // [B * NS] the slices' sums
    unsigned long long* bsum;  // [B][row blocks][2] the fast pass's block sums
    long long nbr;          // blocks per row
    Epilogue ep;
    int B, k, V, NS, SC;    // slices per sequence, chunks per slice
    int force_precise;
    ff c2;
};

// A slice of the decision row as a draw context (rank 0 of a cluster of one).
template <typename DT>
__device__ __forceinline__ DrawCtx<DT> slice_ctx(unsigned char* dyn, const DT* rowp,
                                                 const float* qrow, bool residual, int V, float m,
                                                 ff c2, float u, long long c0, int mych,
                                                 float s_row) {
    DrawCtx<DT> d;
    d.rowp = rowp;
    d.qrow = qrow;
    d.V = V;
    d.residual = residual;
    d.m = m;
    d.c = c2.hi;
    d.clo = c2.lo;
    d.c2 = c2;
    d.u = u;
    d.c0 = c0;
    d.mych = mych > 0 ? mych : 0;
    d.nblk = (d.mych + kBlockChunks - 1) / kBlockChunks;
    d.al_l = (reinterpret_cast<uintptr_t>(rowp) & 15) == 0;
    d.al_q = residual && (reinterpret_cast<uintptr_t>(qrow) & 15) == 0;
    d.rank = 0;
    d.G = 1;
    d.bsum = reinterpret_cast<unsigned long long*>(dyn);
    d.thi = nullptr;
    d.tlo = nullptr;
    d.s_row = s_row;
    d.ecache = nullptr;
    d.pY = nullptr;
    d.pQ = nullptr;
    d.pamb = nullptr;
    return d;
}

// 32-byte slice sums read past L1 (another SM wrote them).
__device__ __forceinline__ FastTotals load_totals_cg(const FastTotals* p) {
    const uint4* v = reinterpret_cast<const uint4*>(p);
    const uint4 x = __ldcg(v), y = __ldcg(v + 1);
    FastTotals t;
    t.S.hi = __uint_as_float(x.x);
    t.S.lo = __uint_as_float(x.y);
    t.Y = ((unsigned long long)x.w << 32) | x.z;
    t.Q = ((unsigned long long)y.y << 32) | y.x;
    t.Aq = __uint_as_float(y.z);
    t.qmin = __uint_as_float(y.w);
    return t;
}

struct SplitShared {
    FastTotals tot;
    unsigned long long woffY[kWarps], woffQ[kWarps];
    unsigned long long M, tau, Y0, Q0;
    int ok, owner, last;
};

template <typename DT, bool EXACT>
__global__ void __launch_bounds__(kThreads, 2) sv_split_draw_kernel(SplitArgs a) {
    __shared__ DrawShared ds;
    __shared__ ScanShared sc;
    __shared__ SplitShared ss;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NS = a.NS;
    const int b = blockIdx.x / NS, s = blockIdx.x % NS;
    const int k = a.k, V = a.V;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the row records are complete
    // The precise launch (a programmatic dependent) may start now: its CTAs
    // wait for this grid's results, and it returns at once with no draw listed.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    scan_sequence(sc, a.rows, a.ua, a.ur, b, k);
    const int n = sc.n;
    int32_t* o = a.out + (long long)b * (k + 1);
    if (sc.bits) {  // an invalid sequence: no draw (every slice returns here)
        if (s == 0) {
            for (int i = tid; i <= k; i += kThreads) o[i] = -1;
            if (tid == 0) {
                a.nacc[b] = -1;
                a.seqstat[b] = (uint32_t)sc.bits;
                commit_sequence(a.ep, b, -1, k);
            }
        }
        return;
    }
    const bool res = n < k;
    const DT* drow = static_cast<const DT*>(a.logits) + ((long long)b * (k + 1) + n) * V;
    const float* qrow = res ? a.q + ((long long)b * k + n) * V : nullptr;
    const long long nch = ((long long)V + kChunk - 1) / kChunk;
    const float m = sc.recs[n].mraw, s_row = sc.recs[n].S, u = sc.ur;
    const FastScale f = make_fast_scale(m, a.c2, s_row, res);
    unsigned long long* rowblk = a.bsum + (long long)b * a.nbr * 2;  // this row's block sums
    {
        const long long c0 = (long long)s * a.SC;
        const DrawCtx<DT> d =
            slice_ctx<DT>(reinterpret_cast<unsigned char*>(rowblk + (c0 / kFastGroup) * 2), drow,
                          qrow, res, V, m, a.c2, u, c0, (int)min((long long)a.SC, nch - c0), s_row);
        const FastTotals t =
            res ? fast_pass<DT, true, EXACT, true>(d, f) : fast_pass<DT, false, EXACT, true>(d, f);
        cta_fast_totals(ds, t, &ss.tot);
    }
    if (tid == 0) {
        a.srec[(long long)b * NS + s] = ss.tot;
        __threadfence();
        ss.last = atomicAdd(&a.arrive[b], 1u) == (uint32_t)(NS - 1);
    }
    __syncthreads();
    if (!ss.last) return;

    // ---- the last CTA of the sequence: the totals, the owning slice, the token
    __threadfence();
    if (tid == 0) a.arrive[b] = 0;  // for the next call on this workspace
    FastTotals mine = tid < NS ? load_totals_cg(a.srec + (long long)b * NS + tid) : zero_totals();
    if (tid >= NS) mine.qmin = 0.0f;
    // Exclusive prefix of (Y, Q) over the slices (one slice per thread).
    unsigned long long iy = mine.Y, iq = mine.Q;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long yo = __shfl_up_sync(0xffffffffu, iy, off);
        const unsigned long long qo = __shfl_up_sync(0xffffffffu, iq, off);
        if (lane >= off) {
            iy += yo;
            iq += qo;
        }
    }
    if (lane == 31) {
        ss.woffY[warp] = iy;
        ss.woffQ[warp] = iq;
    }
    cta_fast_totals(ds, mine, &ss.tot);  // (its barriers also publish woff*)
    unsigned long long wy = 0ull, wq = 0ull;
    for (int w = 0; w < warp; ++w) {
        wy += ss.woffY[w];
        wq += ss.woffQ[w];
    }
    const unsigned long long yend = wy + iy, qend = wq + iq;  // through this slice
    const FastBound fb = fast_bound<EXACT>(ss.tot, s_row, u, f.ey, nch);
    const bool past = !a.force_precise && fb.ok && tid < NS &&
                      fast_cval(yend, qend, fb.M) > (long long)fb.tau;
    const unsigned bw = __ballot_sync(0xffffffffu, past);
    if (lane == 0) ds.red_f[warp] = bw ? (float)(__ffs(bw) - 1) : -1.0f;
    __syncthreads();
    int owner = -1;
    for (int w = 0; w < kWarps && owner < 0; ++w)
        if (ds.red_f[w] >= 0.0f) owner = w * 32 + (int)ds.red_f[w];
    if (tid == owner) {
        ss.Y0 = yend - mine.Y;
        ss.Q0 = qend - mine.Q;
    }
    __syncthreads();
    bool cert = false;
    int token = -1;
    if (owner >= 0) {  // uniform across the CTA
        const long long c0 = (long long)owner * a.SC;
        const DrawCtx<DT> d =
            slice_ctx<DT>(reinterpret_cast<unsigned char*>(rowblk + (c0 / kFastGroup) * 2), drow,
                          qrow, res, V, m, a.c2, u, c0, (int)min((long long)a.SC, nch - c0), s_row);
        if (res)
            fast_search<DT, true, EXACT, true>(ds, d, f, fb.M, fb.tau, ss.Y0, ss.Q0, fb.c);
        else
            fast_search<DT, false, EXACT, true>(ds, d, f, fb.M, fb.tau, ss.Y0, ss.Q0, fb.c);
        cert = ds.cert != 0 && ds.token >= 0;
        token = ds.token;
    }
    for (int i = tid; i <= k; i += kThreads)
        if (i != n) o[i] = i < n ? a.x[(long long)b * k + i] : -1;
    if (tid == 0) {
        if (cert) o[n] = token;
        a.nacc[b] = n;
        a.seqstat[b] = cert ? 0u : SV_DEV_PRECISE;
        commit_sequence(a.ep, b, n, k);
        if (!cert) {
            const uint32_t j = atomicAdd(a.plist_count, 1u);
            if (j < (uint32_t)a.B) {  // at most B entries
                a.parrive[j] = 0u;
                a.pambn[j] = 0u;
                // The precise pass classifies each element against q with this
                // normaliser: the fast pass's S (within e_S of the exact one)
                // when it is a positive number, else the row stream's.
                const bool sok = fb.S > 0.0f && fb.S < INFINITY;
                a.pS[j] = sok ? fb.S : s_row;
                a.pD[j] = sok ? 2.0f * fb.c.eS + 8.0f * 5.96046448e-08f : 1.0f / 2048.0f;
                a.plist[j] = (uint32_t)b;
            }
        }
    }
}

// ---- the split precise draw
//
// The draws the fast pass could not certify, each cut into slices of whole
// 64-element blocks spread over a persistent grid (as many slices per draw as
// the grid holds, so that the listed draws take one round).  Each slice's CTA
// forms e = exp((l - m)/T) in float-float for its elements and classifies each
// against q with the fast pass's normaliser S' (within e_S of the exact S):
// positive when e / S' > q (1 + delta), zero when e / S' < q (1 - delta) or q
// is not a non-negative number (such entries weigh 0), otherwise ambiguous
// (listed, with its e and q).  The weight max(0, e/S - q) of the positive
// elements is the linear form e/S - q, so as in the fast pass each chunk's
// positive e and q are summed (float-float, in element order) and turned into
// fixed point (Y in units 2^-EY, Q in 2^-62); the block sums go to the
// workspace, the slice's sums of Y, Q and S to its item record.  The last CTA
// of a draw (an arrival counter): S, M = floor(2^(123 - EY) / S), each listed
// element decided exactly (e/S - q > 0 in float-float) and added at its
// position, C = floor(Y M / 2^61) - Q, tau = floor(u C_tot), then the slice,
// block, chunk and element holding tau, recomputed where needed in the same
// arithmetic.  The token equals the exact-arithmetic one unless u C_tot lies
// within a few units of 2^-62 of a bin edge (float-float exponentials to about
// 2^-45, fixed-point sums exact).  A draw with more ambiguous elements than the
// list holds, an S beyond the margin of S', or a residual without mass takes
// the two-pass precise draw in that CTA alone (a zero-mass residual is drawn
// from p there, counted).
struct SplitPreciseArgs {
    const void* logits;
    const float* q;
    const float* ur;
    const RowRec* rows;
    const int32_t* nacc;
    const uint32_t* plist_count;
    const uint32_t* plist;
    uint32_t* parrive;            // [B] per list entry
    uint32_t* pambn;              // [B] per list entry
    const float* pS;              // [B]
    const float* pD;              // [B]
    AmbElem* amb;                 // [B][kAmbCap]
    PreciseItem* items;           // [max(kPreciseGrid, B)]
    unsigned long long* bsum;     // [B][row blocks][2] (the fast pass's array, reused)
    long long nbr;                // blocks per row
    uint32_t* seqstat;
    int32_t* out;
    int B, k, V;
    ff c2;
};

__device__ __forceinline__ void load_exp_table(float* thi, float* tlo) {
    for (int i = threadIdx.x; i < kExpTable; i += blockDim.x) {
        thi[i] = g_exp2_table.hi[i];
        tlo[i] = g_exp2_table.lo[i];
    }
    __syncthreads();
}

// Dynamic shared memory of the precise split kernel: the 2^(i/1024) table and
// the block sums of the two-pass fallback over a whole row.
__host__ __device__ inline size_t split_precise_smem_bytes(int V) {
    const long long nch = ((long long)V + kChunk - 1) / kChunk;
    return 2 * kExpTable * sizeof(float) +
           (size_t)((nch + kBlockChunks - 1) / kBlockChunks) * sizeof(unsigned long long);
}

// Classes of the precise pass.
constexpr int kPcZero = 0, kPcPos = 1, kPcAmb = 2;
struct PreciseCls {
    float inv;         // 1 / S' (rounded)
    float hi, lo;      // 1 + delta, 1 - delta
    int ey;
};
__device__ __forceinline__ int precise_class(ff e, float q, const PreciseCls& c, bool res) {
    if (!res) return kPcPos;
    if (!(q >= 0.0f) || e.hi == 0.0f) return kPcZero;  // NaN or negative q, or e = 0: weight 0
    const float r = __fmul_rn(e.hi, c.inv);
    if (r > __fmul_rn(q, c.hi)) return kPcPos;
    if (r < __fmul_rn(q, c.lo)) return kPcZero;
    return kPcAmb;
}

// One chunk of the precise pass: the fixed-point sums of its positive
// elements' e and q (not counting ambiguous ones); `es`, `cls` receive each
// element's e and class when not null; the chunk's e total goes into S.  (Not
// inlining it, so that a row's last CTA would find its chunk search's code in
// the instruction cache, made the slices' pass twice as slow: measured.)
template <typename DT>
__device__ __forceinline__ void precise_lin_chunk(const DrawCtx<DT>& d, int ci, const float* l,
                                                  const float* q, const PreciseCls& c, bool res,
                                                  ff& S, unsigned long long& cy,
                                                  unsigned long long& cq, ff* es, int* cls) {
    ff Y{0.0f, 0.0f}, Q{0.0f, 0.0f};
#pragma unroll
    for (int e = 0; e < kChunk; ++e) {
        const ff ev = exp_rel(l[e], d.m, d.c2, d.thi, d.tlo);
        ff_accumulate(S, ev);
        const int k = precise_class(ev, q[e], c, res);
        if (k == kPcPos) {
            ff_accumulate(Y, ev);
            if (res) ff_acc1(Q, q[e]);
        }
        if (es) {
            es[e] = ev;
            cls[e] = k;
        }
    }
    cy = ff_fixed(ff_normalize(Y), c.ey);
    cq = res ? ff_fixed(ff_normalize(Q), 62) : 0ull;
}

struct PreciseShared {
    AmbElem amb[kAmbCap];              // the listed elements, sorted by index
    unsigned long long ay[kAmbCap], aq[kAmbCap];  // their fixed-point y and q (0: not positive)
    unsigned long long ry[kWarps], rq[kWarps];
    ff rs[kWarps];
    unsigned long long Y, Q, Y0, Q0, bY, bQ, M, tau;
    ff S;
    int nb_amb, owner, blk, chunk, token, last, fallback;
};

// Sums of the listed positive elements with index in [lo, hi).
__device__ __forceinline__ void amb_in(const PreciseShared& ps, long long lo, long long hi,
                                       unsigned long long& y, unsigned long long& q) {
    for (int i = 0; i < ps.nb_amb; ++i)
        if (ps.amb[i].idx >= lo && ps.amb[i].idx < hi) {
            y += ps.ay[i];
            q += ps.aq[i];
        }
}

template <typename DT>
__global__ void __launch_bounds__(kThreads, 2) sv_split_precise_kernel(SplitPreciseArgs a) {
    extern __shared__ __align__(16) unsigned char dyn[];
    __shared__ DrawShared ds;
    __shared__ PreciseShared ps;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = lane / kFastGroup, gl = lane % kFastGroup;
    float* thi = reinterpret_cast<float*>(dyn);
    float* tlo = thi + kExpTable;
    load_exp_table(thi, tlo);  // (a constant table: read while the draw kernel ends)
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the list is complete
    const uint32_t cnt = min(*a.plist_count, (uint32_t)a.B);
    if (cnt == 0) return;
    const int P = gridDim.x;
    const long long nbr = a.nbr;
    const long long nch = ((long long)a.V + kChunk - 1) / kChunk;
    // Slices per draw: as many as the grid holds (whole blocks each).
    long long nsl = P / (long long)cnt;
    if (nsl < 1) nsl = 1;
    if (nsl > nbr) nsl = nbr;
    const long long slb = (nbr + nsl - 1) / nsl;  // blocks per slice
    nsl = (nbr + slb - 1) / slb;
    const long long items = (long long)cnt * nsl;
    if (blockIdx.x >= items) return;
    cg::cluster_group cluster = cg::this_cluster();
    const int k = a.k, V = a.V;
    for (long long it = blockIdx.x; it < items; it += P) {
        const int j = (int)(it / nsl), s = (int)(it % nsl);
        const int b = (int)a.plist[j];
        const int n = a.nacc[b];
        const bool res = n < k;
        const RowRec rec = a.rows[(long long)b * (k + 1) + n];
        const DT* drow = static_cast<const DT*>(a.logits) + ((long long)b * (k + 1) + n) * V;
        const float* qrow = res ? a.q + ((long long)b * k + n) * V : nullptr;
        unsigned long long* rowblk = a.bsum + (long long)b * nbr * 2;
        PreciseCls cl;
        const float Sc = a.pS[j], dl = a.pD[j];
        cl.inv = __frcp_rn(Sc);
        cl.hi = 1.0f + dl;
        cl.lo = 1.0f - dl;
        cl.ey = fast_ey(Sc);
        const float u = a.ur[b];
        // ---- the slice's pass
        {
            const long long c0 = (long long)s * slb * kFastGroup;
            DrawCtx<DT> d = slice_ctx<DT>(reinterpret_cast<unsigned char*>(rowblk + (c0 / kFastGroup) * 2),
                                          drow, qrow, res, V, rec.mraw, a.c2, u, c0,
                                          (int)min(slb * kFastGroup, nch - c0), rec.S);
            d.thi = thi;
            d.tlo = tlo;
            const int fnb = (d.mych + kFastGroup - 1) / kFastGroup;
            ff S{0.0f, 0.0f};
            unsigned long long Yt = 0ull, Qt = 0ull;
            for (int base = warp * 32; base < d.mych; base += kThreads) {
                const int ci = base + lane;
                unsigned long long cy = 0ull, cq = 0ull;
                if (ci < d.mych) {
                    float l[kChunk], q[kChunk] = {};
                    load_l(d, ci, l);
                    load_q(d, ci, res, q);
                    ff es[kChunk];
                    int cls[kChunk];
                    precise_lin_chunk<DT>(d, ci, l, q, cl, res, S, cy, cq, es, cls);
#pragma unroll
                    for (int e = 0; e < kChunk; ++e)
                        if (cls[e] == kPcAmb) {  // rare: list it
                            const uint32_t w = atomicAdd(a.pambn + j, 1u);
                            if (w < (uint32_t)kAmbCap) {
                                AmbElem ae;
                                ae.idx = (int)((d.c0 + ci) * kChunk + e);
                                ae.q = q[e];
                                ae.ehi = es[e].hi;
                                ae.elo = es[e].lo;
                                a.amb[(long long)j * kAmbCap + w] = ae;
                            }
                        }
                }
                Yt += cy;
                Qt += cq;
                const unsigned long long by = group_sum_u64(cy);
                const unsigned long long bq = group_sum_u64(cq);
                const int blk = (base + grp * kFastGroup) / kFastGroup;
                if (gl == 0 && blk < fnb)
                    reinterpret_cast<ulonglong2*>(d.bsum)[blk] = make_ulonglong2(by, bq);
            }
            // the slice's sums
            Yt = warp_sum(Yt);
            Qt = warp_sum(Qt);
            S = warp_sum_ff(ff_normalize(S));
            if (lane == 0) {
                ps.ry[warp] = Yt;
                ps.rq[warp] = Qt;
                ps.rs[warp] = S;
            }
            __syncthreads();
            if (tid == 0) {
                PreciseItem r;
                r.Y = 0ull;
                r.Q = 0ull;
                r.S = ff{0.0f, 0.0f};
                r.pad = 0ull;
                for (int w = 0; w < kWarps; ++w) {
                    r.Y += ps.ry[w];
                    r.Q += ps.rq[w];
                    r.S = ff_add(r.S, ps.rs[w]);
                }
                a.items[it] = r;
                __threadfence();
                ps.last = atomicAdd(a.parrive + j, 1u) == (uint32_t)(nsl - 1);
            }
            __syncthreads();
        }
        if (!ps.last) continue;

        // ---- the last slice of entry j: the token
        __threadfence();
        const long long ib = (long long)j * nsl;  // this entry's items: it - s .. + nsl
        const long long it0 = it - s;
        (void)ib;
        PreciseItem mine;
        mine.Y = 0ull;
        mine.Q = 0ull;
        mine.S = ff{0.0f, 0.0f};
        const uint32_t na = tid == 0 ? __ldcg(a.pambn + j) : 0u;  // (read with the items)
        if (tid < nsl) {
            const ulonglong2 v0 = __ldcg(reinterpret_cast<const ulonglong2*>(a.items + it0 + tid));
            const ulonglong2 v1 = __ldcg(reinterpret_cast<const ulonglong2*>(a.items + it0 + tid) + 1);
            mine.Y = v0.x;
            mine.Q = v0.y;
            mine.S = ff{__uint_as_float((uint32_t)v1.x), __uint_as_float((uint32_t)(v1.x >> 32))};
        }
        // S, Y, Q totals (a block reduction in a fixed order)
        {
            const unsigned long long y = warp_sum(mine.Y), q = warp_sum(mine.Q);
            const ff sw = warp_sum_ff(ff_normalize(mine.S));
            if (lane == 0) {
                ps.ry[warp] = y;
                ps.rq[warp] = q;
                ps.rs[warp] = sw;
            }
            __syncthreads();
            if (tid == 0) {
                unsigned long long Y = 0ull, Q = 0ull;
                ff St{0.0f, 0.0f};
                for (int w = 0; w < kWarps; ++w) {
                    Y += ps.ry[w];
                    Q += ps.rq[w];
                    St = ff_add(St, ps.rs[w]);
                }
                ps.Y = Y;
                ps.Q = Q;
                ps.S = ff_normalize(St);
                ps.nb_amb = (int)min(na, (uint32_t)kAmbCap);
                ps.fallback = na > (uint32_t)kAmbCap ||
                              !(fabsf(__fsub_rn(ps.S.hi, Sc)) <= 0.5f * dl * ps.S.hi);
                ps.token = -1;
            }
            __syncthreads();
        }
        const ff inv = ff_recip(ps.S);
        if (!ps.fallback && warp == 0) {
            // the listed elements: decided exactly, then sorted by index
            AmbElem ae;
            ae.idx = 0x7fffffff;
            ae.q = 0.0f;
            ae.ehi = 0.0f;
            ae.elo = 0.0f;
            if (lane < ps.nb_amb) {
                const uint4 v = __ldcg(reinterpret_cast<const uint4*>(a.amb + (long long)j * kAmbCap + lane));
                ae.idx = (int)v.x;
                ae.q = __uint_as_float(v.y);
                ae.ehi = __uint_as_float(v.z);
                ae.elo = __uint_as_float(v.w);
            }
            unsigned long long y = 0ull, qq = 0ull;
            if (lane < ps.nb_amb) {
                const ff e{ae.ehi, ae.elo};
                const ff pr = ff_mul(e, inv);
                const ff d = two_sum(pr.hi, -ae.q);
                const float w = __fadd_rn(d.hi, __fadd_rn(d.lo, pr.lo));
                if (w > 0.0f) {
                    y = ff_fixed(ff_normalize(e), cl.ey);
                    qq = fix_pow2(ae.q, 62);
                }
            }
            int rank = 0;
            for (int o = 0; o < ps.nb_amb; ++o) {
                const int oi = __shfl_sync(0xffffffffu, ae.idx, o);
                rank += (oi < ae.idx || (oi == ae.idx && o < lane)) ? 1 : 0;
            }
            if (lane < ps.nb_amb) {
                ps.amb[rank] = ae;
                ps.ay[rank] = y;
                ps.aq[rank] = qq;
            }
        }
        __syncthreads();
        if (!ps.fallback && tid == 0) {
            unsigned long long Y = ps.Y, Q = ps.Q;
            for (int i = 0; i < ps.nb_amb; ++i) {
                Y += ps.ay[i];
                Q += ps.aq[i];
            }
            ps.M = ff_fixed(inv, 123 - cl.ey);
            const long long Ctot = fast_cval(Y, Q, ps.M);
            if (Ctot <= 0) ps.fallback = 1;  // no mass: the two-pass draw, from p
            else ps.tau = scale_floor(u, (unsigned long long)Ctot);
            ps.owner = -1;
        }
        __syncthreads();
        bool degenerate = false;
        if (ps.fallback) {
            DrawCtx<DT> w = slice_ctx<DT>(dyn + 2 * kExpTable * sizeof(float), drow, qrow, res, V,
                                          rec.mraw, a.c2, u, 0, (int)nch, rec.S);
            w.thi = thi;
            w.tlo = tlo;
            if (tid == 0) ds.token = -1;
            __syncthreads();
            draw_precise<DT>(cluster, ds, w, degenerate);
            __syncthreads();
            if (tid == 0) ps.token = ds.token;
            __syncthreads();
        } else {
            const unsigned long long M = ps.M, tau = ps.tau;
            // Warp 0 alone from here (no block-wide barrier until the token):
            // the slice, then the block inside it, each a warp scan over
            // contiguous ranges (one per lane) and a walk of the first range
            // whose end passes tau; then the chunk and the element.
            int first = -1;
            if (warp == 0) {
                const long long Ls = (nsl + 31) / 32;
                const long long sb = min(nsl, (long long)lane * Ls), se = min(nsl, sb + Ls);
                const long long eps = slb * kFastGroup * kChunk;  // elements per slice
                unsigned long long sy = 0ull, sq = 0ull;
                for (long long i = sb; i < se; ++i) {
                    const ulonglong2 v = __ldcg(reinterpret_cast<const ulonglong2*>(a.items + it0 + i));
                    sy += v.x;
                    sq += v.y;
                }
                if (se > sb) amb_in(ps, sb * eps, se * eps, sy, sq);
                unsigned long long iy = sy, iq = sq;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const unsigned long long yo = __shfl_up_sync(0xffffffffu, iy, off);
                    const unsigned long long qo = __shfl_up_sync(0xffffffffu, iq, off);
                    if (lane >= off) {
                        iy += yo;
                        iq += qo;
                    }
                }
                const unsigned bs1 =
                    __ballot_sync(0xffffffffu, se > sb && fast_cval(iy, iq, M) > (long long)tau);
                const int fl = bs1 ? __ffs(bs1) - 1 : 0;
                long long own = -1;
                unsigned long long y0 = 0ull, q0 = 0ull;
                if (lane == fl && bs1) {
                    unsigned long long ry = iy - sy, rq = iq - sq;
                    long long i = sb;
                    for (; i < se - 1; ++i) {
                        const ulonglong2 v = __ldcg(reinterpret_cast<const ulonglong2*>(a.items + it0 + i));
                        unsigned long long y = v.x, q = v.y;
                        amb_in(ps, i * eps, (i + 1) * eps, y, q);
                        if (fast_cval(ry + y, rq + q, M) > (long long)tau) break;
                        ry += y;
                        rq += q;
                    }
                    own = i;
                    y0 = ry;
                    q0 = rq;
                }
                own = __shfl_sync(0xffffffffu, own, fl);
                y0 = __shfl_sync(0xffffffffu, y0, fl);
                q0 = __shfl_sync(0xffffffffu, q0, fl);
                if (bs1) {
                    // the block inside slice `own`
                    const long long b0 = own * slb;
                    const long long nbs = min(slb, nbr - b0);
                    const long long Lb = (nbs + 31) / 32;
                    const long long cb = min(nbs, (long long)lane * Lb), ce = min(nbs, cb + Lb);
                    const unsigned long long* bsp = rowblk + b0 * 2;
                    unsigned long long my = 0ull, mq = 0ull;
                    for (long long i = cb; i < ce; ++i) {
                        const ulonglong2 v = __ldcg(reinterpret_cast<const ulonglong2*>(bsp) + i);
                        my += v.x;
                        mq += v.y;
                    }
                    if (ce > cb) amb_in(ps, (b0 + cb) * 64, (b0 + ce) * 64, my, mq);
                    unsigned long long jy = my, jq = mq;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const unsigned long long yo = __shfl_up_sync(0xffffffffu, jy, off);
                        const unsigned long long qo = __shfl_up_sync(0xffffffffu, jq, off);
                        if (lane >= off) {
                            jy += yo;
                            jq += qo;
                        }
                    }
                    const bool bp = ce > cb && fast_cval(y0 + jy, q0 + jq, M) > (long long)tau;
                    const unsigned bb = __ballot_sync(0xffffffffu, bp);
                    first = bb ? __ffs(bb) - 1 : -1;
                    if (lane == first) {
                        unsigned long long ry = y0 + jy - my, rq = q0 + jq - mq;
                        long long i = cb;
                        for (; i < ce - 1; ++i) {
                            const ulonglong2 v = __ldcg(reinterpret_cast<const ulonglong2*>(bsp) + i);
                            unsigned long long y = v.x, q = v.y;
                            amb_in(ps, (b0 + i) * 64, (b0 + i + 1) * 64, y, q);
                            if (fast_cval(ry + y, rq + q, M) > (long long)tau) break;
                            ry += y;
                            rq += q;
                        }
                        ps.blk = (int)(b0 + i);
                        ps.bY = ry;
                        ps.bQ = rq;
                    }
                    __syncwarp();
                }
            }
            {
                if (first >= 0 && warp == 0) {
                    // the chunk: lanes 0..7 recompute the block's chunks
                    DrawCtx<DT> d = slice_ctx<DT>(dyn, drow, qrow, res, V, rec.mraw, a.c2, u, 0,
                                                  (int)nch, rec.S);
                    d.thi = thi;
                    d.tlo = tlo;
                    const int ci = ps.blk * kFastGroup + (lane & (kFastGroup - 1));
                    const bool have = lane < kFastGroup && ci < nch;
                    float l[kChunk] = {}, q[kChunk] = {};
                    ff es[kChunk];
                    int cls[kChunk];
                    ff Sd{0.0f, 0.0f};
                    unsigned long long cy = 0ull, cq = 0ull;
                    if (have) {
                        load_l(d, ci, l);
                        load_q(d, ci, res, q);
                        precise_lin_chunk<DT>(d, ci, l, q, cl, res, Sd, cy, cq, es, cls);
                        amb_in(ps, (long long)ci * kChunk, (long long)(ci + 1) * kChunk, cy, cq);
                    } else {
#pragma unroll
                        for (int e = 0; e < kChunk; ++e) {
                            es[e] = ff{0.0f, 0.0f};
                            cls[e] = kPcZero;
                        }
                    }
                    unsigned long long iy2 = cy, iq2 = cq;
#pragma unroll
                    for (int off = 1; off < kFastGroup; off <<= 1) {
                        const unsigned long long yo = __shfl_up_sync(0xffffffffu, iy2, off);
                        const unsigned long long qo = __shfl_up_sync(0xffffffffu, iq2, off);
                        if (lane >= off) {
                            iy2 += yo;
                            iq2 += qo;
                        }
                    }
                    const unsigned long long ly = ps.bY + iy2 - cy, lq = ps.bQ + iq2 - cq;
                    const bool lp = have && fast_cval(ly + cy, lq + cq, M) > (long long)tau;
                    const unsigned bl = __ballot_sync(0xffffffffu, lp);
                    // The element: lane e < 8 takes element e of the chunk of
                    // lane oc (its class, e and q shuffled from there) and forms
                    // the cumulative weight through e, in the pass's order; the
                    // first positive element past tau is the token.
                    const int oc = bl ? __ffs(bl) - 1 : 0;
                    ff ese[kChunk];
                    float qe[kChunk];
                    int ce[kChunk];
#pragma unroll
                    for (int j = 0; j < kChunk; ++j) {
                        ese[j] = ff{__shfl_sync(0xffffffffu, es[j].hi, oc),
                                    __shfl_sync(0xffffffffu, es[j].lo, oc)};
                        qe[j] = __shfl_sync(0xffffffffu, q[j], oc);
                        ce[j] = __shfl_sync(0xffffffffu, cls[j], oc);
                    }
                    const unsigned long long cly = __shfl_sync(0xffffffffu, ly, oc);
                    const unsigned long long clq = __shfl_sync(0xffffffffu, lq, oc);
                    const long long c8 = ((long long)ps.blk * kFastGroup + oc) * kChunk;
                    const int e = lane & (kChunk - 1);
                    ff Y{0.0f, 0.0f}, Q{0.0f, 0.0f};
                    bool pe = false;
#pragma unroll
                    for (int j = 0; j < kChunk; ++j) {
                        if (j <= e && ce[j] == kPcPos) {
                            ff_accumulate(Y, ese[j]);
                            if (res) ff_acc1(Q, qe[j]);
                        }
                        if (j == e) pe = ce[j] == kPcPos;
                    }
                    unsigned long long ea = 0ull, eq = 0ull;
                    amb_in(ps, c8, c8 + e + 1, ea, eq);
                    for (int i = 0; i < ps.nb_amb; ++i)
                        if (ps.amb[i].idx == c8 + e && ps.ay[i] > 0ull) pe = true;
                    const unsigned long long py = ff_fixed(ff_normalize(Y), cl.ey);
                    const unsigned long long pq = res ? ff_fixed(ff_normalize(Q), 62) : 0ull;
                    const bool hit = bl && lane < kChunk && pe &&
                                     fast_cval(cly + py + ea, clq + pq + eq, M) > (long long)tau;
                    const unsigned bh = __ballot_sync(0xffffffffu, hit);
                    if (lane == 0 && bh) ps.token = (int)(c8 + __ffs(bh) - 1);
                }
            }
            __syncthreads();
        }
        if (tid == 0) {
            if (ps.token >= 0) a.out[(long long)b * (k + 1) + n] = ps.token;
            if (degenerate) a.seqstat[b] = SV_DEV_PRECISE | SV_DEV_DEGENERATE;
            a.parrive[j] = 0u;
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------ sample-and-match

// Sample-and-match ("Decodificação especulativa explicada", §"A regra de
// amostragem por rejeição", the simpler exact scheme some engines use): a
// target token y_i is drawn from p_i at every position and the draft is kept
// while y_i == x_i; the first position where they differ (or position k)
// emits y_i.  Here every row's draw runs at once, one cluster per row, after
// the row stream has left each row's max and validity; out_tokens[b, i]
// receives y_i, and sv_finish_match_kernel then finds the first mismatch.
struct MatchArgs {
    const void* logits;
    const float* ua;   // u for the draw at positions 0..k-1
    const float* ur;   // u for the draw at position k
    const RowRec* rows;
    int32_t* out;
    int B, k, V, G;
    int draw_level, force_precise;
    float c;
    ff c2;
};

template <typename DT>
__global__ void __launch_bounds__(kThreads, 2) sv_match_draw_kernel(MatchArgs a) {
    extern __shared__ __align__(16) unsigned char dyn[];
    __shared__ DrawShared ds;
    __shared__ RowRec rec;
    __shared__ float s_u;
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x, G = a.G, k = a.k, V = a.V;
    const long long row = blockIdx.x / G;
    const int rank = blockIdx.x % G;
    const int b = (int)(row / (k + 1)), i = (int)(row % (k + 1));
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the row records are complete
    if (tid == 0) {
        rec = a.rows[row];
        s_u = i < k ? a.ua[(long long)b * k + i] : a.ur[b];
    }
    __syncthreads();
    // A bad row or uniform draws nothing (the finish kernel marks the sequence
    // if its scan reaches the row); every CTA of the cluster sees the same values.
    if ((rec.flags & (kRowBad | kRowSkipped)) || !(s_u >= 0.0f && s_u < 1.0f)) return;
    const DT* rowp = static_cast<const DT*>(a.logits) + row * (long long)V;
    const DrawCtx<DT> dc = make_draw_ctx<DT>(dyn, a.draw_level, rowp, nullptr,
                                             false, V, rec.mraw, a.c, a.c2, s_u, rank, G, rec.S);
    bool degenerate = false, fallback = false;
    draw<DT, true>(cluster, ds, dc, a.force_precise != 0, false, a.out + row, degenerate,
                   fallback);
}

// One warp per sequence: lanes test positions in parallel (a bad row, a bad
// draft token, a bad uniform, or the first y_i != x_i, or position k, ends the
// scan), in the order of the oracle's checks; then the outputs past n are -1.
__global__ void sv_finish_match_kernel(const int32_t* __restrict__ x,
                                       const float* __restrict__ ua,
                                       const float* __restrict__ ur,
                                       const RowRec* __restrict__ rows,
                                       uint32_t* __restrict__ seqstat, int B, int k, int V,
                                       int32_t* __restrict__ out, int32_t* __restrict__ nacc,
                                       Epilogue ep) {
    const int wi = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * 4 + wi;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the draws are complete
    if (b >= B) return;
    const RowRec* rr = rows + (long long)b * (k + 1);
    const int32_t* xx = x + (long long)b * k;
    int32_t* o = out + (long long)b * (k + 1);
    int first = k, code = 0;  // 1 emit, 2 bad row, 3 bad token, 4 bad uniform
    for (int base = 0; base <= k; base += 32) {
        const int i = base + lane;
        int c = 0;
        if (i <= k) {
            const float u = i < k ? ua[(long long)b * k + i] : ur[b];
            const int xi = i < k ? xx[i] : -1;
            if (rr[i].flags & (kRowBad | kRowSkipped)) c = 2;
            else if (i < k && (xi < 0 || xi >= V)) c = 3;
            else if (!(u >= 0.0f && u < 1.0f)) c = 4;
            else c = (i == k || o[i] != xi) ? 1 : 0;
        }
        const unsigned m = __ballot_sync(0xffffffffu, c != 0);
        if (m) {  // uniform across the warp
            const int src = __ffs(m) - 1;
            first = base + src;
            code = __shfl_sync(0xffffffffu, c, src);
            break;
        }
    }
    const bool bad = code != 1;
    const int n = first;
    __syncwarp();
    for (int i = lane; i <= k; i += 32)
        if (bad || i > n) o[i] = -1;
    if (lane == 0) {
        nacc[b] = bad ? -1 : n;
        seqstat[b] = code == 2 ? SV_DEV_BAD_ROW : code == 3 ? SV_DEV_BAD_TOKEN
                   : code == 4 ? SV_DEV_BAD_UNIFORM : 0u;
        commit_sequence(ep, b, bad ? -1 : n, k);
    }
}

// ------------------------------------------------------------------ n-gram drafter

// Prompt-lookup / n-gram drafting ("Decodificação especulativa explicada",
// §"A família de rascunhos": find the last tokens earlier in the context and
// propose what followed them there; "Speculative Decoding" (ch15), §"What
// proposes the tokens", the NgramDrafter).  Rule: for n = n_max down to n_min
// the last n tokens are looked for earlier in the history (an occurrence ends
// at e <= L - 2); the first n that occurs wins, and of its occurrences the most
// recent; the draft is the up to k tokens after it.
//
// One CTA per sequence.  The last n_max tokens sit in shared memory; each
// thread takes candidate end positions e (coalesced loads of h[e]) and extends
// the common suffix of h[..e] and h[..L-1] only while it matches.  The winner
// maximises (min(suffix, n_max), e): the longest n with an occurrence, then
// the most recent one, which is the rule above.
constexpr int kNgramThreads = 256;
constexpr int kNgramMaxN = 32;

__global__ void __launch_bounds__(kNgramThreads) sv_ngram_kernel(
    const int32_t* __restrict__ history, const int32_t* __restrict__ lengths, int Lmax, int k,
    int n_min, int n_max, int32_t* __restrict__ draft, int32_t* __restrict__ num) {
    __shared__ int32_t suf[kNgramMaxN];
    __shared__ unsigned long long red[kNgramThreads / 32];
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t* h = history + (long long)b * Lmax;
    int L = lengths[b];
    L = L < 0 ? 0 : (L > Lmax ? Lmax : L);
    for (int t = tid; t < n_max; t += kNgramThreads) suf[t] = t < L ? h[L - 1 - t] : -1;
    __syncthreads();
    unsigned long long best = 0;  // (match length << 32) | (e + 1); 0 = none
    // Eight candidates per thread in flight: their last tokens are loaded
    // together; only those equal to the history's last token extend the match.
    constexpr int U = 8;
    const int32_t last = suf[0];
    for (int base = L - 2 - tid; base >= 0; base -= U * kNgramThreads) {
        int32_t v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = base - u * kNgramThreads;
            v[u] = e >= 0 ? __ldg(h + e) : ~last;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = base - u * kNgramThreads;
            if (e >= 0 && v[u] == last) {
                int t = 1;
                const int tmax = min(n_max, e + 1);
                while (t < tmax && __ldg(h + e - t) == suf[t]) ++t;
                if (t >= n_min) {
                    const unsigned long long key =
                        ((unsigned long long)t << 32) | (unsigned)(e + 1);
                    best = key > best ? key : best;
                }
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
        best = o > best ? o : best;
    }
    if (lane == 0) red[warp] = best;
    __syncthreads();
    if (warp == 0) {
        best = lane < kNgramThreads / 32 ? red[lane] : 0ull;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
            best = o > best ? o : best;
        }
        const int e = best ? (int)(best & 0xFFFFFFFFull) - 1 : -1;
        const int cnt = e >= 0 ? min(k, L - 1 - e) : 0;
        for (int i = lane; i < k; i += 32)
            draft[(long long)b * k + i] = i < cnt ? h[e + 1 + i] : -1;
        if (lane == 0) num[b] = cnt;
    }
}

// ------------------------------------------------------------------ debug kernel

__global__ void sv_debug_ffexp_kernel(const float* l, float m, int n, ff c2, double* out) {
    __shared__ float thi[kExpTable], tlo[kExpTable];
    for (int t = threadIdx.x; t < kExpTable; t += blockDim.x) {
        thi[t] = g_exp2_table.hi[t];
        tlo[t] = g_exp2_table.lo[t];
    }
    __syncthreads();
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    ff e = exp_rel(l[i], m, c2, thi, tlo);
    out[i] = (double)e.hi + (double)e.lo;
}

// Worst relative error of ex2.approx over n consecutive negative-float bit
// patterns starting at b_lo, against the float-float exponential.
__global__ void sv_debug_ex2_kernel(uint32_t b_lo, unsigned long long n, float* out) {
    __shared__ float thi[kExpTable], tlo[kExpTable];
    for (int t = threadIdx.x; t < kExpTable; t += blockDim.x) {
        thi[t] = g_exp2_table.hi[t];
        tlo[t] = g_exp2_table.lo[t];
    }
    __syncthreads();
    float worst = 0.0f;
    const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
    for (unsigned long long i = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += stride) {
        const float a = __uint_as_float(b_lo + (uint32_t)i);
        const float y = ex2_approx(a);
        ff r = a >= kExp2Min ? exp2_ff(a, 0.0f, thi, tlo) : ff{0.0f, 0.0f};
        if (a < kExp2Min) {  // 2^a = 2^-64 * 2^(a + 64), both factors exact or in range
            ff t = exp2_ff(a + 64.0f, 0.0f, thi, tlo);
            r = ff{t.hi * 5.42101086e-20f, t.lo * 5.42101086e-20f};
        }
        const float err = fabsf((y - r.hi) - r.lo) / r.hi;
        worst = fmaxf(worst, err);
    }
    worst = fmaxf(worst, __shfl_xor_sync(0xffffffffu, worst, 16));
    worst = fmaxf(worst, __shfl_xor_sync(0xffffffffu, worst, 8));
    worst = fmaxf(worst, __shfl_xor_sync(0xffffffffu, worst, 4));
    worst = fmaxf(worst, __shfl_xor_sync(0xffffffffu, worst, 2));
    worst = fmaxf(worst, __shfl_xor_sync(0xffffffffu, worst, 1));
    if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<int*>(out), __float_as_int(worst));
}

// ------------------------------------------------------------------ host side

static ff log2e_over(float T) {
    const double v = 1.4426950408889634074 / (double)T;
    const float hi = (float)v;
    return ff{hi, (float)(v - (double)hi)};
}

// The options of one call (sv_tuning, specverify_debug.h): all zero, the
// automatic choices, for the entry points of specverify.h; the caller's for
// the _tuned entry points, so that a test's or a tuning script's setting
// affects its own calls only.
static const sv_tuning kAuto = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0};


struct DeviceInfo {
    int sms = 0;
    int clusters[5] = {0, 0, 0, 0, 0};  // resident clusters of 1, 2, 4, 8, 16 drawing CTAs
    bool ok = false;
    bool configured = false;
};
static std::mutex g_mu;
static DeviceInfo g_dev[64];

constexpr size_t kDynSmemMax = 160 * 1024;  // attribute of the kernels that draw

// Cache level of a draw with G CTAs per row: 2 (the precise pass keeps its
// exponentials) when that fits the budget, else 0.
static int draw_level(int V, int G) {
    return draw_smem_bytes(V, G, 2) <= kDrawSmemBudget ? 2 : 0;
}

template <typename K> static cudaError_t cluster_attrs(K kernel, bool dyn) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess && dyn)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kDynSmemMax);
    return e;
}

static cudaLaunchAttribute cluster_attr(int G) {
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = G;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    return at;
}

static sv_status device_setup(int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
    if (dev < 0 || dev >= 64) return SV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.configured) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SV_ERR_CUDA;
        d.ok = (major == 10 && minor == 3);
        if (d.ok) {
            cudaError_t e = cudaSuccess;
#define SV_TRY(x) if (e == cudaSuccess) e = (x)
            SV_TRY(cluster_attrs(sv_verify_kernel<__nv_bfloat16, true>, true));
            SV_TRY(cluster_attrs(sv_verify_kernel<float, true>, true));
            SV_TRY(cluster_attrs(sv_verify_kernel<__nv_bfloat16, false>, false));
            SV_TRY(cluster_attrs(sv_verify_kernel<float, false>, false));
            SV_TRY(cluster_attrs(sv_finish_sample_kernel<__nv_bfloat16, true>, true));
            SV_TRY(cluster_attrs(sv_finish_sample_kernel<float, true>, true));
            SV_TRY(cluster_attrs(sv_finish_sample_kernel<__nv_bfloat16, false>, true));
            SV_TRY(cluster_attrs(sv_finish_sample_kernel<float, false>, true));
            SV_TRY(cluster_attrs(sv_precise_kernel<__nv_bfloat16>, true));
            SV_TRY(cluster_attrs(sv_match_draw_kernel<__nv_bfloat16>, true));
            SV_TRY(cluster_attrs(sv_match_draw_kernel<float>, true));
            SV_TRY(cluster_attrs(sv_precise_kernel<float>, true));
            SV_TRY(cluster_attrs(sv_split_precise_kernel<__nv_bfloat16>, true));
            SV_TRY(cluster_attrs(sv_split_precise_kernel<float>, true));
            SV_TRY(cluster_attrs(sv_rows_kernel<__nv_bfloat16, true, 128>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<__nv_bfloat16, true, 256>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<__nv_bfloat16, true, 512>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<__nv_bfloat16, true, 1024>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<__nv_bfloat16, false, 128>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<__nv_bfloat16, false, 256>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<__nv_bfloat16, false, 512>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<__nv_bfloat16, false, 1024>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<float, true, 128>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<float, true, 256>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<float, true, 512>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<float, true, 1024>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<float, false, 128>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<float, false, 256>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<float, false, 512>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<float, false, 1024>, false));
            SV_TRY(cudaFuncSetAttribute(sv_tree_kernel<__nv_bfloat16, true>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)tree_bsum_bytes(kMaxV)));
            SV_TRY(cudaFuncSetAttribute(sv_tree_kernel<float, true>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)tree_bsum_bytes(kMaxV)));
#undef SV_TRY
            if (e != cudaSuccess) return SV_ERR_CUDA;
            // How many clusters of the drawing kernel fit at once, per cluster
            // size, at the largest shared memory a draw uses.
            for (int lg = 0; lg < 5; ++lg) {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(1u << lg, 1, 1);
                cfg.blockDim = dim3(kThreads, 1, 1);
                cfg.dynamicSmemBytes = kDrawSmemBudget;
                cudaLaunchAttribute at = cluster_attr(1 << lg);
                cfg.attrs = &at;
                cfg.numAttrs = 1;
                int n = 0;
                if (cudaOccupancyMaxActiveClusters(&n, sv_finish_sample_kernel<__nv_bfloat16, true>,
                                                   &cfg) != cudaSuccess)
                    n = 0;
                d.clusters[lg] = n;
            }
            (void)cudaGetLastError();
        }
        d.configured = true;
    }
    if (!d.ok) return SV_ERR_UNSUPPORTED;
    *sms = d.sms;
    return SV_OK;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

static sv_status check_common(const void* logits, sv_dtype dt, const int32_t* x, int B, int k,
                              int V, void* ws, size_t ws_bytes, bool base_ws = false) {
    if (dt != SV_BF16 && dt != SV_F32) return SV_ERR_INVALID_ARG;
    if (B < 0 || k < 1 || V < 1) return SV_ERR_INVALID_ARG;
    if (k > kMaxK || V > kMaxV) return SV_ERR_UNSUPPORTED;
    if ((long double)B * (k + 1) * V >= (long double)(1ll << 40)) return SV_ERR_UNSUPPORTED;
    if ((long long)B * (k + 1) * 16 >= (1ll << 31)) return SV_ERR_UNSUPPORTED;  // grid size
    if (B > 0 && (!logits || !x)) return SV_ERR_INVALID_ARG;
    if (B > 0 && (!aligned16(logits) || !aligned16(x))) return SV_ERR_INVALID_ARG;
    if (!ws) return SV_ERR_WORKSPACE;
    if (!aligned16(ws)) return SV_ERR_INVALID_ARG;
    if (ws_bytes < (base_ws ? ws_base_bytes(B, k) : ws_bytes_for(B, k, V))) return SV_ERR_WORKSPACE;
    return SV_OK;
}

static sv_status check_outputs(const int32_t* out, const int32_t* nacc, int B) {
    if (B > 0 && (!out || !nacc)) return SV_ERR_INVALID_ARG;
    if (B > 0 && (!aligned16(out) || !aligned16(nacc))) return SV_ERR_INVALID_ARG;
    return SV_OK;
}

static sv_status check_sample(const float* q, const float* ua, const float* ur, float T, int B) {
    if (!(T > 0.0f) || !std::isfinite(T)) return SV_ERR_INVALID_ARG;
    if (B > 0 && (!q || !ua || !ur)) return SV_ERR_INVALID_ARG;
    if (B > 0 && (!aligned16(q) || !aligned16(ua) || !aligned16(ur))) return SV_ERR_INVALID_ARG;
    return SV_OK;
}

// Resident clusters of G drawing CTAs on the current device (0 if unknown).
static int resident_clusters(int G) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int lg = 0;
    while ((1 << lg) < G && lg < 4) ++lg;
    std::lock_guard<std::mutex> lk(g_mu);
    return g_dev[dev].clusters[lg];
}

// Cluster size of the per-sequence kernels.  Sampled: the whole batch resident
// at once (B clusters of G CTAs, as the occupancy query counts them, else two
// 512-thread CTAs per SM), but no CTA draws from more than kSliceMax elements
// of a row and none from fewer than 2048.
// Greedy: enough CTAs to give each SM four, with at least 4 KiB of every row
// per CTA.
static int seq_split(bool sampled, int B, int V, int esz, int sms) {
    int G = 1;
    if (sampled) {
        while (G < 16 && (V + G - 1) / G > kSliceMax) G *= 2;
        while (G < 16 && V / (2 * G) >= 2048) {
            const int rc = resident_clusters(2 * G);
            if (rc > 0 ? B > rc : (long long)B * 2 * G > 2LL * sms) break;
            G *= 2;
        }
    } else {
        while (G < 16 && (long long)B * G < 4LL * sms && (long long)V * esz / (2LL * G) >= 4096)
            G *= 2;
    }
    return G;
}

// Rows per wave of the fused kernel.  One wave costs about one HBM round trip
// whatever its size, so a wave should carry enough bytes across the batch to
// cover the bandwidth-latency product (taken as 32 MiB); beyond that, waves of
// one row stop at the first rejection and never read the later rows.
static int wave_rows(int B, int k, int V, int esz) {
    const double wave_bytes = (double)B * V * esz;
    int W = (int)std::ceil((32.0 * 1024 * 1024) / (wave_bytes > 1.0 ? wave_bytes : 1.0));
    if (W < 1) W = 1;
    if (W > k + 1) W = k + 1;
    return W > kWarps ? kWarps : W;
}

// The precise draws listed by a draw kernel of a large batch (plist_count and
// plist in the workspace): persistent 16-CTA clusters, launched as a
// programmatic dependent of that kernel.
// Cluster size of sv_precise_kernel (sv_tuning.precise_split overrides it).
// Four CTAs per draw:
// each draw's chain of barriers and single-warp search costs about the same at
// any size, so more clusters at once (76 of 4 against 14 of 16 on GB300)
// finish a batch's precise draws sooner (measured on B=256, V=151936: the
// draws take 157 us with clusters of 4, 192 us with 16, 172 with 8).
constexpr int kPreciseG = 4;

static sv_status launch_precise(const void* logits, sv_dtype dt, const float* q, const float* ur,
                                const RowRec* rows, const int32_t* nacc,
                                const uint32_t* plist_count, const uint32_t* plist,
                                uint32_t* seqstat, int32_t* out, int B, int k, int V, float c,
                                ff c2, cudaStream_t stream, const sv_tuning& tu) {
    cudaError_t e;
    cudaLaunchAttribute pdl;
    pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl.val.programmaticStreamSerializationAllowed = 1;
    PreciseArgs pa;
    pa.logits = logits;
    pa.q = q;
    pa.ur = ur;
    pa.rows = rows;
    pa.nacc = nacc;
    pa.plist_count = plist_count;
    pa.plist = plist;
    pa.seqstat = seqstat;
    pa.out = out;
    pa.B = B;
    pa.k = k;
    pa.V = V;
    pa.G = tu.precise_split ? tu.precise_split : kPreciseG;
    pa.draw_level = draw_level(V, pa.G);
    pa.c = c;
    pa.c2 = c2;
    const size_t psmem = draw_smem_bytes(V, pa.G, pa.draw_level);
    if (psmem > kDynSmemMax) return SV_ERR_UNSUPPORTED;
    int ncl = resident_clusters(pa.G);
    if (ncl <= 0) ncl = 8;
    if (ncl > B) ncl = B;
    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3((unsigned)(ncl * pa.G), 1, 1);
    pc.blockDim = dim3(kThreads, 1, 1);
    pc.dynamicSmemBytes = psmem;
    pc.stream = stream;
    cudaLaunchAttribute pattr[2] = {cluster_attr(pa.G), pdl};
    pc.attrs = pattr;
    pc.numAttrs = 2;
    e = dt == SV_BF16 ? cudaLaunchKernelEx(&pc, sv_precise_kernel<__nv_bfloat16>, pa)
                      : cudaLaunchKernelEx(&pc, sv_precise_kernel<float>, pa);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

static sv_status launch_fused(bool sampled, const void* logits, sv_dtype dt, const float* q,
                              const int32_t* x, const float* ua, const float* ur, float T, int B,
                              int k, int V, int32_t* out, int32_t* nacc, void* ws,
                              cudaStream_t stream, int sms, Epilogue ep, const sv_tuning& tu) {
    VerifyArgs a;
    a.ep = ep;
    a.logits = logits;
    a.q = q;
    a.x = x;
    a.ua = ua;
    a.ur = ur;
    a.hdr = static_cast<Header*>(ws);
    a.rows = reinterpret_cast<RowRec*>(static_cast<char*>(ws) + ws_rows_offset());
    a.seqstat = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + ws_seq_offset(B, k));
    a.out = out;
    a.nacc = nacc;
    a.B = B;
    a.k = k;
    a.V = V;
    const int esz = dt == SV_BF16 ? 2 : 4;
    a.G = seq_split(sampled, B, V, esz, sms);
    a.W = wave_rows(B, k, V, esz);
    a.c2 = log2e_over(sampled ? T : 1.0f);
    a.c = a.c2.hi;
    a.force_precise = tu.force_precise != 0;
    a.plist_count = nullptr;
    a.plist = nullptr;
    size_t smem = 0;
    a.draw_level = 0;
    // Large sampled batches defer the precise draws to sv_precise_kernel.
    const int dmode = tu.fused_defer;
    const bool defer = sampled && (dmode == 1 || (dmode == 0 && B >= sms));
    if (sampled) {
        a.draw_level = draw_level(V, a.G);
        smem = draw_smem_bytes(V, a.G, a.draw_level);
        if (const int pad = tu.fused_pad_kib) smem = std::max(smem, (size_t)pad * 1024);
        if (smem > kDynSmemMax) return SV_ERR_UNSUPPORTED;
        if (defer) {
            a.plist_count =
                reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + ws_plist_offset(B, k));
            a.plist = a.plist_count + 4;
            if (cudaMemsetAsync(a.plist_count, 0, 16, stream) != cudaSuccess) return SV_ERR_CUDA;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((long long)B * a.G), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {cluster_attr(a.G)};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (dt == SV_BF16)
        e = sampled ? cudaLaunchKernelEx(&cfg, sv_verify_kernel<__nv_bfloat16, true>, a)
                    : cudaLaunchKernelEx(&cfg, sv_verify_kernel<__nv_bfloat16, false>, a);
    else
        e = sampled ? cudaLaunchKernelEx(&cfg, sv_verify_kernel<float, true>, a)
                    : cudaLaunchKernelEx(&cfg, sv_verify_kernel<float, false>, a);
    if (e != cudaSuccess) return SV_ERR_CUDA;
    if (!defer) return SV_OK;
    return launch_precise(logits, dt, q, ur, a.rows, nacc, a.plist_count, a.plist, a.seqstat, out,
                          B, k, V, a.c, a.c2, stream, tu);
}

// Vocabulary split of the per-row kernel: rows are split over a cluster only
// while there are fewer than two CTAs per SM (the cluster barriers and the
// DSMEM merge cost more than the imbalance of whole rows beyond that), and each
// CTA keeps at least 512 16-byte vectors (8 KiB) of its row.
static int rows_split(long long R, long long nvec_row, int sms) {
    int G = 1;
    while (G < 16 && R * G < 2LL * sms && nvec_row / (2LL * G) >= 512) G *= 2;
    return G;
}

// Threads per CTA: at least two vectors per thread, and the whole grid resident
// at once when it can be (2048 threads per SM), so that no wave tail forms.
static int rows_threads(long long ctas, long long nvec_cta, int sms) {
    int t = 512;
    while (t > 128 && (nvec_cta < 2LL * t || ctas * t > 2048LL * sms)) t /= 2;
    return t;
}

// With `skip`: one 512-thread CTA per row, rows position-major, stop[] reset
// first (a memset on the same stream).  sv_tuning.rows_split / rows_threads
// fix the split and thread count of the two-kernel path's stream (which also
// keeps greedy batches off the flat stream, as sv_tuning.flat_off does).

// Plan of the flat greedy stream: P ranges, one per resident CTA (two per SM)
// and at least one per SM, each at least a third of a row long (a row meets at
// most kFlatSlots ranges) and at most three rows long (a range meets at most
// kFlatSlots rows).  Rows must be whole 16-byte vectors of an aligned tensor.
static bool flat_plan(int B, int k, int V, int esz, const void* logits, int sms, FlatArgs* f) {
    if (((long long)V * esz) % 16 != 0 || (reinterpret_cast<uintptr_t>(logits) & 15) != 0)
        return false;
    const long long w = (long long)V * esz / 16;
    const long long n = (long long)B * (k + 1) * w;
    if (n >= (1LL << 31)) return false;
    const long long p = std::min<long long>(2LL * sms, n / ((w + 2) / 3));
    if (p < sms || (n + p - 1) / p > 3 * w) return false;
    f->P = (int)p;
    f->vpr = (int)w;
    f->per = (int)(n / p);
    f->rem = (int)(n % p);
    return true;
}

// `flat_ok`: a greedy stream may leave the flat layout (only the greedy finish
// kernel reads it).
static sv_status launch_rows(bool sampled, const void* logits, sv_dtype dt, const float* q,
                             const int32_t* x, const float* ua, float T, int B, int k, int V,
                             void* ws, cudaStream_t stream, int sms, bool skip,
                             const sv_tuning& tu, bool flat_ok = true, bool full_ws = false,
                             bool zero_split = false) {
    const long long R = (long long)B * (k + 1);
    RowsArgs a;
    a.logits = logits;
    a.q = q;
    a.x = x;
    a.ua = ua;
    a.hdr = static_cast<Header*>(ws);
    a.rows = reinterpret_cast<RowRec*>(static_cast<char*>(ws) + ws_rows_offset());
    a.stop = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + ws_stop_offset(B, k));
    a.skip = skip ? 1 : 0;
    // With zero_split the split draw that follows finds its list counter, list
    // and arrival counters cleared by this launch (so it needs no memset).
    a.zero = zero_split ? reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + ws_plist_offset(B, k))
                        : nullptr;
    a.nzero = zero_split ? (int)((ws_split_offset(B, k) - ws_plist_offset(B, k)) / 4 + B) : 0;
    a.B = B;
    a.k = k;
    a.V = V;
    a.mode = sampled ? SV_MODE_SAMPLE : SV_MODE_GREEDY;
    a.c2 = log2e_over(sampled ? T : 1.0f);
    a.c = a.c2.hi;
    const int esz = dt == SV_BF16 ? 2 : 4;
    FlatArgs f;
    if (!sampled && !skip && flat_ok && !tu.flat_off && !tu.rows_split && !tu.rows_threads &&
        flat_plan(B, k, V, esz, logits, sms, &f)) {
        f.logits = logits;
        f.rows = a.rows;
        f.hdr = a.hdr;
        f.B = B;
        f.k = k;
        f.V = V;
        cudaLaunchConfig_t fc = {};
        fc.gridDim = dim3((unsigned)f.P, 1, 1);
        fc.blockDim = dim3(kFlatThreads, 1, 1);
        fc.stream = stream;
        cudaLaunchAttribute pdl;
        pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pdl.val.programmaticStreamSerializationAllowed = 1;
        fc.attrs = &pdl;
        fc.numAttrs = 1;
        const cudaError_t fe = dt == SV_BF16
                                   ? cudaLaunchKernelEx(&fc, sv_flat_greedy_kernel<__nv_bfloat16>, f)
                                   : cudaLaunchKernelEx(&fc, sv_flat_greedy_kernel<float>, f);
        return fe == cudaSuccess ? SV_OK : SV_ERR_CUDA;
    }
    const long long nvec_row = ((long long)V * esz + 15) / 16;
    a.G = skip ? 1 : rows_split(R, nvec_row, sms);
    int nt = skip ? 512 : rows_threads(R * a.G, nvec_row / a.G, sms);
    if (!skip && tu.rows_split) a.G = tu.rows_split;
    if (tu.rows_threads) nt = tu.rows_threads;
    if (skip && cudaMemsetAsync(a.stop, 0xFF, (size_t)B * sizeof(uint32_t), stream) != cudaSuccess)
        return SV_ERR_CUDA;
    // The row-skipping stream with rows cut into G CTAs (a full workspace only;
    // a tuning option: on B = 256, k = 8, V = 151936 fp32, 4 CTAs per row took
    // 36 us longer than one, the many short CTAs costing more than the earlier
    // decisions save).
    const int gs = tu.rows_split ? std::min(tu.rows_split, kRowSplitMax) : 1;
    if (skip && full_ws && gs > 1) {
        a.G = gs;
        char* w = static_cast<char*>(ws);
        RowSplitArgs rs;
        const size_t ro = ws_rowsplit_offset(B, k, V);
        rs.rowcnt = reinterpret_cast<uint32_t*>(w + ro);
        rs.parts = reinterpret_cast<RowPart*>(w + ro + ((R * 4 + 15) & ~15ll));
        rs.gath = reinterpret_cast<RowGather*>(reinterpret_cast<char*>(rs.parts) + R * 8 * 16);
        if (cudaMemsetAsync(rs.rowcnt, 0, (size_t)R * 4, stream) != cudaSuccess) return SV_ERR_CUDA;
        cudaLaunchConfig_t sc = {};
        sc.gridDim = dim3((unsigned)(R * gs), 1, 1);
        sc.blockDim = dim3(512, 1, 1);
        sc.stream = stream;
        cudaError_t se;
        if (dt == SV_BF16)
            se = sampled ? cudaLaunchKernelEx(&sc, sv_rows_skip_kernel<__nv_bfloat16, true>, a, rs)
                         : cudaLaunchKernelEx(&sc, sv_rows_skip_kernel<__nv_bfloat16, false>, a, rs);
        else
            se = sampled ? cudaLaunchKernelEx(&sc, sv_rows_skip_kernel<float, true>, a, rs)
                         : cudaLaunchKernelEx(&sc, sv_rows_skip_kernel<float, false>, a, rs);
        return se == cudaSuccess ? SV_OK : SV_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(R * a.G), 1, 1);
    cfg.blockDim = dim3(nt, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {cluster_attr(a.G)};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
#define SV_ROWS(DTY, S)                                                          \
    e = nt == 1024  ? cudaLaunchKernelEx(&cfg, sv_rows_kernel<DTY, S, 1024>, a)    \
        : nt == 512 ? cudaLaunchKernelEx(&cfg, sv_rows_kernel<DTY, S, 512>, a)     \
        : nt == 256 ? cudaLaunchKernelEx(&cfg, sv_rows_kernel<DTY, S, 256>, a)     \
                    : cudaLaunchKernelEx(&cfg, sv_rows_kernel<DTY, S, 128>, a)
    if (dt == SV_BF16) {
        if (sampled) SV_ROWS(__nv_bfloat16, true);
        else SV_ROWS(__nv_bfloat16, false);
    } else {
        if (sampled) SV_ROWS(float, true);
        else SV_ROWS(float, false);
    }
#undef SV_ROWS
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}


// Cluster size of the draw kernel of a large batch (B >= SMs): one CTA per
// sequence (no cluster barriers, every CTA resident at once, the scheduler
// starting each as a slot frees), unless a row exceeds the largest slice one
// CTA draws from.  The precise draws go to sv_precise_kernel's 16-CTA clusters.
static int draw_split_wide(int B, int V, int sms) {
    (void)B;
    (void)sms;
    int G = 1;
    while (G < 16 && (V + G - 1) / G > kSliceMax) G *= 2;
    return G;
}

// The split draw of a sampled verify: a memset of the list's counter and the
// arrival counters, sv_split_draw_kernel (B * NS CTAs), then the precise launch
// (persistent, 2 CTAs per SM, a programmatic dependent; it returns at once when
// no draw was listed).
static sv_status launch_split(const void* logits, sv_dtype dt, const float* q, const int32_t* x,
                              const float* ua, const float* ur, float T, int B, int k, int V,
                              int32_t* out, int32_t* nacc, void* ws, cudaStream_t stream, int sms,
                              Epilogue ep, const sv_tuning& tu, bool zeroed) {
    char* w = static_cast<char*>(ws);
    SplitArgs a;
    a.logits = logits;
    a.q = q;
    a.x = x;
    a.ua = ua;
    a.ur = ur;
    a.rows = reinterpret_cast<const RowRec*>(w + ws_rows_offset());
    a.seqstat = reinterpret_cast<uint32_t*>(w + ws_seq_offset(B, k));
    a.out = out;
    a.nacc = nacc;
    a.plist_count = reinterpret_cast<uint32_t*>(w + ws_plist_offset(B, k));
    a.plist = a.plist_count + 4;
    const size_t so = ws_split_offset(B, k);
    const SplitLayout lay = split_layout(B, V);
    a.arrive = reinterpret_cast<uint32_t*>(w + so);
    a.parrive = reinterpret_cast<uint32_t*>(w + so + lay.parrive);
    a.pambn = reinterpret_cast<uint32_t*>(w + so + lay.pambn);
    a.pS = reinterpret_cast<float*>(w + so + lay.pS);
    a.pD = reinterpret_cast<float*>(w + so + lay.pD);
    a.srec = reinterpret_cast<FastTotals*>(w + so + lay.srec);
    a.bsum = reinterpret_cast<unsigned long long*>(w + so + lay.bsum);
    a.nbr = split_row_blocks(V);
    a.ep = ep;
    a.B = B;
    a.k = k;
    a.V = V;
    a.NS = split_slices(B, V, &a.SC);
    if (tu.draw_split && tu.draw_split < a.NS) {  // fewer, longer slices (tuning)
        const long long nch = ((long long)V + kChunk - 1) / kChunk;
        long long c = (nch + tu.draw_split - 1) / tu.draw_split;
        c = (c + kFastGroup - 1) / kFastGroup * kFastGroup;
        a.SC = (int)c;
        a.NS = (int)((nch + c - 1) / c);
    }
    a.force_precise = tu.force_precise != 0;
    a.c2 = log2e_over(T);
    // The list's counter, its entries and the arrival counters: cleared by the
    // row stream just before (`zeroed`: then this launch is its programmatic
    // dependent), else here in one memset.
    cudaLaunchAttribute dep;
    dep.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    dep.val.programmaticStreamSerializationAllowed = 1;
    if (!zeroed) {
        const size_t zlen =
            ws_split_offset(B, k) + (size_t)B * sizeof(uint32_t) - ws_plist_offset(B, k);
        if (cudaMemsetAsync(a.plist_count, 0, zlen, stream) != cudaSuccess) return SV_ERR_CUDA;
    }
    cudaError_t e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((long long)B * a.NS), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = stream;
    cfg.attrs = &dep;
    cfg.numAttrs = zeroed ? 1 : 0;
    // float-float chunk sums (a tighter bound, fewer precise draws) on small
    // batches, whose draws are latency; pairwise on large ones, whose fast pass
    // is instruction-bound
    if (B < sms)
        e = dt == SV_BF16 ? cudaLaunchKernelEx(&cfg, sv_split_draw_kernel<__nv_bfloat16, true>, a)
                          : cudaLaunchKernelEx(&cfg, sv_split_draw_kernel<float, true>, a);
    else
        e = dt == SV_BF16 ? cudaLaunchKernelEx(&cfg, sv_split_draw_kernel<__nv_bfloat16, false>, a)
                          : cudaLaunchKernelEx(&cfg, sv_split_draw_kernel<float, false>, a);
    if (e != cudaSuccess) return SV_ERR_CUDA;

    SplitPreciseArgs pa;
    pa.logits = logits;
    pa.q = q;
    pa.ur = ur;
    pa.rows = a.rows;
    pa.nacc = nacc;
    pa.plist_count = a.plist_count;
    pa.plist = a.plist;
    pa.parrive = a.parrive;
    pa.pambn = a.pambn;
    pa.pS = a.pS;
    pa.pD = a.pD;
    pa.amb = reinterpret_cast<AmbElem*>(w + so + lay.amb);
    pa.items = reinterpret_cast<PreciseItem*>(w + so + lay.items);
    pa.bsum = a.bsum;
    pa.nbr = a.nbr;
    pa.seqstat = a.seqstat;
    pa.out = out;
    pa.B = B;
    pa.k = k;
    pa.V = V;
    pa.c2 = a.c2;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1] = cluster_attr(1);
    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3((unsigned)std::min(2 * sms, kPreciseGrid), 1, 1);
    pc.blockDim = dim3(kThreads, 1, 1);
    pc.dynamicSmemBytes = split_precise_smem_bytes(V);
    pc.stream = stream;
    pc.attrs = attr;
    pc.numAttrs = 2;
    e = dt == SV_BF16 ? cudaLaunchKernelEx(&pc, sv_split_precise_kernel<__nv_bfloat16>, pa)
                      : cudaLaunchKernelEx(&pc, sv_split_precise_kernel<float>, pa);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// The split draw (automatic, or when asked for) if the workspace has its
// region; the cluster draw with draw_mode 2.  Measured on B = 256, k = 8,
// V = 151936 fp32 (222.9 against 242 us per verify) and B = 1, k = 8,
// V = 256000 bf16 (19.3 against 21.4 us).
static bool uses_split(const sv_tuning& tu, bool wide, int B, int V) {
    (void)wide;
    return tu.draw_mode != 2 && split_fits(B, V);
}

// `wide`: the draw kernel of a large batch (draw_split_wide), else seq_split.
static sv_status launch_finish(bool sampled, const void* logits, sv_dtype dt, const float* q,
                               const int32_t* x, const float* ua, const float* ur, float T,
                               int B, int k, int V, int32_t* out, int32_t* nacc, void* ws,
                               cudaStream_t stream, int sms, bool wide, Epilogue ep,
                               const sv_tuning& tu, bool split_zeroed = false) {
    const RowRec* rows =
        reinterpret_cast<const RowRec*>(static_cast<char*>(ws) + ws_rows_offset());
    uint32_t* seqstat = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + ws_seq_offset(B, k));
    cudaError_t e;
    cudaLaunchAttribute pdl;
    pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl.val.programmaticStreamSerializationAllowed = 1;
    if (!sampled) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)((B + 3) / 4), 1, 1);
        cfg.blockDim = dim3(128, 1, 1);
        cfg.stream = stream;
        cfg.attrs = &pdl;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, sv_finish_greedy_kernel, x, rows,
                               static_cast<const Header*>(ws), seqstat, B, k, out, nacc,
                               ep);
        return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
    }
    if (uses_split(tu, wide, B, V))
        return launch_split(logits, dt, q, x, ua, ur, T, B, k, V, out, nacc, ws, stream, sms, ep,
                            tu, split_zeroed);
    FinishArgs a;
    a.ep = ep;
    a.logits = logits;
    a.q = q;
    a.x = x;
    a.ua = ua;
    a.ur = ur;
    a.rows = rows;
    a.seqstat = seqstat;
    a.out = out;
    a.nacc = nacc;
    a.B = B;
    a.k = k;
    a.V = V;
    a.G = wide ? draw_split_wide(B, V, sms) : seq_split(true, B, V, dt == SV_BF16 ? 2 : 4, sms);
    if (const int fg = tu.draw_split) a.G = fg;
    a.c2 = log2e_over(T);
    a.c = a.c2.hi;
    a.force_precise = tu.force_precise != 0;
    a.draw_level = draw_level(V, a.G);
    a.plist_count = nullptr;
    a.plist = nullptr;
    const size_t smem = draw_smem_bytes(V, a.G, a.draw_level);
    if (smem > kDynSmemMax) return SV_ERR_UNSUPPORTED;
    // Large batches: the precise draws go to sv_precise_kernel through a list
    // whose counter is reset here (so this kernel follows a memset, not the row
    // stream, and is launched without the programmatic dependency).
    if (wide) {
        a.plist_count = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + ws_plist_offset(B, k));
        a.plist = a.plist_count + 4;
        if (cudaMemsetAsync(a.plist_count, 0, 16, stream) != cudaSuccess) return SV_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((long long)B * a.G), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2] = {cluster_attr(a.G), pdl};
    cfg.attrs = attr;
    cfg.numAttrs = wide ? 1 : 2;
    if (wide)  // large batches: the cheaper fast pass (its precise draws are deferred)
        e = dt == SV_BF16 ? cudaLaunchKernelEx(&cfg, sv_finish_sample_kernel<__nv_bfloat16, false>, a)
                          : cudaLaunchKernelEx(&cfg, sv_finish_sample_kernel<float, false>, a);
    else
        e = dt == SV_BF16 ? cudaLaunchKernelEx(&cfg, sv_finish_sample_kernel<__nv_bfloat16, true>, a)
                          : cudaLaunchKernelEx(&cfg, sv_finish_sample_kernel<float, true>, a);
    if (e != cudaSuccess || !wide) return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;

    return launch_precise(logits, dt, q, ur, rows, nacc, a.plist_count, a.plist, seqstat, out, B,
                          k, V, a.c, a.c2, stream, tu);
}

// Sample-and-match: the row stream (greedy statistics: max, argmax, validity),
// one draw per row (a cluster of G CTAs per row, G by the row stream's rule for
// the draw: rows split only while there are fewer than two CTAs per SM and each
// keeps 2048 elements), then the scan.  Both later kernels are programmatic
// dependents of the one before.
static sv_status launch_match(const void* logits, sv_dtype dt, const int32_t* x, const float* ua,
                              const float* ur, float T, int B, int k, int V, int32_t* out,
                              int32_t* nacc, void* ws, cudaStream_t stream, int sms,
                              Epilogue ep, const sv_tuning& tu) {
    sv_status st = launch_rows(false, logits, dt, nullptr, x, nullptr, 1.0f, B, k, V, ws, stream,
                               sms, false, tu, false);
    if (st != SV_OK) return st;
    const RowRec* rows =
        reinterpret_cast<const RowRec*>(static_cast<char*>(ws) + ws_rows_offset());
    uint32_t* seqstat = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + ws_seq_offset(B, k));
    const long long R = (long long)B * (k + 1);
    MatchArgs a;
    a.logits = logits;
    a.ua = ua;
    a.ur = ur;
    a.rows = rows;
    a.out = out;
    a.B = B;
    a.k = k;
    a.V = V;
    int G = 1;
    while (G < 16 && R * G < 2LL * sms && V / (2 * G) >= 2048) G *= 2;
    while (G < 16 && (V + G - 1) / G > kSliceMax) G *= 2;
    a.G = G;
    a.draw_level = draw_level(V, G);
    a.force_precise = tu.force_precise != 0;
    a.c2 = log2e_over(T);
    a.c = a.c2.hi;
    const size_t smem = draw_smem_bytes(V, G, a.draw_level);
    if (smem > kDynSmemMax) return SV_ERR_UNSUPPORTED;
    cudaLaunchAttribute pdl;
    pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(R * G), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2] = {cluster_attr(G), pdl};
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = dt == SV_BF16 ? cudaLaunchKernelEx(&cfg, sv_match_draw_kernel<__nv_bfloat16>, a)
                                  : cudaLaunchKernelEx(&cfg, sv_match_draw_kernel<float>, a);
    if (e != cudaSuccess) return SV_ERR_CUDA;
    cudaLaunchConfig_t fc = {};
    fc.gridDim = dim3((unsigned)((B + 3) / 4), 1, 1);
    fc.blockDim = dim3(128, 1, 1);
    fc.stream = stream;
    fc.attrs = &pdl;
    fc.numAttrs = 1;
    e = cudaLaunchKernelEx(&fc, sv_finish_match_kernel, x, ua, ur, rows, seqstat, B, k, V, out,
                           nacc, ep);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// Paths of the one-call entry points.  Batches with a sequence for every SM (for
// sampled batches, every other SM) take the row-skipping path (the row stream
// in position-major order, rows past a sequence's first stop never read, then
// one draw CTA per sequence and the precise draws in 4-CTA clusters).  Smaller sampled batches whose clusters
// still cover every SM take the fused per-sequence kernel (rows in waves, early
// exit, the draw in the same launch, no second launch); the rest take the
// two-kernel path, whose row stream spreads every row over all SMs.
enum Path { kPathTwoKernel = 1, kPathFused = 2, kPathSkip = 3 };
// sv_tuning.path: 0 automatic, else a Path.
static Path choose_path(bool sampled, int B, int V, int esz, int sms, const sv_tuning& tu) {
    const int f = tu.path;
    if (f >= kPathTwoKernel && f <= kPathSkip) return (Path)f;
    if (B >= sms) return kPathSkip;
    // Sampled batches of at least half an SM count: measured on B = 80..128 at
    // k = 8, V = 151936 fp32 (skipping 15-18 % faster) and B = 96 at k = 5,
    // V = 128256 bf16 (12 % faster; 4 % slower at B = 128).
    if (sampled && 2 * B >= sms) return kPathSkip;
    // Rows of at most 1 KiB (toy vocabularies): the whole verify is launch
    // latency, and one launch beats two (B = 1, V = 32: 11.3 against 12.0 us;
    // B = 64: 11.7 against 13.6 us).
    if (sampled && (long long)V * esz <= 1024) return kPathFused;
    if (sampled && (long long)B * seq_split(true, B, V, esz, sms) >= sms) return kPathFused;
    return kPathTwoKernel;
}
static Path choose_path(bool sampled, int B, int V, int esz, int sms) {
    return choose_path(sampled, B, V, esz, sms, kAuto);
}

static sv_status run_verify(bool sampled, const void* logits, sv_dtype dt, const float* q,
                            const int32_t* x, const float* ua, const float* ur, float T, int B,
                            int k, int V, int32_t* out, int32_t* nacc, void* ws,
                            cudaStream_t stream, int sms, Epilogue ep, const sv_tuning& tu,
                            bool full_ws = true) {
    const Path path = choose_path(sampled, B, V, dt == SV_BF16 ? 2 : 4, sms, tu);
    if (path == kPathFused)
        return launch_fused(sampled, logits, dt, q, x, ua, ur, T, B, k, V, out, nacc, ws, stream,
                            sms, ep, tu);
    const bool skip = path == kPathSkip;
    // the split draw's counters cleared by the row stream (one launch fewer)
    const bool zs = sampled && full_ws && uses_split(tu, skip, B, V);
    sv_status st = launch_rows(sampled, logits, dt, q, x, ua, T, B, k, V, ws, stream, sms, skip,
                               tu, true, full_ws, zs);
    if (st != SV_OK) return st;
    return launch_finish(sampled, logits, dt, q, x, ua, ur, T, B, k, V, out, nacc, ws, stream,
                         sms, skip, ep, tu, zs);
}

// Tree verification: the row stream over all B*N rows (statistics only, no
// gathers; greedy batches may take the flat stream), then the walk kernel as
// its programmatic dependent, one CTA per sequence.
static sv_status run_tree(bool sampled, const void* logits, sv_dtype dt, const float* q,
                          const int32_t* tok, const int32_t* par, const float* ua,
                          const float* ur, float T, int B, int N, int V, int32_t* out,
                          int32_t* nodes, int32_t* nacc, void* ws, cudaStream_t stream, int sms,
                          const sv_tuning& tu) {
    const int k = N - 1;
    sv_status st = launch_rows(sampled, logits, dt, nullptr, nullptr, nullptr, T, B, k, V, ws,
                               stream, sms, false, tu, !sampled);
    if (st != SV_OK) return st;
    TreeArgs a;
    a.logits = logits;
    a.q = q;
    a.tok = tok;
    a.par = par;
    a.ua = ua;
    a.ur = ur;
    a.hdr = static_cast<const Header*>(ws);
    a.rows = reinterpret_cast<RowRec*>(static_cast<char*>(ws) + ws_rows_offset());
    a.seqstat = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + ws_seq_offset(B, k));
    a.out = out;
    a.nodes = nodes;
    a.nacc = nacc;
    a.B = B;
    a.N = N;
    a.V = V;
    a.c2 = log2e_over(sampled ? T : 1.0f);
    cudaLaunchAttribute pdl;
    pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)B, 1, 1);
    cfg.blockDim = dim3(sampled ? kThreads : 64, 1, 1);
    // the final draw's block sums: a double per 32 chunks of 8 elements
    cfg.dynamicSmemBytes = sampled ? tree_bsum_bytes(V) : 0;
    cfg.stream = stream;
    cfg.attrs = &pdl;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (sampled)
        e = dt == SV_BF16 ? cudaLaunchKernelEx(&cfg, sv_tree_kernel<__nv_bfloat16, true>, a)
                          : cudaLaunchKernelEx(&cfg, sv_tree_kernel<float, true>, a);
    else
        e = dt == SV_BF16 ? cudaLaunchKernelEx(&cfg, sv_tree_kernel<__nv_bfloat16, false>, a)
                          : cudaLaunchKernelEx(&cfg, sv_tree_kernel<float, false>, a);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// The row record that the flat greedy stream's partial keys of row r stand
// for, merged on the host the way the finish kernel merges them on the device:
// the largest key names the maximum and the lowest index holding it, an
// all-ones key a NaN in the row.
static RowRec merge_flat_keys_host(const RowRec& raw, long long r, int vpr, int per, int rem,
                                   bool drafted) {
    const int c0 = flat_owner((int)r * vpr, per, rem);
    const int c1 = flat_owner((int)(r + 1) * vpr - 1, per, rem);
    unsigned long long w[kFlatSlots];
    std::memcpy(w, &raw, sizeof(w));
    unsigned long long key = 0ull;
    for (int c = c0; c <= c1 && c - c0 < kFlatSlots; ++c) key = w[c - c0] > key ? w[c - c0] : key;
    const bool nan = key == ~0ull;
    const uint32_t o = (uint32_t)(key >> 32);
    const uint32_t bits = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
    float m;
    std::memcpy(&m, &bits, sizeof(m));
    RowRec rec;
    rec.mraw = nan ? NAN : m;
    rec.S = 0.0f;
    rec.px = drafted ? 0.0 : (double)NAN;
    rec.lx = NAN;
    rec.qx = NAN;
    rec.argmax = nan ? 0 : (int32_t)(0xFFFFFFFFu - (uint32_t)key);
    rec.flags = (nan || !(m > -INFINITY) || m == INFINITY) ? kRowBad : 0u;
    return rec;
}
static_assert(kFlatSlots * sizeof(unsigned long long) == sizeof(RowRec), "flat key slots");

}  // namespace sv

using namespace sv;

extern "C" {

size_t spec_verify_workspace_size(int B, int k, int V, sv_dtype dtype) {
    if (B < 0 || k < 1 || V < 1 || k > kMaxK || V > kMaxV) return 0;
    if (dtype != SV_BF16 && dtype != SV_F32) return 0;
    return ws_bytes_for(B, k, V);
}

}  // extern "C"

namespace sv {

// The options of a _tuned call are checked like any other argument.
static sv_tuning cluster_draw(sv_tuning t) {
    t.draw_mode = 2;
    return t;
}
static bool tuning_valid(const sv_tuning& t) {
    auto pow2 = [](int g) { return g == 0 || g == 1 || g == 2 || g == 4 || g == 8 || g == 16; };
    return t.path >= 0 && t.path <= 3 && pow2(t.draw_split) && pow2(t.precise_split) &&
           pow2(t.rows_split) && t.fused_defer >= 0 && t.fused_defer <= 2 &&
           t.fused_pad_kib >= 0 && t.fused_pad_kib <= 160 &&
           (t.rows_threads == 0 || t.rows_threads == 128 || t.rows_threads == 256 ||
            t.rows_threads == 512 || t.rows_threads == 1024) &&
           t.draw_mode >= 0 && t.draw_mode <= 2;
}

static sv_status rows_impl(sv_mode mode, const void* logits, sv_dtype dtype,
                           const float* draft_probs, const int32_t* draft_tokens, float T, int B,
                           int k, int V, void* ws, size_t ws_bytes, cudaStream_t stream,
                           const sv_tuning& tu) {
    if (mode != SV_MODE_SAMPLE && mode != SV_MODE_GREEDY) return SV_ERR_INVALID_ARG;
    sv_status st = check_common(logits, dtype, draft_tokens, B, k, V, ws, ws_bytes);
    if (st != SV_OK) return st;
    const bool sampled = mode == SV_MODE_SAMPLE;
    if (sampled) {
        if (!(T > 0.0f) || !std::isfinite(T)) return SV_ERR_INVALID_ARG;
        if (B > 0 && (!draft_probs || !aligned16(draft_probs))) return SV_ERR_INVALID_ARG;
    }
    int sms = 0;
    if ((st = device_setup(&sms)) != SV_OK) return st;
    if (B == 0) return SV_OK;
    return launch_rows(sampled, logits, dtype, draft_probs, draft_tokens, nullptr, T, B, k, V, ws,
                       stream, sms, false, tu);
}

static sv_status finish_impl(sv_mode mode, const void* logits, sv_dtype dtype,
                             const float* draft_probs, const int32_t* draft_tokens,
                             const float* u_accept, const float* u_resample, float T, int B,
                             int k, int V, int32_t* out_tokens, int32_t* num_accepted, void* ws,
                             size_t ws_bytes, cudaStream_t stream, const sv_tuning& tu) {
    if (mode != SV_MODE_SAMPLE && mode != SV_MODE_GREEDY) return SV_ERR_INVALID_ARG;
    sv_status st = check_common(logits, dtype, draft_tokens, B, k, V, ws, ws_bytes);
    if (st != SV_OK) return st;
    if ((st = check_outputs(out_tokens, num_accepted, B)) != SV_OK) return st;
    const bool sampled = mode == SV_MODE_SAMPLE;
    if (sampled && (st = check_sample(draft_probs, u_accept, u_resample, T, B)) != SV_OK) return st;
    int sms = 0;
    if ((st = device_setup(&sms)) != SV_OK) return st;
    if (B == 0) return SV_OK;
    return launch_finish(sampled, logits, dtype, draft_probs, draft_tokens, u_accept, u_resample,
                         T, B, k, V, out_tokens, num_accepted, ws, stream, sms, B >= sms,
                         Epilogue{nullptr, nullptr}, tu);
}

// spec_verify_greedy[_kv] (sampled = false: q, u_accept, u_resample unused, T
// ignored) and spec_verify_sample[_kv].
static sv_status verify_impl(bool sampled, const void* logits, sv_dtype dtype,
                             const float* draft_probs, const int32_t* draft_tokens,
                             const float* u_accept, const float* u_resample, float T, int B,
                             int k, int V, int32_t* out_tokens, int32_t* num_accepted, void* ws,
                             size_t ws_bytes, int32_t* kv_len, sv_spec_stats* stats,
                             cudaStream_t stream, const sv_tuning& tu, bool base_ws = false) {
    // base_ws: a workspace without the split draw's region (the no-allocation
    // entry point), so the draw is the cluster draw
    sv_status st = check_common(logits, dtype, draft_tokens, B, k, V, ws, ws_bytes, base_ws);
    if (st != SV_OK) return st;
    if ((st = check_outputs(out_tokens, num_accepted, B)) != SV_OK) return st;
    if (sampled && (st = check_sample(draft_probs, u_accept, u_resample, T, B)) != SV_OK) return st;
    if ((kv_len && !aligned16(kv_len)) || (stats && !aligned16(stats))) return SV_ERR_INVALID_ARG;
    int sms = 0;
    if ((st = device_setup(&sms)) != SV_OK) return st;
    if (B == 0) return SV_OK;
    return run_verify(sampled, logits, dtype, sampled ? draft_probs : nullptr, draft_tokens,
                      sampled ? u_accept : nullptr, sampled ? u_resample : nullptr,
                      sampled ? T : 1.0f, B, k, V, out_tokens, num_accepted, ws, stream, sms,
                      Epilogue{kv_len, reinterpret_cast<unsigned long long*>(stats)},
                      base_ws ? cluster_draw(tu) : tu, !base_ws);
}

static sv_status tree_impl(sv_mode mode, const void* logits, sv_dtype dtype,
                           const float* draft_probs, const int32_t* tree_tokens,
                           const int32_t* tree_parents, const float* u_accept,
                           const float* u_resample, float T, int B, int N, int V,
                           int32_t* out_tokens, int32_t* out_nodes, int32_t* num_accepted,
                           void* ws, size_t ws_bytes, cudaStream_t stream, const sv_tuning& tu) {
    if (mode != SV_MODE_SAMPLE && mode != SV_MODE_GREEDY) return SV_ERR_INVALID_ARG;
    if (N < 2) return SV_ERR_INVALID_ARG;
    if (N > kTreeMaxN) return SV_ERR_UNSUPPORTED;
    sv_status st = check_common(logits, dtype, tree_tokens, B, N - 1, V, ws, ws_bytes);
    if (st != SV_OK) return st;
    if ((st = check_outputs(out_tokens, num_accepted, B)) != SV_OK) return st;
    if (B > 0 && (!tree_parents || !aligned16(tree_parents) || !out_nodes || !aligned16(out_nodes)))
        return SV_ERR_INVALID_ARG;
    const bool sampled = mode == SV_MODE_SAMPLE;
    if (sampled && (st = check_sample(draft_probs, u_accept, u_resample, T, B)) != SV_OK) return st;
    int sms = 0;
    if ((st = device_setup(&sms)) != SV_OK) return st;
    if (B == 0) return SV_OK;
    return run_tree(sampled, logits, dtype, draft_probs, tree_tokens, tree_parents, u_accept,
                    u_resample, T, B, N, V, out_tokens, out_nodes, num_accepted, ws, stream, sms,
                    tu);
}

static sv_status match_impl(const void* logits, sv_dtype dtype, const int32_t* draft_tokens,
                            const float* u_draw, const float* u_bonus, float T, int B, int k,
                            int V, int32_t* out_tokens, int32_t* num_accepted, void* ws,
                            size_t ws_bytes, cudaStream_t stream, const sv_tuning& tu) {
    sv_status st = check_common(logits, dtype, draft_tokens, B, k, V, ws, ws_bytes);
    if (st != SV_OK) return st;
    if ((st = check_outputs(out_tokens, num_accepted, B)) != SV_OK) return st;
    if (!(T > 0.0f) || !std::isfinite(T)) return SV_ERR_INVALID_ARG;
    if (B > 0 && (!u_draw || !u_bonus || !aligned16(u_draw) || !aligned16(u_bonus)))
        return SV_ERR_INVALID_ARG;
    int sms = 0;
    if ((st = device_setup(&sms)) != SV_OK) return st;
    if (B == 0) return SV_OK;
    return launch_match(logits, dtype, draft_tokens, u_draw, u_bonus, T, B, k, V, out_tokens,
                        num_accepted, ws, stream, sms, Epilogue{nullptr, nullptr}, tu);
}

}  // namespace sv

extern "C" {

sv_status spec_verify_rows(sv_mode mode, const void* logits, sv_dtype dtype,
                           const float* draft_probs, const int32_t* draft_tokens, float T, int B,
                           int k, int V, void* ws, size_t ws_bytes, cudaStream_t stream) {
    return rows_impl(mode, logits, dtype, draft_probs, draft_tokens, T, B, k, V, ws, ws_bytes,
                     stream, kAuto);
}

sv_status spec_verify_finish(sv_mode mode, const void* logits, sv_dtype dtype,
                             const float* draft_probs, const int32_t* draft_tokens,
                             const float* u_accept, const float* u_resample, float T, int B,
                             int k, int V, int32_t* out_tokens, int32_t* num_accepted, void* ws,
                             size_t ws_bytes, cudaStream_t stream) {
    return finish_impl(mode, logits, dtype, draft_probs, draft_tokens, u_accept, u_resample, T, B,
                       k, V, out_tokens, num_accepted, ws, ws_bytes, stream, kAuto);
}

sv_status spec_verify_greedy(const void* logits, sv_dtype dtype, const int32_t* draft_tokens,
                             int B, int k, int V, int32_t* out_tokens, int32_t* num_accepted,
                             void* ws, size_t ws_bytes, cudaStream_t stream) {
    return verify_impl(false, logits, dtype, nullptr, draft_tokens, nullptr, nullptr, 1.0f, B, k,
                       V, out_tokens, num_accepted, ws, ws_bytes, nullptr, nullptr, stream, kAuto);
}

sv_status spec_verify_greedy_kv(const void* logits, sv_dtype dtype, const int32_t* draft_tokens,
                                int B, int k, int V, int32_t* out_tokens, int32_t* num_accepted,
                                void* ws, size_t ws_bytes, int32_t* kv_len, sv_spec_stats* stats,
                                cudaStream_t stream) {
    return verify_impl(false, logits, dtype, nullptr, draft_tokens, nullptr, nullptr, 1.0f, B, k,
                       V, out_tokens, num_accepted, ws, ws_bytes, kv_len, stats, stream, kAuto);
}

sv_status spec_verify_sample(const void* logits, sv_dtype dtype, const float* draft_probs,
                             const int32_t* draft_tokens, const float* u_accept,
                             const float* u_resample, float T, int B, int k, int V,
                             int32_t* out_tokens, int32_t* num_accepted, void* ws,
                             size_t ws_bytes, cudaStream_t stream) {
    return verify_impl(true, logits, dtype, draft_probs, draft_tokens, u_accept, u_resample, T, B,
                       k, V, out_tokens, num_accepted, ws, ws_bytes, nullptr, nullptr, stream,
                       kAuto);
}

sv_status spec_verify_sample_kv(const void* logits, sv_dtype dtype, const float* draft_probs,
                                const int32_t* draft_tokens, const float* u_accept,
                                const float* u_resample, float T, int B, int k, int V,
                                int32_t* out_tokens, int32_t* num_accepted, void* ws,
                                size_t ws_bytes, int32_t* kv_len, sv_spec_stats* stats,
                                cudaStream_t stream) {
    return verify_impl(true, logits, dtype, draft_probs, draft_tokens, u_accept, u_resample, T, B,
                       k, V, out_tokens, num_accepted, ws, ws_bytes, kv_len, stats, stream, kAuto);
}

sv_status spec_verify_tree(sv_mode mode, const void* logits, sv_dtype dtype,
                           const float* draft_probs, const int32_t* tree_tokens,
                           const int32_t* tree_parents, const float* u_accept,
                           const float* u_resample, float T, int B, int N, int V,
                           int32_t* out_tokens, int32_t* out_nodes, int32_t* num_accepted,
                           void* ws, size_t ws_bytes, cudaStream_t stream) {
    return tree_impl(mode, logits, dtype, draft_probs, tree_tokens, tree_parents, u_accept,
                     u_resample, T, B, N, V, out_tokens, out_nodes, num_accepted, ws, ws_bytes,
                     stream, kAuto);
}

sv_status spec_verify_match(const void* logits, sv_dtype dtype, const int32_t* draft_tokens,
                            const float* u_draw, const float* u_bonus, float T, int B, int k,
                            int V, int32_t* out_tokens, int32_t* num_accepted, void* ws,
                            size_t ws_bytes, cudaStream_t stream) {
    return match_impl(logits, dtype, draft_tokens, u_draw, u_bonus, T, B, k, V, out_tokens,
                      num_accepted, ws, ws_bytes, stream, kAuto);
}

// The same calls with the options of sv_tuning (specverify_debug.h); a null
// `tuning` means the automatic choices.
#define SV_TUNING_OR_AUTO(t)                                         \
    const sv_tuning& tu = (t) ? *(t) : kAuto;                        \
    if (!tuning_valid(tu)) return SV_ERR_INVALID_ARG

sv_status spec_verify_rows_tuned(sv_mode mode, const void* logits, sv_dtype dtype,
                                 const float* draft_probs, const int32_t* draft_tokens, float T,
                                 int B, int k, int V, void* ws, size_t ws_bytes,
                                 cudaStream_t stream, const sv_tuning* tuning) {
    SV_TUNING_OR_AUTO(tuning);
    return rows_impl(mode, logits, dtype, draft_probs, draft_tokens, T, B, k, V, ws, ws_bytes,
                     stream, tu);
}

sv_status spec_verify_finish_tuned(sv_mode mode, const void* logits, sv_dtype dtype,
                                   const float* draft_probs, const int32_t* draft_tokens,
                                   const float* u_accept, const float* u_resample, float T,
                                   int B, int k, int V, int32_t* out_tokens,
                                   int32_t* num_accepted, void* ws, size_t ws_bytes,
                                   cudaStream_t stream, const sv_tuning* tuning) {
    SV_TUNING_OR_AUTO(tuning);
    return finish_impl(mode, logits, dtype, draft_probs, draft_tokens, u_accept, u_resample, T, B,
                       k, V, out_tokens, num_accepted, ws, ws_bytes, stream, tu);
}

sv_status spec_verify_greedy_tuned(const void* logits, sv_dtype dtype,
                                   const int32_t* draft_tokens, int B, int k, int V,
                                   int32_t* out_tokens, int32_t* num_accepted, void* ws,
                                   size_t ws_bytes, int32_t* kv_len, sv_spec_stats* stats,
                                   cudaStream_t stream, const sv_tuning* tuning) {
    SV_TUNING_OR_AUTO(tuning);
    return verify_impl(false, logits, dtype, nullptr, draft_tokens, nullptr, nullptr, 1.0f, B, k,
                       V, out_tokens, num_accepted, ws, ws_bytes, kv_len, stats, stream, tu);
}

sv_status spec_verify_sample_tuned(const void* logits, sv_dtype dtype, const float* draft_probs,
                                   const int32_t* draft_tokens, const float* u_accept,
                                   const float* u_resample, float T, int B, int k, int V,
                                   int32_t* out_tokens, int32_t* num_accepted, void* ws,
                                   size_t ws_bytes, int32_t* kv_len, sv_spec_stats* stats,
                                   cudaStream_t stream, const sv_tuning* tuning) {
    SV_TUNING_OR_AUTO(tuning);
    return verify_impl(true, logits, dtype, draft_probs, draft_tokens, u_accept, u_resample, T, B,
                       k, V, out_tokens, num_accepted, ws, ws_bytes, kv_len, stats, stream, tu);
}

sv_status spec_verify_tree_tuned(sv_mode mode, const void* logits, sv_dtype dtype,
                                 const float* draft_probs, const int32_t* tree_tokens,
                                 const int32_t* tree_parents, const float* u_accept,
                                 const float* u_resample, float T, int B, int N, int V,
                                 int32_t* out_tokens, int32_t* out_nodes, int32_t* num_accepted,
                                 void* ws, size_t ws_bytes, cudaStream_t stream,
                                 const sv_tuning* tuning) {
    SV_TUNING_OR_AUTO(tuning);
    return tree_impl(mode, logits, dtype, draft_probs, tree_tokens, tree_parents, u_accept,
                     u_resample, T, B, N, V, out_tokens, out_nodes, num_accepted, ws, ws_bytes,
                     stream, tu);
}

sv_status spec_verify_match_tuned(const void* logits, sv_dtype dtype, const int32_t* draft_tokens,
                                  const float* u_draw, const float* u_bonus, float T, int B, int k,
                                  int V, int32_t* out_tokens, int32_t* num_accepted, void* ws,
                                  size_t ws_bytes, cudaStream_t stream, const sv_tuning* tuning) {
    SV_TUNING_OR_AUTO(tuning);
    return match_impl(logits, dtype, draft_tokens, u_draw, u_bonus, T, B, k, V, out_tokens,
                      num_accepted, ws, ws_bytes, stream, tu);
}
#undef SV_TUNING_OR_AUTO

sv_status spec_ngram_draft(const int32_t* history, const int32_t* lengths, int B, int Lmax,
                           int k, int n_min, int n_max, int32_t* draft_tokens,
                           int32_t* num_drafted, cudaStream_t stream) {
    if (B < 0 || Lmax < 0 || k < 1 || k > kMaxK || n_min < 1 || n_max < n_min ||
        n_max > kNgramMaxN)
        return SV_ERR_INVALID_ARG;
    if (B > 0 && (!history || !lengths || !draft_tokens || !num_drafted)) return SV_ERR_INVALID_ARG;
    if (B > 0 && (!aligned16(history) || !aligned16(lengths) || !aligned16(draft_tokens) ||
                  !aligned16(num_drafted)))
        return SV_ERR_INVALID_ARG;
    if ((long long)B * Lmax >= (1LL << 40) || B >= (1 << 30)) return SV_ERR_UNSUPPORTED;
    int sms = 0;
    sv_status st = device_setup(&sms);
    if (st != SV_OK) return st;
    if (B == 0) return SV_OK;
    sv_ngram_kernel<<<B, kNgramThreads, 0, stream>>>(history, lengths, Lmax, k, n_min, n_max,
                                                     draft_tokens, num_drafted);
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

sv_status spec_verify_read_status(const void* ws, cudaStream_t stream, uint32_t* device_status,
                                  uint32_t* n_degenerate) {
    if (!ws || !device_status) return SV_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SV_ERR_CUDA;
    Header h;
    if (cudaMemcpy(&h, ws, sizeof(Header), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SV_ERR_CUDA;
    if (h.magic != kMagic || h.k < 1 || h.k > (uint32_t)kMaxK) return SV_ERR_INVALID_ARG;
    uint32_t* st = new (std::nothrow) uint32_t[h.B > 0 ? h.B : 1];
    if (!st) return SV_ERR_INVALID_ARG;
    cudaError_t e = cudaMemcpy(st, static_cast<const char*>(ws) + ws_seq_offset(h.B, (int)h.k),
                               (size_t)h.B * sizeof(uint32_t), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
        delete[] st;
        return SV_ERR_CUDA;
    }
    uint32_t bits = 0, ndeg = 0;
    for (uint32_t b = 0; b < h.B; ++b) {
        bits |= st[b];
        ndeg += (st[b] & SV_DEV_DEGENERATE) ? 1u : 0u;
    }
    delete[] st;
    *device_status = bits;
    if (n_degenerate) *n_degenerate = ndeg;
    return (bits & ~(SV_DEV_DEGENERATE | SV_DEV_PRECISE)) ? SV_ERR_DATA : SV_OK;
}

sv_status spec_verify_row_stats(const void* ws, cudaStream_t stream, int B, int k, float* m,
                                float* S, int32_t* argmax, float* px, float* qx) {
    if (!ws || B < 0 || k < 1 || k > kMaxK) return SV_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SV_ERR_CUDA;
    Header h;
    if (cudaMemcpy(&h, ws, sizeof(Header), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SV_ERR_CUDA;
    if (h.magic != kMagic || (int)h.B != B || (int)h.k != k) return SV_ERR_INVALID_ARG;
    const long long R = (long long)B * (k + 1);
    RowRec* host = new (std::nothrow) RowRec[R > 0 ? R : 1];
    if (!host) return SV_ERR_INVALID_ARG;
    cudaError_t e = cudaMemcpy(host, static_cast<const char*>(ws) + ws_rows_offset(),
                               R * sizeof(RowRec), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
        delete[] host;
        return SV_ERR_CUDA;
    }
    for (long long r = 0; r < R; ++r) {
        RowRec rec = host[r];
        // After the flat greedy stream the records hold per-range partial keys
        // until a reader merges them (the finish kernel merges its own copies).
        if (h.flat_ctas) rec = merge_flat_keys_host(rec, r, (int)h.flat_vpr, (int)h.flat_per,
                                                    (int)h.flat_rem, (int)(r % (k + 1)) < k);
        if (m) m[r] = rec.mraw;
        if (S) S[r] = rec.S;
        if (argmax) argmax[r] = rec.argmax;
        if (px) px[r] = (float)rec.px;
        if (qx) qx[r] = rec.qx;
    }
    delete[] host;
    return SV_OK;
}

const char* spec_verify_status_string(sv_status s) {
    switch (s) {
        case SV_OK: return "ok";
        case SV_ERR_INVALID_ARG: return "invalid argument";
        case SV_ERR_WORKSPACE: return "workspace missing or too small";
        case SV_ERR_UNSUPPORTED: return "unsupported size or device";
        case SV_ERR_CUDA: return "CUDA runtime error";
        case SV_ERR_DATA: return "device-detected invalid data";
        case SV_ERR_TIMEOUT: return "bounded device wait gave up";
    }
    return "unknown status";
}

// Test hook (declared in include/specverify_debug.h): e[i] = exp((l[i] - m)/T)
// evaluated by the draw's float-float exponential, returned as hi + lo in double.
sv_status spec_verify_debug_ffexp(const float* l, float m, float T, int n, double* out,
                                  cudaStream_t stream) {
    if (n < 0 || (n > 0 && (!l || !out)) || !(T > 0.0f)) return SV_ERR_INVALID_ARG;
    if (n == 0) return SV_OK;
    sv_debug_ffexp_kernel<<<(n + 255) / 256, 256, 0, stream>>>(l, m, n, log2e_over(T), out);
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// Introspection (declared in include/specverify_debug.h): per status bit, the
// number of sequences of the last call on `ws` whose status word has it.
sv_status spec_verify_debug_status_counts(const void* ws, cudaStream_t stream,
                                          uint32_t counts[8]) {
    if (!ws || !counts) return SV_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return SV_ERR_CUDA;
    Header h;
    if (cudaMemcpy(&h, ws, sizeof(Header), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SV_ERR_CUDA;
    if (h.magic != kMagic || h.k < 1 || h.k > (uint32_t)kMaxK) return SV_ERR_INVALID_ARG;
    uint32_t* st = new (std::nothrow) uint32_t[h.B > 0 ? h.B : 1];
    if (!st) return SV_ERR_INVALID_ARG;
    const cudaError_t e = cudaMemcpy(st, static_cast<const char*>(ws) + ws_seq_offset(h.B, (int)h.k),
                                     (size_t)h.B * sizeof(uint32_t), cudaMemcpyDeviceToHost);
    for (int i = 0; i < 8; ++i) counts[i] = 0;
    if (e == cudaSuccess)
        for (uint32_t b = 0; b < h.B; ++b)
            for (int i = 0; i < 8; ++i) counts[i] += (st[b] >> i) & 1u;
    delete[] st;
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// Introspection (declared in include/specverify_debug.h): the path the one-call
// entry points take for these sizes on the current device (1 two-kernel, 2
// fused, 3 row-skipping), -1 on error.
int spec_verify_debug_path(sv_mode mode, int B, int V, sv_dtype dtype) {
    int sms = 0;
    if (device_setup(&sms) != SV_OK) return -1;
    if (B < 1 || V < 1 || (dtype != SV_BF16 && dtype != SV_F32)) return -1;
    return (int)choose_path(mode == SV_MODE_SAMPLE, B, V, dtype == SV_BF16 ? 2 : 4, sms);
}

// Introspection (declared in include/specverify_debug.h): the flat greedy
// stream's CTA count for these sizes (16-byte aligned logits) on the current
// device, 0 when a greedy verify would not take it, -1 on error.
int spec_verify_debug_flat_ctas(int B, int k, int V, sv_dtype dtype) {
    int sms = 0;
    if (device_setup(&sms) != SV_OK) return -1;
    if (B < 1 || k < 1 || k > kMaxK || V < 1 || (dtype != SV_BF16 && dtype != SV_F32)) return -1;
    if (choose_path(false, B, V, dtype == SV_BF16 ? 2 : 4, sms) != kPathTwoKernel) return 0;
    FlatArgs f;
    static const uint4 aligned = {};
    return flat_plan(B, k, V, dtype == SV_BF16 ? 2 : 4, &aligned, sms, &f) ? f.P : 0;
}

// Test / timing hook: the first stage of the row-skipping path alone (the reset
// of the stop rows and the position-major row stream).  Argument checks as for
// spec_verify_rows; u_accept is required in sampled mode.
sv_status spec_verify_debug_rows_skip(sv_mode mode, const void* logits, sv_dtype dtype,
                                      const float* draft_probs, const int32_t* draft_tokens,
                                      const float* u_accept, float T, int B, int k, int V,
                                      void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (mode != SV_MODE_SAMPLE && mode != SV_MODE_GREEDY) return SV_ERR_INVALID_ARG;
    sv_status st = check_common(logits, dtype, draft_tokens, B, k, V, ws, ws_bytes);
    if (st != SV_OK) return st;
    const bool sampled = mode == SV_MODE_SAMPLE;
    if (sampled) {
        if (!(T > 0.0f) || !std::isfinite(T)) return SV_ERR_INVALID_ARG;
        if (B > 0 && (!draft_probs || !u_accept || !aligned16(draft_probs) || !aligned16(u_accept)))
            return SV_ERR_INVALID_ARG;
    }
    int sms = 0;
    if ((st = device_setup(&sms)) != SV_OK) return st;
    if (B == 0) return SV_OK;
    return launch_rows(sampled, logits, dtype, draft_probs, draft_tokens, u_accept, T, B, k, V, ws,
                       stream, sms, true, kAuto, true, true);
}

// Test hook: the largest relative error of ex2.approx.ftz.f32 against the
// float-float 2^a over every float a in [a0, a1] (a0 <= a1 <= 0, a0 >= -126),
// written to *out (a DEVICE float).  Synchronous.
sv_status spec_verify_debug_ex2_error(float a0, float a1, float* out, cudaStream_t stream) {
    if (!out || !(a0 <= a1) || !(a1 <= 0.0f) || !(a0 >= -126.0f)) return SV_ERR_INVALID_ARG;
    if (cudaMemsetAsync(out, 0, sizeof(float), stream) != cudaSuccess) return SV_ERR_CUDA;
    // floats in [a0, a1] are the bit patterns from bits(a1) up to bits(a0) (negative)
    const uint32_t b_hi = __builtin_bit_cast(uint32_t, a0);
    const uint32_t b_lo = __builtin_bit_cast(uint32_t, a1 == 0.0f ? -0.0f : a1);
    const unsigned long long n = (unsigned long long)(b_hi - b_lo) + 1ull;
    sv_debug_ex2_kernel<<<1216, 256, 0, stream>>>(b_lo, n, out);
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
    return cudaStreamSynchronize(stream) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // extern "C"

// ------------------------------------------------------------------ entry point without allocation
//
// spec_verify_sample with its scratch in a fixed device array of this library
// instead of a caller-provided workspace.  The array's name is only a host-side
// handle; its device address is looked up once per device with
// cudaGetSymbolAddress and then passed to the kernels like any workspace.
namespace sv {

constexpr size_t kNoAllocScratchBytes = SV_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes >= 256 + 32 * (size_t)SV_NOALLOC_MAX_ROWS +
                                          12 * (size_t)(SV_NOALLOC_MAX_ROWS / 2) + 31 + 255,
              "scratch size");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

static std::mutex g_noalloc_mu;
static void* g_noalloc_addr[64];

// Device address of the scratch array on the current device (looked up on the
// first call made with that device current, then cached).
static sv_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SV_ERR_CUDA;
    if (dev < 0 || dev >= 64) return SV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return SV_ERR_CUDA;
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return SV_OK;
}

}  // namespace sv

extern "C" sv_status spec_verify_sample_noalloc(const void* logits, sv_dtype dtype,
                                                const float* draft_probs,
                                                const int32_t* draft_tokens,
                                                const float* u_accept, const float* u_resample,
                                                float T, int B, int k, int V,
                                                int32_t* out_tokens, int32_t* num_accepted,
                                                cudaStream_t stream) {
    if (B < 0 || k < 1 || V < 1) return SV_ERR_INVALID_ARG;
    if (k > sv::kMaxK || V > sv::kMaxV) return SV_ERR_UNSUPPORTED;
    if ((long long)B * (k + 1) > SV_NOALLOC_MAX_ROWS) return SV_ERR_WORKSPACE;
    void* ws = nullptr;
    sv_status st = sv::noalloc_scratch(&ws);
    if (st != SV_OK) return st;
    return sv::verify_impl(true, logits, dtype, draft_probs, draft_tokens, u_accept, u_resample,
                           T, B, k, V, out_tokens, num_accepted, ws, sv::kNoAllocScratchBytes,
                           nullptr, nullptr, stream, sv::kAuto, true);
}
