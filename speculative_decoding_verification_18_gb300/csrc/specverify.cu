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
#include <atomic>
#include <mutex>
#include <new>

#include "../../include/specverify.h"
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
    uint32_t pad[59];
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

// Layout: header | B*(k+1) row records | B per-sequence status words.
__host__ __device__ inline size_t ws_rows_offset() { return sizeof(Header); }
__host__ __device__ inline size_t ws_seq_offset(long long B, int k) {
    return sizeof(Header) + (size_t)B * (k + 1) * sizeof(RowRec);
}
__host__ __device__ inline size_t ws_bytes_for(long long B, int k) {
    size_t b = ws_seq_offset(B, k) + (size_t)B * sizeof(uint32_t);
    return (b + 255) & ~(size_t)255;
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
template <typename DT, bool SAMPLED, int U>
__device__ __forceinline__ Partial stream_slice(const DT* __restrict__ rowp, int V, long long vb,
                                                long long ve, int head, long long tail0,
                                                bool head_here, bool tail_here, int tg, int ng,
                                                float c) {
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
    long long v = vb + tg;
    for (; v + (long long)(U - 1) * ng < ve; v += (long long)U * ng) {
        uint4 buf[U];
#pragma unroll
        for (int u = 0; u < U; ++u) buf[u] = ld_stream16(vp + v + (long long)u * ng);
#pragma unroll
        for (int u = 0; u < U; ++u) vector(buf[u], head + (v + (long long)u * ng) * VW);
    }
    for (; v < ve; v += ng) vector(ld_stream16(vp + v), head + v * VW);
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
constexpr int kSliceMax = 163840;   // largest slice of a row one CTA draws from (chunk sums in smem)

// Error model of the fast fp32 draw.  ex2.approx.ftz.f32 is taken to be within
// kEx2RelErr of 2^a (relative) on [-126, 0]; a test measures its worst case
// exhaustively on that range and checks it is at least 2x below this bound.
constexpr float kEx2RelErr = 4.76837158e-07f;  // 2^-21
// Relative error bound of p = ex2(a)/S per element, apart from the argument
// term: ex2 itself, the normaliser's ex2 errors, and the roundings of 1/S
// (with S carried to 2^-47), of e * (1/S) and of p - q.
constexpr float kFastE0 = 2.0f * kEx2RelErr + 4.0f * 5.96046448e-08f;
// The fp32 argument a = fl(fl(l - m) * fl(log2(e)/T)) is off by at most
// 3 * 2^-24 * |a|, i.e. 2^a by a relative 3 * 2^-24 * ln2 * |a|.
constexpr float kFastKappa = 3.0f * 5.96046448e-08f * 0.693147181f;
// Elements with p < q (1 - kRelSlack) for sure weigh exactly 0 in both passes.
constexpr float kRelSlack = 4.0e-5f;

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

// Shared memory of the draw besides its dynamic chunk-sum array.
struct DrawShared {
    float thi[kExpTable], tlo[kExpTable];
    ff red_ff[kWarps];
    float red_f[kWarps];
    unsigned long long red_u[kWarps];
    unsigned long long woff[kWarps];
    // per-CTA values read by the other CTAs of the cluster through DSMEM
    ff slot_S;
    float slot_A;
    unsigned long long slot_W[3];
    float slot_D;
    int slot_cert;
    // cluster-wide values, identical in every CTA
    ff S_tot;
    float A_tot, D_tot;
    unsigned long long prefix, total;
    int cert_all;
    int token;
};

__device__ const Exp2Table g_exp2_table = make_exp2_table();

__device__ __forceinline__ void load_exp_table(DrawShared& sh) {
    for (int i = threadIdx.x; i < kExpTable; i += blockDim.x) {
        sh.thi[i] = g_exp2_table.hi[i];
        sh.tlo[i] = g_exp2_table.lo[i];
    }
}

// Block sum of a float-float value, then the cluster sum over ranks 0..G-1 in a
// fixed order (the same tree in every CTA, so every CTA gets the same value).
__device__ __forceinline__ ff cluster_sum_ff(cg::cluster_group& cluster, DrawShared& sh, ff v,
                                             int G) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum_ff(ff_normalize(v));
    if (lane == 0) sh.red_ff[warp] = v;
    __syncthreads();
    if (warp == 0) {
        ff w = lane < kWarps ? sh.red_ff[lane] : ff{0.0f, 0.0f};
        w = warp_sum_ff(w);
        if (lane == 0) sh.slot_S = w;
    }
    cluster.sync();
    if (warp == 0) {
        ff w = lane < G ? *cluster.map_shared_rank(&sh.slot_S, lane) : ff{0.0f, 0.0f};
        w = warp_sum_ff(w);
        if (lane == 0) sh.S_tot = w;
    }
    __syncthreads();
    return sh.S_tot;
}

// Block sum of the chunk-weight totals, then the exclusive prefix of this rank
// and the grand total over the cluster (sh.prefix, sh.total); `slot` selects
// which of the three DSMEM slots carries this round.  Also sums one float over
// the cluster into sh.D_tot (pass 0.0f when unused).
__device__ __forceinline__ void cluster_prefix(cg::cluster_group& cluster, DrawShared& sh,
                                               unsigned long long t, float d, int slot, int rank,
                                               int G) {
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
        w = warp_sum(w);
        f = warp_sum(f);
        if (lane == 0) {
            sh.slot_W[slot] = w;
            sh.slot_D = f;
        }
    }
    cluster.sync();
    if (warp == 0) {
        unsigned long long v = lane < G ? cluster.map_shared_rank(sh.slot_W, lane)[slot] : 0ull;
        float f = lane < G ? *cluster.map_shared_rank(&sh.slot_D, lane) : 0.0f;
        unsigned long long incl = v;  // inclusive prefix over ranks
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            unsigned long long o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        f = warp_sum(f);
        unsigned long long tot = __shfl_sync(0xffffffffu, incl, 31);
        unsigned long long pre = __shfl_sync(0xffffffffu, incl - v, rank);
        if (lane == 0) {
            sh.prefix = pre;
            sh.total = tot;
            sh.D_tot = f;
        }
    }
    __syncthreads();
}

// Inside the CTA that owns `want` (0 <= want < sum of csum[0..mych)), the
// thread whose contiguous chunk range holds it returns true with the chunk
// index and the cumulative weight before that chunk; other threads return false.
__device__ __forceinline__ bool find_chunk(DrawShared& sh, const unsigned long long* csum,
                                           int mych, unsigned long long want, int* cstar,
                                           unsigned long long* before) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = (mych + kThreads - 1) / kThreads;
    const int cb = tid * L, ce = min(mych, cb + L);
    unsigned long long mine = 0;
    for (int ci = cb; ci < ce; ++ci) mine += csum[ci];
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
    if (!(mine > 0 && excl <= want && want - excl < mine)) return false;
    unsigned long long run = excl;
    int c = cb;
    for (; c < ce; ++c) {
        if (want - run < csum[c]) break;
        run += csum[c];
    }
    if (c >= ce) c = ce - 1;  // unreachable: `mine` covers `want`
    *cstar = c;
    *before = run;
    return true;
}

// ---- fast pass: fp32 exponentials, exact integer prefix sums, error bound

// Fixed-point weights of one chunk from fp32 arithmetic, with the error-bound
// contribution of its elements.  With `want` < ~0ull, also the first element
// whose cumulative weight exceeds `want` and the cumulative weights around it.
template <typename DT>
__device__ __forceinline__ unsigned long long fast_chunk(
    const DT* __restrict__ rowp, const float* __restrict__ qrow, long long j0, int V, bool al_l,
    bool al_q, bool residual, float m, float c, float inv, float* bound, unsigned long long want,
    int* token, unsigned long long* lo_out, unsigned long long* hi_out) {
    float lf[kChunk], qf[kChunk];
    load_chunk<DT>(rowp, j0, V, al_l, lf);
    if (residual) load_q_chunk(qrow, j0, V, al_q, qf);
    unsigned long long cs = 0;
    float bd = 0.0f;
#pragma unroll
    for (int e = 0; e < kChunk; ++e) {
        const float a = (lf[e] - m) * c;
        const float p = ex2_approx(a) * inv;
        const float w = residual ? fmaxf(p - qf[e], 0.0f) : p;
        const bool rel = !residual || p >= qf[e] * (1.0f - kRelSlack);
        bd += rel ? p * (kFastE0 + kFastKappa * fabsf(a)) : 0.0f;
        const unsigned long long W = fix_mag(w);
        if (token && *token < 0 && W > 0 && cs + W > want) {
            *token = (int)(j0 + e);
            *lo_out = cs;
            *hi_out = cs + W;
        }
        cs += W;
    }
    *bound += bd;
    return cs;
}

// The fast draw by the G CTAs of a cluster.  Returns true (in every thread of
// every CTA) when the token is certified, i.e. u*C lies farther than twice the
// accumulated error bound from both edges of the chosen bin, so the exact
// draw picks the same bin; the owner CTA then holds it in sh.token.
template <typename DT>
__device__ bool draw_fast(cg::cluster_group& cluster, DrawShared& sh, unsigned long long* csum,
                          const DT* __restrict__ rowp, const float* __restrict__ qrow,
                          bool residual, int V, float m, float c, float u, int rank, int G) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool al_l = (reinterpret_cast<uintptr_t>(rowp) & 15) == 0;
    const bool al_q = residual && (reinterpret_cast<uintptr_t>(qrow) & 15) == 0;
    const long long nch = (V + kChunk - 1) / kChunk;
    const long long c0 = nch * rank / G, c1 = nch * (rank + 1) / G;
    const int mych = (int)(c1 - c0);

    // Pass A: S = sum_j ex2(a_j), carried in float-float.
    ff accS{0.0f, 0.0f};
    for (int ci = tid; ci < mych; ci += kThreads) {
        float f[kChunk];
        load_chunk<DT>(rowp, (c0 + ci) * kChunk, V, al_l, f);
#pragma unroll
        for (int e = 0; e < kChunk; ++e) {
            ff s = two_sum(accS.hi, ex2_approx((f[e] - m) * c));
            accS.hi = s.hi;
            accS.lo = __fadd_rn(accS.lo, s.lo);
        }
    }
    const ff S = cluster_sum_ff(cluster, sh, accS, G);
    const float inv = __frcp_rn(S.hi);

    // Pass B: fixed-point weights, chunk sums, the error bound, cluster prefix.
    unsigned long long tacc = 0;
    float bound = 0.0f;
    for (int ci = tid; ci < mych; ci += kThreads) {
        unsigned long long cs = fast_chunk<DT>(rowp, qrow, (c0 + ci) * kChunk, V, al_l, al_q,
                                               residual, m, c, inv, &bound, 0ull, nullptr,
                                               nullptr, nullptr);
        csum[ci] = cs;
        tacc += cs;
    }
    cluster_prefix(cluster, sh, tacc, bound, 0, rank, G);
    const unsigned long long prefix = sh.prefix, total = sh.total, mytot = sh.slot_W[0];
    // Bound in fixed-point units: the element bounds (with margin for their own
    // fp32 summation), the rounding of p - q (2^-24 of the total), and one unit
    // of truncation per element.
    const float dunits = sh.D_tot * 1.0009765625f * 1.152921504606847e18f +
                         (float)total * 5.96046448e-08f + (float)V + 2.0f;
    const unsigned long long D = (unsigned long long)dunits + 1ull;

    const unsigned long long tau = scale_floor(u, total);
    const bool owner = total > 0 && mytot > 0 && prefix <= tau && tau - prefix < mytot;
    if (tid == 0) {
        sh.token = -1;
        sh.slot_cert = owner ? 0 : 1;
    }
    __syncthreads();
    if (owner) {
        const unsigned long long want = tau - prefix;
        int cstar;
        unsigned long long before;
        if (find_chunk(sh, csum, mych, want, &cstar, &before)) {
            float unused = 0.0f;
            int tok = -1;
            unsigned long long lo = 0, hi = 0;
            fast_chunk<DT>(rowp, qrow, (c0 + cstar) * kChunk, V, al_l, al_q, residual, m, c, inv,
                           &unused, want - before, &tok, &lo, &hi);
            // bin edges relative to `want`: want - (before + lo) >= 2D and
            // (before + hi) - want > 2D + 1 certify the bin
            const unsigned long long below = want - before - lo, above = before + hi - want;
            sh.token = tok;
            sh.slot_cert = (tok >= 0 && below >= 2 * D && above > 2 * D + 1) ? 1 : 0;
        }
    }
    cluster.sync();
    if (warp == 0) {
        int ok = lane < G ? *cluster.map_shared_rank(&sh.slot_cert, lane) : 1;
        ok = __all_sync(0xffffffffu, ok);
        if (lane == 0) sh.cert_all = ok && total > 0;
    }
    __syncthreads();
    return sh.cert_all != 0;
}

// ---- precise pass: float-float exponentials, exact integer prefix sums

// Chunk-level weight of the chunk starting at element j0: the float-float sum of
// its eight weights, quantised.  Element-level cumulative values inside the
// chunk are quantisations of the partial sums in the same order, so the last
// one equals the chunk value exactly.  With `token` set, the first element
// whose cumulative value exceeds `want` is stored there.
template <typename DT>
__device__ __forceinline__ unsigned long long chunk_weight(
    const DT* __restrict__ rowp, const float* __restrict__ qrow, long long j0, int V, bool al_l,
    bool al_q, bool residual, float m, ff c, ff inv, const DrawShared& sh,
    unsigned long long want, int* token) {
    float lf[kChunk], qf[kChunk];
    load_chunk<DT>(rowp, j0, V, al_l, lf);
    if (residual) load_q_chunk(qrow, j0, V, al_q, qf);
    ff acc{0.0f, 0.0f};
#pragma unroll
    for (int e = 0; e < kChunk; ++e) {
        ff ev = exp_rel(lf[e], m, c, sh.thi, sh.tlo);
        ff w = draw_weight(ev, inv, residual ? qf[e] : 0.0f, residual);
        ff_accumulate(acc, w);
        if (token && *token < 0 && w.hi > 0.0f && to_fixed(ff_normalize(acc)) > want)
            *token = (int)(j0 + e);
    }
    return to_fixed(ff_normalize(acc));
}

// The precise draw on one row by the G CTAs of a cluster (rank r owns chunks
// [nch*r/G, nch*(r+1)/G)).  The owner CTA holds the token in sh.token;
// `degenerate` is set in all threads.
template <typename DT>
__device__ void draw_precise(cg::cluster_group& cluster, DrawShared& sh,
                             unsigned long long* csum, const DT* __restrict__ rowp,
                             const float* __restrict__ qrow, bool residual, int V, float m, ff c,
                             float u, int rank, int G, bool& degenerate) {
    const int tid = threadIdx.x;
    const bool al_l = (reinterpret_cast<uintptr_t>(rowp) & 15) == 0;
    const bool al_q = residual && (reinterpret_cast<uintptr_t>(qrow) & 15) == 0;
    const long long nch = (V + kChunk - 1) / kChunk;
    const long long c0 = nch * rank / G, c1 = nch * (rank + 1) / G;
    const int mych = (int)(c1 - c0);

    // Pass A: e_j = exp((l_j - m)/T) and the normaliser S = sum_j e_j.
    ff acc{0.0f, 0.0f};
    for (int ci = tid; ci < mych; ci += kThreads) {
        float f[kChunk];
        load_chunk<DT>(rowp, (c0 + ci) * kChunk, V, al_l, f);
#pragma unroll
        for (int e = 0; e < kChunk; ++e) ff_accumulate(acc, exp_rel(f[e], m, c, sh.thi, sh.tlo));
    }
    const ff inv = ff_recip(cluster_sum_ff(cluster, sh, acc, G));

    // Pass B: chunk weights, CTA total, cluster prefix; a second round draws
    // from p when the residual has no mass.
    bool use_res = residual;
    degenerate = false;
    unsigned long long prefix = 0, total = 0, mytot = 0;
    for (int round = 0; round < 2; ++round) {
        unsigned long long tacc = 0;
        for (int ci = tid; ci < mych; ci += kThreads) {
            unsigned long long cs = chunk_weight<DT>(rowp, qrow, (c0 + ci) * kChunk, V, al_l,
                                                     al_q, use_res, m, c, inv, sh, 0ull, nullptr);
            csum[ci] = cs;
            tacc += cs;
        }
        cluster_prefix(cluster, sh, tacc, 0.0f, 1 + round, rank, G);
        prefix = sh.prefix;
        total = sh.total;
        mytot = sh.slot_W[1 + round];
        if (total > 0 || !use_res) break;
        use_res = false;  // zero residual mass: draw from p (counted)
        degenerate = true;
    }

    const unsigned long long tau = scale_floor(u, total);
    const bool owner = mytot > 0 && prefix <= tau && tau - prefix < mytot;
    if (owner) {
        const unsigned long long want = tau - prefix;
        int cstar;
        unsigned long long before;
        if (find_chunk(sh, csum, mych, want, &cstar, &before)) {
            int tok = -1;
            chunk_weight<DT>(rowp, qrow, (c0 + cstar) * kChunk, V, al_l, al_q, use_res, m, c,
                             inv, sh, want - before, &tok);
            sh.token = tok;
        }
    }
}

// The draw: the certified fast pass, and the precise pass when the fast one
// cannot certify its bin (or when `force_precise`).  Every CTA calls it; the
// owner CTA's thread 0 writes the token to *token_out.  Sets `degenerate` and
// `fallback` in all threads.
template <typename DT>
__device__ void draw(cg::cluster_group& cluster, DrawShared& sh, unsigned long long* csum,
                     const DT* __restrict__ rowp, const float* __restrict__ qrow, bool residual,
                     int V, float m, float c, ff c2, float u, int rank, int G, bool force_precise,
                     int32_t* token_out, bool& degenerate, bool& fallback) {
    degenerate = false;
    fallback = true;
    if (!force_precise && draw_fast<DT>(cluster, sh, csum, rowp, qrow, residual, V, m, c, u, rank,
                                        G)) {
        fallback = false;
        if (threadIdx.x == 0 && sh.token >= 0) *token_out = sh.token;
        return;
    }
    if (threadIdx.x == 0) sh.token = -1;
    __syncthreads();
    draw_precise<DT>(cluster, sh, csum, rowp, qrow, residual, V, m, c2, u, rank, G, degenerate);
    __syncthreads();
    if (threadIdx.x == 0 && sh.token >= 0) *token_out = sh.token;
}

// ------------------------------------------------------------------ the fused kernel

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
    int B, k, V, G, W;
    int force_precise;  // test hook: skip the fast draw
    float c;     // log2(e)/T (float, for the row statistics and the fast draw)
    ff c2;       // log2(e)/T in float-float (p(x) and the precise draw)
};

struct FusedShared {
    Partial wpart[kWarps];
    Partial part[2][kWarps];   // this CTA's per-row partials of a wave (read through DSMEM)
    Partial rowstat[kWarps];   // merged statistics of the wave's rows
    float lx[kMaxK], qx[kMaxK], ua[kMaxK];
    int xs[kMaxK];
    uint32_t gfl[kMaxK];
    float px[kWarps];
    int n, bits;
};

template <typename DT, bool SAMPLED>
__global__ void __launch_bounds__(kThreads) sv_verify_kernel(VerifyArgs a) {
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
    if (SAMPLED) load_exp_table(ds);
    if (tid == 0) {
        fs.n = -1;
        fs.bits = 0;
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
        const long long vb = nvec * rank / G, ve = nvec * (rank + 1) / G;
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
        if (tid == 0) {  // the scan over this wave's rows
            int n = -1, bits = 0;
            for (int ww = 0; ww < Wc; ++ww) {
                const int i = i0 + ww;
                const Partial& r = fs.rowstat[ww];
                if (row_flags<SAMPLED>(r) & kRowBad) { bits = SV_DEV_BAD_ROW; break; }
                if (i == k) { n = k; break; }
                if (fs.gfl[i] & kRowTokenBad) { bits = SV_DEV_BAD_TOKEN; break; }
                bool accept;
                if (SAMPLED) {
                    const float u = fs.ua[i];
                    if (!(u >= 0.0f && u < 1.0f)) { bits = SV_DEV_BAD_UNIFORM; break; }
                    if (fs.gfl[i] & kRowQBad) { bits = SV_DEV_BAD_Q; break; }
                    ff ex = exp_rel(fs.lx[i], r.m, a.c2, ds.thi, ds.tlo);
                    const float P = __fdiv_rn(ex.hi, r.s);
                    const float Q = fs.qx[i];
                    fs.px[ww] = P;
                    accept = (P >= Q) || (u < __fdiv_rn(P, Q));
                } else {
                    accept = fs.xs[i] == r.idx;
                }
                if (!accept) { n = i; break; }
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
        for (int i = last_wave_end + tid; i <= k; i += kThreads) {
            RowRec rec;
            rec.mraw = NAN;
            rec.S = NAN;
            rec.px = NAN;
            rec.lx = NAN;
            rec.qx = NAN;
            rec.argmax = -1;
            rec.flags = kRowSkipped;
            a.rows[(long long)b * (k + 1) + i] = rec;
        }

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
            }
        }
        if (G > 1) cluster.sync();  // partial slots may still be read by other ranks
        return;
    }

    // ---- the draw on row n, then the outputs
    const float u = a.ur[b];
    if (!(u >= 0.0f && u < 1.0f)) {  // every CTA sees the same uniform
        if (rank == 0) {
            for (int i = tid; i <= k; i += kThreads) o[i] = -1;
            if (tid == 0) {
                a.nacc[b] = -1;
                a.seqstat[b] = SV_DEV_BAD_UNIFORM;
            }
        }
        if (G > 1) cluster.sync();
        return;
    }
    const DT* drow = seq_logits + (long long)n * V;
    const float* qrow = n < k ? a.q + ((long long)b * k + n) * V : nullptr;
    const float m = fs.rowstat[n - wave_row0].m;
    bool degenerate = false, fallback = false;
    draw<DT>(cluster, ds, reinterpret_cast<unsigned long long*>(dyn), drow, qrow, n < k, V, m, a.c,
             a.c2, u, rank, G, a.force_precise != 0, o + n, degenerate, fallback);
    if (rank == 0) {
        for (int i = tid; i <= k; i += kThreads)
            if (i != n) o[i] = i < n ? fs.xs[i] : -1;
        if (tid == 0) {
            a.nacc[b] = n;
            a.seqstat[b] = (degenerate ? SV_DEV_DEGENERATE : 0u) | (fallback ? SV_DEV_PRECISE : 0u);
        }
    }
    cluster.sync();  // no CTA leaves while another may still read its slots
}

// ------------------------------------------------------------------ two-stage kernels

struct RowsArgs {
    const void* logits;
    const float* q;
    const int32_t* x;
    Header* hdr;
    RowRec* rows;
    int B, k, V, G, mode;
    float c;        // log2(e) / T
    ff c2;          // log2(e) / T in float-float (p(x))
};

// One CTA (or a cluster of G CTAs splitting the vocabulary) per row.
template <typename DT, bool SAMPLED, int NT>
__global__ void __launch_bounds__(NT) sv_rows_kernel(RowsArgs a) {
    using E = Elt<DT>;
    constexpr int NW = NT / 32;
    __shared__ Partial wpart[NW];
    __shared__ Partial cta_part;  // read by cluster rank 0 through DSMEM
    __shared__ float thi[SAMPLED ? kExpTable : 1], tlo[SAMPLED ? kExpTable : 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.G;
    const long long row = blockIdx.x / G;
    const int rank = blockIdx.x % G;
    const int V = a.V;
    const DT* rowp = static_cast<const DT*>(a.logits) + row * (long long)V;
    const int b = (int)(row / (a.k + 1));
    const int i = (int)(row % (a.k + 1));
    // The finish kernel is launched as a programmatic dependent: let it start
    // its launch now; it waits (griddepcontrol.wait) for this grid's results.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (blockIdx.x == 0 && tid == 0) {
        a.hdr->magic = kMagic;
        a.hdr->B = a.B;
        a.hdr->k = a.k;
        a.hdr->V = V;
        a.hdr->mode = a.mode;
    }
    int head;
    long long nvec, tail0;
    row_layout<DT>(rowp, V, head, nvec, tail0);
    const long long vb = nvec * rank / G, ve = nvec * (rank + 1) / G;
    Partial p = stream_slice<DT, SAMPLED, 4>(rowp, V, vb, ve, head, tail0, rank == 0,
                                             rank == G - 1, tid, NT, a.c);
    p = warp_merge<SAMPLED>(p, a.c);
    if (lane == 0) wpart[warp] = p;
    __syncthreads();
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
    if (rank != 0) return;
    if (SAMPLED && i < a.k) {
        for (int t = tid; t < kExpTable; t += NT) {
            thi[t] = g_exp2_table.hi[t];
            tlo[t] = g_exp2_table.lo[t];
        }
        __syncthreads();
    }
    if (tid != 0) return;
    RowRec rec;
    rec.mraw = p.m;
    rec.S = SAMPLED ? p.s : 0.0f;
    rec.argmax = p.idx < 0 ? 0 : p.idx;
    rec.px = 0.0;
    rec.lx = NAN;
    rec.qx = NAN;
    uint32_t fl = row_flags<SAMPLED>(p);
    if (i < a.k) {
        const int xi = a.x[(long long)b * a.k + i];
        if (xi < 0 || xi >= V) {
            fl |= kRowTokenBad;
        } else {
            rec.lx = E::load1(rowp + xi);
            if (SAMPLED) {
                rec.qx = a.q[((long long)b * a.k + i) * V + xi];
                if (!(rec.qx >= 0.0f)) fl |= kRowQBad;
                if (!(fl & kRowBad)) {
                    ff ex = exp_rel(rec.lx, p.m, a.c2, thi, tlo);
                    rec.px = (double)__fdiv_rn(ex.hi, p.s);
                }
            }
        }
    } else {
        rec.px = NAN;
    }
    rec.flags = fl;
    a.rows[row] = rec;
}

// One warp per sequence: the lanes load the records in parallel, lane 0 scans.
__global__ void sv_finish_greedy_kernel(const int32_t* __restrict__ x,
                                        const RowRec* __restrict__ rows,
                                        uint32_t* __restrict__ seqstat, int B, int k,
                                        int32_t* __restrict__ out, int32_t* __restrict__ nacc) {
    __shared__ RowRec recs[4][kMaxK + 1];
    __shared__ int xs[4][kMaxK];
    const int wi = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * 4 + wi;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the row records are complete
    if (b >= B) return;
    RowRec* rr = recs[wi];
    int* xx = xs[wi];
    for (int i = lane; i <= k; i += 32) rr[i] = rows[(long long)b * (k + 1) + i];
    for (int i = lane; i < k; i += 32) xx[i] = x[(long long)b * k + i];
    __syncwarp();
    if (lane != 0) return;
    int32_t* o = out + (long long)b * (k + 1);
    uint32_t bits = 0;
    int n = k;
    for (int i = 0; i < k; ++i) {
        if (rr[i].flags & kRowBad) { bits = SV_DEV_BAD_ROW; break; }
        if (rr[i].flags & kRowTokenBad) { bits = SV_DEV_BAD_TOKEN; break; }
        if (xx[i] != rr[i].argmax) { n = i; break; }
    }
    if (!bits && (rr[n].flags & kRowBad)) bits = SV_DEV_BAD_ROW;
    seqstat[b] = bits;
    if (bits) {
        for (int i = 0; i <= k; ++i) o[i] = -1;
        nacc[b] = -1;
        return;
    }
    for (int i = 0; i < n; ++i) o[i] = xx[i];
    o[n] = rr[n].argmax;
    for (int i = n + 1; i <= k; ++i) o[i] = -1;
    nacc[b] = n;
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
    int B, k, V, G;
    int force_precise;
    float c;
    ff c2;
};

template <typename DT>
__global__ void __launch_bounds__(kThreads) sv_finish_sample_kernel(FinishArgs a) {
    extern __shared__ __align__(16) unsigned char dyn[];
    __shared__ DrawShared ds;
    __shared__ RowRec recs[kMaxK + 1];
    __shared__ float uas[kMaxK];
    __shared__ int s_n, s_bits;
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x;
    const int G = a.G;
    const int b = blockIdx.x / G;
    const int rank = blockIdx.x % G;
    const int k = a.k, V = a.V;
    load_exp_table(ds);
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the row records are complete
    for (int i = tid; i <= k; i += kThreads) recs[i] = a.rows[(long long)b * (k + 1) + i];
    for (int i = tid; i < k; i += kThreads) uas[i] = a.ua[(long long)b * k + i];
    __syncthreads();
    if (tid == 0) {
        int bits = 0, n = k;
        for (int i = 0; i < k; ++i) {
            const RowRec& r = recs[i];
            if (r.flags & kRowBad) { bits = SV_DEV_BAD_ROW; break; }
            if (r.flags & kRowTokenBad) { bits = SV_DEV_BAD_TOKEN; break; }
            const float u = uas[i];
            if (!(u >= 0.0f && u < 1.0f)) { bits = SV_DEV_BAD_UNIFORM; break; }
            if (r.flags & kRowQBad) { bits = SV_DEV_BAD_Q; break; }
            const float P = (float)r.px, Q = r.qx;
            if (!((P >= Q) || (u < __fdiv_rn(P, Q)))) { n = i; break; }
        }
        if (!bits && (recs[n].flags & kRowBad)) bits = SV_DEV_BAD_ROW;
        if (!bits) {
            const float u = a.ur[b];
            if (!(u >= 0.0f && u < 1.0f)) bits = SV_DEV_BAD_UNIFORM;
        }
        s_n = n;
        s_bits = bits;
    }
    __syncthreads();
    const int n = s_n;
    int32_t* o = a.out + (long long)b * (k + 1);
    if (s_bits) {
        if (rank == 0) {
            for (int i = tid; i <= k; i += kThreads) o[i] = -1;
            if (tid == 0) {
                a.nacc[b] = -1;
                a.seqstat[b] = (uint32_t)s_bits;
            }
        }
        return;  // every CTA of the cluster takes this branch together
    }
    const DT* drow = static_cast<const DT*>(a.logits) + ((long long)b * (k + 1) + n) * V;
    const float* qrow = n < k ? a.q + ((long long)b * k + n) * V : nullptr;
    bool degenerate = false, fallback = false;
    draw<DT>(cluster, ds, reinterpret_cast<unsigned long long*>(dyn), drow, qrow, n < k, V,
             recs[n].mraw, a.c, a.c2, a.ur[b], rank, G, a.force_precise != 0, o + n, degenerate,
             fallback);
    if (rank == 0) {
        for (int i = tid; i <= k; i += kThreads)
            if (i != n) o[i] = i < n ? a.x[(long long)b * k + i] : -1;
        if (tid == 0) {
            a.nacc[b] = n;
            a.seqstat[b] = (degenerate ? SV_DEV_DEGENERATE : 0u) | (fallback ? SV_DEV_PRECISE : 0u);
        }
    }
    cluster.sync();
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

// Test hook (spec_verify_debug_force_precise): every draw takes the precise pass.
static std::atomic<int> g_force_precise{0};


struct DeviceInfo {
    int sms = 0;
    bool ok = false;
    bool configured = false;
};
static std::mutex g_mu;
static DeviceInfo g_dev[64];

constexpr size_t kDynSmemMax = 160 * 1024;  // chunk sums: up to kSliceMax bytes

template <typename K> static cudaError_t cluster_attrs(K kernel, bool dyn) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess && dyn)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kDynSmemMax);
    return e;
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
            SV_TRY(cluster_attrs(sv_finish_sample_kernel<__nv_bfloat16>, true));
            SV_TRY(cluster_attrs(sv_finish_sample_kernel<float>, true));
            SV_TRY(cluster_attrs(sv_rows_kernel<__nv_bfloat16, true, 128>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<__nv_bfloat16, true, 256>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<__nv_bfloat16, true, 512>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<__nv_bfloat16, false, 128>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<__nv_bfloat16, false, 256>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<__nv_bfloat16, false, 512>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<float, true, 128>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<float, true, 256>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<float, true, 512>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<float, false, 128>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<float, false, 256>, false));
            SV_TRY(cluster_attrs(sv_rows_kernel<float, false, 512>, false));
#undef SV_TRY
            if (e != cudaSuccess) return SV_ERR_CUDA;
        }
        d.configured = true;
    }
    if (!d.ok) return SV_ERR_UNSUPPORTED;
    *sms = d.sms;
    return SV_OK;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

static sv_status check_common(const void* logits, sv_dtype dt, const int32_t* x, int B, int k,
                              int V, void* ws, size_t ws_bytes) {
    if (dt != SV_BF16 && dt != SV_F32) return SV_ERR_INVALID_ARG;
    if (B < 0 || k < 1 || V < 1) return SV_ERR_INVALID_ARG;
    if (k > kMaxK || V > kMaxV) return SV_ERR_UNSUPPORTED;
    if ((long double)B * (k + 1) * V >= (long double)(1ll << 40)) return SV_ERR_UNSUPPORTED;
    if ((long long)B * (k + 1) * 16 >= (1ll << 31)) return SV_ERR_UNSUPPORTED;  // grid size
    if (B > 0 && (!logits || !x)) return SV_ERR_INVALID_ARG;
    if (B > 0 && (!aligned16(logits) || !aligned16(x))) return SV_ERR_INVALID_ARG;
    if (!ws) return SV_ERR_WORKSPACE;
    if (!aligned16(ws)) return SV_ERR_INVALID_ARG;
    if (ws_bytes < ws_bytes_for(B, k)) return SV_ERR_WORKSPACE;
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

static cudaLaunchAttribute cluster_attr(int G) {
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = G;
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    return at;
}

// Cluster size of the per-sequence kernels.  Sampled: about four CTAs per SM
// over the whole batch (a 512-thread CTA of these kernels needs little shared
// memory, so four fit on an SM), but no CTA draws from more than kSliceMax
// elements of a row and none from fewer than 2048.  Greedy: enough CTAs to give
// each SM four, with at least 4 KiB of every row per CTA.
static int seq_split(bool sampled, int B, int V, int esz, int sms) {
    int G = 1;
    if (sampled) {
        while (G < 16 && (V + G - 1) / G > kSliceMax) G *= 2;
        while (G < 16 && (long long)B * G * 2 <= 4LL * sms && V / (2 * G) >= 2048) G *= 2;
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

static sv_status launch_fused(bool sampled, const void* logits, sv_dtype dt, const float* q,
                              const int32_t* x, const float* ua, const float* ur, float T, int B,
                              int k, int V, int32_t* out, int32_t* nacc, void* ws,
                              cudaStream_t stream, int sms) {
    VerifyArgs a;
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
    a.force_precise = g_force_precise.load();
    size_t smem = 0;
    if (sampled) {
        const long long nch = (V + kChunk - 1) / kChunk;
        smem = (size_t)((nch + a.G - 1) / a.G) * 8;  // chunk sums of this CTA's slice
        if (smem > kDynSmemMax) return SV_ERR_UNSUPPORTED;
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
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// Vocabulary split of the per-row kernel: enough CTAs to give every SM about
// four, while keeping each CTA's slice at 512 16-byte vectors (8 KiB) or more.
static int rows_split(long long R, long long nvec_row, int sms) {
    int G = 1;
    while (G < 16 && R * G < 4LL * sms && nvec_row / (2LL * G) >= 512) G *= 2;
    return G;
}

// Threads per CTA: at least two vectors per thread, and the whole grid resident
// at once when it can be (2048 threads per SM), so that no wave tail forms.
static int rows_threads(long long ctas, long long nvec_cta, int sms) {
    int t = 512;
    while (t > 128 && (nvec_cta < 2LL * t || ctas * t > 2048LL * sms)) t /= 2;
    return t;
}

static sv_status launch_rows(bool sampled, const void* logits, sv_dtype dt, const float* q,
                             const int32_t* x, float T, int B, int k, int V, void* ws,
                             cudaStream_t stream, int sms) {
    const long long R = (long long)B * (k + 1);
    RowsArgs a;
    a.logits = logits;
    a.q = q;
    a.x = x;
    a.hdr = static_cast<Header*>(ws);
    a.rows = reinterpret_cast<RowRec*>(static_cast<char*>(ws) + ws_rows_offset());
    a.B = B;
    a.k = k;
    a.V = V;
    a.mode = sampled ? SV_MODE_SAMPLE : SV_MODE_GREEDY;
    a.c2 = log2e_over(sampled ? T : 1.0f);
    a.c = a.c2.hi;
    const int esz = dt == SV_BF16 ? 2 : 4;
    const long long nvec_row = ((long long)V * esz + 15) / 16;
    a.G = rows_split(R, nvec_row, sms);
    const int nt = rows_threads(R * a.G, nvec_row / a.G, sms);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(R * a.G), 1, 1);
    cfg.blockDim = dim3(nt, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {cluster_attr(a.G)};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
#define SV_ROWS(DTY, S)                                                          \
    e = nt == 512   ? cudaLaunchKernelEx(&cfg, sv_rows_kernel<DTY, S, 512>, a)     \
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

static sv_status launch_finish(bool sampled, const void* logits, sv_dtype dt, const float* q,
                               const int32_t* x, const float* ua, const float* ur, float T,
                               int B, int k, int V, int32_t* out, int32_t* nacc, void* ws,
                               cudaStream_t stream, int sms) {
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
        e = cudaLaunchKernelEx(&cfg, sv_finish_greedy_kernel, x, rows, seqstat, B, k, out, nacc);
        return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
    }
    FinishArgs a;
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
    a.G = seq_split(true, B, V, dt == SV_BF16 ? 2 : 4, sms);
    a.c2 = log2e_over(T);
    a.c = a.c2.hi;
    a.force_precise = g_force_precise.load();
    const long long nch = (V + kChunk - 1) / kChunk;
    const size_t smem = (size_t)((nch + a.G - 1) / a.G) * 8;
    if (smem > kDynSmemMax) return SV_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((long long)B * a.G), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2] = {cluster_attr(a.G), pdl};
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = dt == SV_BF16 ? cudaLaunchKernelEx(&cfg, sv_finish_sample_kernel<__nv_bfloat16>, a)
                      : cudaLaunchKernelEx(&cfg, sv_finish_sample_kernel<float>, a);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

// The one-call entry points run the fused per-sequence kernel (rows read in
// waves, early exit) when the batch alone has a sequence for every SM; smaller
// batches take the two-kernel path, whose row stream spreads every row over
// all SMs.
// Test hook (spec_verify_debug_force_path): 0 automatic, 1 two-kernel, 2 fused.
static std::atomic<int> g_force_path{0};
static bool prefer_fused(int B, int sms) {
    const int f = g_force_path.load();
    return f == 2 || (f == 0 && B >= sms);
}

}  // namespace sv

using namespace sv;

extern "C" {

size_t spec_verify_workspace_size(int B, int k, int V, sv_dtype dtype) {
    if (B < 0 || k < 1 || V < 1 || k > kMaxK || V > kMaxV) return 0;
    if (dtype != SV_BF16 && dtype != SV_F32) return 0;
    return ws_bytes_for(B, k);
}

sv_status spec_verify_rows(sv_mode mode, const void* logits, sv_dtype dtype,
                           const float* draft_probs, const int32_t* draft_tokens, float T, int B,
                           int k, int V, void* ws, size_t ws_bytes, cudaStream_t stream) {
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
    return launch_rows(sampled, logits, dtype, draft_probs, draft_tokens, T, B, k, V, ws, stream,
                       sms);
}

sv_status spec_verify_finish(sv_mode mode, const void* logits, sv_dtype dtype,
                             const float* draft_probs, const int32_t* draft_tokens,
                             const float* u_accept, const float* u_resample, float T, int B,
                             int k, int V, int32_t* out_tokens, int32_t* num_accepted, void* ws,
                             size_t ws_bytes, cudaStream_t stream) {
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
                         T, B, k, V, out_tokens, num_accepted, ws, stream, sms);
}

sv_status spec_verify_greedy(const void* logits, sv_dtype dtype, const int32_t* draft_tokens,
                             int B, int k, int V, int32_t* out_tokens, int32_t* num_accepted,
                             void* ws, size_t ws_bytes, cudaStream_t stream) {
    sv_status st = check_common(logits, dtype, draft_tokens, B, k, V, ws, ws_bytes);
    if (st != SV_OK) return st;
    if ((st = check_outputs(out_tokens, num_accepted, B)) != SV_OK) return st;
    int sms = 0;
    if ((st = device_setup(&sms)) != SV_OK) return st;
    if (B == 0) return SV_OK;
    if (prefer_fused(B, sms))
        return launch_fused(false, logits, dtype, nullptr, draft_tokens, nullptr, nullptr, 1.0f, B,
                            k, V, out_tokens, num_accepted, ws, stream, sms);
    st = launch_rows(false, logits, dtype, nullptr, draft_tokens, 1.0f, B, k, V, ws, stream, sms);
    if (st != SV_OK) return st;
    return launch_finish(false, logits, dtype, nullptr, draft_tokens, nullptr, nullptr, 1.0f, B, k,
                         V, out_tokens, num_accepted, ws, stream, sms);
}

sv_status spec_verify_sample(const void* logits, sv_dtype dtype, const float* draft_probs,
                             const int32_t* draft_tokens, const float* u_accept,
                             const float* u_resample, float T, int B, int k, int V,
                             int32_t* out_tokens, int32_t* num_accepted, void* ws,
                             size_t ws_bytes, cudaStream_t stream) {
    sv_status st = check_common(logits, dtype, draft_tokens, B, k, V, ws, ws_bytes);
    if (st != SV_OK) return st;
    if ((st = check_outputs(out_tokens, num_accepted, B)) != SV_OK) return st;
    if ((st = check_sample(draft_probs, u_accept, u_resample, T, B)) != SV_OK) return st;
    int sms = 0;
    if ((st = device_setup(&sms)) != SV_OK) return st;
    if (B == 0) return SV_OK;
    if (prefer_fused(B, sms))
        return launch_fused(true, logits, dtype, draft_probs, draft_tokens, u_accept, u_resample,
                            T, B, k, V, out_tokens, num_accepted, ws, stream, sms);
    st = launch_rows(true, logits, dtype, draft_probs, draft_tokens, T, B, k, V, ws, stream, sms);
    if (st != SV_OK) return st;
    return launch_finish(true, logits, dtype, draft_probs, draft_tokens, u_accept, u_resample, T,
                         B, k, V, out_tokens, num_accepted, ws, stream, sms);
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
        if (m) m[r] = host[r].mraw;
        if (S) S[r] = host[r].S;
        if (argmax) argmax[r] = host[r].argmax;
        if (px) px[r] = (float)host[r].px;
        if (qx) qx[r] = host[r].qx;
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

// Test hook (declared in include/specverify_debug.h): route every sampled draw
// through the precise float-float pass (on != 0) or back to the certified fast
// pass with fallback (on == 0).  Affects launches made after the call.
void spec_verify_debug_force_precise(int on) { g_force_precise.store(on != 0 ? 1 : 0); }

// Test hook (declared in include/specverify_debug.h): choose the one-call path.
void spec_verify_debug_force_path(int path) { g_force_path.store(path >= 0 && path <= 2 ? path : 0); }

// Introspection (declared in include/specverify_debug.h): 1 if the one-call
// entry points run the fused per-sequence kernel for a batch of B sequences on
// the current device, 0 for the two-kernel path, -1 on error.
int spec_verify_debug_uses_fused(int B) {
    int sms = 0;
    if (device_setup(&sms) != SV_OK) return -1;
    return prefer_fused(B, sms) ? 1 : 0;
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
                                          4 * (size_t)(SV_NOALLOC_MAX_ROWS / 2) + 255,
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
    return spec_verify_sample(logits, dtype, draft_probs, draft_tokens, u_accept, u_resample, T,
                              B, k, V, out_tokens, num_accepted, ws, sv::kNoAllocScratchBytes,
                              stream);
}
