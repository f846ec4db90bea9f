// specverify: batched speculative-decoding verify on GB300 (sm_103a).
//
// Three kernels, launched back to back on the caller's stream:
//
//  1. sv_rows_kernel — the only pass over the whole logits tensor.  One CTA (or
//     one thread-block cluster of G CTAs splitting the vocabulary when there are
//     too few rows to fill the 152 SMs) streams each row once with 16-byte
//     coalesced loads and keeps an online max / sum-of-exponentials per thread
//     (one ex2 per element, rescaled only when the running max moves), plus the
//     first index of the maximum.  Threads merge with warp shuffles, warps through
//     shared memory, and the CTAs of a cluster through distributed shared memory
//     (DSMEM) into rank 0, which gathers l(x) and q(x) for the row's draft token
//     and writes one 32-byte record per row to the workspace.
//     Softmax statistics: "Speculative Decoding" (ch15, LLM serving from
//     scratch), §"Why the result is exactly the target model" (accept_sampled
//     takes the target logits); p = softmax(l/T).
//  2. sv_scan_greedy_kernel (greedy) — one thread per sequence: accept while the
//     draft equals the row's argmax, emit argmax at the first mismatch or the
//     bonus ("Decodificação especulativa explicada: rascunhe barato, verifique
//     numa passada", §"A regra de amostragem por rejeição", greedy case).
//  3. sv_draw_kernel (sampled) — one cluster per sequence: the accept scan on
//     the row records (min(1, p/q) in double, §"A regra de amostragem por
//     rejeição", rule 1), then the draw from the one decision row: the residual
//     norm(max(0, p - q)) at a rejection (rule 2) or p itself for the bonus
//     (rule 3).  The draw recomputes that row's exponentials in float-float,
//     sums them exactly enough (~2^-47) for the normaliser, turns every weight
//     into a 62-bit fixed-point integer so that all prefix sums are exact and
//     order-independent, and locates the first j with C_j > u * C_{V-1} (the
//     right-sided search of §"Amostragem especulativa em numpy, com prova")
//     with a cluster-wide exclusive scan through DSMEM.
//
// Nothing here allocates memory, synchronises the host, or waits on another
// CTA outside hardware cluster barriers.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/specverify.h"
#include "ff.cuh"

namespace cg = cooperative_groups;

namespace sv {

// ------------------------------------------------------------------ workspace

constexpr uint32_t kMagic = 0x53564631u;  // "SVF1"
constexpr int kMaxK = 64;
constexpr int kMaxV = 1 << 21;

struct alignas(16) Header {
    uint32_t status;
    uint32_t n_degenerate;
    uint32_t B, k, V, mode, magic;
    uint32_t pad[57];
};
static_assert(sizeof(Header) == 256, "header size");

// One record per logits row.
struct alignas(16) RowRec {
    float mraw;       // max_j l_j (raw logits)
    float S;          // sum_j 2^((l_j - mraw) * log2(e)/T)  (sampled mode)
    double px;        // p(x) = exp((l_x - mraw)/T) / S in double (sampled, rows < k)
    float lx;         // l[x]
    float qx;         // q[x]
    int32_t argmax;   // lowest index of the maximum raw logit
    uint32_t flags;   // kRow* bits
};
static_assert(sizeof(RowRec) == 32, "row record size");

constexpr uint32_t kRowBad = 1u, kRowTokenBad = 2u, kRowQBad = 4u;

__host__ __device__ inline size_t ws_bytes_for(long long R) {
    size_t b = sizeof(Header) + (size_t)R * sizeof(RowRec);
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

// Online softmax partial of one thread: running max m, sum s of 2^((l-m)c),
// index of the first maximum (or the first index of the 16-byte vector holding
// it, resolved at the end), and a NaN flag (greedy mode, which forms no sum).
struct Partial {
    float m, s;
    int idx;
    int vec;   // 1 if idx is the start of an unresolved vector
    int nan;
};

// Merge b into a (a holds lower-or-equal indices on ties only by the explicit
// index comparison, so the merge order does not matter).
template <bool SAMPLED>
__device__ __forceinline__ void merge(Partial& a, float bm, float bs, int bidx, int bnan,
                                      float c) {
    float mn = fmaxf(a.m, bm);
    if (SAMPLED) {
        float fa = (a.m == mn) ? 1.0f : ex2_approx((a.m - mn) * c);
        float fb = (bm == mn) ? 1.0f : ex2_approx((bm - mn) * c);
        a.s = a.s * fa + bs * fb;
    }
    if (bm > a.m || (bm == a.m && (unsigned)bidx < (unsigned)a.idx)) a.idx = bidx;
    a.m = mn;
    a.nan |= bnan;
}

// ------------------------------------------------------------------ kernel 1: row stream

struct RowsArgs {
    const void* logits;
    const float* q;
    const int32_t* x;
    Header* hdr;
    RowRec* rows;
    int B, k, V, G, mode;
    float c;        // log2(e) / T
    double T;
};

template <typename DT, bool SAMPLED, int kThreads>
__global__ void __launch_bounds__(kThreads) sv_rows_kernel(RowsArgs a) {
    using E = Elt<DT>;
    constexpr int VW = E::kVec;
    constexpr int kWarps = kThreads / 32;
    const int tid = threadIdx.x;
    const int G = a.G;
    const long long row = blockIdx.x / G;
    const int rank = blockIdx.x % G;  // == cluster rank: clusters are (G,1,1) along x
    const int V = a.V;
    const DT* rowp = static_cast<const DT*>(a.logits) + row * (long long)V;

    if (blockIdx.x == 0 && tid == 0) {
        a.hdr->status = 0;
        a.hdr->n_degenerate = 0;
        a.hdr->B = a.B;
        a.hdr->k = a.k;
        a.hdr->V = V;
        a.hdr->mode = a.mode;
        a.hdr->magic = kMagic;
    }

    // Gather of the draft token's logit and q (rank 0, last thread: issued early,
    // consumed at the end).
    const int b = (int)(row / (a.k + 1));
    const int i = (int)(row % (a.k + 1));
    int xi = -1;
    float lx = NAN, qx = NAN;
    uint32_t gflags = 0;
    if (rank == 0 && tid == kThreads - 1 && i < a.k) {
        xi = a.x[(long long)b * a.k + i];
        if (xi < 0 || xi >= V) {
            gflags |= kRowTokenBad;
        } else {
            lx = E::load1(rowp + xi);
            if (SAMPLED) qx = a.q[((long long)b * a.k + i) * V + xi];
        }
    }

    // Row layout: [0, head) unaligned scalars, then nvec 16-byte vectors, then a
    // scalar tail.  The vectors are split evenly over the G ranks.
    const uintptr_t addr = reinterpret_cast<uintptr_t>(rowp);
    int head = (int)(((16 - (addr & 15)) & 15) / sizeof(DT));
    if (head > V) head = V;
    const long long nvec = (V - head) / VW;
    const long long tail0 = head + nvec * VW;
    const long long vb = nvec * rank / G, ve = nvec * (rank + 1) / G;
    const uint4* vp = reinterpret_cast<const uint4*>(rowp + head);

    Partial p{-INFINITY, 0.0f, -1, 0, 0};
    const float c = a.c;

    auto scalar = [&](long long j) {
        float v = E::load1(rowp + j);
        if (!SAMPLED) p.nan |= (v != v);
        if (v > p.m) {
            if (SAMPLED) p.s *= ex2_approx((p.m - v) * c);
            p.m = v;
            p.idx = (int)j;
            p.vec = 0;
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
            p.vec = 1;
        }
        if (SAMPLED) {
            float acc = 0.0f;
#pragma unroll
            for (int e = 0; e < VW; ++e) acc += ex2_approx((f[e] - p.m) * c);
            p.s += acc;
        }
    };

    if (rank == 0)
        for (long long j = tid; j < head; j += kThreads) scalar(j);
    constexpr int U = 4;
    long long v = vb + tid;
    for (; v + (U - 1) * kThreads < ve; v += U * kThreads) {
        uint4 buf[U];
#pragma unroll
        for (int u = 0; u < U; ++u) buf[u] = ld_stream16(vp + v + u * kThreads);
#pragma unroll
        for (int u = 0; u < U; ++u) vector(buf[u], head + (v + u * kThreads) * VW);
    }
    for (; v < ve; v += kThreads) vector(ld_stream16(vp + v), head + v * VW);
    if (rank == G - 1)
        for (long long j = tail0 + tid; j < V; j += kThreads) scalar(j);

    // Resolve the index of the first maximum inside its vector.
    if (p.vec) {
        float f[VW];
        E::unpack(*reinterpret_cast<const uint4*>(rowp + p.idx), f);
        int e = 0;
        while (e < VW - 1 && !(f[e] == p.m)) ++e;
        p.idx += e;
        p.vec = 0;
    }

    // Warp, then CTA reduction.
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        float om = __shfl_xor_sync(0xffffffffu, p.m, off);
        float os = __shfl_xor_sync(0xffffffffu, p.s, off);
        int oi = __shfl_xor_sync(0xffffffffu, p.idx, off);
        int on = __shfl_xor_sync(0xffffffffu, p.nan, off);
        merge<SAMPLED>(p, om, os, oi, on, c);
    }
    __shared__ float sm_m[kWarps], sm_s[kWarps];
    __shared__ int sm_i[kWarps], sm_n[kWarps];
    __shared__ Partial cta_part;  // read by cluster rank 0 through DSMEM
    const int warp = tid >> 5, lane = tid & 31;
    if (lane == 0) {
        sm_m[warp] = p.m;
        sm_s[warp] = p.s;
        sm_i[warp] = p.idx;
        sm_n[warp] = p.nan;
    }
    __syncthreads();
    if (warp == 0) {
        Partial w{-INFINITY, 0.0f, -1, 0, 0};
        if (lane < kWarps) w = Partial{sm_m[lane], sm_s[lane], sm_i[lane], 0, sm_n[lane]};
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            float om = __shfl_xor_sync(0xffffffffu, w.m, off);
            float os = __shfl_xor_sync(0xffffffffu, w.s, off);
            int oi = __shfl_xor_sync(0xffffffffu, w.idx, off);
            int on = __shfl_xor_sync(0xffffffffu, w.nan, off);
            merge<SAMPLED>(w, om, os, oi, on, c);
        }
        p = w;
        if (lane == 0) cta_part = w;
    }

    if (G > 1) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        if (rank == 0 && warp == 0) {
            Partial w{-INFINITY, 0.0f, -1, 0, 0};
            if (lane < G) w = *cluster.map_shared_rank(&cta_part, lane);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                float om = __shfl_xor_sync(0xffffffffu, w.m, off);
                float os = __shfl_xor_sync(0xffffffffu, w.s, off);
                int oi = __shfl_xor_sync(0xffffffffu, w.idx, off);
                int on = __shfl_xor_sync(0xffffffffu, w.nan, off);
                merge<SAMPLED>(w, om, os, oi, on, c);
            }
            p = w;
        }
        cluster.sync();  // keep every CTA's shared memory alive until rank 0 has read it
    }

    if (rank != 0) return;
    // The gather lives in the last thread; hand it to thread 0 through shared memory.
    __shared__ int g_x;
    __shared__ float g_lx, g_qx;
    __shared__ uint32_t g_fl;
    if (tid == kThreads - 1) {
        g_x = xi;
        g_lx = lx;
        g_qx = qx;
        g_fl = gflags;
    }
    __syncthreads();
    if (tid != 0) return;
    RowRec rec;
    rec.mraw = p.m;
    rec.S = SAMPLED ? p.s : 0.0f;
    rec.argmax = p.idx < 0 ? 0 : p.idx;
    rec.lx = g_lx;
    rec.qx = g_qx;
    rec.px = 0.0;
    uint32_t fl = (i < a.k) ? g_fl : 0u;
    bool bad = !(p.m > -INFINITY) || p.m == INFINITY || p.nan;
    if (SAMPLED) bad = bad || !(p.s > 0.0f) || !(p.s < INFINITY);
    if (bad) fl |= kRowBad;
    if (SAMPLED && i < a.k && !(fl & (kRowBad | kRowTokenBad))) {
        if (!(rec.qx >= 0.0f)) fl |= kRowQBad;  // NaN or negative
        rec.px = exp(((double)rec.lx - (double)p.m) / a.T) / (double)p.s;
    }
    if (i == a.k) {
        rec.lx = NAN;
        rec.qx = NAN;
        rec.px = NAN;
    }
    rec.flags = fl;
    a.rows[row] = rec;
}

// ------------------------------------------------------------------ kernel 2: greedy scan

__global__ void sv_scan_greedy_kernel(const int32_t* __restrict__ x, const RowRec* __restrict__ rows,
                                      Header* hdr, int B, int k, int32_t* __restrict__ out,
                                      int32_t* __restrict__ nacc) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const RowRec* r = rows + (long long)b * (k + 1);
    int32_t* o = out + (long long)b * (k + 1);
    uint32_t bits = 0;
    int n = k;
    for (int i = 0; i < k; ++i) {
        uint32_t fl = r[i].flags;
        if (fl & kRowBad) { bits |= SV_DEV_BAD_ROW; break; }
        if (fl & kRowTokenBad) { bits |= SV_DEV_BAD_TOKEN; break; }
        if (x[(long long)b * k + i] != r[i].argmax) { n = i; break; }
    }
    if (!bits && (r[n].flags & kRowBad)) bits |= SV_DEV_BAD_ROW;
    if (bits) {
        for (int i = 0; i <= k; ++i) o[i] = -1;
        nacc[b] = -1;
        atomicOr(&hdr->status, bits);
        return;
    }
    for (int i = 0; i < n; ++i) o[i] = x[(long long)b * k + i];
    o[n] = r[n].argmax;
    for (int i = n + 1; i <= k; ++i) o[i] = -1;
    nacc[b] = n;
}

// ------------------------------------------------------------------ kernel 3: sampled scan + draw

constexpr int kDrawThreads = 512;
constexpr int kChunk = 8;           // contiguous elements per work item
constexpr int kSegMax = 16384;      // elements of one CTA's segment kept in shared memory

struct DrawArgs {
    const void* logits;
    const float* q;
    const int32_t* x;
    const float* ua;
    const float* ur;
    Header* hdr;
    const RowRec* rows;
    int32_t* out;
    int32_t* nacc;
    int B, k, V, G;
    ff rT;          // 1/T in float-float
    FFExpConst fc;
};

// uint64 fixed point: a weight w in [0, 1] becomes round(w * 2^62).
__device__ __forceinline__ unsigned long long quantize(ff w) {
    const float s = 4611686018427387904.0f;  // 2^62
    long long h = __float2ll_rn(__fmul_rn(w.hi, s));
    long long l = __float2ll_rn(__fmul_rn(w.lo, s));
    return (unsigned long long)(h + l);
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
    return (lo >> sh) | (sh == 0 ? 0ull : (hi << (64 - sh)));
}

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

// e_j = exp((l_j - m)/T) in float-float; 0 below exp(-44) (such a weight is
// below the 2^-62 resolution of the fixed-point sums once divided by S >= 1).
__device__ __forceinline__ ff exp_elem(float l, float m, ff rT, const float* thi,
                                       const float* tlo, const FFExpConst& fc) {
    ff d = two_sum(l, -m);
    ff y = ff_mul(d, rT);
    if (!(y.hi >= -44.0f)) return ff{0.0f, 0.0f};  // also -inf logits
    return ff_exp_neg(y, thi, tlo, fc.c1, fc.c2, fc.c3, fc.inv_l);
}

__device__ __forceinline__ ff weight(ff e, ff inv, float qv, bool residual) {
    ff p = ff_mul(e, inv);
    if (!residual) return p;
    ff s = two_sum(p.hi, -qv);
    ff w = fast_two_sum(s.hi, __fadd_rn(s.lo, p.lo));
    if (!(w.hi > 0.0f)) return ff{0.0f, 0.0f};
    if (w.hi > 1.0f) return ff{1.0f, 0.0f};  // only reachable with a negative q entry
    return w;
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

template <typename DT, bool STORE>
__global__ void __launch_bounds__(kDrawThreads) sv_draw_kernel(DrawArgs a) {
    constexpr int kWarps = kDrawThreads / 32;
    extern __shared__ __align__(16) unsigned char dyn[];
    __shared__ RowRec recs[kMaxK + 1];
    __shared__ float s_ua[kMaxK];
    __shared__ float thi[64], tlo[64];
    __shared__ int s_n, s_valid;
    __shared__ uint32_t s_bits;
    __shared__ ff red_ff[kWarps];
    __shared__ unsigned long long red_u[kWarps];
    __shared__ ff slot_S;                      // this CTA's partial normaliser (DSMEM)
    __shared__ unsigned long long slot_W[2];   // this CTA's residual / fallback totals (DSMEM)
    __shared__ unsigned long long s_scan[kDrawThreads];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.G;
    const int b = blockIdx.x / G;
    const int rank = blockIdx.x % G;
    const int k = a.k, V = a.V;

    if (tid < 64) {
        thi[tid] = a.fc.tbl_hi[tid];
        tlo[tid] = a.fc.tbl_lo[tid];
    }
    for (int i = tid; i <= k; i += kDrawThreads) recs[i] = a.rows[(long long)b * (k + 1) + i];
    for (int i = tid; i < k; i += kDrawThreads) s_ua[i] = a.ua[(long long)b * k + i];
    __syncthreads();

    // ---- accept scan (every CTA of the cluster computes the same result)
    if (tid == 0) {
        uint32_t bits = 0;
        int n = k;
        for (int i = 0; i < k; ++i) {
            const RowRec& r = recs[i];
            if (r.flags & kRowBad) { bits |= SV_DEV_BAD_ROW; break; }
            if (r.flags & kRowTokenBad) { bits |= SV_DEV_BAD_TOKEN; break; }
            float u = s_ua[i];
            if (!(u >= 0.0f && u < 1.0f)) { bits |= SV_DEV_BAD_UNIFORM; break; }
            if (r.flags & kRowQBad) { bits |= SV_DEV_BAD_Q; break; }
            double P = r.px, Q = (double)r.qx;
            bool accept = (P >= Q) || ((double)u < P / Q);
            if (!accept) { n = i; break; }
        }
        if (!bits && (recs[n].flags & kRowBad)) bits |= SV_DEV_BAD_ROW;
        if (!bits) {
            float u = a.ur[b];
            if (!(u >= 0.0f && u < 1.0f)) bits |= SV_DEV_BAD_UNIFORM;
        }
        s_n = n;
        s_bits = bits;
        s_valid = bits == 0;
    }
    __syncthreads();
    const int n = s_n;
    if (!s_valid) {
        if (rank == 0) {
            int32_t* o = a.out + (long long)b * (k + 1);
            for (int i = tid; i <= k; i += kDrawThreads) o[i] = -1;
            if (tid == 0) {
                a.nacc[b] = -1;
                atomicOr(&a.hdr->status, s_bits);
            }
        }
        return;  // every CTA of the cluster takes this branch together
    }

    // ---- the draw on row n
    cg::cluster_group cluster = cg::this_cluster();
    const long long rowid = (long long)b * (k + 1) + n;
    const DT* rowp = static_cast<const DT*>(a.logits) + rowid * V;
    const bool residual = n < k;
    const float* qrow = residual ? a.q + ((long long)b * k + n) * V : nullptr;
    const float m = recs[n].mraw;
    const float u = a.ur[b];
    const bool al_l = (reinterpret_cast<uintptr_t>(rowp) & 15) == 0;
    const bool al_q = residual && (reinterpret_cast<uintptr_t>(qrow) & 15) == 0;

    const long long nch = (V + kChunk - 1) / kChunk;
    const long long c0 = nch * rank / G, c1 = nch * (rank + 1) / G;
    const int mych = (int)(c1 - c0);
    float* ehi = reinterpret_cast<float*>(dyn);
    float* elo = ehi + (STORE ? kSegMax : 0);
    unsigned long long* csum =
        reinterpret_cast<unsigned long long*>(dyn + (STORE ? 2 * kSegMax * sizeof(float) : 0));

    // Pass A: e_j and the normaliser S = sum_j e_j.
    ff acc{0.0f, 0.0f};
    for (int c = tid; c < mych; c += kDrawThreads) {
        const long long j0 = (c0 + c) * kChunk;
        float f[kChunk];
        load_chunk<DT>(rowp, j0, V, al_l, f);
#pragma unroll
        for (int e = 0; e < kChunk; ++e) {
            ff ev = exp_elem(f[e], m, a.rT, thi, tlo, a.fc);
            if (STORE) {
                ehi[c * kChunk + e] = ev.hi;
                elo[c * kChunk + e] = ev.lo;
            }
            acc = ff_add(acc, ev);
        }
    }
    acc = warp_sum_ff(acc);
    if (lane == 0) red_ff[warp] = acc;
    __syncthreads();
    if (warp == 0) {
        ff w = lane < kWarps ? red_ff[lane] : ff{0.0f, 0.0f};
        w = warp_sum_ff(w);
        if (lane == 0) slot_S = w;
    }
    cluster.sync();
    ff S{0.0f, 0.0f};
    for (int r = 0; r < G; ++r) S = ff_add(S, *cluster.map_shared_rank(&slot_S, r));
    const ff inv = ff_recip(S);

    // Pass B: fixed-point weights, per-chunk sums, CTA total; cluster prefix.
    // A second round draws from p when the residual has no mass.
    unsigned long long prefix = 0, total = 0, mytot = 0;
    bool use_res = residual;
    bool degenerate = false;
    for (int round = 0; round < 2; ++round) {
        unsigned long long tacc = 0;
        for (int c = tid; c < mych; c += kDrawThreads) {
            const long long j0 = (c0 + c) * kChunk;
            float lf[kChunk], qf[kChunk];
            if (!STORE) load_chunk<DT>(rowp, j0, V, al_l, lf);
            if (use_res) load_q_chunk(qrow, j0, V, al_q, qf);
            unsigned long long cs = 0;
#pragma unroll
            for (int e = 0; e < kChunk; ++e) {
                ff ev = STORE ? ff{ehi[c * kChunk + e], elo[c * kChunk + e]}
                              : exp_elem(lf[e], m, a.rT, thi, tlo, a.fc);
                cs += quantize(weight(ev, inv, use_res ? qf[e] : 0.0f, use_res));
            }
            csum[c] = cs;
            tacc += cs;
        }
        tacc = warp_sum(tacc);
        if (lane == 0) red_u[warp] = tacc;
        __syncthreads();
        if (warp == 0) {
            unsigned long long w = lane < kWarps ? red_u[lane] : 0ull;
            w = warp_sum(w);
            if (lane == 0) slot_W[round] = w;
        }
        cluster.sync();
        prefix = 0;
        total = 0;
        for (int r = 0; r < G; ++r) {
            unsigned long long t = cluster.map_shared_rank(slot_W, r)[round];
            if (r < rank) prefix += t;
            total += t;
        }
        mytot = slot_W[round];
        if (total > 0 || !use_res) break;
        use_res = false;  // zero residual mass: draw from p (counted)
        degenerate = true;
    }

    const unsigned long long tau = scale_floor(u, total);
    const bool owner = mytot > 0 && prefix <= tau && tau - prefix < mytot;
    if (owner) {
        // Exclusive scan of the per-chunk sums in index order: thread t owns the
        // contiguous chunk range [t*L, (t+1)*L).
        const unsigned long long want = tau - prefix;
        const int L = (mych + kDrawThreads - 1) / kDrawThreads;
        const int cb = tid * L, ce = min(mych, cb + L);
        unsigned long long mine = 0;
        for (int c = cb; c < ce; ++c) mine += csum[c];
        // inclusive block scan through shared memory (Hillis-Steele)
        s_scan[tid] = mine;
        __syncthreads();
        for (int off = 1; off < kDrawThreads; off <<= 1) {
            unsigned long long add = tid >= off ? s_scan[tid - off] : 0ull;
            __syncthreads();
            s_scan[tid] += add;
            __syncthreads();
        }
        const unsigned long long excl = s_scan[tid] - mine;
        if (mine > 0 && excl <= want && want - excl < mine) {
            unsigned long long run = excl;
            int cstar = cb;
            for (; cstar < ce; ++cstar) {
                if (want - run < csum[cstar]) break;
                run += csum[cstar];
            }
            if (cstar >= ce) cstar = ce - 1;  // unreachable: mine covers `want`
            const long long j0 = (c0 + cstar) * kChunk;
            float lf[kChunk], qf[kChunk];
            if (!STORE) load_chunk<DT>(rowp, j0, V, al_l, lf);
            if (use_res) load_q_chunk(qrow, j0, V, al_q, qf);
            int tok = -1;
#pragma unroll
            for (int e = 0; e < kChunk; ++e) {
                ff ev = STORE ? ff{ehi[cstar * kChunk + e], elo[cstar * kChunk + e]}
                              : exp_elem(lf[e], m, a.rT, thi, tlo, a.fc);
                unsigned long long w = quantize(weight(ev, inv, use_res ? qf[e] : 0.0f, use_res));
                if (tok < 0 && w > 0 && want - run < w) tok = (int)(j0 + e);
                if (tok < 0) run += w;
            }
            a.out[(long long)b * (k + 1) + n] = tok;
        }
    }
    if (rank == 0) {
        int32_t* o = a.out + (long long)b * (k + 1);
        const int32_t* xs = a.x + (long long)b * k;
        for (int i = tid; i <= k; i += kDrawThreads) {
            if (i < n) o[i] = xs[i];
            else if (i > n) o[i] = -1;
        }
        if (tid == 0) {
            a.nacc[b] = n;
            if (degenerate) {
                atomicOr(&a.hdr->status, SV_DEV_DEGENERATE);
                atomicAdd(&a.hdr->n_degenerate, 1u);
            }
        }
    }
    cluster.sync();  // no CTA leaves while another may still read its slots
}

// ------------------------------------------------------------------ debug kernel

__global__ void sv_debug_ffexp_kernel(const float* l, float m, int n, ff rT, FFExpConst fc,
                                      double* out) {
    __shared__ float thi[64], tlo[64];
    if (threadIdx.x < 64) {
        thi[threadIdx.x] = fc.tbl_hi[threadIdx.x];
        tlo[threadIdx.x] = fc.tbl_lo[threadIdx.x];
    }
    __syncthreads();
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    ff e = exp_elem(l[i], m, rT, thi, tlo, fc);
    out[i] = (double)e.hi + (double)e.lo;
}

// ------------------------------------------------------------------ host side

static FFExpConst make_exp_const() {
    FFExpConst c;
    for (int i = 0; i < 64; ++i) {
        double v = std::exp2((double)i / 64.0);
        c.tbl_hi[i] = (float)v;
        c.tbl_lo[i] = (float)(v - (double)c.tbl_hi[i]);
    }
    const double L = std::log(2.0) / 64.0;
    int e;
    double f = std::frexp(L, &e);                      // L = f * 2^e, f in [0.5, 1)
    double c1 = std::ldexp(std::nearbyint(std::ldexp(f, 12)), e - 12);  // 12 significant bits
    c.c1 = (float)c1;
    c.c2 = (float)(L - c1);
    c.c3 = (float)(L - c1 - (double)c.c2);
    c.inv_l = (float)(64.0 / std::log(2.0));
    return c;
}

static const FFExpConst& exp_const() {
    static const FFExpConst c = make_exp_const();
    return c;
}

static ff make_rT(float T) {
    double r = 1.0 / (double)T;
    float hi = (float)r;
    return ff{hi, (float)(r - (double)hi)};
}

struct DeviceInfo {
    int sms = 0;
    bool ok = false;
    bool configured = false;
};
static std::mutex g_mu;
static DeviceInfo g_dev[64];

template <typename DT, bool SAMPLED, int NT> static cudaError_t set_rows_attr() {
    return cudaFuncSetAttribute(sv_rows_kernel<DT, SAMPLED, NT>,
                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}
template <typename DT, bool STORE> static cudaError_t set_draw_attr() {
    cudaError_t e = cudaFuncSetAttribute(sv_draw_kernel<DT, STORE>,
                                         cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(sv_draw_kernel<DT, STORE>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
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
            SV_TRY((set_rows_attr<__nv_bfloat16, true, 128>()));
            SV_TRY((set_rows_attr<__nv_bfloat16, true, 256>()));
            SV_TRY((set_rows_attr<__nv_bfloat16, true, 512>()));
            SV_TRY((set_rows_attr<__nv_bfloat16, false, 128>()));
            SV_TRY((set_rows_attr<__nv_bfloat16, false, 256>()));
            SV_TRY((set_rows_attr<__nv_bfloat16, false, 512>()));
            SV_TRY((set_rows_attr<float, true, 128>()));
            SV_TRY((set_rows_attr<float, true, 256>()));
            SV_TRY((set_rows_attr<float, true, 512>()));
            SV_TRY((set_rows_attr<float, false, 128>()));
            SV_TRY((set_rows_attr<float, false, 256>()));
            SV_TRY((set_rows_attr<float, false, 512>()));
            SV_TRY((set_draw_attr<__nv_bfloat16, true>()));
            SV_TRY((set_draw_attr<__nv_bfloat16, false>()));
            SV_TRY((set_draw_attr<float, true>()));
            SV_TRY((set_draw_attr<float, false>()));
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
    if (ws_bytes < ws_bytes_for((long long)B * (k + 1))) return SV_ERR_WORKSPACE;
    return SV_OK;
}

// Vocabulary split of the row stream: enough CTAs to give every SM about four,
// while keeping each CTA's slice at 512 16-byte vectors (8 KiB) or more.
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
    a.rows = reinterpret_cast<RowRec*>(static_cast<char*>(ws) + sizeof(Header));
    a.B = B;
    a.k = k;
    a.V = V;
    a.mode = sampled ? SV_MODE_SAMPLE : SV_MODE_GREEDY;
    a.T = sampled ? (double)T : 1.0;
    a.c = sampled ? (float)(1.4426950408889634 / (double)T) : 1.0f;
    const int esz = dt == SV_BF16 ? 2 : 4;
    const long long nvec_row = ((long long)V * esz + 15) / 16;
    a.G = rows_split(R, nvec_row, sms);
    const int nt = rows_threads(R * a.G, nvec_row / a.G, sms);

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(R * a.G), 1, 1);
    cfg.blockDim = dim3(nt, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
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

// Cluster size of the draw: each CTA's slice of the decision row fits in shared
// memory when possible (V <= 16 * 16384), and small batches spread wider.
static int draw_split(int B, int V, int sms) {
    int G = 1;
    while (G < 16 && (V + G - 1) / G > kSegMax) G *= 2;
    while (G < 16 && (long long)B * G < 2LL * sms && V / (2 * G) >= 2048) G *= 2;
    return G;
}

static sv_status launch_finish(bool sampled, const void* logits, sv_dtype dt, const float* q,
                               const int32_t* x, const float* ua, const float* ur, float T,
                               int B, int k, int V, int32_t* out, int32_t* nacc, void* ws,
                               cudaStream_t stream, int sms) {
    Header* hdr = static_cast<Header*>(ws);
    const RowRec* rows = reinterpret_cast<const RowRec*>(static_cast<char*>(ws) + sizeof(Header));
    cudaError_t e;
    if (!sampled) {
        const int nt = 128;
        sv_scan_greedy_kernel<<<(B + nt - 1) / nt, nt, 0, stream>>>(x, rows, hdr, B, k, out, nacc);
        e = cudaGetLastError();
        return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
    }
    DrawArgs a;
    a.logits = logits;
    a.q = q;
    a.x = x;
    a.ua = ua;
    a.ur = ur;
    a.hdr = hdr;
    a.rows = rows;
    a.out = out;
    a.nacc = nacc;
    a.B = B;
    a.k = k;
    a.V = V;
    a.G = draw_split(B, V, sms);
    a.rT = make_rT(T);
    a.fc = exp_const();
    const long long seg = ((long long)(V + kChunk - 1) / kChunk + a.G - 1) / a.G * kChunk;
    const bool store = seg <= kSegMax;
    const size_t nchunk_max = (size_t)(seg / kChunk + 1);
    const size_t smem = (store ? 2 * kSegMax * sizeof(float) : 0) + nchunk_max * 8;
    if (smem > 200 * 1024) return SV_ERR_UNSUPPORTED;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((long long)B * a.G), 1, 1);
    cfg.blockDim = dim3(kDrawThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dt == SV_BF16)
        e = store ? cudaLaunchKernelEx(&cfg, sv_draw_kernel<__nv_bfloat16, true>, a)
                  : cudaLaunchKernelEx(&cfg, sv_draw_kernel<__nv_bfloat16, false>, a);
    else
        e = store ? cudaLaunchKernelEx(&cfg, sv_draw_kernel<float, true>, a)
                  : cudaLaunchKernelEx(&cfg, sv_draw_kernel<float, false>, a);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

static sv_status check_sample(const float* q, const float* ua, const float* ur, float T, int B) {
    if (!(T > 0.0f) || !std::isfinite(T)) return SV_ERR_INVALID_ARG;
    if (B > 0 && (!q || !ua || !ur)) return SV_ERR_INVALID_ARG;
    if (B > 0 && (!aligned16(q) || !aligned16(ua) || !aligned16(ur))) return SV_ERR_INVALID_ARG;
    return SV_OK;
}

}  // namespace sv

using namespace sv;

extern "C" {

size_t spec_verify_workspace_size(int B, int k, int V, sv_dtype dtype) {
    if (B < 0 || k < 1 || V < 1 || k > kMaxK || V > kMaxV) return 0;
    if (dtype != SV_BF16 && dtype != SV_F32) return 0;
    return ws_bytes_for((long long)B * (k + 1));
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
    if (B > 0 && (!out_tokens || !num_accepted)) return SV_ERR_INVALID_ARG;
    if (B > 0 && (!aligned16(out_tokens) || !aligned16(num_accepted))) return SV_ERR_INVALID_ARG;
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
    if (B > 0 && (!out_tokens || !num_accepted)) return SV_ERR_INVALID_ARG;
    if (B > 0 && (!aligned16(out_tokens) || !aligned16(num_accepted))) return SV_ERR_INVALID_ARG;
    int sms = 0;
    if ((st = device_setup(&sms)) != SV_OK) return st;
    if (B == 0) return SV_OK;
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
    if (B > 0 && (!out_tokens || !num_accepted)) return SV_ERR_INVALID_ARG;
    if (B > 0 && (!aligned16(out_tokens) || !aligned16(num_accepted))) return SV_ERR_INVALID_ARG;
    if ((st = check_sample(draft_probs, u_accept, u_resample, T, B)) != SV_OK) return st;
    int sms = 0;
    if ((st = device_setup(&sms)) != SV_OK) return st;
    if (B == 0) return SV_OK;
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
    *device_status = h.status;
    if (n_degenerate) *n_degenerate = h.n_degenerate;
    return (h.status & ~SV_DEV_DEGENERATE) ? SV_ERR_DATA : SV_OK;
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
    cudaError_t e = cudaMemcpy(host, static_cast<const char*>(ws) + sizeof(Header),
                               R * sizeof(RowRec), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
        delete[] host;
        return SV_ERR_CUDA;
    }
    // A temperature is not kept in the workspace; m is reported as stored scaled
    // back with the T of the records' px (greedy: T = 1).
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
    sv_debug_ffexp_kernel<<<(n + 255) / 256, 256, 0, stream>>>(l, m, n, make_rT(T), exp_const(), out);
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
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
static_assert(kNoAllocScratchBytes >= 256 + 32 * (size_t)SV_NOALLOC_MAX_ROWS, "scratch size");

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
