// isd_step.cu -- B300 (sm_103a) kernels and C ABI of the ISD verify-and-propose step.
//
// The operation is the one "Introspective Diffusion Language Models" describes as
// Introspective Strided Decoding (ai.arkapp.pw blog, section "I-DLM 如何解決這些問題";
// de.news.hada.io, "Inference & ISD"): clean rows verify the previous step's proposals
// with min(1, p/q), MASK rows propose the next ones.  include/isd.h states the contract.
//
// Design (HBM-bound scan; no tensor cores):
//   isd_stream_kernel   one pass over every logit row the step reads.  The unit of work
//                       is a chunk of 4 KB (2048 bf16 / 1024 fp32) handled by one warp
//                       with eight 16-byte loads per lane in flight; a CTA takes eight
//                       chunks of one sequence at a time.  Per chunk it writes the
//                       chunk max and the sum of 2^((x - max) * log2(e)/T) (sampling) or
//                       the chunk max and its lowest argmax (greedy).  The last CTA to
//                       finish a sequence (atomic ticket, no waiting) combines the chunk
//                       statistics, runs the acceptance tests (one lane per pending
//                       token, warp ballot for the first rejection), and draws the
//                       anchor and MASK tokens by inverse CDF: a walk over the chunk
//                       sums, then a rescan of the one chunk that holds the target.
//   isd_residual_q_kernel   for sequences that rejected at K: statistics of the previous
//                       step's MASK row N+K (the q row of the rejected token).
//   isd_residual_kernel     per chunk sums of max(0, p - q) over the anchor row K and that
//                       q row, then (last CTA per sequence) the inverse-CDF draw of the
//                       replacement token.
// Greedy mode needs only the first kernel.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "isd.h"

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kVec = 8;  // 16-byte vectors per lane per chunk
constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxR = 2 * ISD_MAX_N - 1;
constexpr int kMaxB = 8192;
constexpr double kNearTie = 1e-6;

// ----------------------------------------------------------------------------------------
// element access: a chunk is uint4 v[kVec] per lane; element (k, e) of lane L sits at
// chunk_base + (k*32 + L)*kPerVec + e, so each of the eight loads is one coalesced
// 512-byte access per warp and a lane's elements run in ascending index order.
// ----------------------------------------------------------------------------------------
template <int DT>
struct Elem;

template <>
struct Elem<ISD_BF16> {
    static constexpr int kPerVec = 8;
    static constexpr int kChunk = 32 * kVec * kPerVec;  // 2048
    static constexpr uint32_t kNegInfWord = 0xFF80FF80u;
    static __device__ __forceinline__ float get(const uint4 (&v)[kVec], int k, int e) {
        const uint32_t* w = &v[k].x;
        uint32_t word = w[e >> 1];
        return __uint_as_float((e & 1) ? (word & 0xFFFF0000u) : (word << 16));
    }
    static __device__ __forceinline__ uint32_t scalar_bits(const void* row, int64_t idx) {
        return static_cast<const uint16_t*>(row)[idx];
    }
    static __device__ __forceinline__ void put_scalar(uint4 (&v)[kVec], int k, int e, uint32_t bits) {
        uint32_t* w = &v[k].x;
        w[e >> 1] = (e & 1) ? ((w[e >> 1] & 0x0000FFFFu) | (bits << 16)) : ((w[e >> 1] & 0xFFFF0000u) | bits);
    }
    static constexpr uint32_t kNegInfBits = 0xFF80u;
};

template <>
struct Elem<ISD_F32> {
    static constexpr int kPerVec = 4;
    static constexpr int kChunk = 32 * kVec * kPerVec;  // 1024
    static constexpr uint32_t kNegInfWord = 0xFF800000u;
    static __device__ __forceinline__ float get(const uint4 (&v)[kVec], int k, int e) {
        const uint32_t* w = &v[k].x;
        return __uint_as_float(w[e]);
    }
    static __device__ __forceinline__ uint32_t scalar_bits(const void* row, int64_t idx) {
        return static_cast<const uint32_t*>(row)[idx];
    }
    static __device__ __forceinline__ void put_scalar(uint4 (&v)[kVec], int k, int e, uint32_t bits) {
        uint32_t* w = &v[k].x;
        w[e] = bits;
    }
    static constexpr uint32_t kNegInfBits = 0xFF800000u;
};

template <int DT>
__device__ __forceinline__ float load_elem(const void* row, int64_t idx) {
    uint32_t bits = Elem<DT>::scalar_bits(row, idx);
    return __uint_as_float(DT == ISD_BF16 ? (bits << 16) : bits);
}

// Load one chunk of a row.  Elements at or beyond V read as -inf.  `stream` marks loads
// that are read once (evict-first in L1/L2).
template <int DT>
__device__ __forceinline__ void load_chunk(const void* row, int V, int64_t chunk_base, bool vec_ok,
                                           bool stream, uint4 (&v)[kVec]) {
    using E = Elem<DT>;
    const int lane = threadIdx.x & 31;
    if (vec_ok) {
        const uint4* base = reinterpret_cast<const uint4*>(row);
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
            int64_t first = chunk_base + (int64_t)(k * 32 + lane) * E::kPerVec;
            if (first < V) {
                v[k] = stream ? __ldcs(base + first / E::kPerVec) : __ldg(base + first / E::kPerVec);
            } else {
                v[k] = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
            int64_t first = chunk_base + (int64_t)(k * 32 + lane) * E::kPerVec;
            v[k] = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int e = 0; e < E::kPerVec; ++e) {
                int64_t idx = first + e;
                uint32_t bits = idx < V ? E::scalar_bits(row, idx) : E::kNegInfBits;
                E::put_scalar(v, k, e, bits);
            }
        }
    }
}

__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float fmax_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

__device__ __forceinline__ float ex2_approx(float t) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(t));
    return y;
}

// float -> unsigned key whose order is the float order (NaN excluded by the caller)
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float from_key(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Lane maximum of a chunk, NaN-propagating.
template <int DT>
__device__ __forceinline__ float lane_max(const uint4 (&v)[kVec]) {
    if constexpr (DT == ISD_BF16) {
        uint32_t acc = v[0].x;
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
            acc = bmax2_nan(acc, v[k].x);
            acc = bmax2_nan(acc, v[k].y);
            acc = bmax2_nan(acc, v[k].z);
            acc = bmax2_nan(acc, v[k].w);
        }
        return fmax_nan(__uint_as_float(acc << 16), __uint_as_float(acc & 0xFFFF0000u));
    } else {
        float acc = __uint_as_float(v[0].x);
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
            acc = fmax_nan(acc, __uint_as_float(v[k].x));
            acc = fmax_nan(acc, __uint_as_float(v[k].y));
            acc = fmax_nan(acc, __uint_as_float(v[k].z));
            acc = fmax_nan(acc, __uint_as_float(v[k].w));
        }
        return acc;
    }
}

// Warp maximum; NaN if any lane holds NaN.
__device__ __forceinline__ float warp_max_nan(float x) {
    bool nan = isnan(x);
    uint32_t key = nan ? 0u : order_key(x);
    key = __reduce_max_sync(kFull, key);
    float m = from_key(key);
    return __any_sync(kFull, nan) ? __int_as_float(0x7FC00000) : m;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}

__device__ __forceinline__ double warp_incl_scan(double x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        double y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

__device__ __forceinline__ float warp_excl_scan(float x, float& total) {
    const int lane = threadIdx.x & 31;
    float incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        float y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    total = __shfl_sync(kFull, incl, 31);
    float excl = __shfl_up_sync(kFull, incl, 1);
    return lane == 0 ? 0.f : excl;
}

// weight of one logit relative to a finite reference: 2^((x - ref) * log2(e)/T), with
// log2(e)/T = s_hi + s_lo (s_lo > 0) so the product keeps the precision of x - ref.
__device__ __forceinline__ float weight(float x, float ref, float s_hi, float s_lo) {
    float d = x - ref;
    return ex2_approx(fmaf(d, s_hi, d * s_lo));
}

// Philox4x32-10, Salmon, Moraes, Dror, Shaw, SC'11, section 4.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
    for (int i = 0; i < 10; ++i) {
        if (i > 0) {
            k.x += 0x9E3779B9u;
            k.y += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
    }
    return c;
}

__device__ __forceinline__ uint4 row_words(uint64_t seed, uint64_t step, int b, int r) {
    return philox4x32_10(make_uint4((uint32_t)step, (uint32_t)(step >> 32), (uint32_t)b, (uint32_t)r),
                         make_uint2((uint32_t)seed, (uint32_t)(seed >> 32)));
}
__device__ __forceinline__ float to_uniform(uint32_t w) {
    return (float)(w >> 8) * (1.0f / 16777216.0f);
}

// ----------------------------------------------------------------------------------------
// parameters and workspace
// ----------------------------------------------------------------------------------------
struct RowStat {
    double Z;   // sum over the row of 2^((x - m) * s)
    float m;    // row maximum (the reference of Z)
    int amax;   // greedy: lowest index of the maximum
};

struct Params {
    const void* logits;
    const void* prev;
    const int32_t* pending;
    int pending_ld;
    const float* pending_q;
    int32_t* accepted_len;
    int32_t* tokens_out;
    float* new_q;
    float* p_out;
    int32_t* diag;
    int B, N, V, R, C;  // C = chunks per row
    float s_hi, s_lo;
    int vec_ok;
    uint64_t seed, step;
    // workspace
    uint32_t* seq_ticket;  // [B]
    uint32_t* q_ticket;    // [B]
    uint32_t* r_ticket;    // [B]
    uint32_t* counters;    // [0] residual jobs, [1] residual CTAs done
    int32_t* jobs;         // [B] sequences needing a residual draw
    int32_t* seq_K;        // [B] rejected position, -1 if none
    float2* chunk;         // [B][R][C] (max, sum) or (max, argmax bits)
    RowStat* rowstat;      // [B][R]
    float2* qchunk;        // [B][C]
    RowStat* qstat;        // [B]
    float* rchunk;         // [B][C]
};

__device__ __forceinline__ void set_status(const Params& p, int code) {
    if (p.diag) atomicCAS(&p.diag[ISD_DIAG_STATUS], 0, code);
}
__device__ __forceinline__ void diag_add(const Params& p, int word, int v) {
    if (p.diag && v) atomicAdd(&p.diag[word], v);
}

__device__ __forceinline__ const void* row_ptr(const void* base, int dt_bytes, int64_t row, int V) {
    return static_cast<const char*>(base) + row * (int64_t)V * dt_bytes;
}

// ----------------------------------------------------------------------------------------
// per-chunk statistics (one warp)
// ----------------------------------------------------------------------------------------
// sampling: (chunk max, sum of weights relative to the chunk max)
template <int DT>
__device__ __forceinline__ float2 chunk_stat_sample(const uint4 (&v)[kVec], float s_hi, float s_lo) {
    using E = Elem<DT>;
    const float m = warp_max_nan(lane_max<DT>(v));
    const float ref = isfinite(m) ? m : 0.f;
    float sk[kVec];
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
        float a[E::kPerVec];
#pragma unroll
        for (int e = 0; e < E::kPerVec; ++e) a[e] = weight(E::get(v, k, e), ref, s_hi, s_lo);
        if constexpr (E::kPerVec == 8) {
            sk[k] = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
        } else {
            sk[k] = (a[0] + a[1]) + (a[2] + a[3]);
        }
    }
    const float lane_sum = ((sk[0] + sk[1]) + (sk[2] + sk[3])) + ((sk[4] + sk[5]) + (sk[6] + sk[7]));
    return make_float2(m, warp_sum(lane_sum));
}

// greedy: (chunk max, lowest index of it in the chunk)
template <int DT>
__device__ __forceinline__ float2 chunk_stat_argmax(const uint4 (&v)[kVec], int64_t chunk_base) {
    using E = Elem<DT>;
    const int lane = threadIdx.x & 31;
    const float lm = lane_max<DT>(v);
    const float m = warp_max_nan(lm);
    uint32_t idx = 0xFFFFFFFFu;
    if (lm == m) {
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
#pragma unroll
            for (int e = 0; e < E::kPerVec; ++e) {
                if (idx == 0xFFFFFFFFu && E::get(v, k, e) == m)
                    idx = (uint32_t)(chunk_base + (int64_t)(k * 32 + lane) * E::kPerVec + e);
            }
        }
    }
    idx = __reduce_min_sync(kFull, idx);
    return make_float2(m, __uint_as_float(idx));
}

// weight of a chunk total relative to the row maximum, in double
__device__ __forceinline__ double chunk_weight(float2 st, float m_row, float s_hi, float s_lo) {
    if (!(st.y > 0.f) || st.x == -INFINITY) return 0.0;
    const float d = st.x - m_row;
    return (double)st.y * (double)exp2f(fmaf(d, s_hi, d * s_lo));
}

// Row combine (one warp): row max and, by an ordered scan over the chunks, the row sum.
// Returns false if the row is unusable (NaN/+Inf anywhere, or all -Inf).
__device__ bool combine_row_sample(const float2* cs, int C, float s_hi, float s_lo, RowStat& out) {
    const int lane = threadIdx.x & 31;
    bool nan = false;
    uint32_t key = 0;
    for (int c = lane; c < C; c += 32) {
        float m = __ldcg(&cs[c]).x;
        if (isnan(m)) nan = true;
        else key = max(key, order_key(m));
    }
    key = __reduce_max_sync(kFull, key);
    nan = __any_sync(kFull, nan);
    const float m_row = from_key(key);
    if (nan || !isfinite(m_row)) return false;
    double carry = 0.0;
    for (int g = 0; g * 32 < C; ++g) {
        const int c = g * 32 + lane;
        double w = c < C ? chunk_weight(__ldcg(&cs[c]), m_row, s_hi, s_lo) : 0.0;
        double incl = warp_incl_scan(w);
        carry += __shfl_sync(kFull, incl, 31);
    }
    out.Z = carry;
    out.m = m_row;
    out.amax = -1;
    return true;
}

__device__ bool combine_row_argmax(const float2* cs, int C, RowStat& out) {
    const int lane = threadIdx.x & 31;
    bool nan = false;
    uint32_t key = 0;
    for (int c = lane; c < C; c += 32) {
        float m = __ldcg(&cs[c]).x;
        if (isnan(m)) nan = true;
        else key = max(key, order_key(m));
    }
    key = __reduce_max_sync(kFull, key);
    nan = __any_sync(kFull, nan);
    const float m_row = from_key(key);
    if (nan || !isfinite(m_row)) return false;
    uint32_t first = 0xFFFFFFFFu;
    for (int c = lane; c < C; c += 32) {
        if (__ldcg(&cs[c]).x == m_row) first = min(first, (uint32_t)c);
    }
    first = __reduce_min_sync(kFull, first);
    if (first >= (uint32_t)C) return false;
    out.Z = 0.0;
    out.m = m_row;
    out.amax = (int)__float_as_uint(__ldcg(&cs[first]).y);
    return true;
}

// Inverse-CDF draw over one row (one warp): find the chunk whose running sum first exceeds
// u*Z, then rescan that chunk.  Returns the token; *wx receives its weight relative to the
// row maximum (for q = wx / Z).
template <int DT>
__device__ int draw_row(const Params& p, const void* row, const float2* cs, const RowStat& rs, float u,
                        float* wx) {
    using E = Elem<DT>;
    const int lane = threadIdx.x & 31;
    const int C = p.C;
    const double target = (double)u * rs.Z;
    // 1. walk the chunks (same arithmetic and order as the combine's scan)
    double carry = 0.0;
    int cstar = -1;
    double before = 0.0;
    int last_pos = -1;
    for (int g = 0; g * 32 < C && cstar < 0; ++g) {
        const int c = g * 32 + lane;
        double w = c < C ? chunk_weight(__ldcg(&cs[c]), rs.m, p.s_hi, p.s_lo) : 0.0;
        double incl = warp_incl_scan(w);
        unsigned pos = __ballot_sync(kFull, w > 0.0);
        if (pos) last_pos = g * 32 + 31 - __clz(pos);
        unsigned cross = __ballot_sync(kFull, c < C && carry + incl > target);
        if (cross) {
            const int l = __ffs(cross) - 1;
            cstar = g * 32 + l;
            double excl = __shfl_sync(kFull, incl - w, l);
            double incl_l = __shfl_sync(kFull, incl, l);
            double w_l = __shfl_sync(kFull, w, l);
            before = carry + (incl_l - w_l);
            (void)excl;
        }
        carry += __shfl_sync(kFull, incl, 31);
    }
    bool overshoot = false;
    if (cstar < 0) {  // rounding left no crossing: take the last chunk with weight
        cstar = last_pos < 0 ? 0 : last_pos;
        overshoot = true;
    }
    // 2. rescan chunk cstar with the weights of the statistics pass
    const float2 st = __ldcg(&cs[cstar]);
    const float ref = isfinite(st.x) ? st.x : 0.f;
    const double scale = chunk_weight(make_float2(st.x, 1.0f), rs.m, p.s_hi, p.s_lo);
    const double local_target = overshoot ? INFINITY : (target - before) / scale;
    uint4 v[kVec];
    const int64_t base = (int64_t)cstar * E::kChunk;
    load_chunk<DT>(row, p.V, base, p.vec_ok, false, v);
    float running = 0.f;
    int found = -1;
    float found_x = 0.f;
    uint32_t last_idx = 0;
    bool any_pos = false;
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
        float a[E::kPerVec];
        float lane_tot = 0.f;
#pragma unroll
        for (int e = 0; e < E::kPerVec; ++e) {
            a[e] = weight(E::get(v, k, e), ref, p.s_hi, p.s_lo);
            lane_tot += a[e];
        }
        float slot_tot;
        const float excl = warp_excl_scan(lane_tot, slot_tot);
        int my_e = -1;
        float cum = running + excl;
#pragma unroll
        for (int e = 0; e < E::kPerVec; ++e) {
            cum += a[e];
            if (my_e < 0 && a[e] > 0.f && (double)cum > local_target) my_e = e;
            if (a[e] > 0.f) {
                last_idx = (uint32_t)(base + (int64_t)(k * 32 + lane) * E::kPerVec + e);
                any_pos = true;
            }
        }
        const unsigned hit = __ballot_sync(kFull, my_e >= 0);
        if (found < 0 && hit) {
            const int l = __ffs(hit) - 1;
            const int e = __shfl_sync(kFull, my_e, l);
            found = (int)(base + (int64_t)(k * 32 + l) * E::kPerVec + e);
            float xv = 0.f;
#pragma unroll
            for (int ee = 0; ee < E::kPerVec; ++ee)
                if (ee == my_e) xv = E::get(v, k, ee);
            found_x = __shfl_sync(kFull, xv, l);
        }
        running += slot_tot;
    }
    if (found < 0) {  // overshoot inside the chunk: the last index with positive weight
        uint32_t li = any_pos ? last_idx : 0u;
        li = __reduce_max_sync(kFull, li);
        found = (int)li;
        found_x = load_elem<DT>(row, found);
        if (lane == 0) diag_add(p, ISD_DIAG_NEAR_TIE_CDF, 1);
    }
    *wx = weight(found_x, rs.m, p.s_hi, p.s_lo);
    return found;
}

// ----------------------------------------------------------------------------------------
// decision for one sequence (whole CTA)
// ----------------------------------------------------------------------------------------
template <int DT, bool GREEDY>
__device__ void decide_sequence(const Params& p, int b) {
    __shared__ RowStat s_rs[kMaxR];
    __shared__ int s_bad;
    __shared__ int s_K;
    __shared__ int s_state;  // 0 error, 1 propose, 2 rejected
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = p.N, R = p.R, V = p.V;
    const int dtb = DT == ISD_BF16 ? 2 : 4;
    const int32_t* pend = p.pending + (int64_t)b * p.pending_ld;
    const bool has_pending = pend[0] >= 0;
    const int first_row = has_pending ? 0 : N - 1;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    for (int r = first_row + warp; r < R; r += kWarps) {
        const float2* cs = p.chunk + ((int64_t)b * R + r) * p.C;
        RowStat rs;
        bool ok = GREEDY ? combine_row_argmax(cs, p.C, rs) : combine_row_sample(cs, p.C, p.s_hi, p.s_lo, rs);
        if (lane == 0) {
            if (!ok) atomicOr(&s_bad, 1);
            s_rs[r] = rs;
            p.rowstat[(int64_t)b * R + r] = rs;
        }
    }
    __syncthreads();
    int32_t* tok = p.tokens_out + (int64_t)b * R;
    float* nq = p.new_q + (int64_t)b * (N - 1);
    if (warp == 0) {
        int K = N - 1;
        int state = 1;
        bool bad_pending = false;
        bool accept = true;
        int x = -1;
        if (has_pending && lane < N - 1) {
            x = pend[lane];
            if (x < 0 || x >= V) bad_pending = true;
            if (!GREEDY) {
                const float q = p.pending_q[(int64_t)b * (N - 1) + lane];
                if (!(q > 0.f && q < INFINITY) || p.prev == nullptr) bad_pending = true;
            }
        }
        bad_pending = __any_sync(kFull, bad_pending);
        const bool nonfinite = s_bad != 0;
        if (bad_pending || nonfinite) {
            state = 0;
        } else if (has_pending) {
            if (lane < N - 1) {
                if (GREEDY) {
                    accept = (x == s_rs[lane].amax);
                } else {
                    const RowStat rs = s_rs[lane];
                    const float xl = load_elem<DT>(row_ptr(p.logits, dtb, (int64_t)b * R + lane, V), x);
                    const float d = xl - rs.m;
                    const double pv = (double)exp2f(fmaf(d, p.s_hi, d * p.s_lo)) / rs.Z;
                    const double ratio = pv / (double)p.pending_q[(int64_t)b * (N - 1) + lane];
                    const double u = (double)to_uniform(row_words(p.seed, p.step, b, lane).x);
                    accept = u < ratio;
                    if (p.p_out) p.p_out[(int64_t)b * (N - 1) + lane] = (float)pv;
                    if (fabs(u - ratio) < kNearTie) diag_add(p, ISD_DIAG_NEAR_TIE_ACC, 1);
                }
            }
            const unsigned rej = __ballot_sync(kFull, lane < N - 1 && !accept);
            K = rej ? __ffs(rej) - 1 : N - 1;
            state = K < N - 1 ? 2 : 1;
        }
        // emitted tokens known now: the accepted prefix (and the greedy replacement)
        if (state != 0) {
            for (int i = lane; i < R; i += 32) {
                int t = -1;
                if (has_pending && i < K) t = pend[i];
                if (GREEDY) {
                    if (state == 2 && i == K) t = s_rs[K].amax;
                    if (state == 1) {
                        const int y_pos = has_pending ? N - 1 : 0;
                        if (i == y_pos) t = s_rs[N - 1].amax;
                        if (i >= N) t = s_rs[i].amax;
                    }
                }
                tok[i] = t;
            }
            for (int i = lane; i < N - 1; i += 32) nq[i] = (GREEDY && state == 1) ? 1.f : 0.f;
        } else {
            for (int i = lane; i < R; i += 32) tok[i] = -1;
            for (int i = lane; i < N - 1; i += 32) nq[i] = 0.f;
        }
        if (lane == 0) {
            if (state == 0) {
                p.accepted_len[b] = 0;
                set_status(p, bad_pending ? ISD_ERR_BAD_PENDING : ISD_ERR_NONFINITE);
            } else {
                const int emitted = has_pending ? K + 1 : 1;
                p.accepted_len[b] = emitted;
                diag_add(p, ISD_DIAG_EMITTED, emitted);
                if (has_pending) {
                    diag_add(p, ISD_DIAG_ACCEPTS, K);
                    diag_add(p, ISD_DIAG_TESTS, K < N - 1 ? K + 1 : N - 1);
                } else {
                    diag_add(p, ISD_DIAG_RECOVERY, 1);
                }
                if (!GREEDY && state == 2) {
                    p.seq_K[b] = K;
                    const int j = atomicAdd(&p.counters[0], 1);
                    p.jobs[j] = b;
                    diag_add(p, ISD_DIAG_RESIDUALS, 1);
                }
            }
            if (!has_pending || state == 0 || GREEDY) {
                if (p.p_out)
                    for (int i = 0; i < N - 1; ++i) p.p_out[(int64_t)b * (N - 1) + i] = 0.f;
            }
            s_K = K;
            s_state = state;
        }
    }
    __syncthreads();
    if (!GREEDY && s_state == 1) {
        // bonus token (row N-1) and the N-1 proposals (rows N..2N-2), one warp per row
        for (int j = warp; j < N; j += kWarps) {
            const int r = N - 1 + j;
            const RowStat rs = s_rs[r];
            const float u = to_uniform(row_words(p.seed, p.step, b, r).y);
            float wx;
            const int t = draw_row<DT>(p, row_ptr(p.logits, dtb, (int64_t)b * R + r, V),
                                       p.chunk + ((int64_t)b * R + r) * p.C, rs, u, &wx);
            if (lane == 0) {
                if (j == 0) {
                    tok[has_pending ? N - 1 : 0] = t;
                } else {
                    tok[r] = t;
                    nq[j - 1] = (float)((double)wx / rs.Z);
                }
            }
        }
    }
}

// prefix over sequences of the number of CTA items (8 chunks each) the step needs
__device__ void build_item_prefix(const Params& p, int* s_prefix) {
    const int B = p.B;
    const int per = (B + kThreads - 1) / kThreads;
    const int b0 = threadIdx.x * per;
    int local = 0;
    for (int b = b0; b < min(B, b0 + per); ++b) {
        const int rows = p.pending[(int64_t)b * p.pending_ld] >= 0 ? p.R : p.N;
        local += (rows * p.C + kWarps - 1) / kWarps;
    }
    __shared__ int s_warp[kWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int off = 0;
    for (int w = 0; w < warp; ++w) off += s_warp[w];
    int run = off + incl - local;
    for (int b = b0; b < min(B, b0 + per); ++b) {
        s_prefix[b] = run;
        const int rows = p.pending[(int64_t)b * p.pending_ld] >= 0 ? p.R : p.N;
        run += (rows * p.C + kWarps - 1) / kWarps;
    }
    if (threadIdx.x == kThreads - 1) s_prefix[B] = run;
    __syncthreads();
}

__device__ __forceinline__ int find_seq(const int* s_prefix, int B, int item) {
    int lo = 0, hi = B - 1;  // largest b with s_prefix[b] <= item
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_prefix[mid] <= item) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

template <int DT, bool GREEDY>
__global__ void __launch_bounds__(kThreads) isd_stream_kernel(Params p) {
    extern __shared__ int s_prefix[];
    __shared__ int s_last;
    build_item_prefix(p, s_prefix);
    const int total = s_prefix[p.B];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int dtb = DT == ISD_BF16 ? 2 : 4;
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
        const int b = find_seq(s_prefix, p.B, item);
        const int local = item - s_prefix[b];
        const bool has_pending = p.pending[(int64_t)b * p.pending_ld] >= 0;
        const int first_row = has_pending ? 0 : p.N - 1;
        const int rows = p.R - first_row;
        const int flat = local * kWarps + warp;
        if (flat < rows * p.C) {
            const int r = first_row + flat / p.C;
            const int c = flat % p.C;
            const int64_t base = (int64_t)c * Elem<DT>::kChunk;
            uint4 v[kVec];
            load_chunk<DT>(row_ptr(p.logits, dtb, (int64_t)b * p.R + r, p.V), p.V, base, p.vec_ok, true, v);
            const float2 st = GREEDY ? chunk_stat_argmax<DT>(v, base) : chunk_stat_sample<DT>(v, p.s_hi, p.s_lo);
            if (lane == 0) {
                p.chunk[((int64_t)b * p.R + r) * p.C + c] = st;
                __threadfence();
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            const uint32_t need = (uint32_t)(s_prefix[b + 1] - s_prefix[b]);
            const uint32_t old = atomicAdd(&p.seq_ticket[b], 1u);
            s_last = (old == need - 1);
        }
        __syncthreads();
        if (s_last) {
            __threadfence();
            decide_sequence<DT, GREEDY>(p, b);
            if (threadIdx.x == 0) p.seq_ticket[b] = 0;
            __syncthreads();
        }
    }
}

// ----------------------------------------------------------------------------------------
// residual: statistics of the q row (previous step's MASK row N+K)
// ----------------------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kThreads) isd_residual_q_kernel(Params p) {
    __shared__ int s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int dtb = DT == ISD_BF16 ? 2 : 4;
    const int jobs = *(volatile uint32_t*)&p.counters[0];
    const int slices = (p.C + kWarps - 1) / kWarps;
    for (int item = blockIdx.x; item < jobs * slices; item += gridDim.x) {
        const int j = item / slices, k = item % slices;
        const int b = p.jobs[j];
        const int K = p.seq_K[b];
        const int c = k * kWarps + warp;
        if (c < p.C) {
            const int64_t base = (int64_t)c * Elem<DT>::kChunk;
            uint4 v[kVec];
            load_chunk<DT>(row_ptr(p.prev, dtb, (int64_t)b * p.R + p.N + K, p.V), p.V, base, p.vec_ok, true, v);
            const float2 st = chunk_stat_sample<DT>(v, p.s_hi, p.s_lo);
            if (lane == 0) {
                p.qchunk[(int64_t)b * p.C + c] = st;
                __threadfence();
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            const uint32_t old = atomicAdd(&p.q_ticket[b], 1u);
            s_last = (old == (uint32_t)slices - 1);
        }
        __syncthreads();
        if (s_last) {
            __threadfence();
            if (warp == 0) {
                RowStat rs;
                const bool ok = combine_row_sample(p.qchunk + (int64_t)b * p.C, p.C, p.s_hi, p.s_lo, rs);
                if (lane == 0) {
                    p.qstat[b] = rs;
                    if (!ok) {  // the q row is unusable: the sequence fails
                        p.seq_K[b] = -1;
                        p.accepted_len[b] = 0;
                        for (int i = 0; i < p.R; ++i) p.tokens_out[(int64_t)b * p.R + i] = -1;
                        set_status(p, ISD_ERR_NONFINITE);
                    }
                    p.q_ticket[b] = 0;
                }
            }
            __syncthreads();
        }
    }
}

// ----------------------------------------------------------------------------------------
// residual: chunk sums of max(0, p - q) and the replacement draw
// ----------------------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ float residual_elem(float xp, float xq, float mp, float mq, float izp, float izq,
                                               float s_hi, float s_lo) {
    const float pp = weight(xp, mp, s_hi, s_lo) * izp;
    const float qq = weight(xq, mq, s_hi, s_lo) * izq;
    return fmaxf(pp - qq, 0.f);
}

template <int DT>
__device__ int draw_residual(const Params& p, int b, int K, float u) {
    using E = Elem<DT>;
    const int lane = threadIdx.x & 31;
    const int dtb = DT == ISD_BF16 ? 2 : 4;
    const int C = p.C;
    const float* rc = p.rchunk + (int64_t)b * C;
    // total and walk in one ordered scan
    double carry = 0.0;
    for (int g = 0; g * 32 < C; ++g) {
        const int c = g * 32 + lane;
        double w = c < C ? (double)__ldcg(&rc[c]) : 0.0;
        carry += __shfl_sync(kFull, warp_incl_scan(w), 31);
    }
    const double total = carry;
    const void* prow = row_ptr(p.logits, dtb, (int64_t)b * p.R + K, p.V);
    if (!(total > 0.0)) {
        // no residual mass left by rounding: draw from p (anchor row K) instead
        if (lane == 0) diag_add(p, ISD_DIAG_NEAR_TIE_CDF, 1);
        float wx;
        return draw_row<DT>(p, prow, p.chunk + ((int64_t)b * p.R + K) * C, p.rowstat[(int64_t)b * p.R + K], u, &wx);
    }
    const double target = (double)u * total;
    carry = 0.0;
    int cstar = -1, last_pos = -1;
    double before = 0.0;
    for (int g = 0; g * 32 < C && cstar < 0; ++g) {
        const int c = g * 32 + lane;
        double w = c < C ? (double)__ldcg(&rc[c]) : 0.0;
        double incl = warp_incl_scan(w);
        unsigned pos = __ballot_sync(kFull, w > 0.0);
        if (pos) last_pos = g * 32 + 31 - __clz(pos);
        unsigned cross = __ballot_sync(kFull, c < C && carry + incl > target);
        if (cross) {
            const int l = __ffs(cross) - 1;
            cstar = g * 32 + l;
            before = carry + (__shfl_sync(kFull, incl, l) - __shfl_sync(kFull, w, l));
        }
        carry += __shfl_sync(kFull, incl, 31);
    }
    bool overshoot = false;
    if (cstar < 0) {
        cstar = last_pos < 0 ? 0 : last_pos;
        overshoot = true;
    }
    const double local_target = overshoot ? INFINITY : target - before;
    const RowStat ps = p.rowstat[(int64_t)b * p.R + K];
    const RowStat qs = p.qstat[b];
    const float izp = (float)(1.0 / ps.Z), izq = (float)(1.0 / qs.Z);
    const void* qrow = row_ptr(p.prev, dtb, (int64_t)b * p.R + p.N + K, p.V);
    const int64_t base = (int64_t)cstar * E::kChunk;
    uint4 vp[kVec], vq[kVec];
    load_chunk<DT>(prow, p.V, base, p.vec_ok, false, vp);
    load_chunk<DT>(qrow, p.V, base, p.vec_ok, false, vq);
    float running = 0.f;
    int found = -1;
    uint32_t last_idx = 0;
    bool any_pos = false;
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
        float a[E::kPerVec];
        float lane_tot = 0.f;
#pragma unroll
        for (int e = 0; e < E::kPerVec; ++e) {
            a[e] = residual_elem<DT>(E::get(vp, k, e), E::get(vq, k, e), ps.m, qs.m, izp, izq, p.s_hi, p.s_lo);
            lane_tot += a[e];
        }
        float slot_tot;
        const float excl = warp_excl_scan(lane_tot, slot_tot);
        int my_e = -1;
        float cum = running + excl;
#pragma unroll
        for (int e = 0; e < E::kPerVec; ++e) {
            cum += a[e];
            if (my_e < 0 && a[e] > 0.f && (double)cum > local_target) my_e = e;
            if (a[e] > 0.f) {
                last_idx = (uint32_t)(base + (int64_t)(k * 32 + lane) * E::kPerVec + e);
                any_pos = true;
            }
        }
        const unsigned hit = __ballot_sync(kFull, my_e >= 0);
        if (found < 0 && hit) {
            const int l = __ffs(hit) - 1;
            found = (int)(base + (int64_t)(k * 32 + l) * E::kPerVec + __shfl_sync(kFull, my_e, l));
        }
        running += slot_tot;
    }
    if (found < 0) {
        uint32_t li = any_pos ? last_idx : 0u;
        found = (int)__reduce_max_sync(kFull, li);
        if (lane == 0) diag_add(p, ISD_DIAG_NEAR_TIE_CDF, 1);
    }
    return found;
}

template <int DT>
__global__ void __launch_bounds__(kThreads) isd_residual_kernel(Params p) {
    using E = Elem<DT>;
    __shared__ int s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int dtb = DT == ISD_BF16 ? 2 : 4;
    const int jobs = *(volatile uint32_t*)&p.counters[0];
    const int slices = (p.C + kWarps - 1) / kWarps;
    for (int item = blockIdx.x; item < jobs * slices; item += gridDim.x) {
        const int j = item / slices, k = item % slices;
        const int b = p.jobs[j];
        const int K = p.seq_K[b];
        if (K < 0) continue;  // uniform across the CTA: the sequence already failed
        const int c = k * kWarps + warp;
        if (c < p.C) {
            const RowStat ps = p.rowstat[(int64_t)b * p.R + K];
            const RowStat qs = p.qstat[b];
            const float izp = (float)(1.0 / ps.Z), izq = (float)(1.0 / qs.Z);
            const int64_t base = (int64_t)c * E::kChunk;
            uint4 vp[kVec], vq[kVec];
            load_chunk<DT>(row_ptr(p.logits, dtb, (int64_t)b * p.R + K, p.V), p.V, base, p.vec_ok, true, vp);
            load_chunk<DT>(row_ptr(p.prev, dtb, (int64_t)b * p.R + p.N + K, p.V), p.V, base, p.vec_ok, true, vq);
            float sk[kVec];
#pragma unroll
            for (int kk = 0; kk < kVec; ++kk) {
                float a[E::kPerVec];
#pragma unroll
                for (int e = 0; e < E::kPerVec; ++e)
                    a[e] = residual_elem<DT>(E::get(vp, kk, e), E::get(vq, kk, e), ps.m, qs.m, izp, izq, p.s_hi,
                                             p.s_lo);
                float s = 0.f;
#pragma unroll
                for (int e = 0; e < E::kPerVec; ++e) s += a[e];
                sk[kk] = s;
            }
            const float lane_sum = ((sk[0] + sk[1]) + (sk[2] + sk[3])) + ((sk[4] + sk[5]) + (sk[6] + sk[7]));
            const float tot = warp_sum(lane_sum);
            if (lane == 0) {
                p.rchunk[(int64_t)b * p.C + c] = tot;
                __threadfence();
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            const uint32_t old = atomicAdd(&p.r_ticket[b], 1u);
            s_last = (old == (uint32_t)slices - 1);
        }
        __syncthreads();
        if (s_last) {
            __threadfence();
            if (warp == 0) {
                const float u = to_uniform(row_words(p.seed, p.step, b, K).y);
                const int y = draw_residual<DT>(p, b, K, u);
                if (lane == 0) {
                    p.tokens_out[(int64_t)b * p.R + K] = y;
                    p.r_ticket[b] = 0;
                }
            }
            __syncthreads();
        }
    }
    // the last CTA to leave clears the job list for the next step
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t old = atomicAdd(&p.counters[1], 1u);
        if (old == gridDim.x - 1) {
            p.counters[0] = 0;
            p.counters[1] = 0;
        }
    }
}

// ----------------------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------------------
struct Layout {
    size_t seq_ticket, q_ticket, r_ticket, counters, jobs, seq_K, chunk, rowstat, qchunk, qstat, rchunk, total;
};

size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

int chunk_elems(int dtype) { return dtype == ISD_BF16 ? Elem<ISD_BF16>::kChunk : Elem<ISD_F32>::kChunk; }

bool make_layout(int B, int N, int V, int dtype, Layout& L) {
    if (B < 1 || B > kMaxB || N < 2 || N > ISD_MAX_N || V < 1) return false;
    if (dtype != ISD_BF16 && dtype != ISD_F32) return false;
    const int R = 2 * N - 1;
    if ((int64_t)V * R > (int64_t)INT32_MAX) return false;
    const size_t C = (size_t)((V + chunk_elems(dtype) - 1) / chunk_elems(dtype));
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + bytes);
        return at;
    };
    L.seq_ticket = take(sizeof(uint32_t) * B);
    L.q_ticket = take(sizeof(uint32_t) * B);
    L.r_ticket = take(sizeof(uint32_t) * B);
    L.counters = take(sizeof(uint32_t) * 8);
    L.jobs = take(sizeof(int32_t) * B);
    L.seq_K = take(sizeof(int32_t) * B);
    L.chunk = take(sizeof(float2) * (size_t)B * R * C);
    L.rowstat = take(sizeof(RowStat) * (size_t)B * R);
    L.qchunk = take(sizeof(float2) * (size_t)B * C);
    L.qstat = take(sizeof(RowStat) * (size_t)B);
    L.rchunk = take(sizeof(float) * (size_t)B * C);
    L.total = off;
    return true;
}

thread_local int g_last_launches = 0;

// measurement: CUDA timing events around each launch while a session is open
struct Profile {
    int cap = 0, next = 0;
    cudaEvent_t* ev = nullptr;  // 2 per launch
    int* kind = nullptr;
};
Profile g_prof;

enum { kKindStream = 0, kKindResidualQ = 1, kKindResidual = 2 };

struct ProfileScope {
    int slot = -1;
    cudaStream_t stream;
    ProfileScope(int kind, cudaStream_t s) : stream(s) {
        if (g_prof.cap > 0 && g_prof.next < g_prof.cap) {
            slot = g_prof.next++;
            g_prof.kind[slot] = kind;
            record(g_prof.ev[2 * slot]);
        }
    }
    ~ProfileScope() {
        if (slot >= 0) record(g_prof.ev[2 * slot + 1]);
    }
    void record(cudaEvent_t e) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaStreamIsCapturing(stream, &cs);
        cudaEventRecordWithFlags(e, stream, cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal
                                                                                : cudaEventRecordDefault);
    }
};

// CTAs of `kernel` that fit on the device at once (cached per device and kernel).
template <typename K>
int resident_ctas(K kernel, size_t smem) {
    struct Entry {
        int dev;
        const void* fn;
        size_t smem;
        int value;
    };
    static Entry cache[64];
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const void* fn = reinterpret_cast<const void*>(kernel);
    for (int i = 0; i < used; ++i)
        if (cache[i].dev == dev && cache[i].fn == fn && cache[i].smem == smem) return cache[i].value;
    int sms = 0, per = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, kThreads, smem) != cudaSuccess) return 0;
    const int value = sms * (per > 0 ? per : 1);
    if (used < 64) cache[used++] = Entry{dev, fn, smem, value};
    return value;
}

template <int DT>
int launch_all(const Params& p, int greedy, cudaStream_t stream) {
    const size_t smem = sizeof(int) * (size_t)(p.B + 1);
    const int items_max = p.B * ((p.R * p.C + kWarps - 1) / kWarps);
    int launches = 0;
    if (greedy) {
        auto k = isd_stream_kernel<DT, true>;
        if (smem > 48 * 1024) cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        const int grid = max(1, min(items_max, resident_ctas(k, smem)));
        {
            ProfileScope ps(kKindStream, stream);
            k<<<grid, kThreads, smem, stream>>>(p);
        }
        launches = 1;
    } else {
        auto k = isd_stream_kernel<DT, false>;
        if (smem > 48 * 1024) cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        const int grid = max(1, min(items_max, resident_ctas(k, smem)));
        {
            ProfileScope ps(kKindStream, stream);
            k<<<grid, kThreads, smem, stream>>>(p);
        }
        const int slices = (p.C + kWarps - 1) / kWarps;
        const int rgrid = max(1, min(p.B * slices, resident_ctas(isd_residual_kernel<DT>, 0)));
        {
            ProfileScope ps(kKindResidualQ, stream);
            isd_residual_q_kernel<DT><<<rgrid, kThreads, 0, stream>>>(p);
        }
        {
            ProfileScope ps(kKindResidual, stream);
            isd_residual_kernel<DT><<<rgrid, kThreads, 0, stream>>>(p);
        }
        launches = 3;
    }
    g_last_launches = launches;
    return cudaGetLastError() == cudaSuccess ? ISD_OK : ISD_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t isd_workspace_size(int B, int N, int V, int dtype) {
    Layout L;
    return make_layout(B, N, V, dtype, L) ? L.total : 0;
}

int isd_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
    if (workspace == nullptr) return ISD_ERR_WORKSPACE;
    return cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream) == cudaSuccess ? ISD_OK
                                                                                             : ISD_ERR_CUDA;
}

int isd_step(const void* logits, const void* prev_logits, int dtype, const int32_t* pending_tokens,
             int pending_ld, const float* pending_q, int B, int N, int V, float temperature, int greedy, uint64_t philox_seed,
             uint64_t step, int32_t* accepted_len, int32_t* tokens_out, float* new_q, float* p_out,
             int32_t* diag, void* workspace, size_t workspace_bytes, void* stream) {
    g_last_launches = 0;
    Layout L;
    if (!make_layout(B, N, V, dtype, L)) return ISD_ERR_INVALID_ARG;
    if (!logits || !pending_tokens || !accepted_len || !tokens_out || !new_q) return ISD_ERR_INVALID_ARG;
    if (pending_ld < N - 1) return ISD_ERR_INVALID_ARG;
    if (!greedy && (!pending_q || !(temperature > 0.f) || !isfinite(temperature))) return ISD_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < L.total || ((uintptr_t)workspace & 255)) return ISD_ERR_WORKSPACE;

    Params p;
    memset(&p, 0, sizeof p);
    p.logits = logits;
    p.prev = greedy ? nullptr : prev_logits;
    p.pending = pending_tokens;
    p.pending_ld = pending_ld;
    p.pending_q = pending_q;
    p.accepted_len = accepted_len;
    p.tokens_out = tokens_out;
    p.new_q = new_q;
    p.p_out = p_out;
    p.diag = diag;
    p.B = B;
    p.N = N;
    p.V = V;
    p.R = 2 * N - 1;
    p.C = (V + chunk_elems(dtype) - 1) / chunk_elems(dtype);
    // log2(e)/T split into a float head (rounded down) and a positive float tail
    const double s = greedy ? 1.0 : 1.4426950408889634 / (double)temperature;
    float hi = (float)s;
    if ((double)hi > s) hi = nextafterf(hi, 0.f);
    float lo = (float)(s - (double)hi);
    if (!(lo > 0.f)) lo = 1e-30f;
    p.s_hi = hi;
    p.s_lo = lo;
    const int esz = dtype == ISD_BF16 ? 2 : 4;
    const bool aligned = ((uintptr_t)logits % 16 == 0) && (!p.prev || (uintptr_t)p.prev % 16 == 0);
    p.vec_ok = (aligned && ((int64_t)V * esz) % 16 == 0) ? 1 : 0;
    p.seed = philox_seed;
    p.step = step;
    char* ws = static_cast<char*>(workspace);
    p.seq_ticket = reinterpret_cast<uint32_t*>(ws + L.seq_ticket);
    p.q_ticket = reinterpret_cast<uint32_t*>(ws + L.q_ticket);
    p.r_ticket = reinterpret_cast<uint32_t*>(ws + L.r_ticket);
    p.counters = reinterpret_cast<uint32_t*>(ws + L.counters);
    p.jobs = reinterpret_cast<int32_t*>(ws + L.jobs);
    p.seq_K = reinterpret_cast<int32_t*>(ws + L.seq_K);
    p.chunk = reinterpret_cast<float2*>(ws + L.chunk);
    p.rowstat = reinterpret_cast<RowStat*>(ws + L.rowstat);
    p.qchunk = reinterpret_cast<float2*>(ws + L.qchunk);
    p.qstat = reinterpret_cast<RowStat*>(ws + L.qstat);
    p.rchunk = reinterpret_cast<float*>(ws + L.rchunk);
    cudaStream_t st = (cudaStream_t)stream;
    return dtype == ISD_BF16 ? launch_all<ISD_BF16>(p, greedy, st) : launch_all<ISD_F32>(p, greedy, st);
}

const char* isd_status_string(int status) {
    switch (status) {
        case ISD_OK: return "ok";
        case ISD_ERR_INVALID_ARG: return "invalid argument";
        case ISD_ERR_CUDA: return "CUDA runtime error";
        case ISD_ERR_NONFINITE: return "non-finite logits in a row the step reads";
        case ISD_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case ISD_ERR_TIMEOUT: return "a bounded device wait gave up";
        case ISD_ERR_BAD_PENDING: return "pending token out of range or pending q not positive";
        case ISD_ERR_SCRATCH_LIMIT: return "sizes need more scratch than the static scratch of isd_step_noalloc holds";
        default: return "unknown status";
    }
}

int isd_last_launch_count(void) { return g_last_launches; }

void isd_profile_end(void) {
    if (g_prof.ev) {
        for (int i = 0; i < 2 * g_prof.cap; ++i) cudaEventDestroy(g_prof.ev[i]);
    }
    delete[] g_prof.ev;
    delete[] g_prof.kind;
    g_prof = Profile();
}

int isd_profile_begin(int capacity) {
    if (capacity < 1 || capacity > (1 << 20)) return ISD_ERR_INVALID_ARG;
    isd_profile_end();
    g_prof.ev = new cudaEvent_t[2 * (size_t)capacity];
    g_prof.kind = new int[capacity];
    for (int i = 0; i < 2 * capacity; ++i) {
        if (cudaEventCreate(&g_prof.ev[i]) != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(g_prof.ev[j]);
            delete[] g_prof.ev;
            delete[] g_prof.kind;
            g_prof = Profile();
            return ISD_ERR_CUDA;
        }
    }
    g_prof.cap = capacity;
    g_prof.next = 0;
    return ISD_OK;
}

int isd_profile_read(int kind, double* total_ms, int* launches) {
    if (!total_ms || !launches) return ISD_ERR_INVALID_ARG;
    double tot = 0.0;
    int n = 0;
    for (int i = 0; i < g_prof.next; ++i) {
        if (g_prof.kind[i] != kind) continue;
        if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess) return ISD_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) != cudaSuccess) return ISD_ERR_CUDA;
        tot += ms;
        ++n;
    }
    *total_ms = tot;
    *launches = n;
    return ISD_OK;
}

}  // extern "C"

// ----------------------------------------------------------------------------------------
// isd_step_noalloc: the same step with its scratch in a static device array, for callers
// that cannot allocate device memory where they run the step.
// ----------------------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_static_scratch[ISD_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_addr[kMaxDevices];  // device address of g_static_scratch, per device

// In host code g_static_scratch names a host-side stand-in, not device memory: the
// device address comes from cudaGetSymbolAddress, looked up once per device with that
// device current.
int static_scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ISD_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (g_static_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return ISD_ERR_CUDA;
        g_static_addr[dev] = p;
    }
    *out = g_static_addr[dev];
    return ISD_OK;
}

}  // namespace

extern "C" int isd_step_noalloc(const void* logits, const void* prev_logits, int dtype,
                                const int32_t* pending_tokens, int pending_ld, const float* pending_q, int B,
                                int N, int V, float temperature, int greedy, uint64_t philox_seed,
                                uint64_t step, int32_t* accepted_len, int32_t* tokens_out, float* new_q,
                                float* p_out, int32_t* diag, void* stream) {
    Layout L;
    if (!make_layout(B, N, V, dtype, L)) return ISD_ERR_INVALID_ARG;
    if (L.total > (size_t)ISD_STATIC_SCRATCH_BYTES) return ISD_ERR_SCRATCH_LIMIT;
    // the argument checks of isd_step, made here too so that a rejected call enqueues nothing
    if (!logits || !pending_tokens || !accepted_len || !tokens_out || !new_q) return ISD_ERR_INVALID_ARG;
    if (pending_ld < N - 1) return ISD_ERR_INVALID_ARG;
    if (!greedy && (!pending_q || !(temperature > 0.f) || !isfinite(temperature))) return ISD_ERR_INVALID_ARG;
    void* ws = nullptr;
    const int rc = static_scratch_address(&ws);
    if (rc != ISD_OK) return rc;
    // the tickets and counters at the front of the layout must start at zero
    if (cudaMemsetAsync(ws, 0, L.jobs, (cudaStream_t)stream) != cudaSuccess) return ISD_ERR_CUDA;
    return isd_step(logits, prev_logits, dtype, pending_tokens, pending_ld, pending_q, B, N, V, temperature,
                    greedy, philox_seed, step, accepted_len, tokens_out, new_q, p_out, diag, ws, L.total,
                    stream);
}
