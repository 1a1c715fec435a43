// isd_step.cu -- B300 (sm_103a) kernels and C ABI of the ISD verify-and-propose step.
//
// The operation is the one "Introspective Diffusion Language Models" describes as
// Introspective Strided Decoding (ai.arkapp.pw blog, section "I-DLM 如何解決這些問題";
// de.news.hada.io, "Inference & ISD"): clean rows verify the previous step's proposals
// with min(1, p/q), MASK rows propose the next ones.  include/isd.h states the contract.
//
// Design (an HBM-bound scan; no tensor cores), two launches per step:
//   isd_stats_kernel    one pass over every logit row the step reads, at HBM bandwidth.
//                       Persistent: one CTA of 20 warps per SM.  The unit of work is a
//                       4 KB chunk of a row (2048 bf16 / 1024 fp32); each warp's first
//                       batch of 4 units is fixed and later batches come from an atomic
//                       counter.  Each warp owns a ring of two 4 KB shared-memory
//                       stages filled by 1-D bulk copies (cp.async.bulk, completion on an
//                       mbarrier, L2 evict-first), so a chunk per warp is in flight while
//                       it reduces the previous one.  Per chunk it writes the
//                       chunk max and the sum of 2^((x - max) * log2(e)/T) (sampling) or
//                       the chunk max and its lowest argmax (greedy).  Shapes whose rows
//                       are not 16-byte aligned use isd_stats_plain_kernel (plain loads).
//   isd_decide_kernel   one thread-block cluster per sequence, launched as a programmatic
//                       dependent of the statistics kernel.  Every CTA of the cluster
//                       combines the anchor rows' chunk statistics into row statistics and
//                       runs the acceptance tests (one lane per pending token, warp ballot
//                       for the first rejection); all reach the same decision.  The pending
//                       tokens, their q, their logits, the uniforms and the carried q-row
//                       statistics are read before the wait for the statistics grid.  Then:
//                         - all accepted, or no pending tokens: the cluster combines the
//                           anchor row N-1 and the MASK rows (read only by such a sequence)
//                           and the bonus token and the N-1
//                           proposals are drawn by inverse CDF (a walk over the chunk sums,
//                           then a rescan of the one chunk that holds the target), the draws
//                           spread over the cluster's CTAs and warps;
//                         - rejection at position K: the q row statistics come from the
//                           previous call (carried in the workspace) or from a pass of the
//                           cluster over the previous step's MASK row N+K (the rejected
//                           token's q row); the cluster then splits the chunks of
//                           max(0, p - q) over anchor row K and that q row, with a cluster
//                           barrier after each pass; the leader CTA draws the replacement.
//                       Greedy mode uses clusters of one CTA and no draws.  In the
//                       argmax-proposal mode the proposals are rescans for the row maximum
//                       and a rejection draws from anchor row K without the rejected token.
// isd_step_fused runs the same step as one persistent kernel instead (isd_fused.cuh,
// included below; slower on a B300, kept as an alternative).
#include <cuda_runtime.h>
#include <math.h>
#include <stddef.h>
#include <algorithm>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "isd.h"
#include "isd_internal.h"
#include "isd_chunkstat.cuh"

namespace {

constexpr int kWarps = 6;  // warps of a decide CTA (6 keeps clusters of 8 resident at B=64)
constexpr int kThreads = kWarps * 32;
constexpr int kVec = 8;  // 16-byte vectors per lane per chunk
constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxR = 2 * ISD_MAX_N - 1;
constexpr int kMaxB = 8192;
constexpr double kNearTie = 1e-6;
constexpr int kChunkBytes = 32 * kVec * 16;  // 4096
constexpr int kSWarps = 20;                  // warps of a statistics CTA
constexpr int kSThreads = kSWarps * 32;
constexpr int kDepth = 2;  // bulk-copy stages per statistics warp
constexpr size_t kStatsSmem = (size_t)kSWarps * kDepth * kChunkBytes;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // a bounded wait gives up after ~1 s

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
    static constexpr int kBytes = 2;
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
    static constexpr int kBytes = 4;
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


__device__ __forceinline__ float fmax_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
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
// (a pairwise tree, so that the chain of dependent maxima is short)
__device__ __forceinline__ float lane_max(const uint4 (&v)[kVec]) {
    if constexpr (DT == ISD_BF16) {
        uint32_t acc[kVec];
#pragma unroll
        for (int k = 0; k < kVec; ++k) acc[k] = bmax2_nan(bmax2_nan(v[k].x, v[k].y), bmax2_nan(v[k].z, v[k].w));
#pragma unroll
        for (int w = kVec / 2; w > 0; w >>= 1)
#pragma unroll
            for (int k = 0; k < w; ++k) acc[k] = bmax2_nan(acc[k], acc[k + w]);
        return fmax_nan(__uint_as_float(acc[0] << 16), __uint_as_float(acc[0] & 0xFFFF0000u));
    } else {
        float acc[kVec];
#pragma unroll
        for (int k = 0; k < kVec; ++k)
            acc[k] = fmax_nan(fmax_nan(__uint_as_float(v[k].x), __uint_as_float(v[k].y)),
                              fmax_nan(__uint_as_float(v[k].z), __uint_as_float(v[k].w)));
#pragma unroll
        for (int w = kVec / 2; w > 0; w >>= 1)
#pragma unroll
            for (int k = 0; k < w; ++k) acc[k] = fmax_nan(acc[k], acc[k + w]);
        return acc[0];
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

__device__ __forceinline__ uint64_t warp_incl_scan_u64(uint64_t x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(kFull, x, o);
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

// Weights.  With s = log2(e)/T split into a float head s_hi and a small positive tail
// s_lo, the weight of logit x against an integer exponent reference e is
// 2^(x*s - e): the head product is exact inside the first FMA (one rounding of a result
// near 0 for the heavy entries) and the tail adds x*s_lo.  -inf logits weigh 0.
__device__ __forceinline__ float weight_exp(float x, float e, float s_hi, float s_lo) {
    return fmaf(x, s_lo, fmaf(x, s_hi, -e));
}

// Unsigned fixed point for exact sums and prefix sums of non-negative weights:
// to_fixed(x, k) = floor(x * 2^k) for finite x >= 0 (0 for x <= 0 and for NaN), the
// caller keeping x * 2^k below 2^63; fixed_to_float(v, k) = v * 2^-k, truncated to 24
// significant bits.
__device__ __forceinline__ uint64_t to_fixed(float x, int k) {
    const uint32_t b = __float_as_uint(x);
    if ((b & 0x80000000u) || b == 0u || (b >> 23) == 0xFFu) return 0ull;
    const uint32_t ex = b >> 23;
    const uint64_t mant = ex ? ((b & 0x7FFFFFu) | 0x800000u) : (b & 0x7FFFFFu);
    const int sh = (ex ? (int)ex : 1) - 150 + k;  // x * 2^k = mant * 2^sh
    if (sh >= 0) return sh > 39 ? (mant << 39) : (mant << sh);
    return sh <= -64 ? 0ull : (mant >> (-sh));
}
__device__ __forceinline__ float fixed_to_float(uint64_t v, int k) {
    if (v == 0ull) return 0.f;
    const int msb = 63 - __clzll((long long)v);
    const int sh = msb - 23;
    const uint32_t mant = sh >= 0 ? (uint32_t)(v >> sh) : (uint32_t)(v << (-sh));
    return ldexpf((float)mant, sh - k);
}
// floor(u * Z) for the 24-bit uniform u = (w >> 8) * 2^-24 and a fixed-point total Z.
__device__ __forceinline__ uint64_t scale_by_uniform(uint64_t Z, uint32_t w) {
    return __umul64hi(Z, (uint64_t)(w >> 8) << 40);
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
    uint64_t Zfx;  // sum over the row of 2^(x*s - M), fixed point with fx fraction bits
    float M;       // integer exponent reference of the row (greedy: the row maximum)
    float Zf;      // Zfx as a float (Z in units of 2^M)
    float T;       // tail factor 2^(m*s_lo) of the row maximum m
    int amax;      // greedy: lowest index of the maximum
    float mx;      // the row maximum m
};

// Identity of the call whose MASK-row statistics a carry slot holds.  A later call uses
// them only if its prev_logits is that call's logits and every other input they depend
// on matches; otherwise it reads the q row again (same result, more traffic).
struct CarryKey {
    const void* logits;
    uint64_t step;
    int B, N, V, dtype;
    float s_hi, s_lo;
    uint32_t tag;  // kCarryTag once written by a sampling call
    uint32_t pad;
};
constexpr uint32_t kCarryTag = 0x15D0C4A7u;

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
    int fx, fxr;        // fraction bits of the fixed-point row and residual sums
    float s_hi, s_lo;
    int vec_ok;
    int amode;  // argmax proposals (q = 1) verified by sampling; residual = p without x
    uint64_t seed, step;
    // workspace
    unsigned long long* sched;  // work counter of the statistics kernel (zero between steps)
    float2* chunk;   // [B][R][C] (max, sum) or (max, argmax bits)
    float2* qchunk;  // [B][C] chunk statistics of the residual's q row
    float* rchunk;   // [B][C] chunk sums of max(0, p - q)
    uint64_t* rtotal;  // [B] fixed-point total of rchunk (zeroed by the statistics kernel)
    // Statistics of the MASK rows, kept for the next call (its residual q rows), in two
    // slots chosen by step parity; each slot has a key naming the call that wrote it.
    RowStat* carry;    // [2][B][N-1]
    CarryKey* carry_key;  // [2]
    int dtype;
    uint64_t wait_ns;      // bounded waits give up after this long
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
// PTX: mbarriers, 1-D bulk copies, clusters, programmatic dependent launch
// ----------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// Test the phase of `bar` with parity `parity`; the thread may be suspended a while (until
// the phase completes or a hardware time limit passes).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// The same test without suspending the thread.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for the phase of `bar` with parity `parity` to complete; false after `limit_ns`
// (about 1 s by default).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
    if (limit_ns < 100000u) {
        // a short limit (a test's): poll without suspending, so that the limit holds
        const uint64_t t0 = global_ns();
        while (!mbar_test_wait(bar, parity))
            if (global_ns() - t0 > limit_ns) return false;
        return true;
    }
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;  // (each try may suspend the thread a while)
        if (global_ns() - t0 > limit_ns) return false;
    }
}
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// 1-D bulk copy global -> this CTA's shared memory, completing `bytes` on mbarrier `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}
// Order this thread's earlier generic-proxy shared-memory accesses before later async-proxy ones.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// All threads of all CTAs of the cluster; release/acquire at cluster scope.
__device__ __forceinline__ void cluster_sync() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::
            : "memory");
}
// The address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// Store to another CTA's shared memory in the cluster (visible there after a cluster barrier).
__device__ __forceinline__ void st_shared_cluster(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void wait_for_prerequisite_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ----------------------------------------------------------------------------------------
// per-chunk statistics (one warp)
// ----------------------------------------------------------------------------------------
// Packed fp32 pairs (Blackwell f32x2 arithmetic): two floats in one 64-bit register.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}


// sampling: (chunk maximum m, sum of 2^(x*s - e) with e = exponent_ref(m)), the chunk held
// in registers; the four pair accumulators run the f32x2 pipe.
template <int DT>
__device__ __forceinline__ float2 chunk_stat_sample(const uint4 (&v)[kVec], float s_hi, float s_lo) {
    const float m = warp_max_nan(lane_max<DT>(v));
    const float ref = ref_or_zero(exponent_ref(m, s_hi));
    const uint64_t S2 = pack2(s_hi, s_hi), NE2 = pack2(-ref, -ref);
    uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
        const uint32_t* w = &v[k].x;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            if constexpr (DT == ISD_BF16) {
                // one 32-bit word = two bf16 = two fp32 after a shift / a mask
                const uint64_t x2 = pack2(__uint_as_float(w[h] << 16), __uint_as_float(w[h] & 0xFFFF0000u));
                float t0, t1;
                unpack2(fma2(x2, S2, NE2), t0, t1);
                acc[h] = add2(acc[h], pack2(ex2_approx(t0), ex2_approx(t1)));
            } else if ((h & 1) == 0) {
                // two fp32 words are a pair as loaded
                const uint64_t x2 = pack2(__uint_as_float(w[h]), __uint_as_float(w[h + 1]));
                float t0, t1;
                unpack2(fma2(x2, S2, NE2), t0, t1);
                acc[h >> 1] = add2(acc[h >> 1], pack2(ex2_approx(t0), ex2_approx(t1)));
            }
        }
    }
    float lo, hi;
    unpack2(add2(add2(acc[0], acc[1]), add2(acc[2], acc[3])), lo, hi);
    return make_float2(m, warp_sum(lo + hi) * tail_factor(m, s_lo));
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
        // the lane's first element equal to m: a match mask per vector (independent
        // compares), then the first vector with a match, then its first element
        uint32_t mask[kVec];
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
            mask[k] = 0u;
#pragma unroll
            for (int e = 0; e < E::kPerVec; ++e) mask[k] |= (E::get(v, k, e) == m ? 1u : 0u) << e;
        }
        int kf = kVec;
        uint32_t mf = 0u;
#pragma unroll
        for (int k = kVec - 1; k >= 0; --k)
            if (mask[k]) {
                kf = k;
                mf = mask[k];
            }
        if (kf < kVec) idx = (uint32_t)(chunk_base + (int64_t)(kf * 32 + lane) * E::kPerVec + (__ffs(mf) - 1));
    }
    idx = __reduce_min_sync(kFull, idx);
    return make_float2(m, __uint_as_float(idx));
}

// Fixed-point weight of a chunk relative to the row reference M (2^fx = weight 1).
__device__ __forceinline__ uint64_t chunk_fixed(float2 st, float M, int fx, float s_hi) {
    const float e = exponent_ref(st.x, s_hi);
    if (!(st.y > 0.f) || !isfinite(e)) return 0ull;
    const float d = fmaxf(e - M, -256.f);  // integer-valued, <= 0
    return to_fixed(st.y, (int)d + fx);
}

// Chunk statistics written by an earlier kernel are read through L1 (read-only path);
// those written earlier in the same kernel by other CTAs are read from L2.
template <bool FRESH>
__device__ __forceinline__ float2 ld_stat(const float2* ptr) {
    return FRESH ? __ldcg(ptr) : __ldg(ptr);
}

// Row combine (one warp): the row reference M = exponent_ref(row maximum), and the row
// sum Z = sum of the chunk sums scaled to M, exact in fixed point.  Returns false if the
// row is unusable (NaN or +inf anywhere, or every entry -inf).  The first 128 chunk
// statistics are loaded once into registers.
template <bool FRESH>
__device__ bool combine_row_sample(const float2* cs, int C, int fx, float s_hi, float s_lo, RowStat& out) {
    constexpr int kCache = 4;
    const int lane = threadIdx.x & 31;
    float2 cache[kCache];
#pragma unroll
    for (int i = 0; i < kCache; ++i) {
        const int c = lane + 32 * i;
        cache[i] = c < C ? ld_stat<FRESH>(&cs[c]) : make_float2(-INFINITY, 0.f);
    }
    bool bad = false;
    uint32_t key = 0;
    auto see = [&](float e) {
        if (isnan(e) || e == INFINITY) bad = true;
        else if (e > -INFINITY) key = max(key, order_key(e));
    };
#pragma unroll
    for (int i = 0; i < kCache; ++i) see(cache[i].x);
    for (int c = lane + 32 * kCache; c < C; c += 32) see(ld_stat<FRESH>(&cs[c]).x);
    key = __reduce_max_sync(kFull, key);
    bad = __any_sync(kFull, bad);
    const float m_row = key ? from_key(key) : -INFINITY;
    if (bad || !isfinite(m_row)) return false;
    const float M = exponent_ref(m_row, s_hi);
    uint64_t Z = 0;
#pragma unroll
    for (int i = 0; i < kCache; ++i) Z += chunk_fixed(cache[i], M, fx, s_hi);
    for (int c = lane + 32 * kCache; c < C; c += 32) Z += chunk_fixed(ld_stat<FRESH>(&cs[c]), M, fx, s_hi);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(kFull, Z, o);
    if (Z == 0ull) return false;
    out.Zfx = Z;
    out.M = M;
    out.Zf = fixed_to_float(Z, fx);
    out.T = tail_factor(m_row, s_lo);
    out.amax = -1;
    out.mx = m_row;
    return true;
}

template <bool FRESH>
__device__ bool combine_row_argmax(const float2* cs, int C, RowStat& out) {
    const int lane = threadIdx.x & 31;
    bool nan = false;
    uint32_t key = 0;
    for (int c = lane; c < C; c += 32) {
        float m = ld_stat<FRESH>(&cs[c]).x;
        if (isnan(m)) nan = true;
        else key = max(key, order_key(m));
    }
    key = __reduce_max_sync(kFull, key);
    nan = __any_sync(kFull, nan);
    const float m_row = from_key(key);
    if (nan || !isfinite(m_row)) return false;
    uint32_t first = 0xFFFFFFFFu;
    for (int c = lane; c < C; c += 32) {
        if (ld_stat<FRESH>(&cs[c]).x == m_row) first = min(first, (uint32_t)c);
    }
    first = __reduce_min_sync(kFull, first);
    if (first >= (uint32_t)C) return false;
    out.Zfx = 0ull;
    out.M = m_row;
    out.Zf = 0.f;
    out.T = 1.f;
    out.amax = (int)__float_as_uint(ld_stat<FRESH>(&cs[first]).y);
    out.mx = m_row;
    return true;
}

// Walk of a row's chunks (one warp): the first chunk whose inclusive fixed-point prefix
// exceeds `target`; *before = the prefix in front of it.  Returns -1 if none does
// (rounding), with *last_pos = the last chunk of positive weight (or -1).
template <typename WeightOf>
__device__ __forceinline__ int walk_chunks(int C, uint64_t target, WeightOf weight_of, uint64_t* before,
                                           int* last_pos) {
    const int lane = threadIdx.x & 31;
    uint64_t carry = 0;
    *last_pos = -1;
    for (int g = 0; g * 32 < C; ++g) {
        const int c = g * 32 + lane;
        const uint64_t w = c < C ? weight_of(c) : 0ull;
        const uint64_t incl = warp_incl_scan_u64(w);
        const unsigned pos = __ballot_sync(kFull, w > 0ull);
        if (pos) *last_pos = g * 32 + 31 - __clz(pos);
        const unsigned cross = __ballot_sync(kFull, c < C && carry + incl > target);
        if (cross) {
            const int l = __ffs(cross) - 1;
            *before = carry + (__shfl_sync(kFull, incl, l) - __shfl_sync(kFull, w, l));
            return g * 32 + l;
        }
        carry += __shfl_sync(kFull, incl, 31);
    }
    return -1;
}

// ----------------------------------------------------------------------------------------
// decision-side chunk buffers: each warp of a decide CTA owns two 4 KB shared-memory chunk
// buffers filled by 1-D bulk copies (or plain loads when rows are not 16-byte aligned) and
// works on them in rolled loops, so that code run once per warp stays small.
// ----------------------------------------------------------------------------------------
constexpr int kSlotBytes = 2 * kChunkBytes;
constexpr int kSharedResidualChunks = 512;  // residual chunk sums kept in shared memory up to this C
constexpr size_t kDecideSmem = (size_t)kWarps * kSlotBytes;

struct WarpSlot {
    unsigned char* a;  // first chunk buffer
    unsigned char* b;  // second chunk buffer
    uint32_t bar;      // mbarrier of this warp's copies
    uint32_t phase;    // parity of its next completion
};

__device__ __forceinline__ void bulk_load_plain(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// With bulk copies (p.vec_ok), the two halves of fetch_chunk: start the copies, then wait
// for them to land (whole warp each).
template <int DT>
__device__ __forceinline__ void start_chunk(const Params& p, WarpSlot& s, const void* rowA, const void* rowB, int c) {
    using E = Elem<DT>;
    const int64_t e0 = (int64_t)c * E::kChunk;
    const int n = (int)min((int64_t)E::kChunk, (int64_t)p.V - e0);
    __syncwarp();  // the warp's earlier reads of the buffers are complete
    if ((threadIdx.x & 31) == 0) {
        fence_proxy_async_smem();
        const uint32_t bytes = (uint32_t)n * E::kBytes;
        mbar_expect_tx(s.bar, rowB ? 2 * bytes : bytes);
        bulk_load_plain(smem_u32(s.a), static_cast<const char*>(rowA) + e0 * E::kBytes, bytes, s.bar);
        if (rowB) bulk_load_plain(smem_u32(s.b), static_cast<const char*>(rowB) + e0 * E::kBytes, bytes, s.bar);
    }
}
__device__ __forceinline__ void land_chunk(const Params& p, WarpSlot& s) {
    if (!__all_sync(kFull, mbar_wait_bounded(s.bar, s.phase, p.wait_ns))) {
        if ((threadIdx.x & 31) == 0) set_status(p, ISD_ERR_TIMEOUT);
        mbar_wait_bounded(s.bar, s.phase);  // let the copy land before the buffer is reused
    }
    s.phase ^= 1u;
}

// Copy chunk c of rowA (and of rowB, if given) into the warp's buffers (whole warp).
// Elements at or beyond V are not copied; readers mask them.
template <int DT>
__device__ void fetch_chunk(const Params& p, WarpSlot& s, const void* rowA, const void* rowB, int c) {
    using E = Elem<DT>;
    const int lane = threadIdx.x & 31;
    const int64_t e0 = (int64_t)c * E::kChunk;
    const int n = (int)min((int64_t)E::kChunk, (int64_t)p.V - e0);
    if (p.vec_ok) {
        start_chunk<DT>(p, s, rowA, rowB, c);
        land_chunk(p, s);
        return;
    }
    __syncwarp();  // the warp's earlier reads of the buffers are complete
    // plain loads; the rest of the buffer reads as -inf (the last vector may be partial)
    for (int i = lane; i < E::kChunk; i += 32) {
        if (DT == ISD_BF16) {
            reinterpret_cast<uint16_t*>(s.a)[i] = i < n ? static_cast<const uint16_t*>(rowA)[e0 + i] : 0xFF80u;
            if (rowB) reinterpret_cast<uint16_t*>(s.b)[i] = i < n ? static_cast<const uint16_t*>(rowB)[e0 + i] : 0xFF80u;
        } else {
            reinterpret_cast<uint32_t*>(s.a)[i] = i < n ? static_cast<const uint32_t*>(rowA)[e0 + i] : 0xFF800000u;
            if (rowB)
                reinterpret_cast<uint32_t*>(s.b)[i] = i < n ? static_cast<const uint32_t*>(rowB)[e0 + i] : 0xFF800000u;
        }
    }
    __syncwarp();
}

// Vector k of this lane from a chunk buffer; vectors at or beyond n elements read as -inf.
template <int DT>
__device__ __forceinline__ uint4 buf_vec(const unsigned char* buf, int k, int n) {
    using E = Elem<DT>;
    const int lane = threadIdx.x & 31;
    return (k * 32 + lane) * E::kPerVec < n
               ? reinterpret_cast<const uint4*>(buf)[k * 32 + lane]
               : make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
}
template <int DT>
__device__ __forceinline__ float vec_elem(const uint4& w, int j) {
    using E = Elem<DT>;
    const uint32_t* x = &w.x;
    if (DT == ISD_BF16) return __uint_as_float((j & 1) ? (x[j >> 1] & 0xFFFF0000u) : (x[j >> 1] << 16));
    return __uint_as_float(x[j]);
}

// Inverse CDF inside one chunk (one warp): the first element, in index order, whose
// running sum of weights exceeds `target`.  weights(k, a) fills a[] with the weights of
// this lane's vector k.  Returns the element's offset in the chunk, or -1 when the sum
// never exceeds the target (then *last = the last offset of positive weight, or -1).
template <int PER, typename Weights>
__device__ int rescan_chunk(float target, Weights weights, int* last) {
    const int lane = threadIdx.x & 31;
    float running = 0.f;
    int last_pos = -1;
#pragma unroll 1
    for (int k = 0; k < kVec; ++k) {
        float a[PER];
        weights(k, a);
        float lane_tot = 0.f;
#pragma unroll
        for (int j = 0; j < PER; ++j) lane_tot += a[j];
        float slot_tot;
        float cum = running + warp_excl_scan(lane_tot, slot_tot);
        int my_j = -1;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            cum += a[j];
            if (my_j < 0 && a[j] > 0.f && cum > target) my_j = j;
            if (a[j] > 0.f) last_pos = (k * 32 + lane) * PER + j;
        }
        const unsigned hit = __ballot_sync(kFull, my_j >= 0);
        if (hit) {
            const int l = __ffs(hit) - 1;
            return (k * 32 + l) * PER + __shfl_sync(kFull, my_j, l);
        }
        running += slot_tot;
    }
    *last = __reduce_max_sync(kFull, (unsigned)(last_pos + 1)) - 1;
    return -1;
}

// Inverse-CDF draw over one row (one warp), in two parts.  plan_draw walks the chunk sums
// to the chunk whose running sum first exceeds u*Z and gives the remaining target in that
// chunk's own units (head weights against its reference); finish_draw fetches the chunk
// and rescans it.  The plan needs only the statistics, so it can be made (and the chunk
// prefetched) before the decision that tells whether the draw is needed.
struct DrawPlan {
    int cstar;     // chunk holding the target
    float target;  // in head-weight units of that chunk; +inf when rounding overshot the row
};

__device__ DrawPlan plan_draw(const Params& p, const float2* cs, const RowStat& rs, uint32_t word) {
    const uint64_t target = scale_by_uniform(rs.Zfx, word);
    uint64_t before = 0;
    int last_pos;
    int cstar = walk_chunks(
        p.C, target, [&](int c) { return chunk_fixed(__ldg(&cs[c]), rs.M, p.fx, p.s_hi); }, &before, &last_pos);
    if (cstar < 0) return DrawPlan{last_pos < 0 ? 0 : last_pos, INFINITY};
    const float2 st = __ldg(&cs[cstar]);
    const int d = (int)fmaxf(exponent_ref(st.x, p.s_hi) - rs.M, -256.f);
    // the chunk sum carries the chunk's tail factor; the rescan sums head weights
    return DrawPlan{cstar, fixed_to_float(target - before, p.fx + d) / tail_factor(st.x, p.s_lo)};
}

// Start moving the plan's chunk of `row` into L2 (asynchronous; one lane).
template <int DT>
__device__ __forceinline__ void prefetch_chunk_l2(const Params& p, const void* row, int c) {
    using E = Elem<DT>;
    const int64_t e0 = (int64_t)c * E::kChunk;
    const int n = (int)min((int64_t)E::kChunk, (int64_t)p.V - e0);
    const char* src = static_cast<const char*>(row) + e0 * E::kBytes;
    if (p.vec_ok)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"((uint32_t)n * E::kBytes) : "memory");
    else
        asm volatile("prefetch.global.L2 [%0];" ::"l"(src));
}

template <int DT>
__device__ __noinline__ int finish_draw(const Params& p, WarpSlot& slot, const void* row, const float2* cs,
                                        const RowStat& rs, DrawPlan plan, float* px) {
    using E = Elem<DT>;
    const int lane = threadIdx.x & 31;
    const int cstar = plan.cstar;
    const float ref = ref_or_zero(exponent_ref(__ldg(&cs[cstar]).x, p.s_hi));
    fetch_chunk<DT>(p, slot, row, nullptr, cstar);
    const int n = (int)min((int64_t)E::kChunk, (int64_t)p.V - (int64_t)cstar * E::kChunk);
    const float s_hi = p.s_hi;
    int last;
    int off = rescan_chunk<E::kPerVec>(
        plan.target,
        [&](int k, float* a) {
            const uint4 w = buf_vec<DT>(slot.a, k, n);
#pragma unroll
            for (int j = 0; j < E::kPerVec; ++j) a[j] = weight_head(vec_elem<DT>(w, j), ref, s_hi);
        },
        &last);
    if (off < 0) {  // overshoot inside the chunk: the last index with positive weight
        off = last < 0 ? 0 : last;
        if (lane == 0) diag_add(p, ISD_DIAG_NEAR_TIE_CDF, 1);
    }
    const float x = DT == ISD_BF16 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(slot.a)[off] << 16)
                                   : reinterpret_cast<const float*>(slot.a)[off];
    *px = exp2f(weight_exp(x, rs.M, p.s_hi, p.s_lo)) / rs.Zf;
    return (int)((int64_t)cstar * E::kChunk + off);
}

template <int DT>
__device__ int draw_row(const Params& p, WarpSlot& slot, const void* row, const float2* cs, const RowStat& rs,
                        uint32_t word, float* px) {
    return finish_draw<DT>(p, slot, row, cs, rs, plan_draw(p, cs, rs, word), px);
}

// ----------------------------------------------------------------------------------------
// argmax proposals verified by sampling: a proposal is the argmax of its MASK row (q = 1, a
// point mass), kept with probability p(x); after a rejection the replacement is drawn from
// max(0, p - delta_x), i.e. p without x
// ----------------------------------------------------------------------------------------
// The first chunk of a row whose maximum is the row maximum mx (one warp).
__device__ DrawPlan plan_argmax(const Params& p, const float2* cs, const RowStat& rs) {
    const int lane = threadIdx.x & 31;
    for (int c0 = 0; c0 < p.C; c0 += 32) {
        const int c = c0 + lane;
        const unsigned hit = __ballot_sync(kFull, c < p.C && __ldg(&cs[c]).x == rs.mx);
        if (hit) return DrawPlan{c0 + __ffs(hit) - 1, 0.f};
    }
    return DrawPlan{0, 0.f};
}

// The lowest index of chunk cstar of `row` holding the value mx (one warp).
template <int DT>
__device__ __noinline__ int finish_argmax(const Params& p, WarpSlot& slot, const void* row, int cstar, float mx) {
    using E = Elem<DT>;
    fetch_chunk<DT>(p, slot, row, nullptr, cstar);
    const int n = (int)min((int64_t)E::kChunk, (int64_t)p.V - (int64_t)cstar * E::kChunk);
#pragma unroll 1
    for (int k = 0; k < kVec; ++k) {
        const uint4 w = buf_vec<DT>(slot.a, k, n);
        int my_j = -1;
#pragma unroll
        for (int j = E::kPerVec - 1; j >= 0; --j)
            if (vec_elem<DT>(w, j) == mx) my_j = j;
        const unsigned hit = __ballot_sync(kFull, my_j >= 0);
        if (hit) {
            const int l = __ffs(hit) - 1;
            return (int)((int64_t)cstar * E::kChunk + (k * 32 + l) * E::kPerVec + __shfl_sync(kFull, my_j, l));
        }
    }
    return (int)((int64_t)cstar * E::kChunk);  // not reached: the chunk holds the maximum
}

// Inverse-CDF draw from row `row` without token x (logit xl), one warp: the fixed-point
// weight of x, computed as the statistics pass weighs it, is taken out of its chunk's sum
// and of the row total; the walk and the rescan then skip it.
template <int DT>
__device__ __noinline__ int draw_excluding(const Params& p, WarpSlot& slot, const void* row, const float2* cs,
                                           const RowStat& rs, int x, float xl, uint32_t word) {
    using E = Elem<DT>;
    const int lane = threadIdx.x & 31;
    const int cx = x / E::kChunk;
    const float2 stx = __ldg(&cs[cx]);
    const float ex = ref_or_zero(exponent_ref(stx.x, p.s_hi));
    const int dx = (int)fmaxf(ex - rs.M, -256.f);
    const uint64_t cfx = chunk_fixed(stx, rs.M, p.fx, p.s_hi);
    const uint64_t wx = to_fixed(weight_head(xl, ex, p.s_hi) * tail_factor(stx.x, p.s_lo), p.fx + dx);
    const uint64_t cut = wx < cfx ? wx : cfx;
    const uint64_t total = rs.Zfx - cut;
    if (total == 0ull) {  // all of the row's mass on x: reachable only through rounding
        if (lane == 0) diag_add(p, ISD_DIAG_NEAR_TIE_CDF, 1);
        float px;
        return draw_row<DT>(p, slot, row, cs, rs, word, &px);
    }
    const uint64_t target = scale_by_uniform(total, word);
    uint64_t before = 0;
    int last_pos;
    int cstar = walk_chunks(
        p.C, target,
        [&](int c) {
            const uint64_t w = chunk_fixed(__ldg(&cs[c]), rs.M, p.fx, p.s_hi);
            return c == cx ? w - cut : w;
        },
        &before, &last_pos);
    float local = INFINITY;
    if (cstar < 0) {
        cstar = last_pos < 0 ? 0 : last_pos;
    } else {
        const float2 st = __ldg(&cs[cstar]);
        const int d = (int)fmaxf(exponent_ref(st.x, p.s_hi) - rs.M, -256.f);
        local = fixed_to_float(target - before, p.fx + d) / tail_factor(st.x, p.s_lo);
    }
    const float ref = ref_or_zero(exponent_ref(__ldg(&cs[cstar]).x, p.s_hi));
    fetch_chunk<DT>(p, slot, row, nullptr, cstar);
    const int n = (int)min((int64_t)E::kChunk, (int64_t)p.V - (int64_t)cstar * E::kChunk);
    const int xoff = cstar == cx ? x - cstar * E::kChunk : -1;
    const float s_hi = p.s_hi;
    int last;
    int off = rescan_chunk<E::kPerVec>(
        local,
        [&](int k, float* a) {
            const uint4 w = buf_vec<DT>(slot.a, k, n);
#pragma unroll
            for (int j = 0; j < E::kPerVec; ++j)
                a[j] = (k * 32 + lane) * E::kPerVec + j == xoff ? 0.f : weight_head(vec_elem<DT>(w, j), ref, s_hi);
        },
        &last);
    if (off < 0) {
        off = last < 0 ? 0 : last;
        if (lane == 0) diag_add(p, ISD_DIAG_NEAR_TIE_CDF, 1);
    }
    return (int)((int64_t)cstar * E::kChunk + off);
}

// ----------------------------------------------------------------------------------------
// residual: max(0, p - q) with p = softmax(anchor row K / T), q = softmax(q row / T)
// ----------------------------------------------------------------------------------------
// One entry of max(0, p - q): p = 2^(xp*s_hi - Mp) * ap and q = 2^(xq*s_hi - Mq) * aq, where
// a = T/Z carries the row's normaliser and tail factor (2^(x*s_lo) taken at the row maximum:
// for the entries that carry mass this is exact to ~1e-8 of the mass).  naq = -aq.
__device__ __forceinline__ float residual_elem(float xp, float xq, float Mp, float Mq, float ap, float naq,
                                               float s_hi) {
    const float pw = ex2_approx(fmaf(xp, s_hi, -Mp));
    const float qw = ex2_approx(fmaf(xq, s_hi, -Mq));
    return fmaxf(fmaf(pw, ap, fmaf(qw, naq, 0.f)), 0.f);
}

// Sum of max(0, p - q) over the chunk held in the warp's buffers (a = p row, b = q row),
// entry pairs on the f32x2 pipe with the same per-entry arithmetic as residual_elem.
template <int DT>
__device__ float residual_chunk_sum(const WarpSlot& slot, int n, const RowStat& ps, const RowStat& qs, float ap,
                                    float naq, float s_hi) {
    const uint64_t S2 = pack2(s_hi, s_hi), NMP2 = pack2(-ps.M, -ps.M), NMQ2 = pack2(-qs.M, -qs.M);
    const uint64_t AP2 = pack2(ap, ap), NAQ2 = pack2(naq, naq), Z2 = 0ull;
    uint64_t acc0 = 0ull, acc1 = 0ull;
#pragma unroll 2
    for (int k = 0; k < kVec; ++k) {
        const uint4 wp = buf_vec<DT>(slot.a, k, n), wq = buf_vec<DT>(slot.b, k, n);
        const uint32_t* xp = &wp.x;
        const uint32_t* xq = &wq.x;
#pragma unroll
        for (int h = 0; h < (DT == ISD_BF16 ? 4 : 2); ++h) {
            uint64_t p2, q2;
            if (DT == ISD_BF16) {
                p2 = pack2(__uint_as_float(xp[h] << 16), __uint_as_float(xp[h] & 0xFFFF0000u));
                q2 = pack2(__uint_as_float(xq[h] << 16), __uint_as_float(xq[h] & 0xFFFF0000u));
            } else {
                p2 = pack2(__uint_as_float(xp[2 * h]), __uint_as_float(xp[2 * h + 1]));
                q2 = pack2(__uint_as_float(xq[2 * h]), __uint_as_float(xq[2 * h + 1]));
            }
            float a0, a1, b0, b1;
            unpack2(fma2(p2, S2, NMP2), a0, a1);
            unpack2(fma2(q2, S2, NMQ2), b0, b1);
            const uint64_t d2 = fma2(pack2(ex2_approx(a0), ex2_approx(a1)), AP2,
                                     fma2(pack2(ex2_approx(b0), ex2_approx(b1)), NAQ2, Z2));
            float d0, d1;
            unpack2(d2, d0, d1);
            const uint64_t r2 = pack2(fmaxf(d0, 0.f), fmaxf(d1, 0.f));
            if (h & 1) acc1 = add2(acc1, r2);
            else acc0 = add2(acc0, r2);
        }
    }
    float lo, hi;
    unpack2(add2(acc0, acc1), lo, hi);
    return warp_sum(lo + hi);
}

// Inverse-CDF draw of the replacement token from the residual (one warp): walk the chunk
// sums rc[] (fixed point; *rtotal is their exact total), then rescan the chunk holding
// u * total.  If no residual mass is left (only possible through rounding) the token is
// drawn from p instead.
template <int DT>
__device__ __noinline__ int draw_residual(const Params& p, WarpSlot& slot, const void* prow, const void* qrow,
                                          const float2* pchunk, const float* rc, bool rc_shared,
                                          const uint64_t* rtotal, const RowStat& ps, const RowStat& qs,
                                          uint32_t word) {
    using E = Elem<DT>;
    const int lane = threadIdx.x & 31;
    uint64_t total;
    if (rc_shared) {  // the chunk sums are in this CTA's shared memory: their exact fixed-point total
        total = 0ull;
        for (int c = lane; c < p.C; c += 32) total += to_fixed(rc[c], p.fxr);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(kFull, total, o);
    } else {
        total = __ldcg(reinterpret_cast<const unsigned long long*>(rtotal));
    }
    if (total == 0ull) {
        if (lane == 0) diag_add(p, ISD_DIAG_NEAR_TIE_CDF, 1);
        float px;
        return draw_row<DT>(p, slot, prow, pchunk, ps, word, &px);
    }
    const uint64_t target = scale_by_uniform(total, word);
    uint64_t before = 0;
    int last_pos;
    int cstar = walk_chunks(
        p.C, target, [&](int c) { return to_fixed(rc_shared ? rc[c] : __ldcg(&rc[c]), p.fxr); }, &before, &last_pos);
    const bool overshoot = cstar < 0;
    if (overshoot) cstar = last_pos < 0 ? 0 : last_pos;
    const float local_target = overshoot ? INFINITY : fixed_to_float(target - before, p.fxr);
    const float ap = ps.T / ps.Zf, naq = -(qs.T / qs.Zf);
    fetch_chunk<DT>(p, slot, prow, qrow, cstar);
    const int n = (int)min((int64_t)E::kChunk, (int64_t)p.V - (int64_t)cstar * E::kChunk);
    const float s_hi = p.s_hi;
    int last;
    int off = rescan_chunk<E::kPerVec>(
        local_target,
        [&](int k, float* a) {
            const uint4 wp = buf_vec<DT>(slot.a, k, n), wq = buf_vec<DT>(slot.b, k, n);
#pragma unroll
            for (int j = 0; j < E::kPerVec; ++j)
                a[j] = residual_elem(vec_elem<DT>(wp, j), vec_elem<DT>(wq, j), ps.M, qs.M, ap, naq, s_hi);
        },
        &last);
    if (off < 0) {
        off = last < 0 ? 0 : last;
        if (lane == 0) diag_add(p, ISD_DIAG_NEAR_TIE_CDF, 1);
    }
    return (int)((int64_t)cstar * E::kChunk + off);
}

// ----------------------------------------------------------------------------------------
// statistics pass
// ----------------------------------------------------------------------------------------
// Units are the chunks of all rows, u = (b*R + r)*C + c, dealt round-robin to the grid's
// warps.  A warp walks its units with a cursor (b, r, c) advanced by the grid stride in the
// same mixed radix, so the loop needs no division.  Rows 0..N-2 of a sequence without
// pending tokens are not read.
struct Cursor {
    int b, r, c;
};

__device__ __forceinline__ Cursor cursor_of(int64_t u, int R, int C) {
    const int64_t row = u / C;
    return Cursor{(int)(row / R), (int)(row - (row / R) * R), (int)(u - row * C)};
}
__device__ __forceinline__ void advance(Cursor& x, const Cursor& s, int R, int C) {
    x.c += s.c;
    int carry = x.c >= C;
    if (carry) x.c -= C;
    x.r += s.r + carry;  // < 2R, since s.r < R
    carry = x.r >= R;
    if (carry) x.r -= R;
    x.b += s.b + carry;
}
// Move x forward on the stride to the first unit the step reads; false if none is left.
__device__ __forceinline__ bool next_needed(const Params& p, Cursor& x, const Cursor& s) {
    for (; x.b < p.B; advance(x, s, p.R, p.C)) {
        if (x.r >= p.N - 1) return true;
        if (p.pending[(int64_t)x.b * p.pending_ld] >= 0) return true;
    }
    return false;
}
__device__ __forceinline__ int64_t unit_row(const Params& p, const Cursor& x) { return (int64_t)x.b * p.R + x.r; }

template <int DT, bool GREEDY>
__device__ __forceinline__ void write_chunk_stat(const Params& p, const Cursor& x, const uint4 (&v)[kVec]) {
    const int64_t base = (int64_t)x.c * Elem<DT>::kChunk;
    const float2 st = GREEDY ? chunk_stat_argmax<DT>(v, base) : chunk_stat_sample<DT>(v, p.s_hi, p.s_lo);
    if ((threadIdx.x & 31) == 0) p.chunk[unit_row(p, x) * p.C + x.c] = st;
}

// Units come in batches of kGrab consecutive units from a global counter, so that faster
// SMs take more of the work; within a batch the cursor steps by one unit.
constexpr int kGrab = 4;

struct UnitSource {
    Cursor x;  // next unit of the current batch
    int left;  // units left in the batch
};

__device__ __forceinline__ void step_one(Cursor& x, int R, int C) {
    if (++x.c == C) {
        x.c = 0;
        if (++x.r == R) {
            x.r = 0;
            ++x.b;
        }
    }
}

// A warp's first batch, taken without the counter: at launch every warp would otherwise
// claim at once, and those atomics on one address serialise.
__device__ __forceinline__ UnitSource first_batch(int R, int C, int64_t U, int64_t warp_global) {
    const int64_t base = warp_global * kGrab;
    if (base >= U) return UnitSource{Cursor{0, 0, 0}, 0};
    return UnitSource{cursor_of(base, R, C), (int)min((int64_t)kGrab, U - base)};
}

// The next unit the step reads (whole warp, uniform); false once the counter is exhausted.
__device__ __forceinline__ bool next_unit(const Params& p, UnitSource& q, Cursor& out) {
    const int64_t U = (int64_t)p.B * p.R * p.C;
    for (;;) {
        while (q.left > 0) {
            const Cursor x = q.x;
            --q.left;
            step_one(q.x, p.R, p.C);
            if (x.r >= p.N - 1 || p.pending[(int64_t)x.b * p.pending_ld] >= 0) {
                out = x;
                return true;
            }
        }
        // the first batch of every warp is fixed (first_batch), the counter deals the rest
        const int64_t first = (int64_t)gridDim.x * (blockDim.x >> 5) * kGrab;
        unsigned long long base = 0;
        if ((threadIdx.x & 31) == 0) base = atomicAdd(p.sched, (unsigned long long)kGrab) + (unsigned long long)first;
        base = __shfl_sync(kFull, base, 0);
        if ((int64_t)base >= U) return false;
        q.x = cursor_of((int64_t)base, p.R, p.C);
        q.left = (int)min((int64_t)kGrab, U - (int64_t)base);
    }
}

// Bulk-copy pipeline: rows must start on 16-byte boundaries and V * element size must be a
// multiple of 16 bytes (every copy is then 16-byte aligned and sized).
template <int DT, bool GREEDY>
__global__ void __launch_bounds__(kSThreads, 1) isd_stats_kernel(Params p) {
    using E = Elem<DT>;
    extern __shared__ __align__(128) unsigned char s_stage[];  // [kSWarps][kDepth][kChunkBytes]
    __shared__ __align__(8) uint64_t s_bar[kSWarps][kDepth];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (blockIdx.x == 0 && p.rtotal)  // residual totals of this step start at zero
        for (int i = threadIdx.x; i < p.B; i += blockDim.x) p.rtotal[i] = 0ull;
    unsigned char* stage = s_stage + (size_t)warp * kDepth * kChunkBytes;
    const uint32_t bar = smem_u32(&s_bar[warp][0]);
    if (lane == 0) {
        for (int d = 0; d < kDepth; ++d) mbar_init(bar + 8 * d, 1);
        fence_mbar_init();
    }
    __syncwarp();
    allow_dependent_launch();  // the decide kernel waits for this grid to finish anyway
    const uint64_t policy = evict_first_policy();

    auto issue = [&](const Cursor& x, int d) {
        const int64_t e0 = (int64_t)x.c * E::kChunk;
        const int64_t n = min((int64_t)E::kChunk, (int64_t)p.V - e0);
        const uint32_t bytes = (uint32_t)(n * E::kBytes);
        const char* src = static_cast<const char*>(p.logits) + (unit_row(p, x) * p.V + e0) * E::kBytes;
        mbar_expect_tx(bar + 8 * d, bytes);
        bulk_load(smem_u32(stage + d * kChunkBytes), src, bytes, bar + 8 * d, policy);
    };

    UnitSource src = first_batch(p.R, p.C, (int64_t)p.B * p.R * p.C, (int64_t)blockIdx.x * kSWarps + warp);
    Cursor cur[kDepth];  // unit held by each stage
    bool full[kDepth];
#pragma unroll
    for (int d = 0; d < kDepth; ++d) {
        full[d] = next_unit(p, src, cur[d]);
        if (full[d] && lane == 0) issue(cur[d], d);
    }
    uint32_t phase = 0;
    bool timed_out = false, done = false;
    while (!done) {
#pragma unroll
        for (int d = 0; d < kDepth; ++d) {
            if (done) break;
            if (!full[d]) {  // stages empty in ring order: nothing left in flight
                done = true;
                break;
            }
            if (!__all_sync(kFull, mbar_wait_bounded(bar + 8 * d, (phase >> d) & 1u, p.wait_ns))) {
                timed_out = true;
                done = true;
                break;
            }
            phase ^= 1u << d;
            uint4 v[kVec];
            const Cursor x = cur[d];
            const uint4* sv = reinterpret_cast<const uint4*>(stage + d * kChunkBytes);
            if (x.c + 1 < p.C) {  // a full chunk
#pragma unroll
                for (int k = 0; k < kVec; ++k) v[k] = sv[k * 32 + lane];
            } else {  // the row's last chunk: entries past V read as -inf
                const int n = p.V - x.c * E::kChunk;
#pragma unroll
                for (int k = 0; k < kVec; ++k)
                    v[k] = (k * 32 + lane) * E::kPerVec < n
                               ? sv[k * 32 + lane]
                               : make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
            }
            __syncwarp();
            // refill this stage before reducing the chunk held in registers
            full[d] = next_unit(p, src, cur[d]);
            if (full[d] && lane == 0) {
                fence_proxy_async_smem();
                issue(cur[d], d);
            }
            write_chunk_stat<DT, GREEDY>(p, x, v);
        }
    }
    if (timed_out) {
        if (lane == 0) set_status(p, ISD_ERR_TIMEOUT);
        // let the copies still in flight land before the CTA's shared memory is released
#pragma unroll
        for (int d = 0; d < kDepth; ++d)
            if (full[d]) mbar_wait_bounded(bar + 8 * d, (phase >> d) & 1u);
    }
}

// Plain-load variant for shapes the bulk copies cannot serve (rows not 16-byte aligned).
template <int DT, bool GREEDY>
__global__ void __launch_bounds__(kThreads) isd_stats_plain_kernel(Params p) {
    if (blockIdx.x == 0 && p.rtotal)  // residual totals of this step start at zero
        for (int i = threadIdx.x; i < p.B; i += blockDim.x) p.rtotal[i] = 0ull;
    const int warp = threadIdx.x >> 5;
    const int dtb = DT == ISD_BF16 ? 2 : 4;
    const Cursor stride = cursor_of((int64_t)gridDim.x * kWarps, p.R, p.C);
    allow_dependent_launch();
    Cursor x = cursor_of((int64_t)blockIdx.x * kWarps + warp, p.R, p.C);
    for (; next_needed(p, x, stride); advance(x, stride, p.R, p.C)) {
        uint4 v[kVec];
        load_chunk<DT>(row_ptr(p.logits, dtb, unit_row(p, x), p.V), p.V, (int64_t)x.c * Elem<DT>::kChunk,
                       p.vec_ok, true, v);
        write_chunk_stat<DT, GREEDY>(p, x, v);
    }
}

// ----------------------------------------------------------------------------------------
// decision pass: one cluster of CL CTAs per sequence
// ----------------------------------------------------------------------------------------
template <int DT, bool GREEDY>
__global__ void __launch_bounds__(kThreads, 4) isd_decide_kernel(Params p, int CL) {
    using E = Elem<DT>;
    __shared__ RowStat s_rs[kMaxR];
    __shared__ RowStat s_qs;
    __shared__ int s_bad, s_K, s_state, s_qok, s_carry;
    __shared__ DrawPlan s_plan[ISD_MAX_N];  // draw plans of rows N-1..2N-2 owned by this CTA
    __shared__ float s_rc[kSharedResidualChunks];  // leader CTA: the residual's chunk sums
    extern __shared__ __align__(128) unsigned char s_buf[];  // [kWarps][2][kChunkBytes]
    __shared__ __align__(8) uint64_t s_wbar[kWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WarpSlot slot{s_buf + (size_t)warp * kSlotBytes, s_buf + (size_t)warp * kSlotBytes + kChunkBytes,
                  smem_u32(&s_wbar[warp]), 0u};
    if (lane == 0) {
        mbar_init(slot.bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    const int crank = CL > 1 ? (int)cluster_ctarank() : 0;
    const bool leader = crank == 0;
    const int b = blockIdx.x / CL;
    const int N = p.N, R = p.R, V = p.V, C = p.C;
    const int dtb = DT == ISD_BF16 ? 2 : 4;
    // Inputs that do not come from the statistics kernel are read before waiting for it:
    // the pending tokens, their q and their logits at the anchor rows.
    const int32_t* pend = p.pending + (int64_t)b * p.pending_ld;
    const bool has_pending = pend[0] >= 0;
    const int first_row = has_pending ? 0 : N - 1;
    const int slot_read = (int)((p.step - 1) & 1), slot_write = (int)(p.step & 1);
    int x = -1;
    float xq = 0.f, xl = 0.f, u_acc = 0.f;
    RowStat carried;  // lane i: the previous call's statistics of its MASK row N+i (a residual's q row)
    memset(&carried, 0, sizeof carried);
    if (warp == 0 && has_pending && lane < N - 1) {
        x = pend[lane];
        if (!GREEDY) {
            xq = p.pending_q[(int64_t)b * (N - 1) + lane];
            if (x >= 0 && x < V) xl = load_elem<DT>(row_ptr(p.logits, dtb, (int64_t)b * R + lane, V), x);
            u_acc = to_uniform(row_words(p.seed, p.step, b, lane).x);  // the acceptance test's uniform
            if (!p.amode && p.prev) carried = p.carry[((int64_t)slot_read * p.B + b) * (N - 1) + lane];
        }
    }
    if (threadIdx.x == 0) {
        s_bad = 0;
        int use = 0;
        if (!GREEDY) {  // were the q rows' statistics left by the call that produced prev_logits?
            const CarryKey k = p.carry_key[slot_read];
            use = k.tag == kCarryTag && k.logits == p.prev && k.step + 1 == p.step && k.B == p.B && k.N == p.N &&
                  k.V == p.V && k.dtype == p.dtype && k.s_hi == p.s_hi && k.s_lo == p.s_lo;
        }
        s_carry = use;
        if (blockIdx.x == 0) {  // name this call as the writer of its slot (unused in greedy mode)
            CarryKey k;
            memset(&k, 0, sizeof k);
            k.logits = p.logits;
            k.step = p.step;
            k.B = p.B;
            k.N = p.N;
            k.V = p.V;
            k.dtype = p.dtype;
            k.s_hi = p.s_hi;
            k.s_lo = p.s_lo;
            k.tag = GREEDY ? 0u : kCarryTag;
            p.carry_key[slot_write] = k;
        }
    }
    wait_for_prerequisite_grid();  // the chunk statistics of this step are complete
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.sched = 0ull;  // the next step's work counter
    __syncthreads();

    // 1. the anchor rows' statistics (every CTA of the cluster, identically)
    for (int r = warp; r < (has_pending ? N - 1 : 0); r += kWarps) {
        const float2* cs = p.chunk + ((int64_t)b * R + r) * C;
        RowStat rs;
        const bool ok = GREEDY ? combine_row_argmax<false>(cs, C, rs) : combine_row_sample<false>(cs, C, p.fx, p.s_hi, p.s_lo, rs);
        if (lane == 0) {
            if (!ok) atomicOr(&s_bad, 1);
            s_rs[r] = rs;
        }
    }
    __syncthreads();

    // 2. acceptance tests and the first rejection (warp 0 of every CTA; the leader writes)
    int32_t* tok = p.tokens_out + (int64_t)b * R;
    float* nq = p.new_q + (int64_t)b * (N - 1);
    bool bad_pending = false;  // (warp 0)
    float pv = 0.f;            // (warp 0, lane i < N-1) p(x_i) at anchor row i
    if (warp == 0) {
        int K = N - 1;
        int state = 1;  // 0 error, 1 propose, 2 rejected at K
        bool accept = true;
        if (has_pending && lane < N - 1) {
            if (x < 0 || x >= V) bad_pending = true;
            if (!GREEDY && (!(xq > 0.f && xq < INFINITY) || (p.prev == nullptr && !p.amode))) bad_pending = true;
        }
        bad_pending = __any_sync(kFull, bad_pending);
        if (bad_pending || (s_bad & 1)) {
            state = 0;
        } else if (has_pending) {
            if (lane < N - 1) {
                if (GREEDY) {
                    accept = (x == s_rs[lane].amax);
                } else {
                    const RowStat rs = s_rs[lane];
                    pv = exp2f(weight_exp(xl, rs.M, p.s_hi, p.s_lo)) / rs.Zf;
                    const float q = xq;
                    const float u = u_acc;
                    // u < p/q  <=>  u*q < p, with u*q = prod + err exactly (err from an FMA)
                    const float prod = u * q;
                    accept = prod < pv || (prod == pv && fmaf(u, q, -prod) < 0.f);
                    if (leader && fabsf(u - pv / q) < (float)kNearTie) diag_add(p, ISD_DIAG_NEAR_TIE_ACC, 1);
                }
            }
            const unsigned rej = __ballot_sync(kFull, lane < N - 1 && !accept);
            K = rej ? __ffs(rej) - 1 : N - 1;
            state = K < N - 1 ? 2 : 1;
        }
        if (!GREEDY && !p.amode && state == 2 && s_carry && lane == K) {  // the residual's q row
            s_qs = carried;
            s_qok = carried.Zfx > 0ull;
        }
        if (lane == 0) {
            s_K = K;
            s_state = state;
        }
    }
    __syncthreads();
    // a rejection whose q row's statistics were carried: each warp starts its first chunk pair
    // of the residual now, ahead of the outputs and the rest of the set-up
    const bool early = !GREEDY && !p.amode && p.vec_ok && s_state == 2 && s_carry && s_qok;
    const int c_first = crank * kWarps + warp;
    if (early && c_first < C)
        start_chunk<DT>(p, slot, row_ptr(p.logits, dtb, (int64_t)b * R + s_K, V),
                        row_ptr(p.prev, dtb, (int64_t)b * R + N + s_K, V), c_first);
    // the anchor row N-1 and the MASK rows, read only by a sequence that proposes (every CTA
    // of the cluster, identically).  For the rows this CTA will draw from (row N-1+j belongs
    // to CTA j % CL and to the warp that combines it) the draw is planned now and its chunk
    // prefetched into L2.
    if (s_state == 1) {
        for (int r = N - 1 + warp; r < R; r += kWarps) {
            const float2* cs = p.chunk + ((int64_t)b * R + r) * C;
            RowStat rs;
            const bool ok =
                GREEDY ? combine_row_argmax<false>(cs, C, rs) : combine_row_sample<false>(cs, C, p.fx, p.s_hi, p.s_lo, rs);
            if (lane == 0) {
                if (!ok) atomicOr(&s_bad, 2);
                s_rs[r] = rs;
            }
            if (!GREEDY && ok && (r - (N - 1)) % CL == crank) {
                const DrawPlan plan = p.amode && r >= N ? plan_argmax(p, cs, rs)
                                                        : plan_draw(p, cs, rs, row_words(p.seed, p.step, b, r).y);
                if (lane == 0) {
                    s_plan[r - (N - 1)] = plan;
                    prefetch_chunk_l2<DT>(p, row_ptr(p.logits, dtb, (int64_t)b * R + r, V), plan.cstar);
                }
            }
        }
        __syncthreads();
    }
    if (warp == 0) {
        const int K = s_K;
        int state = s_state;
        const int bad_rows = s_bad;
        // a proposing sequence fails if one of the rows it draws from is unusable
        if (state == 1 && (bad_rows & 2)) state = 0;
        if (!GREEDY && leader && state != 0 && has_pending && lane < N - 1 && p.p_out)
            p.p_out[(int64_t)b * (N - 1) + lane] = pv;
        if (leader) {
            // the leader writes every output the draws below do not write
            const int bonus_pos = has_pending ? N - 1 : 0;
            for (int i = lane; i < R; i += 32) {
                int t = -1;
                bool mine = true;
                if (state != 0) {
                    if (has_pending && i < K) t = pend[i];
                    if (GREEDY) {
                        if (state == 2 && i == K) t = s_rs[K].amax;
                        if (state == 1) {
                            if (i == bonus_pos) t = s_rs[N - 1].amax;
                            if (i >= N) t = s_rs[i].amax;
                        }
                    } else {
                        if (state == 2 && i == K) mine = false;
                        if (state == 1 && (i == bonus_pos || i >= N)) mine = false;
                    }
                }
                if (mine) tok[i] = t;
            }
            if (GREEDY || state != 1)
                for (int i = lane; i < N - 1; i += 32) nq[i] = (GREEDY && state == 1) ? 1.f : 0.f;
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
                    if (!GREEDY && state == 2) diag_add(p, ISD_DIAG_RESIDUALS, 1);
                }
                if ((!has_pending || state == 0 || GREEDY) && p.p_out)
                    for (int i = 0; i < N - 1; ++i) p.p_out[(int64_t)b * (N - 1) + i] = 0.f;
            }
        }
        if (lane == 0) {
            s_K = K;
            s_state = state;
        }
    }
    __syncthreads();
    if (GREEDY) return;
    const int state = s_state, K = s_K;

    if (state == 2 && p.amode) {
        // 3a'. the rejected proposal was a point mass: the replacement comes from anchor row K
        // without it, drawn by the leader alone (no previous row, no residual pass)
        const int xk = __shfl_sync(kFull, x, K);
        const float xlk = __shfl_sync(kFull, xl, K);
        if (leader && warp == 0) {
            const int y = draw_excluding<DT>(p, slot, row_ptr(p.logits, dtb, (int64_t)b * R + K, V),
                                             p.chunk + ((int64_t)b * R + K) * C, s_rs[K], xk, xlk,
                                             row_words(p.seed, p.step, b, K).y);
            if (lane == 0) tok[K] = y;
        }
    } else if (state == 2) {
        // 3a. replacement token from the residual.  Same state in every CTA of the cluster,
        // so all of them reach both cluster barriers.
        const void* qrow = row_ptr(p.prev, dtb, (int64_t)b * R + N + K, V);
        const void* prow = row_ptr(p.logits, dtb, (int64_t)b * R + K, V);
        float2* qc = p.qchunk + (int64_t)b * C;
        float* rc = p.rchunk + (int64_t)b * C;
        // start this CTA's chunks of both rows towards L2 now
        for (int c = crank * kWarps + warp; c < C; c += CL * kWarps) {
            if (lane == 0) prefetch_chunk_l2<DT>(p, prow, c);
            if (lane == 1) prefetch_chunk_l2<DT>(p, qrow, c);
        }
        if (s_carry) {  // the previous call left the q row's statistics (read in the prologue)
            if (warp == 0 && lane == K) {
                s_qs = carried;
                s_qok = carried.Zfx > 0ull;
            }
            __syncthreads();
        } else {
            for (int c = crank * kWarps + warp; c < C; c += CL * kWarps) {
                uint4 v[kVec];
                load_chunk<DT>(qrow, V, (int64_t)c * E::kChunk, p.vec_ok, false, v);
                const float2 st = chunk_stat_sample<DT>(v, p.s_hi, p.s_lo);
                if (lane == 0) qc[c] = st;
            }
            if (CL > 1) cluster_sync();  // release/acquire at cluster scope covers the global writes
            else __syncthreads();
            if (warp == 0) {
                RowStat qs;
                const bool ok = combine_row_sample<true>(qc, C, p.fx, p.s_hi, p.s_lo, qs);
                if (lane == 0) {
                    s_qs = qs;
                    s_qok = ok ? 1 : 0;
                }
            }
            __syncthreads();
        }
        if (!s_qok) {  // the q row is unusable: the sequence fails (same in every CTA)
            if (leader && threadIdx.x == 0) {
                p.accepted_len[b] = 0;
                for (int i = 0; i < R; ++i) tok[i] = -1;
                set_status(p, ISD_ERR_NONFINITE);
            }
            return;
        }
        const RowStat ps = s_rs[K], qs = s_qs;
        const float ap = ps.T / ps.Zf, naq = -(qs.T / qs.Zf);
        // the chunk sums go to the leader CTA's shared memory when they fit (the leader then
        // needs no global round trip to walk them), else to global memory with an exact total
        const bool rc_shared = C <= kSharedResidualChunks;
        const uint32_t rc_leader = CL > 1 ? cluster_map_shared(smem_u32(s_rc), 0) : smem_u32(s_rc);
        for (int c = crank * kWarps + warp; c < C; c += CL * kWarps) {
            if (early && c == c_first) land_chunk(p, slot);  // started after the decision
            else fetch_chunk<DT>(p, slot, prow, qrow, c);
            const int n = (int)min((int64_t)E::kChunk, (int64_t)V - (int64_t)c * E::kChunk);
            const float tot = residual_chunk_sum<DT>(slot, n, ps, qs, ap, naq, p.s_hi);
            if (lane == 0) {
                if (rc_shared) {
                    if (CL > 1) st_shared_cluster(rc_leader + 4u * (uint32_t)c, tot);
                    else s_rc[c] = tot;
                } else {
                    rc[c] = tot;
                    atomicAdd(reinterpret_cast<unsigned long long*>(&p.rtotal[b]),
                              (unsigned long long)to_fixed(tot, p.fxr));
                }
            }
        }
        if (CL > 1) cluster_sync();  // release/acquire at cluster scope covers the global writes
        else __syncthreads();
        if (leader && warp == 0) {
            const uint32_t w = row_words(p.seed, p.step, b, K).y;
            const int y = draw_residual<DT>(p, slot, prow, qrow, p.chunk + ((int64_t)b * R + K) * C,
                                            rc_shared ? s_rc : rc, rc_shared, &p.rtotal[b], ps, qs, w);
            if (lane == 0) tok[K] = y;
        }
    } else if (state == 1) {
        // keep the MASK rows' statistics for the next call's residual
        if (leader && threadIdx.x < N - 1)
            p.carry[((int64_t)slot_write * p.B + b) * (N - 1) + threadIdx.x] = s_rs[N + threadIdx.x];
        // 3b. the bonus token (row N-1) and the N-1 proposals (rows N..2N-2), each finished by
        // the warp that planned it
        for (int r = first_row + warp; r < R; r += kWarps) {
            const int j = r - (N - 1);
            if (j < 0 || j % CL != crank) continue;
            float px = 1.f;  // an argmax proposal's q is a point mass
            const void* row = row_ptr(p.logits, dtb, (int64_t)b * R + r, V);
            const int t = p.amode && j > 0
                              ? finish_argmax<DT>(p, slot, row, s_plan[j].cstar, s_rs[r].mx)
                              : finish_draw<DT>(p, slot, row, p.chunk + ((int64_t)b * R + r) * C, s_rs[r], s_plan[j], &px);
            if (lane == 0) {
                if (j == 0) {
                    tok[has_pending ? N - 1 : 0] = t;
                } else {
                    tok[r] = t;
                    nq[j - 1] = px;
                }
            }
        }
    }
}

#include "isd_fused.cuh"

}  // namespace

// ----------------------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------------------
namespace {

struct Layout {
    size_t sched, chunk, qchunk, rchunk, rtotal, carry, carry_key, total;
    size_t zero_bytes;  // bytes at the front that must be zero when a step starts
    // isd_step_fused: the sections above, then its own
    size_t eng, estat, eqstat, drawcnt, rescnt, seqbad, ertotal, jobs, decw, rowstat, rsum, total_fused;
    int jobs_cap;
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
    L.sched = take(sizeof(unsigned long long));
    L.chunk = take(sizeof(float2) * (size_t)B * R * C);
    L.qchunk = take(sizeof(float2) * (size_t)B * C);
    L.rchunk = take(sizeof(float) * (size_t)B * C);
    L.rtotal = take(sizeof(uint64_t) * (size_t)B);
    L.carry = take(sizeof(RowStat) * 2 * (size_t)B * (N - 1));
    L.carry_key = take(sizeof(CarryKey) * 2);
    L.total = off;
    L.zero_bytes = L.chunk;  // the work counter; each step's decision kernel leaves it at zero
    // the fused step's counters, self-marking statistics, job records and flags (zero when the
    // workspace is initialised; a call leaves them ready for the next), then its row statistics
    L.eng = take(sizeof(EngineCounters));
    L.estat = take(sizeof(unsigned long long) * (size_t)B * R * C);
    L.eqstat = take(sizeof(unsigned long long) * (size_t)B * C);
    L.drawcnt = take(sizeof(unsigned) * (size_t)B);
    L.rescnt = take(sizeof(unsigned) * (size_t)B);
    L.seqbad = take(sizeof(unsigned) * (size_t)B);
    L.ertotal = take(sizeof(uint64_t) * (size_t)B);
    L.jobs_cap = 3 * B;  // a decision publishes two residual halves, behind a q row when needed
    L.jobs = take(sizeof(JobRec) * (size_t)L.jobs_cap);
    L.decw = take(sizeof(unsigned long long) * (size_t)B);
    L.rowstat = take(sizeof(RowStat) * (size_t)B * R);
    L.rsum = take(sizeof(float) * (size_t)B * 2 * C);
    L.total_fused = off;
    return true;
}

thread_local int g_last_launches = 0;
uint64_t g_wait_limit_ns = kWaitLimitNs;  // the kernels' bounded waits give up after this (a test may shorten it)

// measurement: CUDA timing events around each launch while a session is open
struct Profile {
    int cap = 0, next = 0;
    cudaEvent_t* ev = nullptr;  // 2 per launch
    int* kind = nullptr;
};
Profile g_prof;

using isd_detail::kKindDecide;
using isd_detail::kKindStats;
using isd_detail::ProfileScope;

struct DeviceInfo {
    int dev = -1, sms = 0;
};

// The launch caches below may be filled by several host threads at once.
std::mutex g_cache_mu;

int device_sms() {
    static DeviceInfo cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(g_cache_mu);
    if (cache[dev].dev != dev) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev].sms = sms;
        cache[dev].dev = dev;
    }
    return cache[dev].sms;
}

// CTAs of `kernel` that fit on the device at once (cached per device and kernel).
template <typename K>
int resident_ctas(K kernel, int threads, size_t smem) {
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
    const int sms = device_sms();
    std::lock_guard<std::mutex> lock(g_cache_mu);
    const void* fn = reinterpret_cast<const void*>(kernel);
    for (int i = 0; i < used; ++i)
        if (cache[i].dev == dev && cache[i].fn == fn && cache[i].smem == smem) return cache[i].value;
    int per = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kernel, threads, smem) != cudaSuccess) return 0;
    const int value = sms * (per > 0 ? per : 1);
    if (used < 64) cache[used++] = Entry{dev, fn, smem, value};
    return value;
}

int cluster_size(int C, bool greedy) {
    if (greedy) return 1;
    if (C >= 64) return 8;
    if (C >= 16) return 4;
    if (C >= 4) return 2;
    return 1;
}

// The fused step: one persistent kernel, at most one CTA per SM (all of them resident: its
// finishing warps wait, bounded, for rows that the other CTAs stream).
template <int DT, bool GREEDY>
int launch_fused(const FusedParams& p, cudaStream_t stream) {
    ProfileScope ps(isd_detail::kKindFused, stream);
    auto k = isd_fused_step_kernel<DT, GREEDY>;
    static bool attr_set[64] = {};  // per template instance and device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ISD_ERR_CUDA;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kEngineSmem) != cudaSuccess ||
            cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
            return ISD_ERR_CUDA;
        attr_set[dev] = true;
    }
    // every unit of the step, at most: all rows' chunks, plus the residuals' half chunks
    const int64_t units = (int64_t)p.B * (p.R + 2) * p.C;
    const int64_t want = (units + kEStreamers * kGrab - 1) / (kEStreamers * kGrab);
    const int sms = device_sms();
    if (sms <= 0) return ISD_ERR_CUDA;
    const int grid = (int)(want < sms ? want : sms);
    k<<<grid > 0 ? grid : 1, kEThreads, kEngineSmem, stream>>>(p);
    g_last_launches = 1;
    return cudaGetLastError() == cudaSuccess ? ISD_OK : ISD_ERR_CUDA;
}

template <int DT, bool GREEDY>
int launch_step(const Params& p, cudaStream_t stream, bool stats_ready) {
    const int64_t U = (int64_t)p.B * p.R * p.C;
    if (!stats_ready) {
        ProfileScope ps(kKindStats, stream);
        if (p.vec_ok) {
            auto k = isd_stats_kernel<DT, GREEDY>;
            static bool attr_set[64] = {};  // per template instance and device
            int dev = 0;
            if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ISD_ERR_CUDA;
            if (!attr_set[dev]) {
                if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStatsSmem) !=
                        cudaSuccess ||
                    cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
                    return ISD_ERR_CUDA;
                attr_set[dev] = true;
            }
            const int64_t want = (U + kSWarps - 1) / kSWarps;
            const int grid = (int)(want < device_sms() ? want : device_sms());
            k<<<grid > 0 ? grid : 1, kSThreads, kStatsSmem, stream>>>(p);
        } else {
            auto k = isd_stats_plain_kernel<DT, GREEDY>;
            const int64_t want = (U + kWarps - 1) / kWarps;
            const int res = resident_ctas(k, kThreads, 0);
            const int grid = (int)(want < res ? want : res);
            k<<<grid > 0 ? grid : 1, kThreads, 0, stream>>>(p);
        }
    }
    {
        ProfileScope ps(kKindDecide, stream);
        // clusters as large as the chunk count warrants, but all of them resident at once
        auto dk = isd_decide_kernel<DT, GREEDY>;
        static bool dattr_set[64] = {};  // per template instance and device
        int ddev = 0;
        if (cudaGetDevice(&ddev) != cudaSuccess || ddev < 0 || ddev >= 64) return ISD_ERR_CUDA;
        if (!dattr_set[ddev]) {
            if (cudaFuncSetAttribute(dk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDecideSmem) !=
                    cudaSuccess ||
                cudaFuncSetAttribute(dk, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
                return ISD_ERR_CUDA;
            dattr_set[ddev] = true;
        }
        int CL = cluster_size(p.C, GREEDY);
        const int res = resident_ctas(dk, kThreads, kDecideSmem);
        while (CL > 1 && (int64_t)p.B * CL > res) CL >>= 1;
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof cfg);
        cfg.gridDim = dim3((unsigned)(p.B * CL));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kDecideSmem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        int na = 0;
        if (CL > 1) {
            attr[na].id = cudaLaunchAttributeClusterDimension;
            attr[na].val.clusterDim.x = (unsigned)CL;
            attr[na].val.clusterDim.y = 1;
            attr[na].val.clusterDim.z = 1;
            ++na;
        }
        if (!ps.active()) {  // overlap the launch with the statistics kernel's tail
            attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[na].val.programmaticStreamSerializationAllowed = 1;
            ++na;
        }
        cfg.attrs = attr;
        cfg.numAttrs = na;
        if (cudaLaunchKernelEx(&cfg, dk, p, CL) != cudaSuccess) return ISD_ERR_CUDA;
    }
    g_last_launches = stats_ready ? 1 : 2;
    return cudaGetLastError() == cudaSuccess ? ISD_OK : ISD_ERR_CUDA;
}

}  // namespace

namespace isd_detail {
void scale_split(float temperature, int greedy, float* s_hi, float* s_lo) {
    // log2(e)/T split into a float head (rounded down) and a positive float tail
    const double s = greedy == ISD_GREEDY ? 1.0 : 1.4426950408889634 / (double)temperature;
    float hi = (float)s;
    if ((double)hi > s) hi = nextafterf(hi, 0.f);
    float lo = (float)(s - (double)hi);
    if (!(lo > 0.f)) lo = 1e-30f;
    *s_hi = hi;
    *s_lo = lo;
}
bool workspace_sections(int B, int N, int V, int dtype, size_t* chunk, size_t* rtotal, int* C, int* celems) {
    Layout L;
    if (!make_layout(B, N, V, dtype, L)) return false;
    *chunk = L.chunk;
    *rtotal = L.rtotal;
    *celems = chunk_elems(dtype);
    *C = (V + *celems - 1) / *celems;
    return true;
}
}  // namespace isd_detail

namespace isd_detail {
ProfileScope::ProfileScope(int kind, cudaStream_t s) : stream(s) {
    if (g_prof.cap > 0 && g_prof.next < g_prof.cap) {
        slot = g_prof.next++;
        g_prof.kind[slot] = kind;
        record(g_prof.ev[2 * slot]);
    }
}
ProfileScope::~ProfileScope() {
    if (slot >= 0) record(g_prof.ev[2 * slot + 1]);
}
void ProfileScope::record(cudaEvent_t e) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(stream, &cs);
    cudaEventRecordWithFlags(e, stream, cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal
                                                                            : cudaEventRecordDefault);
}
}  // namespace isd_detail

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
    return isd_detail::step_impl(logits, prev_logits, dtype, pending_tokens, pending_ld, pending_q, B, N, V, temperature,
                                 greedy, philox_seed, step, accepted_len, tokens_out, new_q, p_out, diag, workspace,
                                 workspace_bytes, stream, false);
}

size_t isd_fused_workspace_size(int B, int N, int V, int dtype) {
    Layout L;
    return make_layout(B, N, V, dtype, L) ? L.total_fused : 0;
}

int isd_step_fused(const void* logits, const void* prev_logits, int dtype, const int32_t* pending_tokens,
                   int pending_ld, const float* pending_q, int B, int N, int V, float temperature, int greedy,
                   uint64_t philox_seed, uint64_t step, int32_t* accepted_len, int32_t* tokens_out, float* new_q,
                   float* p_out, int32_t* diag, void* workspace, size_t workspace_bytes, void* stream) {
    return isd_detail::step_impl(logits, prev_logits, dtype, pending_tokens, pending_ld, pending_q, B, N, V, temperature,
                                 greedy, philox_seed, step, accepted_len, tokens_out, new_q, p_out, diag, workspace,
                                 workspace_bytes, stream, false, true);
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

int isd_debug_set_wait_limit_ns(uint64_t ns) {
    g_wait_limit_ns = ns ? ns : kWaitLimitNs;
    return ISD_OK;
}

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
    if (greedy < ISD_SAMPLE || greedy > ISD_ARGMAX_PROPOSE) return ISD_ERR_INVALID_ARG;
    if (greedy != ISD_GREEDY && (!pending_q || !(temperature > 0.f) || !isfinite(temperature)))
        return ISD_ERR_INVALID_ARG;
    void* ws = nullptr;
    const int rc = static_scratch_address(&ws);
    if (rc != ISD_OK) return rc;
    // The work counter at the front of the layout must be zero when a step starts.  A step
    // leaves it at zero, but the array is shared by every call and one that gave up early (a
    // timed-out wait) may leave it as it was: clear it.
    if (cudaMemsetAsync(ws, 0, L.zero_bytes, (cudaStream_t)stream) != cudaSuccess) return ISD_ERR_CUDA;
    return isd_step(logits, prev_logits, dtype, pending_tokens, pending_ld, pending_q, B, N, V, temperature,
                    greedy, philox_seed, step, accepted_len, tokens_out, new_q, p_out, diag, ws, L.total,
                    stream);
}

int isd_detail::step_impl(const void* logits, const void* prev_logits, int dtype, const int32_t* pending_tokens,
             int pending_ld, const float* pending_q, int B, int N, int V, float temperature, int greedy, uint64_t philox_seed,
             uint64_t step, int32_t* accepted_len, int32_t* tokens_out, float* new_q, float* p_out,
             int32_t* diag, void* workspace, size_t workspace_bytes, void* stream, bool stats_ready, bool fused) {
    g_last_launches = 0;
    Layout L;
    if (!make_layout(B, N, V, dtype, L)) return ISD_ERR_INVALID_ARG;
    if (!logits || !pending_tokens || !accepted_len || !tokens_out || !new_q) return ISD_ERR_INVALID_ARG;
    if (pending_ld < N - 1) return ISD_ERR_INVALID_ARG;
    if (greedy < ISD_SAMPLE || greedy > ISD_ARGMAX_PROPOSE) return ISD_ERR_INVALID_ARG;
    if (greedy != ISD_GREEDY && (!pending_q || !(temperature > 0.f) || !isfinite(temperature)))
        return ISD_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < (fused ? L.total_fused : L.total) || ((uintptr_t)workspace & 255))
        return ISD_ERR_WORKSPACE;
    if (fused && stats_ready) return ISD_ERR_INVALID_ARG;

    Params p;
    memset(&p, 0, sizeof p);
    p.logits = logits;
    p.prev = greedy == ISD_SAMPLE ? prev_logits : nullptr;
    p.amode = greedy == ISD_ARGMAX_PROPOSE ? 1 : 0;
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
    // Fixed-point fraction bits: a chunk sum of weights is at most 2^11 and a chunk of the
    // residual at most 1, so C of them stay below 2^62.
    int lg = 0;
    while ((1 << lg) < p.C) ++lg;
    p.fx = 51 - lg < 44 ? 51 - lg : 44;
    p.fxr = 62 - lg < 52 ? 62 - lg : 52;
    isd_detail::scale_split(temperature, greedy, &p.s_hi, &p.s_lo);
    const int esz = dtype == ISD_BF16 ? 2 : 4;
    const bool aligned = ((uintptr_t)logits % 16 == 0) && (!p.prev || (uintptr_t)p.prev % 16 == 0);
    p.vec_ok = (aligned && ((int64_t)V * esz) % 16 == 0) ? 1 : 0;
    p.seed = philox_seed;
    p.step = step;
    char* ws = static_cast<char*>(workspace);
    p.sched = reinterpret_cast<unsigned long long*>(ws + L.sched);
    p.chunk = reinterpret_cast<float2*>(ws + L.chunk);
    p.qchunk = reinterpret_cast<float2*>(ws + L.qchunk);
    p.rchunk = reinterpret_cast<float*>(ws + L.rchunk);
    p.rtotal = reinterpret_cast<uint64_t*>(ws + L.rtotal);
    p.carry = reinterpret_cast<RowStat*>(ws + L.carry);
    p.carry_key = reinterpret_cast<CarryKey*>(ws + L.carry_key);
    p.dtype = dtype;
    p.wait_ns = g_wait_limit_ns;
    cudaStream_t st = (cudaStream_t)stream;
    if (fused) {
        FusedParams f;
        memset(&f, 0, sizeof f);
        static_cast<Params&>(f) = p;
        f.rtotal = reinterpret_cast<uint64_t*>(ws + L.ertotal);
        f.eng = reinterpret_cast<EngineCounters*>(ws + L.eng);
        f.jobs = reinterpret_cast<JobRec*>(ws + L.jobs);
        f.jobs_cap = L.jobs_cap;
        f.estat = reinterpret_cast<unsigned long long*>(ws + L.estat);
        f.eqstat = reinterpret_cast<unsigned long long*>(ws + L.eqstat);
        f.drawcnt = reinterpret_cast<unsigned*>(ws + L.drawcnt);
        f.rescnt = reinterpret_cast<unsigned*>(ws + L.rescnt);
        f.seqbad = reinterpret_cast<unsigned*>(ws + L.seqbad);
        f.decw = reinterpret_cast<unsigned long long*>(ws + L.decw);
        f.rowstat = reinterpret_cast<RowStat*>(ws + L.rowstat);
        f.rsum = reinterpret_cast<float*>(ws + L.rsum);
        int lh = 0;
        while ((1 << lh) < 2 * p.C) ++lh;
        f.fxh = 62 - lh < 52 ? 62 - lh : 52;  // 2C half-chunk sums of at most 1 stay below 2^62
        if (dtype == ISD_BF16)
            return greedy == ISD_GREEDY ? launch_fused<ISD_BF16, true>(f, st) : launch_fused<ISD_BF16, false>(f, st);
        return greedy == ISD_GREEDY ? launch_fused<ISD_F32, true>(f, st) : launch_fused<ISD_F32, false>(f, st);
    }
    if (dtype == ISD_BF16)
        return greedy == ISD_GREEDY ? launch_step<ISD_BF16, true>(p, st, stats_ready)
                                    : launch_step<ISD_BF16, false>(p, st, stats_ready);
    return greedy == ISD_GREEDY ? launch_step<ISD_F32, true>(p, st, stats_ready)
                                : launch_step<ISD_F32, false>(p, st, stats_ready);
}

