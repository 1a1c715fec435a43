// lm_head.cu -- the LM-head GEMM of isd_step_from_hidden on the sm_103a tensor cores.
//
// logits[m][v] = bf16( sum_k hidden[m][k] * lm_head[v][k] ), fp32 accumulation, for the
// M = B*(2N-1) query rows of one forward (the rows the ISD step reads; "Introspective
// Diffusion Language Models", ai.arkapp.pw blog, section "I-DLM 如何解決這些問題").
//
// Roles of the operands.  The vocabulary is the MMA's M dimension: a tile is 128 rows of
// the LM-head weight (operand A, K-major), and the query rows form operand B (K-major).  The
// fp32 accumulator of a work item (128 TMEM lanes x its query columns) stays in tensor memory
// for the whole K loop, so each weight tile is read from HBM once and the small hidden-state
// matrix is re-read from L2.
//
// Work items.  A full item is one vocabulary tile against all Mp <= 448 query rows (two MMAs of
// Mp/2 columns per K step).  The vocabulary tiles that would form a last, partial wave over the
// SMs are cut along the query rows into slices of a multiple of 32 rows, so that every SM ends at
// about the same time; a slice re-reads its weight tile (from L2 for all but the first slice).
//
// One CTA per SM, persistent over the items, ten warps:
//   warp 0     TMA producer: per 64-wide K block, the weight tile (128 x 64) and the item's
//              hidden rows (32-row boxes), 128-byte swizzled, into a ring of stages (mbarrier
//              full/empty);
//   warp 1     allocates the tensor memory, and one lane issues tcgen05.mma (kind::f16, bf16
//              inputs, fp32 accumulator) four K-steps of 16 per stage, committing each stage back
//              to the producer and the finished item to the epilogue;
//   warps 2-9  epilogue: warp w reads TMEM lane quarter w % 4 (32 vocabulary rows) and one half
//              of the item's columns into registers as packed bf16, frees the accumulator for the
//              next item, then, 16 query columns at a time, stores 32 consecutive vocabulary
//              entries per query row and (isd_step_from_hidden) computes the tile's softmax
//              statistics of every query row, which isd_lm_head_merge_kernel turns into the
//              decision pass's chunk statistics.
// Every mbarrier wait gives up after about one second: the kernel then records the failure,
// waits (bounded) for its copies in flight and its MMAs, frees its tensor memory and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "isd.h"
#include "isd_chunkstat.cuh"
#include "isd_internal.h"

namespace {

constexpr int kTileV = 128;   // vocabulary rows per tile (MMA M)
constexpr int kBK = 64;       // K elements per stage: one 128-byte swizzle row of bf16
constexpr int kUmmaK = 16;    // K per tcgen05.mma of kind::f16
constexpr int kMaxTok = 448;  // query rows per launch: two MMAs of at most 224 columns
constexpr int kPk = kMaxTok / 4;  // packed bf16 pairs an epilogue lane holds (its column half)
constexpr int kBoxRows = 32;  // hidden rows per TMA box
constexpr int kEpiWarps = 8;
constexpr int kWarps = 2 + kEpiWarps;
constexpr int kThreads = kWarps * 32;
constexpr uint64_t kLimitNs = 1000000000ull;

struct GemmParams {
    __nv_bfloat16* out;  // [M][V]; null: the logits are not stored (greedy from-hidden step)
    int M, Mp, V, K;     // Mp: M rounded up to a multiple of 32
    int n_tiles, n_kb, stages;
    int n_full;          // items 0..n_full-1: tile = item, all Mp columns
    int slice_w, slices; // then tile n_full + (item - n_full) / slices, columns of width slice_w
    int n_items;
    uint32_t tmem_cols;  // power of two >= Mp, at least 32
    uint32_t stage_bytes, w_bytes;
    int* status;         // first error, 0 if none (device)
    // statistics epilogue (isd_step_from_hidden): per vocabulary tile and query row, the
    // partial chunk statistic of those 128 vocabulary entries
    int mode;            // kModeLogits, kModeSample or kModeGreedy
    float s_hi;          // head of log2(e)/T
    float2* partial;     // [n_tiles][Mtot]
    int m_base, Mtot;    // first global query row of this launch; all query rows
};
constexpr int kModeLogits = 0, kModeSample = 1, kModeGreedy = 2;

struct Item {
    int tile, c0, cw;  // vocabulary tile, first query column, number of columns (multiple of 32)
};
__device__ __forceinline__ Item item_of(const GemmParams& g, int i) {
    Item it;
    if (i < g.n_full) {
        it.tile = i;
        it.c0 = 0;
        it.cw = g.Mp;
    } else {
        const int j = i - g.n_full;
        it.tile = g.n_full + j / g.slices;
        it.c0 = (j % g.slices) * g.slice_w;
        it.cw = min(g.slice_w, g.Mp - it.c0);
    }
    return it;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
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
// Wait for the phase of parity `parity` (bounded, about 1 s).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try(bar, parity)) return true;
        if ((i & 63) == 0 && now_ns() - t0 > kLimitNs) return false;
    }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor of a K-major operand stored as 128-byte swizzled rows
// (TMA SWIZZLE_128B): start address, stride between groups of 8 rows = 1024 bytes,
// descriptor version 1, swizzle mode 128B.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);      // start address >> 4, bits 0-13
    d |= (uint64_t)1 << 16;                         // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024u >> 4) << 32;              // stride byte offset, bits 32-45
    d |= (uint64_t)1 << 46;                         // version
    d |= (uint64_t)2 << 61;                         // swizzle: 128B
    return d;
}
// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "setp.ne.b32 P, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, P;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accum)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 16 consecutive fp32 columns of this warp's 32 TMEM lanes (one per lane).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, "
        "[%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ uint32_t pack_bf16(uint32_t lo, uint32_t hi) {
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<const uint32_t*>(&h2);
}

__device__ __forceinline__ void set_error(const GemmParams& g, int code) {
    if (g.status) atomicCAS(g.status, 0, code);
}

// AND of `v` over the 128 threads of named barrier `id` (a barrier for those threads).
__device__ __forceinline__ bool bar_and(int id, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred P, Q;\n\t"
        "setp.ne.u32 P, %2, 0;\n\t"
        "bar.red.and.pred Q, %1, 128, P;\n\t"
        "selp.u32 %0, 1, 0, Q;\n\t}"
        : "=r"(r)
        : "r"(id), "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// x * 2^d for an integer d <= 0 (exact; 0 once 2^d is below the normal range, where the
// weights that the statistics pass sums are flushed to zero as well).
__device__ __forceinline__ float scale_pow2(float x, int d) {
    return d < -126 ? 0.f : x * __int_as_float((127 + d) << 23);
}

// Merge of the partial statistics a, b = (m, y) of two disjoint vocabulary ranges, a before b.
// Sampling: each y is a sum against the exponent reference of its own m; the result's is
// against the reference of the merged maximum.  Greedy: y holds index bits; the first maximum
// wins.  A NaN maximum on either side makes the result's maximum NaN.
__device__ __forceinline__ float2 merge_sample(float2 a, float2 b, float s_hi) {
    if (isnan(a.x) || isnan(b.x)) return make_float2(__int_as_float(0x7FC00000), 0.f);
    const float m = fmaxf(a.x, b.x);
    const float e = ref_or_zero(exponent_ref(m, s_hi));
    float y = 0.f;
    if (a.y > 0.f) y += scale_pow2(a.y, (int)(ref_or_zero(exponent_ref(a.x, s_hi)) - e));
    if (b.y > 0.f) y += scale_pow2(b.y, (int)(ref_or_zero(exponent_ref(b.x, s_hi)) - e));
    return make_float2(m, y);
}
__device__ __forceinline__ float2 merge_greedy(float2 a, float2 b) {
    if (isnan(a.x) || isnan(b.x)) return make_float2(__int_as_float(0x7FC00000), a.y);
    return b.x > a.x ? b : a;
}

__device__ __forceinline__ float fmax_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

// Reduce-scatter step of column maxima on packed bf16 pairs u[0..2n): lanes with bit k set
// keep pairs n..2n-1, the others 0..n-1, each taking the maximum with its partner's copy.
template <int n>
__device__ __forceinline__ void max_scatter_half(uint32_t (&u)[8], int lane, int k) {
    const bool upper = (lane >> k) & 1;
#pragma unroll
    for (int i = 0; i < n; ++i) {
        const uint32_t send = upper ? u[i] : u[i + n];
        const uint32_t keep = upper ? u[i + n] : u[i];
        u[i] = bmax2_nan(keep, __shfl_xor_sync(0xffffffffu, send, 1 << k));
    }
}
// The inverse step: a lane holding pairs u[0..n) (its half, by lane bit k) receives the
// partner's half, so that it holds u[0..2n) in column order.
template <int n>
__device__ __forceinline__ void max_gather(uint32_t (&u)[8], int lane, int k) {
    const bool upper = (lane >> k) & 1;
#pragma unroll
    for (int i = 0; i < n; ++i) {
        const uint32_t other = __shfl_xor_sync(0xffffffffu, u[i], 1 << k);
        const uint32_t mine = u[i];
        u[i] = upper ? other : mine;
        u[i + n] = upper ? mine : other;
    }
}

// One reduce-scatter step over 2n columns held in t[0..2n): lanes with bit k set keep columns
// n..2n-1, the others 0..n-1; each adds its partner's (lane ^ 2^k) copy of the kept half.
template <int n>
__device__ __forceinline__ void scatter_half(float (&t)[16], int lane, int k) {
    const bool upper = (lane >> k) & 1;
#pragma unroll
    for (int i = 0; i < n; ++i) {
        const float send = upper ? t[i] : t[i + n];
        const float keep = upper ? t[i + n] : t[i];
        t[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1 << k);
    }
}

// Statistics of this warp's 32 vocabulary entries (one per lane) for 16 query columns, the
// launch's columns col..col+15, from the bf16 logits held in w[0..8) (pairs of columns 2e,
// 2e+1).  Entries past V count as -inf.  Sampling: (max m, sum of 2^(x*s_hi - e)) with
// e = ref_or_zero(exponent_ref(m)); greedy: (max, lowest vocabulary index holding it).  The
// column maxima are all-reduced on packed bf16 pairs; the sums are reduce-scattered (16
// shuffles for 16 columns), which leaves the sum of column c in lanes 2c and 2c+1.  The four
// warps of a column half then merge their 32-entry statistics into the tile's, which quarter 0
// writes to partial[tile][row].
__device__ __forceinline__ void group_stats(const GemmParams& g, const Item& it, int q, int h, int col, int ncols,
                                            int parity, const uint32_t* pk, float2* comb) {
    const int lane = threadIdx.x & 31;
    const int vbase = it.tile * kTileV + q * 32;
    const bool valid = vbase + lane < g.V;
    uint32_t w[8], mx[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        w[e] = valid ? pk[e] : 0xFF80FF80u;  // a pair of bf16 -inf
        mx[e] = w[e];
    }
    // column maxima: reduce-scatter (9 shuffles) leaves the maximum of column lane >> 1 in my_m,
    // an all-gather (8 shuffles) gives every lane all 16 again, packed in mx
    max_scatter_half<4>(mx, lane, 4);
    max_scatter_half<2>(mx, lane, 3);
    max_scatter_half<1>(mx, lane, 2);
    float my_m;
    {
        const bool up = (lane >> 1) & 1;  // keep the pair's high column (2P+1), or the low one
        const float keep = __uint_as_float(up ? (mx[0] & 0xFFFF0000u) : (mx[0] << 16));
        const float send = __uint_as_float(up ? (mx[0] << 16) : (mx[0] & 0xFFFF0000u));
        my_m = fmax_nan(keep, __shfl_xor_sync(0xffffffffu, send, 2));
        my_m = fmax_nan(my_m, __shfl_xor_sync(0xffffffffu, my_m, 1));
    }
    {
        const uint32_t mine = __float_as_uint(my_m) >> 16;  // bf16 bits of column lane >> 1
        const uint32_t other = __shfl_xor_sync(0xffffffffu, mine, 2);
        mx[0] = ((lane >> 1) & 1) ? (other | (mine << 16)) : (mine | (other << 16));
    }
    max_gather<1>(mx, lane, 2);
    max_gather<2>(mx, lane, 3);
    max_gather<4>(mx, lane, 4);
    const int mycol = lane >> 1;  // the column whose result this lane writes
    float my_y = 0.f;
    if (g.mode == kModeGreedy) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float x0 = __uint_as_float(w[e] << 16), x1 = __uint_as_float(w[e] & 0xFFFF0000u);
            const float m0 = __uint_as_float(mx[e] << 16), m1 = __uint_as_float(mx[e] & 0xFFFF0000u);
            const uint32_t b0 = __ballot_sync(0xffffffffu, x0 == m0), b1 = __ballot_sync(0xffffffffu, x1 == m1);
            const uint32_t i0 = b0 ? (uint32_t)(vbase + __ffs(b0) - 1) : 0xFFFFFFFFu;
            const uint32_t i1 = b1 ? (uint32_t)(vbase + __ffs(b1) - 1) : 0xFFFFFFFFu;
            if (mycol == 2 * e) my_y = __uint_as_float(i0);
            if (mycol == 2 * e + 1) my_y = __uint_as_float(i1);
        }
    } else {
        float t[16];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float x0 = __uint_as_float(w[e] << 16), x1 = __uint_as_float(w[e] & 0xFFFF0000u);
            const float m0 = __uint_as_float(mx[e] << 16), m1 = __uint_as_float(mx[e] & 0xFFFF0000u);
            t[2 * e] = weight_head(x0, ref_or_zero(exponent_ref(m0, g.s_hi)), g.s_hi);
            t[2 * e + 1] = weight_head(x1, ref_or_zero(exponent_ref(m1, g.s_hi)), g.s_hi);
        }
        scatter_half<8>(t, lane, 4);
        scatter_half<4>(t, lane, 3);
        scatter_half<2>(t, lane, 2);
        scatter_half<1>(t, lane, 1);
        my_y = t[0] + __shfl_xor_sync(0xffffffffu, t[0], 1);
    }
    // the four lane quarters of this column half (warps q = 0..3) combine through shared
    // memory; slots alternate with the group's parity, so one barrier per group suffices
    float2* slot = comb + ((parity * 2 + h) * 4) * 16;
    if (q != 0 && (lane & 1) == 0) slot[q * 16 + mycol] = make_float2(my_m, my_y);
    asm volatile("bar.sync %0, 128;" ::"r"(1 + h) : "memory");
    if (q == 0 && (lane & 1) == 0 && mycol < ncols) {
        float2 r = make_float2(my_m, my_y);
#pragma unroll
        for (int k = 1; k < 4; ++k)
            r = g.mode == kModeGreedy ? merge_greedy(r, slot[k * 16 + mycol]) : merge_sample(r, slot[k * 16 + mycol], g.s_hi);
        g.partial[(size_t)it.tile * g.Mtot + g.m_base + col + mycol] = r;
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    isd_lm_head_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_h,
                       GemmParams g) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // stages start on a 1024-byte boundary (the 128-byte swizzle repeats every 8 rows)
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ __align__(8) uint64_t s_full[4], s_empty[4], s_tmem_full, s_tmem_empty, s_mma_done;
    __shared__ uint32_t s_tmem_base;
    __shared__ float2 s_comb[2 * 2 * 4 * 16];  // [group parity][column half][quarter][column]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < g.stages; ++s) {
            mbar_init(smem_u32(&s_full[s]), 1);
            mbar_init(smem_u32(&s_empty[s]), 1);
        }
        mbar_init(smem_u32(&s_tmem_full), 1);
        mbar_init(smem_u32(&s_tmem_empty), kEpiWarps * 32);
        mbar_init(smem_u32(&s_mma_done), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {  // tensor memory for the accumulator (Mp fp32 columns x 128 lanes)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem_base)),
                     "r"(g.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem_base;

    if (warp == 0) {
        if (lane == 0) {  // producer
            int s = 0;
            uint32_t eph = 0;   // bit s: parity of the next wait on empty[s]
            uint32_t used = 0;  // bit s: stage s has been filled at least once
            bool ok = true;
            for (int i = blockIdx.x; i < g.n_items && ok; i += gridDim.x) {
                const Item it = item_of(g, i);
                for (int kb = 0; kb < g.n_kb; ++kb) {
                    // a stage is free once the MMAs that read it are done (its first use is free)
                    if ((used >> s) & 1u) {
                        if (!mbar_wait(smem_u32(&s_empty[s]), (eph >> s) & 1u)) {
                            ok = false;
                            break;
                        }
                        eph ^= 1u << s;
                    }
                    used |= 1u << s;
                    const uint32_t st = smem_u32(smem + (size_t)s * g.stage_bytes);
                    const uint32_t full = smem_u32(&s_full[s]);
                    mbar_expect_tx(full, g.w_bytes + (uint32_t)it.cw * (kBK * 2));
                    tma_load_2d(st, &map_w, kb * kBK, it.tile * kTileV, full);
                    for (int r = 0; r < it.cw; r += kBoxRows)
                        tma_load_2d(st + g.w_bytes + (uint32_t)r * (kBK * 2), &map_h, kb * kBK, it.c0 + r, full);
                    s = s + 1 == g.stages ? 0 : s + 1;
                }
            }
            if (!ok) set_error(g, ISD_ERR_TIMEOUT);
            // no copy may still be writing shared memory when the CTA leaves: the last fill of
            // every stage has completed (bounded; completed phases return at once).  Stage t was
            // filled once more than its empty barrier was waited for, so its last fill completed
            // phase parity (eph >> t) & 1 of full[t].
            for (int t = 0; t < g.stages; ++t)
                if (((used >> t) & 1u) && !mbar_wait(smem_u32(&s_full[t]), (eph >> t) & 1u))
                    set_error(g, ISD_ERR_TIMEOUT);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            int s = 0;
            uint32_t fph = 0;  // bit s: parity of the next wait on full[s]
            uint32_t eph = 0;  // parity of the next wait on tmem_empty
            bool ok = true;
            for (int i = blockIdx.x; i < g.n_items && ok; i += gridDim.x) {
                const Item it = item_of(g, i);
                if (i != (int)blockIdx.x) {  // the epilogue has drained the previous accumulator
                    if (!mbar_wait(smem_u32(&s_tmem_empty), eph)) {
                        ok = false;
                        break;
                    }
                    eph ^= 1u;
                }
                tc_fence_after();
                // one MMA of cw columns, or two of cw/2 (at most 256 columns each)
                const int nw = it.cw > 256 ? it.cw / 2 : it.cw;
                const uint32_t idesc = idesc_bf16(kTileV, nw);
                const uint32_t boff = (uint32_t)nw * (kBK * 2);  // bytes of the first MMA's rows
                for (int kb = 0; kb < g.n_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&s_full[s]), (fph >> s) & 1u)) {
                        ok = false;
                        break;
                    }
                    fph ^= 1u << s;
                    tc_fence_after();
                    const uint32_t st = smem_u32(smem + (size_t)s * g.stage_bytes);
                    const uint64_t a = sw128_desc(st);
                    const uint64_t b0 = sw128_desc(st + g.w_bytes);
                    const uint64_t b1 = sw128_desc(st + g.w_bytes + boff);
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        // K step k: 16 bf16 = 32 bytes further along the swizzled rows
                        const uint64_t adv = (uint64_t)((k * kUmmaK * 2) >> 4);
                        const uint32_t acc = (kb | k) ? 1u : 0u;
                        umma(tmem, a + adv, b0 + adv, idesc, acc);
                        if (nw != it.cw) umma(tmem + (uint32_t)nw, a + adv, b1 + adv, idesc, acc);
                    }
                    umma_commit(smem_u32(&s_empty[s]));  // the stage is free when these are done
                    s = s + 1 == g.stages ? 0 : s + 1;
                }
                if (ok) umma_commit(smem_u32(&s_tmem_full));  // the item's accumulator is complete
            }
            if (!ok) set_error(g, ISD_ERR_TIMEOUT);
            // every MMA issued by this thread has finished before the tensor memory is freed
            umma_commit(smem_u32(&s_mma_done));
            if (!mbar_wait(smem_u32(&s_mma_done), 0)) set_error(g, ISD_ERR_TIMEOUT);
        }
    } else {  // epilogue: TMEM lane quarter warp % 4, column half (warp - 2) / 4
        const int q = warp & 3, h = (warp - 2) >> 2;
        uint32_t fph = 0;
        for (int i = blockIdx.x; i < g.n_items; i += gridDim.x) {
            const Item it = item_of(g, i);
            const bool ok = mbar_wait(smem_u32(&s_tmem_full), fph);
            // the same decision in the four warps of this column half, which meet at named
            // barriers below: none may leave while another waits there
            if (!bar_and(1 + h, __all_sync(0xffffffffu, ok))) {
                if (lane == 0) set_error(g, ISD_ERR_TIMEOUT);
                break;
            }
            fph ^= 1u;
            tc_fence_after();
            const int hw = it.cw >> 1;  // this warp's columns: [h*hw, (h+1)*hw), hw <= 224
            const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * hw);
            uint32_t pk[kPk];  // bf16 pairs of columns (2j, 2j+1)
#pragma unroll
            for (int j = 0; j < kPk / 8; ++j) {
                if (j * 16 < hw) {
                    uint32_t r[16];
                    tmem_ld16(taddr + (uint32_t)(j * 16), r);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 8; ++e) pk[j * 8 + e] = pack_bf16(r[2 * e], r[2 * e + 1]);
                }
            }
            // the accumulator is in registers: the next item's MMAs may overwrite it
            tc_fence_before();
            mbar_arrive(smem_u32(&s_tmem_empty));
            // statistics and stores, 16 columns at a time in a rolled loop (the next group is
            // shifted into pk[0..8) so that every register index stays fixed)
            const int v = it.tile * kTileV + q * 32 + lane;
            const int col0 = it.c0 + h * hw;  // first query column (within the launch) of this warp
            __nv_bfloat16* o = g.out + (int64_t)col0 * g.V + v;
#pragma unroll 1
            for (int j = 0; j < (hw >> 4); ++j) {
                const int c = col0 + j * 16;
                if (g.mode != kModeLogits) group_stats(g, it, q, h, c, min(16, g.M - c), j & 1, pk, s_comb);
                if (g.out && v < g.V) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int m = j * 16 + 2 * e;
                        if (col0 + m < g.M) o[(int64_t)m * g.V] = __ushort_as_bfloat16((unsigned short)(pk[e] & 0xFFFFu));
                        if (col0 + m + 1 < g.M)
                            o[(int64_t)(m + 1) * g.V] = __ushort_as_bfloat16((unsigned short)(pk[e] >> 16));
                    }
                }
#pragma unroll
                for (int e = 0; e < kPk - 8; ++e) pk[e] = pk[e + 8];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(g.tmem_cols) : "memory");
    }
}

// Chunk statistics [Mtot][C] in the decision pass's format from the epilogue's per-tile
// statistics [n_tiles][Mtot]: chunk c covers tiles [c*TPC, (c+1)*TPC), merged in vocabulary
// order; sampling sums are then multiplied by tail_factor of the chunk maximum, as the
// statistics pass does.  Block (0,0) also clears the residual totals.
template <int TPC>
__global__ void __launch_bounds__(128) isd_lm_head_merge_kernel(const float2* __restrict__ partial, int Mtot,
                                                                 int n_tiles, int C, int mode, float s_hi, float s_lo,
                                                                 float2* __restrict__ chunk, uint64_t* rtotal, int B) {
    // launched as a programmatic dependent of the projection: its statistics (and logits)
    // are complete and visible after this.  Only then may the decision pass be scheduled: it
    // reads the logits at the pending tokens before it waits for this grid.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (blockIdx.x == 0 && blockIdx.y == 0)
        for (int i = threadIdx.x; i < B; i += blockDim.x) rtotal[i] = 0ull;
    const int m = blockIdx.x * blockDim.x + threadIdx.x, c = blockIdx.y;
    if (m >= Mtot) return;
    const int t0 = c * TPC;
    float2 v[TPC];  // every tile of the chunk in flight at once
#pragma unroll
    for (int i = 0; i < TPC; ++i)
        v[i] = t0 + i < n_tiles ? __ldg(&partial[(size_t)(t0 + i) * Mtot + m]) : make_float2(-INFINITY, 0.f);
    float2 r = v[0];
#pragma unroll
    for (int i = 1; i < TPC; ++i) r = mode == kModeGreedy ? merge_greedy(r, v[i]) : merge_sample(r, v[i], s_hi);
    if (mode != kModeGreedy) r.y *= tail_factor(r.x, s_lo);
    chunk[(size_t)m * C + c] = r;
}

// ---- host ---------------------------------------------------------------------------------
// 2-D bf16 tensor map of a row-major [rows][cols] matrix, boxes of box_rows x 64, 128-byte
// swizzle, zero fill outside the matrix.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled, looked up through the runtime so that the library loads (and its
// symbols can be listed) on a machine without the driver.
EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
    const cuuint32_t elem[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                                  box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

thread_local int g_lm_head_launches = 0;  // kernels launched by the last call on this thread

// Per-device facts the launches need, looked up once (the values are the same for every
// caller, so concurrent first calls at worst look them up twice).
struct DeviceFacts {
    int sms = 0, optin = 0;
    size_t static_smem = 0;
    size_t smem_attr = 0;  // largest dynamic shared memory set on the kernel so far
};
DeviceFacts g_facts[64];

const DeviceFacts* device_facts(int* dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    DeviceFacts& f = g_facts[dev];
    if (f.sms == 0) {
        int sms = 0, optin = 0;
        cudaFuncAttributes fa;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaFuncGetAttributes(&fa, isd_lm_head_kernel) != cudaSuccess)
            return nullptr;
        f.optin = optin;
        f.static_smem = fa.sharedSizeBytes;
        f.sms = sms;
    }
    *dev_out = dev;
    return &f;
}

// One launch over query rows [0, M) of `hidden` (M <= 448).
int launch_block(const void* hidden, const void* weight, int M, int K, int V, __nv_bfloat16* out, int32_t* status,
                 cudaStream_t stream, int mode = kModeLogits, float s_hi = 0.f, float2* partial = nullptr,
                 int m_base = 0, int Mtot = 0) {
    GemmParams g;
    memset(&g, 0, sizeof g);
    g.out = out;
    g.mode = mode;
    g.s_hi = s_hi;
    g.partial = partial;
    g.m_base = m_base;
    g.Mtot = Mtot;
    g.M = M;
    g.Mp = (M + 31) / 32 * 32;
    g.V = V;
    g.K = K;
    g.n_tiles = (V + kTileV - 1) / kTileV;
    g.n_kb = (K + kBK - 1) / kBK;
    g.w_bytes = kTileV * kBK * 2;
    g.stage_bytes = g.w_bytes + (uint32_t)g.Mp * kBK * 2;
    g.status = status;
    g.tmem_cols = 32;
    while ((int)g.tmem_cols < g.Mp) g.tmem_cols <<= 1;
    int dev = 0;
    const DeviceFacts* facts = device_facts(&dev);
    if (!facts) return ISD_ERR_CUDA;
    const int sms = facts->sms;
    // whole waves of full tiles; the tiles of a last partial wave are cut into query-row slices
    // (multiples of 32 rows) so that the partial wave spreads over the SMs
    g.n_full = g.n_tiles / sms * sms;
    const int rest = g.n_tiles - g.n_full;
    int per_tile = 1;
    if (rest > 0) {
        per_tile = sms / rest;
        if (per_tile > g.Mp / 32) per_tile = g.Mp / 32;
        if (per_tile < 1) per_tile = 1;
    }
    const int units = g.Mp / 32;
    g.slice_w = 32 * ((units + per_tile - 1) / per_tile);
    g.slices = (g.Mp + g.slice_w - 1) / g.slice_w;
    g.n_items = g.n_full + rest * g.slices;
    const size_t budget = (size_t)facts->optin - facts->static_smem - 1024;  // less static + alignment slack
    g.stages = (int)(budget / g.stage_bytes);
    if (g.stages > 4) g.stages = 4;
    if (g.stages < 2) return ISD_ERR_INVALID_ARG;
    const size_t smem = (size_t)g.stages * g.stage_bytes + 1024;
    if (smem > g_facts[dev].smem_attr) {
        if (cudaFuncSetAttribute(isd_lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return ISD_ERR_CUDA;
        g_facts[dev].smem_attr = smem;
    }
    CUtensorMap map_w, map_h;
    if (!make_map(&map_w, weight, (uint64_t)V, (uint64_t)K, kTileV) ||
        !make_map(&map_h, hidden, (uint64_t)M, (uint64_t)K, kBoxRows))
        return ISD_ERR_CUDA;
    const int grid = g.n_items < sms ? g.n_items : sms;
    {
        isd_detail::ProfileScope ps(isd_detail::kKindLmHead, stream);
        isd_lm_head_kernel<<<grid, kThreads, smem, stream>>>(map_w, map_h, g);
    }
    if (cudaGetLastError() != cudaSuccess) return ISD_ERR_CUDA;
    ++g_lm_head_launches;
    return ISD_OK;
}

}  // namespace

extern "C" int isd_lm_head(const void* hidden, const void* lm_head, int M, int K, int V, void* logits,
                           int32_t* status, void* stream) {
    g_lm_head_launches = 0;
    if (!hidden || !lm_head || !logits) return ISD_ERR_INVALID_ARG;
    if (M < 1 || K < 8 || (K % 8) != 0 || V < 1) return ISD_ERR_INVALID_ARG;
    if (((uintptr_t)hidden | (uintptr_t)lm_head) & 15) return ISD_ERR_INVALID_ARG;
    const char* h = static_cast<const char*>(hidden);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(logits);
    // query rows in blocks of at most 448 (the accumulator's tensor-memory columns, and the
    // registers of the epilogue); each block streams the weight once
    for (int m0 = 0; m0 < M; m0 += kMaxTok) {
        const int mb = M - m0 < kMaxTok ? M - m0 : kMaxTok;
        const int rc = launch_block(h + (size_t)m0 * K * 2, lm_head, mb, K, V, out + (size_t)m0 * V, status,
                                    (cudaStream_t)stream);
        if (rc != ISD_OK) return rc;
    }
    return ISD_OK;
}

extern "C" int isd_lm_head_last_launch_count(void) { return g_lm_head_launches; }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

extern "C" size_t isd_from_hidden_workspace_size(int B, int N, int V) {
    const size_t step = isd_workspace_size(B, N, V, ISD_BF16);
    if (step == 0) return 0;
    const size_t M = (size_t)B * (2 * N - 1);
    const size_t n_tiles = ((size_t)V + kTileV - 1) / kTileV;
    return align256(step) + n_tiles * M * sizeof(float2);
}

extern "C" int isd_step_from_hidden(const void* hidden, const void* lm_head, int K, void* logits,
                                    const void* prev_logits, const int32_t* pending_tokens, int pending_ld,
                                    const float* pending_q, int B, int N, int V, float temperature, int greedy,
                                    uint64_t philox_seed, uint64_t step, int32_t* accepted_len, int32_t* tokens_out,
                                    float* new_q, float* p_out, int32_t* diag, void* workspace,
                                    size_t workspace_bytes, void* stream) {
    g_lm_head_launches = 0;
    // the step's own argument checks first, so that a bad call launches nothing
    const size_t need = isd_from_hidden_workspace_size(B, N, V);
    if (need == 0) return ISD_ERR_INVALID_ARG;
    if (!hidden || !lm_head || !logits || !pending_tokens || !accepted_len || !tokens_out || !new_q)
        return ISD_ERR_INVALID_ARG;
    if (K < 8 || (K % 8) != 0 || (((uintptr_t)hidden | (uintptr_t)lm_head) & 15)) return ISD_ERR_INVALID_ARG;
    if (pending_ld < N - 1) return ISD_ERR_INVALID_ARG;
    if (greedy < ISD_SAMPLE || greedy > ISD_ARGMAX_PROPOSE) return ISD_ERR_INVALID_ARG;
    if (greedy != ISD_GREEDY && (!pending_q || !(temperature > 0.f) || !isfinite(temperature)))
        return ISD_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255)) return ISD_ERR_WORKSPACE;
    size_t off_chunk = 0, off_rtotal = 0;
    int C = 0, chunk_elems = 0;
    if (!isd_detail::workspace_sections(B, N, V, ISD_BF16, &off_chunk, &off_rtotal, &C, &chunk_elems) ||
        chunk_elems % kTileV != 0)
        return ISD_ERR_INVALID_ARG;
    float s_hi = 0.f, s_lo = 0.f;
    isd_detail::scale_split(temperature, greedy, &s_hi, &s_lo);
    const int M = B * (2 * N - 1);
    const int n_tiles = (V + kTileV - 1) / kTileV;
    char* ws = static_cast<char*>(workspace);
    float2* partial = reinterpret_cast<float2*>(ws + align256(isd_workspace_size(B, N, V, ISD_BF16)));
    const int mode = greedy == ISD_GREEDY ? kModeGreedy : kModeSample;
    // the greedy decisions need only the argmax statistics: the logits are not stored
    cudaStream_t st = (cudaStream_t)stream;
    const char* h = static_cast<const char*>(hidden);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(logits);
    int32_t* status = diag ? diag + ISD_DIAG_STATUS : nullptr;
    // 1. the projection, whose epilogue leaves per-tile statistics of every row
    for (int m0 = 0; m0 < M; m0 += kMaxTok) {
        const int mb = M - m0 < kMaxTok ? M - m0 : kMaxTok;
        const int rc = launch_block(h + (size_t)m0 * K * 2, lm_head, mb, K, V,
                                    mode == kModeGreedy ? nullptr : out + (size_t)m0 * V, status, st, mode, s_hi,
                                    partial, m0, M);
        if (rc != ISD_OK) return rc;
    }
    // 2. the chunk statistics of the decision pass, from those
    {
        isd_detail::ProfileScope ps(isd_detail::kKindMerge, st);
        const dim3 grid((unsigned)((M + 127) / 128), (unsigned)C);
        if (chunk_elems / kTileV != 16) return ISD_ERR_INVALID_ARG;  // bf16 chunks of 2048 entries
        cudaLaunchConfig_t cfg;
        memset(&cfg, 0, sizeof cfg);
        cfg.gridDim = grid;
        cfg.blockDim = dim3(128);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = ps.active() ? 0 : 1;  // timed on its own while profiling
        if (cudaLaunchKernelEx(&cfg, isd_lm_head_merge_kernel<16>, (const float2*)partial, M, n_tiles, C, mode, s_hi,
                               s_lo, reinterpret_cast<float2*>(ws + off_chunk),
                               reinterpret_cast<uint64_t*>(ws + off_rtotal), B) != cudaSuccess)
            return ISD_ERR_CUDA;
        ++g_lm_head_launches;
    }
    // 3. the decisions (the statistics pass over the logits is not needed)
    return isd_detail::step_impl(logits, prev_logits, ISD_BF16, pending_tokens, pending_ld, pending_q, B, N, V,
                                 temperature, greedy, philox_seed, step, accepted_len, tokens_out, new_q, p_out, diag,
                                 workspace, workspace_bytes, stream, true);
}
