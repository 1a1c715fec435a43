// isd_chunkstat.cuh -- the arithmetic of the per-chunk statistics that the decision pass
// combines into row statistics.  Shared by the statistics pass over stored logits and by the
// LM-head projection's epilogue, so that both produce the same numbers from the same bf16
// logits.
//
// With s = log2(e) / T split into a float head s_hi (rounded down) and a positive tail s_lo,
// a chunk whose maximum logit is m is summarised as
//   sampling: (m, tail_factor(m) * sum_x 2^(x*s_hi - e)),  e = ref_or_zero(exponent_ref(m))
//   greedy:   (m, bits of the lowest vocabulary index holding m)
// ("Introspective Diffusion Language Models", ai.arkapp.pw blog, section "I-DLM 如何解決這些
// 問題": p and q are softmax distributions over the vocabulary; these sums are their
// normalisers, taken in pieces).
#pragma once
#include <stdint.h>

namespace {

__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float ex2_approx(float t) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(t));
    return y;
}

// The head-only weight 2^(x*s_hi - e) that chunk statistics are summed with.
__device__ __forceinline__ float weight_head(float x, float e, float s_hi) { return ex2_approx(fmaf(x, s_hi, -e)); }
// The exponent reference of a chunk (or row) whose maximum logit is m: the integer
// ceil(m * s_hi), so that every weight is at most about 1.  NaN, +inf and -inf (an
// empty chunk) pass through; weights are then taken against 0 (see ref_or_zero).
__device__ __forceinline__ float exponent_ref(float m, float s_hi) { return isfinite(m) ? ceilf(m * s_hi) : m; }
__device__ __forceinline__ float ref_or_zero(float e) { return isfinite(e) ? e : 0.f; }

// The tail factor of a chunk: 2^(m * s_lo) for the chunk maximum m, to second order
// (m * s_lo is below ~1e-5 for logits/T below ~100, so the error is far below 1e-12).
// Chunk sums are taken with the head s_hi alone and multiplied by it; across a chunk
// 2^(x * s_lo) differs from it only for entries whose weight is negligible.
__device__ __forceinline__ float tail_factor(float m, float s_lo) {
    if (!isfinite(m)) return 1.f;
    const float t = m * s_lo * 0.69314718f;
    return fmaf(fmaf(t, 0.5f, 1.f), t, 1.f);
}

}  // namespace
