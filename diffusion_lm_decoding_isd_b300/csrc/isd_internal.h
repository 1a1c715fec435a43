// isd_internal.h -- declarations shared by the library's translation units (not part of the
// C ABI).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace isd_detail {

// Kinds of kernel launches told apart by the timing session (isd_profile_begin/read).
enum { kKindStats = 0, kKindDecide = 1, kKindLmHead = 2, kKindMerge = 3, kKindFused = 4 };

// While a timing session is open, brackets one kernel launch on `stream` with a pair of CUDA
// events (graph nodes under stream capture).  Inactive otherwise.
struct ProfileScope {
    int slot = -1;
    cudaStream_t stream;
    ProfileScope(int kind, cudaStream_t s);
    ~ProfileScope();
    bool active() const { return slot >= 0; }
    void record(cudaEvent_t e);
};

}  // namespace isd_detail

namespace isd_detail {

// log2(e)/T split into a float head s_hi (rounded down) and a positive float tail s_lo.
void scale_split(float temperature, int greedy, float* s_hi, float* s_lo);

// Byte offsets, inside an isd_step workspace, of the chunk statistics [B][2N-1][C] (float2)
// and of the residual totals [B] (uint64); C = chunks per row of chunk_elems elements.  False
// on bad sizes.
bool workspace_sections(int B, int N, int V, int dtype, size_t* chunk, size_t* rtotal, int* C, int* chunk_elems);

// isd_step; with stats_ready the chunk statistics (and zeroed residual totals) are already in
// the workspace and only the decision pass is launched; with fused, isd_step_fused (one
// persistent kernel).
int step_impl(const void* logits, const void* prev_logits, int dtype, const int32_t* pending_tokens, int pending_ld,
              const float* pending_q, int B, int N, int V, float temperature, int greedy, uint64_t philox_seed,
              uint64_t step, int32_t* accepted_len, int32_t* tokens_out, float* new_q, float* p_out, int32_t* diag,
              void* workspace, size_t workspace_bytes, void* stream, bool stats_ready, bool fused = false);

}  // namespace isd_detail
