// isd_internal.h -- declarations shared by the library's translation units (not part of the
// C ABI).
#pragma once
#include <cuda_runtime.h>

namespace isd_detail {

// Kinds of kernel launches told apart by the timing session (isd_profile_begin/read).
enum { kKindStats = 0, kKindDecide = 1, kKindLmHead = 2 };

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
