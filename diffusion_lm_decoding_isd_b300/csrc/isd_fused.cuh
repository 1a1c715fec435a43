// isd_fused.cuh -- the fused ISD step (isd_step_fused): one persistent kernel reads every
// logit row the step needs once, and each sequence's decisions run as soon as the rows they
// depend on are summarised, while other rows are still streaming.  It is the alternative to
// the two-kernel step of isd_step (statistics pass, then decision pass) with no second launch
// and no grid-wide boundary between the two.  Included by isd_step.cu inside its anonymous
// namespace (it uses that file's element access, chunk statistics, Philox, fixed-point, draw
// planning and PTX helpers).
//
// The operation is the verify-and-propose step of Introspective Strided Decoding
// ("Introspective Diffusion Language Models"; ai.arkapp.pw blog, section "I-DLM 如何解決這些
// 問題"; de.news.hada.io, "Inference & ISD"): clean rows verify the pending tokens with
// min(1, p/q), the first rejection is resampled from norm(max(0, p - q)), MASK rows propose.
//
// Work.  A row job is one logit row cut into C units of one 4 KB chunk.  The row jobs follow
// from the pending state alone and take the first job numbers: the anchor rows 0..N-2 of every
// sequence with pending tokens (first, so that decisions come early), rows N-1..2N-2 of every
// sequence without, then rows N-1..2N-2 of every sequence with pending tokens.  Those last rows
// are read ahead of their sequence's decision; they are drawn from only if it keeps every
// pending token.  A sequence that rejects reads none of them (its bonus and MASK rows would
// only feed proposals that a rejection discards: the schedule under which the closed form of
// de.news.hada.io, "Speedup Factor Explorer", holds): once its decision is known, its units
// still to be taken are counted without a copy, and a NaN in them changes nothing.  A decision
// to reject at K (sampling) publishes the two halves of the residual, each C units of half a
// chunk of anchor row K and half a chunk of the previous call's MASK row N+K (and, when the
// previous call left no statistics of that row, the row itself first).  Units are numbered:
// job s owns units s*C .. s*C + C-1.  Warps take units in batches of 4 from one counter.
//
// Each streaming warp runs a ring of 3 shared-memory stages filled by 1-D bulk copies
// (cp.async.bulk, completion on an mbarrier, L2 evict-first).  A unit whose job is not
// published yet is kept aside while the warp works on its other stages; a warp waits
// (bounded) only when it has nothing else in flight.
//
// Completion.  Each unit writes its chunk statistic and takes a ticket on its job (an
// acquire-release atomic); the warp that takes a job's last ticket marks the job done with
// the call's tag.  Finishing warp f of F (the last warps of each CTA) takes the jobs numbered
// f + i*F in order, waits (bounded) for each to be marked done, and finishes it:
//   - an anchor row: its row statistics and p(x) of the pending token it verifies, then a
//     ticket on the sequence; the last anchor row's warp makes the sequence's decisions and
//     publishes its residual;
//   - a row N-1..2N-2 (of a sequence that proposes; for one with pending tokens, once its
//     decision says so): the draw (inverse CDF over the chunk sums, then a rescan of one chunk
//     read into registers) or the argmax, then a ticket on the sequence; the last one writes
//     the sequence's accepted length (or its error state);
//   - the residual: the replacement token (inverse CDF over the half-chunk sums of
//     max(0, p - q), then a rescan of one half chunk of both rows).
// No wait depends on a warp that is itself waiting: a decision depends only on anchor rows,
// which every finishing warp takes before any other job, and a published job only on
// decisions and on jobs numbered before it.  Counters and tickets are left at zero for the
// next call by their last user; the last warp to leave resets the unit counter and advances
// the epoch that names the next call.

// Per anchor row of a sequence with pending tokens (one lane each): p(x) of the pending token
// the row verifies, its logit, the row's argmax (greedy) and whether the row is usable.
struct AncStat {
    float pv, xl;
    int amax, ok;
};

// A published job: a row to summarise, or half of a residual.
struct JobRec {
    float ps_M, qs_M, ap, naq;  // residual: exponent references of p and q, and their scales
    unsigned long long head;    // call epoch << 32 | valid | skip | kind << 24 | half << 23 | row << 16 | b
    unsigned long long pad;
};
static_assert(sizeof(JobRec) == 32 && offsetof(JobRec, head) == 16, "job records are 32 bytes, constants first");

// Counters of the fused step, each busy one on a cache line of its own.  Zero between calls,
// except the epoch, which names the call (job records and completion flags carry the name of
// the call that wrote them, so they need no clearing between calls).
struct alignas(128) EngineLine {
    unsigned long long v;
    unsigned long long pad[15];
};
struct EngineCounters {
    EngineLine claim;                      // units handed out beyond the warps' first batches
    alignas(128) unsigned int dyn_count;   // job slots reserved by decisions
    unsigned int dec_done;                 // decisions made (sequences with pending tokens)
    alignas(128) unsigned int exit_count;  // warps that have left
    unsigned int epoch;                    // names the current call (never 0xFFFFFFFF)
};

// The step's parameters plus the fused kernel's own workspace (after the two-kernel step's
// sections; see isd_fused_workspace_size).  rtotal points at a residual-total array of its own.
struct FusedParams : Params {
    EngineCounters* eng;   // zero between calls, but for the epoch
    JobRec* jobs;          // [jobs_cap] published jobs
    int jobs_cap;
    unsigned long long* estat;   // [B][R][C] chunk statistics, self-marking (zero: not written yet)
    unsigned long long* eqstat;  // [B][C] the same for the q row of a residual
    unsigned* drawcnt;     // [B] rows N-1..2N-2 of a sequence done
    unsigned* rescnt;      // [B] residual units done (left at zero by the residual's finishing warp)
    unsigned* seqbad;      // [B] a row N-1..2N-2 was unusable
    unsigned long long* decw;  // [B] (epoch + 1) << 32 | outcome of the sequence's decision
    RowStat* rowstat;      // [B][R] statistics of the anchor rows
    float* rsum;           // [B][2C] sums of max(0, p - q) over half chunks
    int fxh;               // fraction bits of the fixed-point half-chunk residual sums
};

constexpr int kEWarps = 16;                 // warps of an engine CTA (one CTA per SM)
constexpr int kEFinishers = 1;              // warps of a CTA that finish jobs (the last ones)
constexpr int kEStreamers = kEWarps - kEFinishers;  // warps that stream units
constexpr int kEThreads = kEWarps * 32;
constexpr int kEDepth = 3;                  // bulk-copy stages per warp
constexpr size_t kEngineSmem = (size_t)kEStreamers * kEDepth * kChunkBytes;
constexpr int kMaskWords = kMaxB / 32;
constexpr int kHalf = kVec / 2;             // vectors per lane in half a chunk
constexpr int kECache = 4;                  // chunk statistics per lane kept in registers by a draw

enum : int { kUnitRow = 0, kUnitQRow = 1, kUnitResid = 2 };
// a unit counted without a copy: of a row that its sequence's decision leaves unread, or of a
// residual whose q row is unusable
constexpr int kUnitSkipRow = -1 - kUnitRow, kUnitSkipResid = -1 - kUnitResid;
// a decision's outcome (low word of its record): draw from rows N-1..2N-2, or not
constexpr unsigned kDecDraw = 1u, kDecNone = 2u;

// ----------------------------------------------------------------------------------------
// memory-model helpers (gpu scope)
// ----------------------------------------------------------------------------------------
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* a, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ unsigned atom_add_release(unsigned* a, unsigned v) {
    unsigned old;
    asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ void red_add_release(unsigned* a, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* a) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long* a) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
    return v;
}
__device__ __forceinline__ void st_release64(unsigned long long* a, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(a), "l"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// A ticket on a row, a sequence or a residual: lane 0 adds n units of work done to
// `counter`, and the warp learns whether they were the last of `count`.  The add has
// release semantics (this warp's earlier writes come first); the last taker then fences
// with acquire semantics, so that it reads after every other taker's writes, and leaves
// the counter at zero for the next call.
__device__ __forceinline__ bool take_ticket(unsigned* counter, unsigned n, unsigned count) {
    unsigned last = 0;
    if ((threadIdx.x & 31) == 0) last = atom_add_release(counter, n) + n == count;
    last = __shfl_sync(kFull, last, 0);
    if (last) {
        fence_acq_rel_gpu();
        if ((threadIdx.x & 31) == 0) *counter = 0u;
    }
    __syncwarp();
    return last != 0;
}

// ----------------------------------------------------------------------------------------
// units
// ----------------------------------------------------------------------------------------
// A unit: its sequence, row (for a residual: the rejected position K), chunk, kind, half
// (residual), the job slot it came from (published jobs), and a residual's constants.
struct Uint4x2 {
    uint4 a, b;
};
__device__ __forceinline__ Uint4x2 make_uint4x2(uint4 a, uint4 b) { return Uint4x2{a, b}; }

struct Unit {
    int b, r, c, kind, half, slot;
};
// A unit as a stage keeps it: sequence, row, kind and half packed in one word.
struct PackedUnit {
    int info, c, slot;
};
__device__ __forceinline__ PackedUnit pack_unit(const Unit& u, bool batch_end) {
    return PackedUnit{u.b | (u.r << 16) | ((u.kind + 4) << 22) | (u.half << 25) | ((int)batch_end << 26), u.c, u.slot};
}
__device__ __forceinline__ bool batch_end_of(const PackedUnit& q) { return (q.info >> 26) & 1; }
__device__ __forceinline__ Unit unpack_unit(const PackedUnit& q) {
    return Unit{q.info & 0xFFFF, (q.info >> 16) & 0x3F, q.c, ((q.info >> 22) & 7) - 4, (q.info >> 25) & 1, q.slot};
}
// The constants of a residual job: exponent references of p and q, and their scales.
struct ResidConst {
    float ps_M, qs_M, ap, naq;
};
__device__ __forceinline__ ResidConst load_resid_const(const JobRec* j) {
    const float4 c = __ldcg(reinterpret_cast<const float4*>(&j->ps_M));
    return ResidConst{c.x, c.y, c.z, c.w};
}

constexpr uint32_t kHeadValid = 1u << 31;
constexpr uint32_t kHeadSkip = 1u << 30;  // a residual whose q row is unusable: its units only count

__device__ __forceinline__ unsigned long long job_head(uint32_t epoch, int b, int r, int kind, int half, bool skip) {
    const uint32_t lo = kHeadValid | (skip ? kHeadSkip : 0u) | ((uint32_t)kind << 24) | ((uint32_t)half << 23) |
                        ((uint32_t)r << 16) | (uint32_t)b;
    return ((unsigned long long)epoch << 32) | lo;
}

// The k-th (0-based) set bit of w.
__device__ __forceinline__ int select_bit(uint32_t w, int k) {
    int pos = 0;
#pragma unroll
    for (int width = 16; width > 0; width >>= 1) {
        const int c = __popc(w & ((1u << width) - 1u));
        if (k >= c) {
            k -= c;
            w >>= width;
            pos += width;
        }
    }
    return pos;
}

struct EngineShared {
    uint32_t mask[kMaskWords];   // bit b: sequence b has pending tokens
    int pre[kMaskWords + 1];     // sequences with pending tokens in words before w
    int nwords, P;               // words, pending sequences
    int A, D0, S0;               // row jobs: anchors [0, A), rows N-1.. without pending tokens
                                 // [A, D0), with pending tokens [D0, S0)
    int carry;                   // the previous call left the q rows' statistics
    uint32_t epoch, tag;         // the call's epoch; tag = epoch + 1 marks what it completed
};

// The sequence of the k-th sequence with (pending) or without (!pending) pending tokens.
__device__ __forceinline__ int kth_sequence(const EngineShared& sh, int B, int k, bool pending) {
    int lo = 0, hi = sh.nwords - 1;  // last word w whose prefix is <= k
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        const int before = pending ? sh.pre[mid] : min(32 * mid, B) - sh.pre[mid];
        if (before <= k) lo = mid;
        else hi = mid - 1;
    }
    const int before = pending ? sh.pre[lo] : min(32 * lo, B) - sh.pre[lo];
    uint32_t w = sh.mask[lo];
    if (!pending) {
        const int valid = min(32, B - 32 * lo);
        w = ~w & (valid == 32 ? 0xFFFFFFFFu : ((1u << valid) - 1u));
    }
    return 32 * lo + select_bit(w, k - before);
}

enum : int { kReady = 0, kNotYet = 1, kNoMore = 2 };

__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long* a) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed64(unsigned long long* a, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(a), "l"(v) : "memory");
}

// Chunk statistics as this kernel stores them: one 64-bit word per chunk, written and read
// whole (single-copy atomic), the maximum's bits complemented in the low half and the sum (or,
// greedy, the index of the maximum) in the high half.  No statistic has a maximum with every
// bit set (a NaN maximum is stored as the canonical NaN), so a zero word marks a chunk not
// summarised yet: the words start at zero (a zero-filled workspace), a finishing warp waits
// until every word of its row is nonzero, and sets them back to zero once it has used them.
typedef unsigned long long EStat;
constexpr EStat kSkippedChunk = 1ull;  // a chunk counted without a copy: never read as a statistic
__device__ __forceinline__ EStat enc_stat(float2 st) {
    return (EStat)(~__float_as_uint(st.x)) | ((EStat)__float_as_uint(st.y) << 32);
}
__device__ __forceinline__ float2 dec_stat(EStat w) {
    return make_float2(__uint_as_float(~(uint32_t)w), __uint_as_float((uint32_t)(w >> 32)));
}
__device__ __forceinline__ float2 ld_estat(const EStat* cs, int c) { return dec_stat(ld_relaxed64(cs + c)); }

// q = x / d, r = x - q*d for non-negative x and positive d (32-bit when x fits).
__device__ __forceinline__ long long div_rem(long long x, int d, int* r) {
    if (x < 0x7FFFFFFFll) {
        const unsigned q = (unsigned)x / (unsigned)d;
        *r = (int)((unsigned)x - q * (unsigned)d);
        return q;
    }
    const long long q = x / d;
    *r = (int)(x - q * d);
    return q;
}

// Row job s < S0 -> its sequence and row; returns 0 (an anchor row), 1 (a row N-1.. of a
// sequence without pending tokens) or 2 (of a sequence with pending tokens).
__device__ __forceinline__ int row_job(const FusedParams& p, const EngineShared& sh, long long s, int& b, int& r) {
    if (s < sh.A) {
        const int k = (int)div_rem(s, p.N - 1, &r);
        b = kth_sequence(sh, p.B, k, true);
        return 0;
    }
    const bool pend = s >= sh.D0;
    const int k = (int)div_rem(s - (pend ? sh.D0 : sh.A), p.N, &r);
    r += p.N - 1;
    b = kth_sequence(sh, p.B, k, pend);
    return pend ? 2 : 1;
}

// Job slot s -> the job's units (all but the chunk), if the job is known (whole warp;
// uniform result).  An unknown job is kNotYet; with check_end, kNoMore when every decision
// has been made and the slot lies past every published job.
__device__ int resolve_slot(const FusedParams& p, const EngineShared& sh, long long s, Unit& u, bool check_end) {
    u.c = 0;
    u.half = 0;
    u.slot = -1;
    if (s < sh.S0) {
        u.kind = kUnitRow;
        if (row_job(p, sh, s, u.b, u.r) == 2) {
            // read ahead of the decision: skipped once the decision says the row is not drawn from
            unsigned long long w = 0ull;
            if ((threadIdx.x & 31) == 0) w = ld_relaxed64(&p.decw[u.b]);
            w = __shfl_sync(kFull, w, 0);
            if ((uint32_t)(w >> 32) == sh.tag && (uint32_t)w != kDecDraw) u.kind = kUnitSkipRow;
        }
        return kReady;
    }
    const long long k = s - sh.S0;
    unsigned long long head = 0ull;
    if (k < p.jobs_cap && (threadIdx.x & 31) == 0) head = ld_relaxed64(&p.jobs[k].head);
    head = __shfl_sync(kFull, head, 0);
    const uint32_t lo = (uint32_t)head;
    if ((uint32_t)(head >> 32) == sh.epoch && (lo & kHeadValid)) {
        u.b = (int)(lo & 0xFFFFu);
        u.r = (int)((lo >> 16) & 0x3Fu);
        u.half = (int)((lo >> 23) & 1u);
        u.kind = (int)((lo >> 24) & 3u);
        u.slot = (int)k;
        if (u.kind == kUnitResid) {
            fence_acq_rel_gpu();  // the job's constants were written before its head
            if (lo & kHeadSkip) u.kind = kUnitSkipResid;  // count only
        }
        return kReady;
    }
    if (!check_end) return kNotYet;
    // not published: is more work still to come?
    unsigned more = 1u;
    if ((threadIdx.x & 31) == 0) {
        if (ld_acquire(&p.eng->dec_done) == (unsigned)sh.P && k >= (long long)ld_acquire(&p.eng->dyn_count)) more = 0u;
    }
    more = __shfl_sync(kFull, more, 0);
    return more ? kNotYet : kNoMore;
}

// Plain loads of n elements into a stage buffer of `len` elements, -inf past n (whole warp;
// for rows that are not 16-byte aligned).
template <int DT>
__device__ __noinline__ void fill_plain(unsigned char* buf, const char* src, int n, int len) {
    const int lane = threadIdx.x & 31;
    for (int i = lane; i < len; i += 32) {
        if (DT == ISD_BF16)
            reinterpret_cast<uint16_t*>(buf)[i] = i < n ? reinterpret_cast<const uint16_t*>(src)[i] : 0xFF80u;
        else
            reinterpret_cast<uint32_t*>(buf)[i] = i < n ? reinterpret_cast<const uint32_t*>(src)[i] : 0xFF800000u;
    }
    __syncwarp();
}

// Start filling a stage with unit u (whole warp).  Rows must be 16-byte aligned with
// V * element size a multiple of 16 bytes for the bulk copies; otherwise the warp fills the
// stage with plain loads now.
template <int DT>
__device__ void issue_unit(const FusedParams& p, const Unit& u, unsigned char* buf, uint32_t bar, uint64_t pol) {
    using E = Elem<DT>;
    const int lane = threadIdx.x & 31;
    const char* logits = static_cast<const char*>(p.logits);
    const char* prev = static_cast<const char*>(p.prev);
    if (u.kind == kUnitSkipRow) {  // nothing to copy: the stage's phase completes at once
        if (p.vec_ok && lane == 0) mbar_expect_tx(bar, 0u);
        return;
    }
    if (u.kind == kUnitResid || u.kind == kUnitSkipResid) {
        constexpr int H = E::kChunk / 2;
        const int64_t e0 = (int64_t)u.c * E::kChunk + u.half * H;
        const int n = (int)max((int64_t)0, min((int64_t)H, (int64_t)p.V - e0));
        const char* pa = logits + ((int64_t)u.b * p.R + u.r) * p.V * E::kBytes + e0 * E::kBytes;
        const char* qa = prev + ((int64_t)u.b * p.R + p.N + u.r) * p.V * E::kBytes + e0 * E::kBytes;
        if (p.vec_ok) {
            if (lane == 0) {
                fence_proxy_async_smem();
                mbar_expect_tx(bar, 2u * (uint32_t)n * E::kBytes);
                if (n > 0) {
                    bulk_load(smem_u32(buf), pa, (uint32_t)n * E::kBytes, bar, pol);
                    bulk_load(smem_u32(buf + kChunkBytes / 2), qa, (uint32_t)n * E::kBytes, bar, pol);
                }
            }
        } else {
            fill_plain<DT>(buf, pa, n, H);
            fill_plain<DT>(buf + kChunkBytes / 2, qa, n, H);
        }
        return;
    }
    const char* base = u.kind == kUnitQRow ? prev : logits;
    const int64_t e0 = (int64_t)u.c * E::kChunk;
    const int n = (int)min((int64_t)E::kChunk, (int64_t)p.V - e0);
    const char* src = base + ((int64_t)u.b * p.R + u.r) * p.V * E::kBytes + e0 * E::kBytes;
    if (p.vec_ok) {
        if (lane == 0) {
            fence_proxy_async_smem();
            mbar_expect_tx(bar, (uint32_t)n * E::kBytes);
            // a row that is drawn from (N-1 and after) is read again, one chunk, by its draw:
            // it is not marked evict-first
            if (u.kind == kUnitRow && u.r >= p.N - 1) bulk_load_plain(smem_u32(buf), src, (uint32_t)n * E::kBytes, bar);
            else bulk_load(smem_u32(buf), src, (uint32_t)n * E::kBytes, bar, pol);
        }
    } else {
        fill_plain<DT>(buf, src, n, E::kChunk);
    }
}

// ----------------------------------------------------------------------------------------
// draws from registers
// ----------------------------------------------------------------------------------------
// Row statistics written earlier in this kernel, read from L2.
__device__ __forceinline__ RowStat load_rowstat_cg(const RowStat* a) {
    static_assert(sizeof(RowStat) == 32, "RowStat is two 16-byte words");
    const float4 x = __ldcg(reinterpret_cast<const float4*>(a));
    const float4 y = __ldcg(reinterpret_cast<const float4*>(a) + 1);
    RowStat r;
    memcpy(&r, &x, 16);
    memcpy(reinterpret_cast<char*>(&r) + 16, &y, 16);
    return r;
}

// Row statistics from the chunk statistics (written in this kernel: read from L2), the
// first kECache*32 of them kept in registers as fixed-point weights for the walk.
struct RowWalk {
    uint64_t w[kECache];  // fixed-point weights of chunks lane + 32*i
    float2 st[kECache];   // their statistics
};

// The first kECache*32 chunk statistics of a row, one per lane and slot (-inf past C).
__device__ __forceinline__ void load_stat_cache(const EStat* cs, int C, float2 (&cache)[kECache]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < kECache; ++i) {
        const int c = lane + 32 * i;
        cache[i] = c < C ? ld_estat(cs, c) : make_float2(-INFINITY, 0.f);
    }
}

// Row statistics from its chunk statistics, the first kECache*32 of them given in `cache`
// (the rest read from L2), kept in registers as fixed-point weights for a walk.
__device__ __forceinline__ bool combine_from_cache(const float2 (&cache)[kECache], const EStat* cs, int C, int fx,
                                                   float s_hi, float s_lo, RowStat& out, RowWalk& rw) {
    const int lane = threadIdx.x & 31;
    bool bad = false;
    uint32_t key = 0;
    auto see = [&](float e) {
        if (isnan(e) || e == INFINITY) bad = true;
        else if (e > -INFINITY) key = max(key, order_key(e));
    };
#pragma unroll
    for (int i = 0; i < kECache; ++i) see(cache[i].x);
    for (int c = lane + 32 * kECache; c < C; c += 32) see(ld_estat(cs, c).x);
    key = __reduce_max_sync(kFull, key);
    bad = __any_sync(kFull, bad);
    const float m_row = key ? from_key(key) : -INFINITY;
    if (bad || !isfinite(m_row)) return false;
    const float M = exponent_ref(m_row, s_hi);
    uint64_t Z = 0;
#pragma unroll
    for (int i = 0; i < kECache; ++i) {
        rw.w[i] = chunk_fixed(cache[i], M, fx, s_hi);
        rw.st[i] = cache[i];
        Z += rw.w[i];
    }
    for (int c = lane + 32 * kECache; c < C; c += 32) Z += chunk_fixed(ld_estat(cs, c), M, fx, s_hi);
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

__device__ __forceinline__ bool combine_row_cached(const EStat* cs, int C, int fx, float s_hi, float s_lo,
                                                   RowStat& out, RowWalk& rw) {
    float2 cache[kECache];
    load_stat_cache(cs, C, cache);
    return combine_from_cache(cache, cs, C, fx, s_hi, s_lo, out, rw);
}

// Greedy: the row maximum and the lowest index holding it, from chunk statistics (maximum,
// lowest index of it in the chunk) given as for combine_from_cache.  False if a chunk
// maximum is NaN or the row has no finite maximum.
__device__ __forceinline__ bool argmax_from_cache(const float2 (&cache)[kECache], const EStat* cs, int C,
                                                  RowStat& out) {
    const int lane = threadIdx.x & 31;
    bool nan = false;
    uint32_t key = 0;
#pragma unroll
    for (int i = 0; i < kECache; ++i) {
        if (isnan(cache[i].x)) nan = true;
        else key = max(key, order_key(cache[i].x));
    }
    for (int c = lane + 32 * kECache; c < C; c += 32) {
        const float m = ld_estat(cs, c).x;
        if (isnan(m)) nan = true;
        else key = max(key, order_key(m));
    }
    key = __reduce_max_sync(kFull, key);
    nan = __any_sync(kFull, nan);
    const float m_row = from_key(key);
    if (nan || !isfinite(m_row)) return false;
    // the first chunk holding the maximum, and its index there
    uint32_t first = 0xFFFFFFFFu, idx = 0u;
#pragma unroll
    for (int i = kECache - 1; i >= 0; --i)
        if (cache[i].x == m_row) {
            first = (uint32_t)(lane + 32 * i);
            idx = __float_as_uint(cache[i].y);
        }
    if (first == 0xFFFFFFFFu)
        for (int c = lane + 32 * kECache; c < C; c += 32) {
            const float2 st = ld_estat(cs, c);
            if (st.x == m_row) {
                first = (uint32_t)c;
                idx = __float_as_uint(st.y);
                break;
            }
        }
    const uint32_t fmin = __reduce_min_sync(kFull, first);
    if (fmin >= (uint32_t)C) return false;
    const unsigned holder = __ballot_sync(kFull, first == fmin);
    out.Zfx = 0ull;
    out.M = m_row;
    out.Zf = 0.f;
    out.T = 1.f;
    out.amax = (int)__shfl_sync(kFull, idx, __ffs(holder) - 1);
    out.mx = m_row;
    return true;
}

// Statistics of chunk c (warp-uniform c): from the lane that keeps it, else from L2.
__device__ __forceinline__ float2 cached_stat(const EStat* cs, const RowWalk& rw, int c) {
    if (c >= 32 * kECache) return ld_estat(cs, c);
    float2 x = rw.st[0];
#pragma unroll
    for (int i = 1; i < kECache; ++i)
        if (i == (c >> 5)) x = rw.st[i];
    return make_float2(__shfl_sync(kFull, x.x, c & 31), __shfl_sync(kFull, x.y, c & 31));
}

// The chunk holding the target of an inverse-CDF draw over a row's chunk sums, and the
// remaining target in that chunk's head-weight units (see plan_draw).
__device__ DrawPlan plan_draw_cached(const FusedParams& p, const EStat* cs, const RowStat& rs, const RowWalk& rw,
                                     uint64_t target) {
    uint64_t before = 0;
    int last_pos;
    const int cstar = walk_chunks(
        p.C, target,
        [&](int c) {
            const int i = c >> 5;
            uint64_t w = 0;
#pragma unroll
            for (int k = 0; k < kECache; ++k)
                if (k == i) w = rw.w[k];
            return i < kECache ? w : chunk_fixed(ld_estat(cs, c), rs.M, p.fx, p.s_hi);
        },
        &before, &last_pos);
    if (cstar < 0) return DrawPlan{last_pos < 0 ? 0 : last_pos, INFINITY};
    const float2 st = cached_stat(cs, rw, cstar);
    const int d = (int)fmaxf(exponent_ref(st.x, p.s_hi) - rs.M, -256.f);
    return DrawPlan{cstar, fixed_to_float(target - before, p.fx + d) / tail_factor(st.x, p.s_lo)};
}

// Inverse CDF inside NV vectors per lane held in registers (one warp): the first element, in
// index order (vector k of lane L holds elements (k*32 + L)*PER .. +PER-1), whose running sum
// of weights exceeds target.  vec(k) gives vector k (k known at compile time) and
// wt(vector, j) the weight of its element j.  Returns the offset, or -1 when rounding leaves
// no such element (*last = the last offset with positive weight, or -1).
struct NoValue {
    template <typename X>
    __device__ float operator()(const X&, int) const { return 0.f; }
};

template <int NV, int PER, typename Vec, typename Wt, typename Val = NoValue>
__device__ __forceinline__ int rescan_regs(float target, Vec vec, Wt wt, int* last, Val val = Val(),
                                           float* value = nullptr) {
    const int lane = threadIdx.x & 31;
    float incl[NV];
    int lastpos = -1;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const auto x = vec(k);
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const float a = wt(x, j);
            s += a;
            if (a > 0.f) lastpos = (k * 32 + lane) * PER + j;
        }
        incl[k] = s;
    }
    // inclusive scans of the NV lane totals across the warp, side by side
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const float y = __shfl_up_sync(kFull, incl[k], o);
            if (lane >= o) incl[k] += y;
        }
    }
    *last = (int)__reduce_max_sync(kFull, (unsigned)(lastpos + 1)) - 1;
    float base = 0.f;
    int ks = -1;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const float tot = __shfl_sync(kFull, incl[k], 31);
        if (ks < 0) {
            if (base + tot > target) ks = k;
            else base += tot;
        }
    }
    if (ks < 0) return -1;
    float mine = 0.f;
    auto x = vec(0);
#pragma unroll
    for (int k = 0; k < NV; ++k)
        if (k == ks) {
            mine = incl[k];
            x = vec(k);
        }
    const unsigned hit = __ballot_sync(kFull, base + mine > target);
    const int L = hit ? __ffs(hit) - 1 : 31;
    const float before = __shfl_sync(kFull, mine, L > 0 ? L - 1 : 0);
    float cum = base + (L > 0 ? before : 0.f);
    int my_j = -1, my_last = -1;
    float my_v = 0.f, my_lv = 0.f;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const float a = wt(x, j);
        cum += a;
        if (my_j < 0 && a > 0.f && cum > target) {
            my_j = j;
            my_v = val(x, j);
        }
        if (a > 0.f) {
            my_last = j;
            my_lv = val(x, j);
        }
    }
    if (my_j < 0) {  // rounding inside the lane: its last weighted element
        my_j = my_last;
        my_v = my_lv;
    }
    my_j = __shfl_sync(kFull, my_j, L);
    my_v = __shfl_sync(kFull, my_v, L);
    if (my_j < 0) return -1;
    if (value) *value = my_v;
    return (ks * 32 + L) * PER + my_j;
}

// Draw one token from a row (whole warp): walk the chunk sums, read the target chunk into
// registers, rescan it.  *px = p(token).
template <int DT>
__device__ int draw_from_row(const FusedParams& p, const void* row, const EStat* cs, const RowStat& rs,
                             const RowWalk& rw, uint32_t word, float* px) {
    using E = Elem<DT>;
    const int lane = threadIdx.x & 31;
    const DrawPlan plan = plan_draw_cached(p, cs, rs, rw, scale_by_uniform(rs.Zfx, word));
    const int64_t base = (int64_t)plan.cstar * E::kChunk;
    uint4 v[kVec];
    load_chunk<DT>(row, p.V, base, p.vec_ok, false, v);
    const float ref = ref_or_zero(exponent_ref(cached_stat(cs, rw, plan.cstar).x, p.s_hi));
    const float s_hi = p.s_hi;
    int last;
    float x;
    int off = rescan_regs<kVec, E::kPerVec>(
        plan.target, [&](int k) { return v[k]; },
        [&](const uint4& w, int j) { return weight_head(vec_elem<DT>(w, j), ref, s_hi); }, &last,
        [&](const uint4& w, int j) { return vec_elem<DT>(w, j); }, &x);
    if (off < 0) {
        off = last < 0 ? 0 : last;
        if (lane == 0) diag_add(p, ISD_DIAG_NEAR_TIE_CDF, 1);
        x = load_elem<DT>(row, base + off);
    }
    *px = exp2f(weight_exp(x, rs.M, p.s_hi, p.s_lo)) / rs.Zf;
    return (int)(base + off);
}

// The lowest index of a row holding its maximum mx (whole warp): the first chunk whose
// maximum is mx, then that chunk read into registers.
template <int DT>
__device__ int argmax_of_row(const FusedParams& p, const void* row, const EStat* cs, float mx) {
    using E = Elem<DT>;
    const int lane = threadIdx.x & 31;
    int cstar = 0;
    for (int c0 = 0; c0 < p.C; c0 += 32) {
        const int c = c0 + lane;
        const unsigned hit = __ballot_sync(kFull, c < p.C && ld_estat(cs, c).x == mx);
        if (hit) {
            cstar = c0 + __ffs(hit) - 1;
            break;
        }
    }
    const int64_t base = (int64_t)cstar * E::kChunk;
    uint4 v[kVec];
    load_chunk<DT>(row, p.V, base, p.vec_ok, false, v);
    uint32_t idx = 0xFFFFFFFFu;
#pragma unroll
    for (int k = kVec - 1; k >= 0; --k)
#pragma unroll
        for (int j = E::kPerVec - 1; j >= 0; --j)
            if (E::get(v, k, j) == mx) idx = (uint32_t)((k * 32 + lane) * E::kPerVec + j);
    idx = __reduce_min_sync(kFull, idx);
    return (int)(base + (idx == 0xFFFFFFFFu ? 0u : idx));
}

// Draw from a row without token x (logit xl), whole warp: x's weight, computed as the
// chunk statistics weigh it, is taken out of its chunk's sum and of the row total.
template <int DT>
__device__ int draw_from_row_excluding(const FusedParams& p, const void* row, const EStat* cs, const RowStat& rs,
                                       const RowWalk& rw, int x, float xl, uint32_t word) {
    using E = Elem<DT>;
    const int lane = threadIdx.x & 31;
    const int cx = x / E::kChunk;
    const float2 stx = ld_estat(cs, cx);
    const float ex = ref_or_zero(exponent_ref(stx.x, p.s_hi));
    const int dx = (int)fmaxf(ex - rs.M, -256.f);
    const uint64_t cfx = chunk_fixed(stx, rs.M, p.fx, p.s_hi);
    const uint64_t wx = to_fixed(weight_head(xl, ex, p.s_hi) * tail_factor(stx.x, p.s_lo), p.fx + dx);
    const uint64_t cut = wx < cfx ? wx : cfx;
    const uint64_t total = rs.Zfx - cut;
    if (total == 0ull) {  // all of the row's mass on x: reachable only through rounding
        if (lane == 0) diag_add(p, ISD_DIAG_NEAR_TIE_CDF, 1);
        float px;
        return draw_from_row<DT>(p, row, cs, rs, rw, word, &px);
    }
    const uint64_t target = scale_by_uniform(total, word);
    uint64_t before = 0;
    int last_pos;
    int cstar = walk_chunks(
        p.C, target,
        [&](int c) {
            const uint64_t w = chunk_fixed(ld_estat(cs, c), rs.M, p.fx, p.s_hi);
            return c == cx ? w - cut : w;
        },
        &before, &last_pos);
    float local = INFINITY;
    if (cstar < 0) {
        cstar = last_pos < 0 ? 0 : last_pos;
    } else {
        const float2 st = ld_estat(cs, cstar);
        const int d = (int)fmaxf(exponent_ref(st.x, p.s_hi) - rs.M, -256.f);
        local = fixed_to_float(target - before, p.fx + d) / tail_factor(st.x, p.s_lo);
    }
    const int64_t base = (int64_t)cstar * E::kChunk;
    uint4 v[kVec];
    load_chunk<DT>(row, p.V, base, p.vec_ok, false, v);
    const float ref = ref_or_zero(exponent_ref(ld_estat(cs, cstar).x, p.s_hi));
    const int xoff = cstar == cx ? x - cstar * E::kChunk : -1;
    const float s_hi = p.s_hi;
    int last;
    // x's own weight is left out by its offset (vector k of lane L holds (k*32 + L)*PER + j)
    int off = rescan_regs<kVec, E::kPerVec>(
        local, [&](int k) { return make_int2(k, 0); },
        [&](const int2& kk, int j) {
            const int k = kk.x;
            uint4 w = v[0];
#pragma unroll
            for (int i = 1; i < kVec; ++i)
                if (i == k) w = v[i];
            return (k * 32 + lane) * E::kPerVec + j == xoff ? 0.f : weight_head(vec_elem<DT>(w, j), ref, s_hi);
        },
        &last);
    if (off < 0) {
        off = last < 0 ? 0 : last;
        if (lane == 0) diag_add(p, ISD_DIAG_NEAR_TIE_CDF, 1);
    }
    return (int)(base + off);
}

// Sum of max(0, p - q) over half a chunk held in registers: p in v[0..kHalf), q in
// v[kHalf..kVec), with the arithmetic of residual_elem on the f32x2 pipe.
template <int DT>
__device__ __forceinline__ float residual_half_sum(const uint4 (&v)[kVec], const ResidConst& u, float s_hi) {
    const uint64_t S2 = pack2(s_hi, s_hi), NMP2 = pack2(-u.ps_M, -u.ps_M), NMQ2 = pack2(-u.qs_M, -u.qs_M);
    const uint64_t AP2 = pack2(u.ap, u.ap), NAQ2 = pack2(u.naq, u.naq), Z2 = 0ull;
    uint64_t acc0 = 0ull, acc1 = 0ull;
#pragma unroll
    for (int k = 0; k < kHalf; ++k) {
        const uint32_t* xp = &v[k].x;
        const uint32_t* xq = &v[kHalf + k].x;
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

// ----------------------------------------------------------------------------------------
// finishing rows and sequences (one warp each)
// ----------------------------------------------------------------------------------------
// Error outputs of sequence b: no token, no proposal, no probability.
__device__ void fail_outputs(const FusedParams& p, int b, int code) {
    const int lane = threadIdx.x & 31;
    for (int i = lane; i < p.R; i += 32) p.tokens_out[(int64_t)b * p.R + i] = -1;
    for (int i = lane; i < p.N - 1; i += 32) {
        p.new_q[(int64_t)b * (p.N - 1) + i] = 0.f;
        if (p.p_out) p.p_out[(int64_t)b * (p.N - 1) + i] = 0.f;
    }
    if (lane == 0) {
        p.accepted_len[b] = 0;
        set_status(p, code);
    }
}

// Reserve n job slots and write them (lane 0).  Returns the first slot.
__device__ __forceinline__ int reserve_jobs(const FusedParams& p, int n) {
    return (int)atomicAdd(&p.eng->dyn_count, (unsigned)n);
}

// The decision record of sequence b (lane 0), after the decision's outputs: whoever reads it
// with acquire semantics reads after them.
__device__ __forceinline__ void post_decision(const FusedParams& p, const EngineShared& sh, int b, unsigned outcome) {
    if ((threadIdx.x & 31) == 0) st_release64(&p.decw[b], ((unsigned long long)sh.tag << 32) | outcome);
}

// What lane i < N-1 of a sequence's finishing warp knows about pending position i: the
// pending token, its q, what anchor row i gave, and (sampling) the references and scales of
// row i and of the previous call's MASK row N+i (carried), for a residual at i.
struct AnchorLane {
    int x;
    float xq;
    AncStat a;
    float ps_M, ap;       // row i: exponent reference, T / Zf
    float qs_M, naq;      // MASK row N+i of the previous call: exponent reference, -T / Zf
    bool q_ok;            // that row was usable
};

// The decisions of sequence b (whole warp; lane i < N-1 holds position i).  What waits on
// them goes first: the residual's jobs, then (for a rejection) the decision record; the
// outputs follow.  A decision to draw from rows N-1.. is recorded after the outputs, with
// release semantics, since the draws' last finisher may overwrite them (failure).  Returns the
// anchor row whose statistic words a residual still reads (K), or -1.
template <int DT, bool GREEDY>
__device__ __forceinline__ int decide_sequence(const FusedParams& p, const EngineShared& sh, int b, const AnchorLane& L) {
    const int lane = threadIdx.x & 31;
    const int N = p.N, R = p.R;
    int32_t* tok = p.tokens_out + (int64_t)b * R;
    float* nq = p.new_q + (int64_t)b * (N - 1);
    const int x = L.x;
    const AncStat& a = L.a;
    bool bad_pending = false;
    if (lane < N - 1) {
        if (x < 0 || x >= p.V) bad_pending = true;
        if (!GREEDY && (!(L.xq > 0.f && L.xq < INFINITY) || (p.prev == nullptr && !p.amode))) bad_pending = true;
    }
    bad_pending = __any_sync(kFull, bad_pending);
    const bool bad_rows = __any_sync(kFull, lane < N - 1 && !a.ok);
    bool accept = true;
    if (lane < N - 1 && !bad_pending && !bad_rows) {
        if (GREEDY) {
            accept = x == a.amax;
        } else {
            const float u = to_uniform(row_words(p.seed, p.step, b, lane).x);
            // u < p/q  <=>  u*q < p, with u*q = prod + err exactly (err from an FMA)
            const float prod = u * L.xq;
            accept = prod < a.pv || (prod == a.pv && fmaf(u, L.xq, -prod) < 0.f);
            if (fabsf(u - a.pv / L.xq) < (float)kNearTie) diag_add(p, ISD_DIAG_NEAR_TIE_ACC, 1);
        }
    }
    const unsigned rej = __ballot_sync(kFull, lane < N - 1 && !accept);
    const int K = rej ? __ffs(rej) - 1 : N - 1;
    // a residual at K whose carried q row is unusable fails the sequence at once
    const bool resid = !GREEDY && !p.amode && K < N - 1;
    const bool q_bad = resid && sh.carry && !__shfl_sync(kFull, L.q_ok, K);
    if (bad_pending || bad_rows || q_bad) {
        fail_outputs(p, b, bad_pending ? ISD_ERR_BAD_PENDING : ISD_ERR_NONFINITE);
        post_decision(p, sh, b, kDecNone);
        if (lane == 0) red_add_release(&p.eng->dec_done, 1u);
        return -1;
    }
    if (resid && sh.carry) {
        // residual from max(0, p - q), q the previous call's MASK row N+K (carried statistics)
        const float psM = __shfl_sync(kFull, L.ps_M, K), ap = __shfl_sync(kFull, L.ap, K);
        const float qsM = __shfl_sync(kFull, L.qs_M, K), naq = __shfl_sync(kFull, L.naq, K);
        if (lane == 0) {
            const int s = reserve_jobs(p, 2);
            for (int h = 0; h < 2; ++h) {
                JobRec* j = &p.jobs[s + h];
                j->ps_M = psM;
                j->qs_M = qsM;
                j->ap = ap;
                j->naq = naq;
            }
            fence_acq_rel_gpu();  // the constants before the heads (a release for both)
            for (int h = 0; h < 2; ++h)
                st_relaxed64(&p.jobs[s + h].head, job_head(sh.epoch, b, K, kUnitResid, h, false));
        }
    }
    if (K < N - 1) post_decision(p, sh, b, kDecNone);
    // outputs: the kept prefix, the -1 of positions nothing will fill, p(x)
    for (int i = lane; i < R; i += 32) {
        if (i < K) tok[i] = x;  // lane i < K < N-1 holds pending token i
        else if (K < N - 1 && i > K) tok[i] = -1;
    }
    if (lane < N - 1) {
        if (p.p_out) p.p_out[(int64_t)b * (N - 1) + lane] = GREEDY ? 0.f : a.pv;
        if (K < N - 1) nq[lane] = 0.f;
    }
    if (lane == 0) {
        p.accepted_len[b] = K < N - 1 ? K + 1 : N;
        diag_add(p, ISD_DIAG_EMITTED, K < N - 1 ? K + 1 : N);
        diag_add(p, ISD_DIAG_ACCEPTS, K);
        diag_add(p, ISD_DIAG_TESTS, K < N - 1 ? K + 1 : N - 1);
        if (!GREEDY && K < N - 1) diag_add(p, ISD_DIAG_RESIDUALS, 1);
    }
    if (K == N - 1) {
        // all kept: the anchor row N-1 and the MASK rows (read ahead) are drawn from
        post_decision(p, sh, b, kDecDraw);
    } else if (GREEDY) {
        const int amax_k = __shfl_sync(kFull, a.amax, K);
        if (lane == 0) tok[K] = amax_k;
    } else if (p.amode) {
        // the rejected proposal was a point mass: the replacement comes from anchor row K
        // without it (no previous row, no residual pass)
        const int xk = __shfl_sync(kFull, x, K);
        const float xlk = __shfl_sync(kFull, a.xl, K);
        const EStat* cs = p.estat + ((int64_t)b * R + K) * p.C;
        RowStat rs;
        RowWalk rw;
        combine_row_cached(cs, p.C, p.fx, p.s_hi, p.s_lo, rs, rw);  // usable: checked with the row
        const void* row = row_ptr(p.logits, Elem<DT>::kBytes, (int64_t)b * R + K, p.V);
        const int y = draw_from_row_excluding<DT>(p, row, cs, rs, rw, xk, xlk, row_words(p.seed, p.step, b, K).y);
        if (lane == 0) tok[K] = y;
    } else if (!sh.carry) {
        // no carried statistics of the q row: it is read first; its finishing warp publishes
        // the residual's jobs (after these outputs: its head is a release)
        if (lane == 0) {
            const int s = reserve_jobs(p, 3);
            st_release64(&p.jobs[s].head, job_head(sh.epoch, b, N + K, kUnitQRow, 0, false));
        }
    }
    if (lane == 0) red_add_release(&p.eng->dec_done, 1u);
    return resid ? K : -1;
}

// Wait (whole warp; lane 0 polls) until the units counted in *counter reach n, then leave
// it at zero for the next call.  The acquire load that sees n reads after every unit's
// writes (each unit's count is a release).  False, with the timeout status set, after the
// wait limit.
__device__ __forceinline__ bool wait_count(const FusedParams& p, unsigned* counter, unsigned n) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) {
        uint64_t t0 = 0;
        while (ld_acquire(counter) != n) {
            const uint64_t now = global_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > p.wait_ns) {
                set_status(p, ISD_ERR_TIMEOUT);
                ok = 0;
                break;
            }
            __nanosleep(96);
        }
        if (ok) *counter = 0u;
    }
    return __shfl_sync(kFull, ok, 0) != 0;
}

// Wait (whole warp) until every statistic word of G rows is written: row j at cs + j*stride,
// for j < n.  The first kECache*32 words of each come back decoded in cache[j] (past C:
// -inf, 0).  False, with the timeout status set, after the wait limit.
template <int G>
__device__ __forceinline__ bool poll_rows(const FusedParams& p, const EStat* cs, int64_t stride, int n,
                                          float2 (&cache)[G][kECache]) {
    const int lane = threadIdx.x & 31;
    uint64_t t0 = 0;
    for (;;) {
        bool mine = true;
#pragma unroll
        for (int j = 0; j < G; ++j) {
#pragma unroll
            for (int i = 0; i < kECache; ++i) {
                const int c = lane + 32 * i;
                const bool in = j < n && c < p.C;
                const EStat w = in ? ld_relaxed64(cs + j * stride + c) : 0ull;
                if (in && w == 0ull) mine = false;
                cache[j][i] = in ? dec_stat(w) : make_float2(-INFINITY, 0.f);
            }
            if (j < n)
                for (int c = lane + 32 * kECache; c < p.C; c += 32)
                    if (ld_relaxed64(cs + j * stride + c) == 0ull) mine = false;
        }
        if (__all_sync(kFull, mine)) return true;
        const uint64_t now = global_ns();
        if (t0 == 0) t0 = now;
        else if (now - t0 > p.wait_ns) {
            if (lane == 0) set_status(p, ISD_ERR_TIMEOUT);
            return false;
        }
        __nanosleep(96);
    }
}

// Set a used row's statistic words back to zero for the next call (whole warp).
__device__ __forceinline__ void clear_row(const FusedParams& p, EStat* cs) {
    for (int c = threadIdx.x & 31; c < p.C; c += 32) cs[c] = 0ull;
}

// The anchor rows 0..N-2 of pending sequence b (whole warp): their statistics and p(x) of the
// pending tokens they verify, then the sequence's decisions.  What does not depend on this
// call's work (the pending tokens, their q and logits, the carried statistics of the previous
// call's MASK rows) is read before the rows are waited for; the chunk statistics of
// kAnchorGroup rows are read together.
constexpr int kAnchorGroup = 3;
template <int DT, bool GREEDY>
__device__ __forceinline__ void finish_anchors(const FusedParams& p, const EngineShared& sh, int b) {
    const int lane = threadIdx.x & 31;
    const int N = p.N, R = p.R;
    AnchorLane L;
    L.x = -1;
    L.xq = 0.f;
    L.a = AncStat{0.f, 0.f, -1, 1};
    L.ps_M = L.ap = L.qs_M = L.naq = 0.f;
    L.q_ok = false;
    if (lane < N - 1) {
        L.x = p.pending[(int64_t)b * p.pending_ld + lane];
        if (!GREEDY) {
            L.xq = p.pending_q[(int64_t)b * (N - 1) + lane];
            if (L.x >= 0 && L.x < p.V)
                L.a.xl = load_elem<DT>(row_ptr(p.logits, Elem<DT>::kBytes, (int64_t)b * R + lane, p.V), L.x);
            if (!p.amode && sh.carry) {
                const RowStat qs = load_rowstat_cg(&p.carry[((int64_t)((p.step - 1) & 1) * p.B + b) * (N - 1) + lane]);
                L.q_ok = qs.Zfx > 0ull;
                L.qs_M = L.q_ok ? qs.M : 0.f;
                L.naq = L.q_ok ? -(qs.T / qs.Zf) : 0.f;
            }
        }
    }
    for (int r0 = 0; r0 < N - 1; r0 += kAnchorGroup) {
        float2 cache[kAnchorGroup][kECache];
        if (!poll_rows<kAnchorGroup>(p, p.estat + ((int64_t)b * R + r0) * p.C, p.C, min(kAnchorGroup, N - 1 - r0),
                                     cache))
            return;
#pragma unroll
        for (int j = 0; j < kAnchorGroup; ++j) {
            const int r = r0 + j;
            if (r >= N - 1) break;
            const EStat* cs = p.estat + ((int64_t)b * R + r) * p.C;
            RowStat rs;
            bool ok;
            if (GREEDY) {
                ok = argmax_from_cache(cache[j], cs, p.C, rs);
            } else {
                RowWalk rw;
                ok = combine_from_cache(cache[j], cs, p.C, p.fx, p.s_hi, p.s_lo, rs, rw);
            }
            const int xr = __shfl_sync(kFull, L.x, r);
            const float xlr = __shfl_sync(kFull, L.a.xl, r);
            float pv = 0.f;
            if (!GREEDY && ok && xr >= 0 && xr < p.V) pv = exp2f(weight_exp(xlr, rs.M, p.s_hi, p.s_lo)) / rs.Zf;
            if (lane == r) {
                L.a.pv = pv;
                L.a.amax = ok ? rs.amax : -1;
                L.a.ok = ok ? 1 : 0;
                L.ps_M = rs.M;
                L.ap = ok ? rs.T / rs.Zf : 0.f;
            }
            // a residual at r without carried statistics reads them back once its q row is done
            if (!GREEDY && !sh.carry && lane == 0) p.rowstat[(int64_t)b * R + r] = rs;
        }
    }
    const int keep = decide_sequence<DT, GREEDY>(p, sh, b, L);
    for (int r = 0; r < N - 1; ++r)
        if (r != keep) clear_row(p, p.estat + ((int64_t)b * R + r) * p.C);
}

// A row N-1..2N-2 of a sequence that proposes, all its units done: the draw or argmax, then a
// ticket on the sequence; the last row writes what the sequence's decision left open.
template <int DT, bool GREEDY>
__device__ __forceinline__ void finish_draw(const FusedParams& p, int b, int r, bool has_pending,
                                            const float2 (&cache)[kECache]) {
    const int lane = threadIdx.x & 31;
    const int N = p.N, R = p.R;
    EStat* cs = p.estat + ((int64_t)b * R + r) * p.C;
    const void* row = row_ptr(p.logits, Elem<DT>::kBytes, (int64_t)b * R + r, p.V);
    RowStat rs;
    RowWalk rw;
    const bool ok = GREEDY ? argmax_from_cache(cache, cs, p.C, rs)
                           : combine_from_cache(cache, cs, p.C, p.fx, p.s_hi, p.s_lo, rs, rw);
    if (!ok) {
        if (lane == 0) atomicOr(&p.seqbad[b], 1u);
    } else {
        int t;
        float q = 1.f;  // an argmax proposal's q is a point mass
        if (GREEDY) t = rs.amax;
        else if (p.amode && r >= N) t = argmax_of_row<DT>(p, row, cs, rs.mx);
        else t = draw_from_row<DT>(p, row, cs, rs, rw, row_words(p.seed, p.step, b, r).y, &q);
        if (lane == 0) {
            p.tokens_out[(int64_t)b * R + (r == N - 1 && !has_pending ? 0 : r)] = t;
            if (r >= N) {
                p.new_q[(int64_t)b * (N - 1) + r - N] = q;
                if (!GREEDY) p.carry[((int64_t)(p.step & 1) * p.B + b) * (N - 1) + r - N] = rs;
            }
        }
    }
    clear_row(p, cs);
    if (take_ticket(&p.drawcnt[b], 1u, (unsigned)N)) {
        unsigned bad = 0;
        if (lane == 0) bad = atomicExch(&p.seqbad[b], 0u);
        bad = __shfl_sync(kFull, bad, 0);
        if (bad) {
            fail_outputs(p, b, ISD_ERR_NONFINITE);
        } else if (!has_pending) {
            // no pending tokens: one token from row N-1, then the proposals
            for (int i = 1 + lane; i < N; i += 32) p.tokens_out[(int64_t)b * R + i] = -1;
            if (p.p_out)
                for (int i = lane; i < N - 1; i += 32) p.p_out[(int64_t)b * (N - 1) + i] = 0.f;
            if (lane == 0) {
                p.accepted_len[b] = 1;
                diag_add(p, ISD_DIAG_EMITTED, 1);
                diag_add(p, ISD_DIAG_RECOVERY, 1);
            }
        }
    }
}

// The last unit of a q row (the previous call left no statistics of it): its statistics,
// then the two residual jobs reserved behind it are filled in and published.
__device__ __forceinline__ void finish_qrow(const FusedParams& p, const EngineShared& sh, int b, int r, int slot,
                                            const float2 (&cache)[kECache]) {
    const int K = r - p.N;
    RowStat qs;
    RowWalk rw;
    EStat* cs = p.eqstat + (int64_t)b * p.C;
    const bool ok = combine_from_cache(cache, cs, p.C, p.fx, p.s_hi, p.s_lo, qs, rw);
    clear_row(p, cs);
    if ((threadIdx.x & 31) == 0) {
        const RowStat ps = load_rowstat_cg(&p.rowstat[(int64_t)b * p.R + K]);
        for (int h = 0; h < 2; ++h) {
            JobRec* j = &p.jobs[slot + 1 + h];
            j->ps_M = ps.M;
            j->qs_M = ok ? qs.M : 0.f;
            j->ap = ps.T / ps.Zf;
            j->naq = ok ? -(qs.T / qs.Zf) : 0.f;
            st_release64(&j->head, job_head(sh.epoch, b, K, kUnitResid, h, !ok));
        }
    }
}

// The last unit of a residual: the replacement token.
template <int DT>
__device__ __forceinline__ void finish_residual(const FusedParams& p, const Unit& u, const ResidConst& rc) {
    using E = Elem<DT>;
    const int lane = threadIdx.x & 31;
    const int b = u.b, K = u.r, R = p.R;
    EStat* const ks = p.estat + ((int64_t)b * R + K) * p.C;  // anchor row K's words: cleared here
    if (u.kind < 0) {  // the q row was unusable
        fail_outputs(p, b, ISD_ERR_NONFINITE);
        if (lane == 0) p.rtotal[b] = 0ull;
        clear_row(p, ks);
        return;
    }
    uint64_t total = 0ull;
    if (lane == 0) {
        total = __ldcg(reinterpret_cast<const unsigned long long*>(&p.rtotal[b]));
        p.rtotal[b] = 0ull;
    }
    total = __shfl_sync(kFull, total, 0);
    const uint32_t word = row_words(p.seed, p.step, b, K).y;
    const void* prow = row_ptr(p.logits, E::kBytes, (int64_t)b * R + K, p.V);
    int y;
    if (total == 0ull) {  // no residual mass left (only through rounding): draw from p
        if (lane == 0) diag_add(p, ISD_DIAG_NEAR_TIE_CDF, 1);
        RowStat ps;
        RowWalk rw;
        combine_row_cached(ks, p.C, p.fx, p.s_hi, p.s_lo, ps, rw);
        float px;
        y = draw_from_row<DT>(p, prow, ks, ps, rw, word, &px);
    } else {
        const void* qrow = row_ptr(p.prev, E::kBytes, (int64_t)b * R + p.N + K, p.V);
        const float* hs = p.rsum + (int64_t)b * 2 * p.C;
        const uint64_t target = scale_by_uniform(total, word);
        uint64_t before = 0;
        int last_pos;
        int hstar = walk_chunks(2 * p.C, target, [&](int i) { return to_fixed(__ldcg(&hs[i]), p.fxh); }, &before,
                                &last_pos);
        const bool overshoot = hstar < 0;
        if (overshoot) hstar = last_pos < 0 ? 0 : last_pos;
        const float local = overshoot ? INFINITY : fixed_to_float(target - before, p.fxh);
        constexpr int H = E::kChunk / 2;
        const int64_t e0 = (int64_t)(hstar >> 1) * E::kChunk + (hstar & 1) * H;
        uint4 v[kVec];
        // half a chunk of each row: vectors k < kHalf of this lane, elements past V read as -inf
#pragma unroll
        for (int k = 0; k < kHalf; ++k) {
            const int64_t first = e0 + (int64_t)(k * 32 + lane) * E::kPerVec;
            uint4 a = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord), c = a;
            if (p.vec_ok) {
                if (first < p.V) {
                    a = __ldg(reinterpret_cast<const uint4*>(prow) + first / E::kPerVec);
                    c = __ldg(reinterpret_cast<const uint4*>(qrow) + first / E::kPerVec);
                }
            } else {
                uint32_t* aw = &a.x;
                uint32_t* cw = &c.x;
#pragma unroll
                for (int e = 0; e < E::kPerVec; ++e) {
                    const int64_t idx = first + e;
                    const uint32_t pb = idx < p.V ? E::scalar_bits(prow, idx) : E::kNegInfBits;
                    const uint32_t qb = idx < p.V ? E::scalar_bits(qrow, idx) : E::kNegInfBits;
                    if (DT == ISD_BF16) {
                        aw[e >> 1] = (e & 1) ? ((aw[e >> 1] & 0x0000FFFFu) | (pb << 16)) : ((aw[e >> 1] & 0xFFFF0000u) | pb);
                        cw[e >> 1] = (e & 1) ? ((cw[e >> 1] & 0x0000FFFFu) | (qb << 16)) : ((cw[e >> 1] & 0xFFFF0000u) | qb);
                    } else {
                        aw[e] = pb;
                        cw[e] = qb;
                    }
                }
            }
            v[k] = a;
            v[kHalf + k] = c;
        }
        const float s_hi = p.s_hi;
        const float Mp = rc.ps_M, Mq = rc.qs_M, ap = rc.ap, naq = rc.naq;
        int last;
        int off = rescan_regs<kHalf, E::kPerVec>(
            local, [&](int k) { return make_uint4x2(v[k], v[kHalf + k]); },
            [&](const Uint4x2& x, int j) {
                return residual_elem(vec_elem<DT>(x.a, j), vec_elem<DT>(x.b, j), Mp, Mq, ap, naq, s_hi);
            },
            &last);
        if (off < 0) {
            off = last < 0 ? 0 : last;
            if (lane == 0) diag_add(p, ISD_DIAG_NEAR_TIE_CDF, 1);
        }
        y = (int)(e0 + off);
    }
    if (lane == 0) p.tokens_out[(int64_t)b * R + K] = y;
    clear_row(p, ks);
}

// Whether two units belong to the same job (sequence, row or rejected position, kind; the two
// halves of a residual share one ticket).
__device__ __forceinline__ bool same_job(const PackedUnit& a, const PackedUnit& b) {
    const int m = 0xFFFF | (0x3F << 16) | (7 << 22);
    return (a.info & m) == (b.info & m);
}

// The loop state of one warp of the engine and its two operations, force-inlined so that the
// state stays in registers.
template <int DT, bool GREEDY>
struct EngineWarp {
    PackedUnit c0, c1, c2;  // the units the stages hold (a select picks one: no indexed array)
    unsigned fullm;         // bit d: stage d holds a unit whose copy was issued
    uint32_t phase;         // bit d: parity of stage d's next completion
    int left;               // units left in the current batch
    unsigned long long ahead;  // lane 0: the next batch's first unit, claimed halfway through this one
    bool have_ahead;
    int nc;                 // the next unit's chunk and job slot
    long long nslot;
    long long cslot;        // the job slot last looked up, and its unit
    PackedUnit cunit;
    uint32_t retry_at;      // an unpublished next unit is looked up again after this time (low bits)
    bool no_more;
    // residual units done on one residual, reported with one count
    unsigned tk_n;
    PackedUnit tk_u;
    bool batch_done;

    // The first batch is fixed (units first_unit .. first_unit + kGrab - 1); later batches of
    // kGrab consecutive units come from the counter, each claimed halfway through the batch
    // before it.
    __device__ __forceinline__ void init(const FusedParams& p, long long first_unit) {
        c0 = c1 = c2 = cunit = tk_u = PackedUnit{0, 0, -1};
        fullm = 0u;
        phase = 0u;
        left = kGrab;
        ahead = 0ull;
        have_ahead = false;
        nslot = div_rem(first_unit, p.C, &nc);
        cslot = -1;
        retry_at = 0u;
        no_more = false;
        tk_n = 0u;
        batch_done = false;
    }

    __device__ __forceinline__ PackedUnit unit_of(int d) const { return d == 0 ? c0 : (d == 1 ? c1 : c2); }

    // Fill stage d with the next unit if its job is known (whole warp).
    __device__ __forceinline__ void fill(const FusedParams& p, const EngineShared& sh, int d, bool check_end,
                                         unsigned char* stage0, uint32_t bar0, uint64_t pol, long long first_all) {
        const int lane = threadIdx.x & 31;
        if (no_more) return;
        if (!check_end && retry_at != 0u && (int32_t)((uint32_t)global_ns() - retry_at) < 0) return;
        if (left == 0) {
            unsigned long long base = ahead;
            if (!have_ahead && lane == 0)
                base = atomicAdd(&p.eng->claim.v, (unsigned long long)kGrab) + (unsigned long long)first_all;
            have_ahead = false;
            left = kGrab;
            nslot = div_rem((long long)__shfl_sync(kFull, base, 0), p.C, &nc);
        }
        Unit u;
        if (nslot == cslot) {  // the job of the previous unit: nothing to look up
            u = unpack_unit(cunit);
        } else {
            const int st = resolve_slot(p, sh, nslot, u, check_end);
            if (st == kNoMore) {
                no_more = true;
                return;
            }
            if (st == kNotYet) {
                retry_at = ((uint32_t)global_ns() + 400u) | 1u;
                return;
            }
            cslot = nslot;
            cunit = pack_unit(u, false);
        }
        u.c = nc;
        retry_at = 0u;
        if (--left == kGrab / 2 && !have_ahead) {
            // claim the next batch now: the atomic's round trip overlaps this batch's work
            if (lane == 0) ahead = atomicAdd(&p.eng->claim.v, (unsigned long long)kGrab) + (unsigned long long)first_all;
            have_ahead = true;
        }
        const bool batch_end = left == 0;
        if (++nc == p.C) {
            nc = 0;
            ++nslot;
        }
        issue_unit<DT>(p, u, stage0 + d * kChunkBytes, bar0 + 8 * d, pol);
        const PackedUnit pu = pack_unit(u, batch_end);
        if (d == 0) c0 = pu;
        else if (d == 1) c1 = pu;
        else c2 = pu;
        fullm |= 1u << d;
    }

    // Report the residual units done (whole warp): a release add to the residual's counter,
    // which its finishing warp waits on.
    __device__ __forceinline__ void flush(const FusedParams& p) {
        if (tk_n == 0u) return;
        if ((threadIdx.x & 31) == 0) red_add_release(&p.rescnt[unpack_unit(tk_u).b], tk_n);
        tk_n = 0u;
    }
};

// The step's counters, reset by the last warp to leave, which also names the next call (the
// epoch skips 0xFFFFFFFF, so that a tag, epoch + 1, is never the zero of a cleared flag).
__device__ __forceinline__ void reset_counters(const FusedParams& p, const EngineShared& sh) {
    p.eng->claim.v = 0ull;
    p.eng->dyn_count = 0u;
    p.eng->dec_done = 0u;
    p.eng->exit_count = 0u;
    p.eng->epoch = sh.epoch + 1u == 0xFFFFFFFFu ? 0u : sh.epoch + 1u;
}

// Wait (whole warp) for the decision of sequence b; returns its outcome, or 0 after the wait
// limit (timeout status set).
__device__ __forceinline__ unsigned wait_decision(const FusedParams& p, const EngineShared& sh, int b) {
    unsigned out = 0u;
    if ((threadIdx.x & 31) == 0) {
        uint64_t t0 = 0;
        for (;;) {
            const unsigned long long w = ld_acquire64(&p.decw[b]);
            if ((uint32_t)(w >> 32) == sh.tag) {
                out = (uint32_t)w;
                break;
            }
            const uint64_t now = global_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > p.wait_ns) {
                set_status(p, ISD_ERR_TIMEOUT);
                break;
            }
            __nanosleep(128);
        }
    }
    return __shfl_sync(kFull, out, 0);
}

// Wait (whole warp) for published job k; false when there is none and will be none (every
// decision made, k past the reserved slots), or after the wait limit (timeout status set).
__device__ __forceinline__ bool wait_published(const FusedParams& p, const EngineShared& sh, long long k,
                                               unsigned long long& head) {
    int ok = 0;
    unsigned long long h = 0ull;
    if ((threadIdx.x & 31) == 0 && k < p.jobs_cap) {
        uint64_t t0 = 0;
        for (;;) {
            h = ld_acquire64(&p.jobs[k].head);
            if ((uint32_t)(h >> 32) == sh.epoch && ((uint32_t)h & kHeadValid)) {
                ok = 1;
                break;
            }
            if (ld_acquire(&p.eng->dec_done) == (unsigned)sh.P && k >= (long long)ld_acquire(&p.eng->dyn_count)) break;
            const uint64_t now = global_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > p.wait_ns) {
                set_status(p, ISD_ERR_TIMEOUT);
                break;
            }
            __nanosleep(128);
        }
    }
    head = __shfl_sync(kFull, h, 0);
    return __shfl_sync(kFull, ok, 0) != 0;
}

// Finishing warp f of F (whole warp): jobs f + i*F, in order.  Job j < P: the anchor rows of
// the j-th sequence with pending tokens; then, from P on, the rows N-1..2N-2 in the order of
// the row jobs; then the published jobs in slot order.
template <int DT, bool GREEDY>
__device__ __forceinline__ void run_finisher(const FusedParams& p, const EngineShared& sh, int f, int F) {
    const long long rows_end = (long long)sh.P + (long long)p.B * p.N;
    for (long long j = f;; j += F) {
        if (j < sh.P) {
            finish_anchors<DT, GREEDY>(p, sh, kth_sequence(sh, p.B, (int)j, true));
            continue;
        }
        if (j < rows_end) {
            int b, r;
            const int group = row_job(p, sh, sh.A + (j - sh.P), b, r);
            bool draw = true;
            if (group == 2) {  // read ahead of the decision: drawn from only if it says so
                const unsigned out = wait_decision(p, sh, b);
                if (out == 0u) return;
                draw = out == kDecDraw;
            }
            float2 cache[1][kECache];
            EStat* cs = p.estat + ((int64_t)b * p.R + r) * p.C;
            if (!poll_rows<1>(p, cs, 0, 1, cache)) return;
            if (draw) finish_draw<DT, GREEDY>(p, b, r, group == 2, cache[0]);
            else clear_row(p, cs);  // every unit has said "done": set the words back to zero
            continue;
        }
        const long long k = j - rows_end;
        unsigned long long head;
        if (!wait_published(p, sh, k, head)) return;
        const uint32_t lo = (uint32_t)head;
        const int b = (int)(lo & 0xFFFFu), r = (int)((lo >> 16) & 0x3Fu);
        const int kind = (int)((lo >> 24) & 3u), half = (int)((lo >> 23) & 1u);
        if (kind == kUnitQRow) {
            float2 cache[1][kECache];
            if (!poll_rows<1>(p, p.eqstat + (int64_t)b * p.C, 0, 1, cache)) return;
            finish_qrow(p, sh, b, r, (int)k, cache[0]);
        } else if (half == 1) {  // a residual is finished once, with its second half
            // (its constants were written before its head, which was read with acquire semantics)
            const ResidConst rc = load_resid_const(&p.jobs[k]);
            if (!wait_count(p, &p.rescnt[b], (unsigned)(2 * p.C))) return;
            Unit u;
            u.b = b;
            u.r = r;
            u.c = 0;
            u.half = 1;
            u.slot = (int)k;
            u.kind = (lo & kHeadSkip) ? kUnitSkipResid : kUnitResid;
            finish_residual<DT>(p, u, rc);
        }
    }
}

// ----------------------------------------------------------------------------------------
// the kernel
// ----------------------------------------------------------------------------------------
template <int DT, bool GREEDY>
__global__ void __launch_bounds__(kEThreads, 1) isd_fused_step_kernel(const FusedParams params) {
    using E = Elem<DT>;
    extern __shared__ __align__(128) unsigned char s_stage[];  // [kEStreamers][kEDepth][kChunkBytes]
    __shared__ __align__(8) uint64_t s_bar[kEWarps][kEDepth];
    __shared__ EngineShared sh;
    // The parameters live in shared memory: the finishing functions take them by reference,
    // which would otherwise give the kernel's parameters a copy in local memory.
    __shared__ __align__(16) FusedParams s_params;
    if (threadIdx.x == 0) s_params = params;
    __syncthreads();
    const FusedParams& p = s_params;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char* stage = s_stage + (size_t)warp * kEDepth * kChunkBytes;
    const uint32_t bar = smem_u32(&s_bar[warp][0]);
    if (lane == 0) {
        for (int d = 0; d < kEDepth; ++d) mbar_init(bar + 8 * d, 1);
        fence_mbar_init();
    }
    // which sequences have pending tokens, and how many before each 32
    const int nw = (p.B + 31) >> 5;
    for (int w = warp; w < nw; w += kEWarps) {
        const int b = 32 * w + lane;
        const unsigned word = __ballot_sync(kFull, b < p.B && p.pending[(int64_t)b * p.pending_ld] >= 0);
        if (lane == 0) sh.mask[w] = word;
    }
    const int slot_read = (int)((p.step - 1) & 1), slot_write = (int)(p.step & 1);
    if (threadIdx.x == kEThreads - 1) {
        int use = 0;
        if (!GREEDY) {  // were the q rows' statistics left by the call that produced prev_logits?
            const CarryKey k = p.carry_key[slot_read];
            use = k.tag == kCarryTag && k.logits == p.prev && k.step + 1 == p.step && k.B == p.B && k.N == p.N &&
                  k.V == p.V && k.dtype == p.dtype && k.s_hi == p.s_hi && k.s_lo == p.s_lo;
        }
        sh.carry = use;
        sh.epoch = *(volatile unsigned*)&p.eng->epoch;
        sh.tag = sh.epoch + 1u;
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
    __syncthreads();
    if (warp == 0) {
        int cnt[8];
        int tot = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int w = lane * 8 + i;
            cnt[i] = w < nw ? __popc(sh.mask[w]) : 0;
            tot += cnt[i];
        }
        int incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        int run = incl - tot;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int w = lane * 8 + i;
            if (w < nw) sh.pre[w] = run;
            run += cnt[i];
        }
        if (lane == 31) {
            sh.pre[nw] = incl;
            sh.nwords = nw;
            sh.P = incl;
            sh.A = (p.N - 1) * incl;
            sh.D0 = sh.A + p.N * (p.B - incl);
            sh.S0 = sh.A + p.N * p.B;
        }
    }
    __syncthreads();
    if (warp >= kEStreamers) {  // a finishing warp
        run_finisher<DT, GREEDY>(p, sh, blockIdx.x * kEFinishers + warp - kEStreamers, gridDim.x * kEFinishers);
        if (lane == 0 && atom_add_acq_rel(&p.eng->exit_count, 1u) == gridDim.x * kEWarps - 1u) reset_counters(p, sh);
        return;
    }
    const uint64_t pol = evict_first_policy();
    const long long first_all = (long long)gridDim.x * kEStreamers * kGrab;
    EngineWarp<DT, GREEDY> w;
    w.init(p, ((long long)blockIdx.x * kEStreamers + warp) * kGrab);
    unsigned char* const stage0 = stage;
    uint64_t idle_since = 0;
    bool timed_out = false;
    int d = 0;
    // One pass per stage in turn: take the stage's unit into registers, refill the stage, then
    // work on the unit.  The stages start empty; the first passes fill them.  Each place of the
    // loop appears once, so that the loop stays small in the instruction cache.
    for (;;) {
        const bool full = (w.fullm >> d) & 1u;
        const PackedUnit pu = w.unit_of(d);
        const Unit u = unpack_unit(pu);
        const bool nothing = !full && w.fullm == 0u;  // no copy in flight in any stage
        // report the residual units done: at the end of a batch, before a unit of another job,
        // and before waiting for work
        if (w.tk_n && (w.batch_done || nothing || (full && !same_job(pu, w.tk_u)))) w.flush(p);
        w.batch_done = false;
        const bool resid = u.kind == kUnitResid || u.kind == kUnitSkipResid;
        uint4 v[kVec];
        if (full) {
            if (p.vec_ok && !__all_sync(kFull, mbar_wait_bounded(bar + 8 * d, (w.phase >> d) & 1u, p.wait_ns))) {
                timed_out = true;
                break;
            }
            if (p.vec_ok) w.phase ^= 1u << d;
            const uint4* sv = reinterpret_cast<const uint4*>(stage0 + d * kChunkBytes);
            if (resid) {
                constexpr int H = E::kChunk / 2;
                const int n =
                    (int)max((int64_t)0, min((int64_t)H, (int64_t)p.V - ((int64_t)u.c * E::kChunk + u.half * H)));
#pragma unroll
                for (int k = 0; k < kHalf; ++k) {
                    const bool in = (k * 32 + lane) * E::kPerVec < n;
                    const uint4 ninf = make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
                    v[k] = in ? sv[k * 32 + lane] : ninf;
                    v[kHalf + k] = in ? sv[kHalf * 32 + k * 32 + lane] : ninf;
                }
            } else if ((int64_t)(u.c + 1) * E::kChunk <= (int64_t)p.V) {  // a whole chunk
#pragma unroll
                for (int k = 0; k < kVec; ++k) v[k] = sv[k * 32 + lane];
            } else {  // the row's last chunk: -inf past V
                const int n = (int)((int64_t)p.V - (int64_t)u.c * E::kChunk);
#pragma unroll
                for (int k = 0; k < kVec; ++k)
                    v[k] = (k * 32 + lane) * E::kPerVec < n
                               ? sv[k * 32 + lane]
                               : make_uint4(E::kNegInfWord, E::kNegInfWord, E::kNegInfWord, E::kNegInfWord);
            }
            __syncwarp();
            w.fullm &= ~(1u << d);
        }
        // refill the stage before working on the unit in registers; with nothing in flight, also
        // learn whether more work will come
        w.fill(p, sh, d, nothing, stage0, bar, pol, first_all);
        if (full) {
            idle_since = 0;
            if (u.kind == kUnitSkipRow) {
                // a row its sequence's decision leaves unread: its word only says "done"
                if (lane == 0) st_relaxed64(&p.estat[((int64_t)u.b * p.R + u.r) * p.C + u.c], kSkippedChunk);
            } else if (!resid) {  // a chunk of a row of logits, or of a q row of the previous logits
                const float2 st = GREEDY ? chunk_stat_argmax<DT>(v, (int64_t)u.c * E::kChunk)
                                         : chunk_stat_sample<DT>(v, p.s_hi, p.s_lo);
                if (lane == 0)
                    st_relaxed64(u.kind == kUnitRow ? &p.estat[((int64_t)u.b * p.R + u.r) * p.C + u.c]
                                                    : &p.eqstat[(int64_t)u.b * p.C + u.c],
                                 enc_stat(st));
            } else {
                const float sum =
                    u.kind == kUnitResid ? residual_half_sum<DT>(v, load_resid_const(&p.jobs[u.slot]), p.s_hi) : 0.f;
                if (lane == 0) {
                    p.rsum[(int64_t)u.b * 2 * p.C + 2 * u.c + u.half] = sum;
                    atomicAdd(reinterpret_cast<unsigned long long*>(&p.rtotal[u.b]),
                              (unsigned long long)to_fixed(sum, p.fxh));
                }
            }
            if (resid) {  // residual units are counted (their sums are added up by atomics)
                w.tk_u = pu;
                ++w.tk_n;
            }
            w.batch_done = batch_end_of(pu);
        } else if (nothing && !((w.fullm >> d) & 1u)) {
            // nothing in flight and no unit to start: done, or wait for a decision to publish one
            if (w.no_more) break;
            const uint64_t now = global_ns();
            if (idle_since == 0) idle_since = now;
            else if (now - idle_since > p.wait_ns) {
                timed_out = true;
                break;
            }
            __nanosleep(256);
        }
        d = d + 1 == kEDepth ? 0 : d + 1;
    }
    // (leaving normally, the last pass found nothing in flight and nothing to report)
    const unsigned fullm = w.fullm;
    const uint32_t phase = w.phase;
    if (timed_out) {
        if (lane == 0) set_status(p, ISD_ERR_TIMEOUT);
        // let the copies still in flight land before the CTA's shared memory is released
        if (p.vec_ok)
            for (int s = 0; s < kEDepth; ++s)
                if ((fullm >> s) & 1u) mbar_wait_bounded(bar + 8 * s, (phase >> s) & 1u);
    }
    // the last warp to leave resets the counters and names the next call's job records
    if (lane == 0 && atom_add_acq_rel(&p.eng->exit_count, 1u) == gridDim.x * kEWarps - 1u) reset_counters(p, sh);
}
