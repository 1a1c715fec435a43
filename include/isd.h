/*
 * isd.h -- C ABI of the B300 (sm_103a) Introspective Strided Decoding step.
 *
 * The operation ("Introspective Diffusion Language Models"; ai.arkapp.pw blog,
 * section "I-DLM 如何解決這些問題"; de.news.hada.io, "Inference & ISD" and
 * "Speedup Factor Explorer"; zhuanzhiai.com, introduction):
 * one forward of B sequences gives 2N-1 logit rows per sequence.  The clean
 * rows verify the N-1 tokens proposed on the previous step: pending token x_i
 * is kept with probability min(1, p(x)/q(x)), p = softmax(clean row i-1 / T)
 * the anchor distribution and q(x) the proposal probability saved when x was
 * drawn.  At the first rejection the replacement token is drawn from the
 * normalised residual max(0, p - q) and the remaining proposals are dropped;
 * if all N-1 are kept, one more token is drawn from clean row N-1.  When the
 * sequence ends the step with a valid prefix (all kept, or it had no pending
 * tokens), the MASK rows propose the next N-1 tokens and their q is saved.
 * So a forward emits 1..N tokens, and tokens per forward follows the pages'
 * closed form (2+p+...+p^(N-2)) / (2-p^(N-1)).
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" are device memory owned by the caller; the
 *    library allocates nothing and keeps no pointer after the call returns.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  Argument errors are detected on the host, return a
 *    negative isd_status and launch nothing.  Conditions found on the device
 *    (non-finite logits, an unusable pending state) are written to diag and
 *    to the affected sequence's outputs, visible once the stream has synced.
 *  - Layout of logits: [B][2N-1][V], row-major, V contiguous.  Row r of
 *    sequence b starts at element (b*(2N-1) + r)*V.
 *      rows 0..N-2  clean rows; row i-1 is the anchor for pending token x_i
 *      row  N-1     clean anchor row for the token after the pending ones
 *      rows N..2N-2 MASK rows; row N-1+j proposes the j-th next token
 *  - Rows read: a sequence with pending tokens reads its anchor rows 0..N-2;
 *    one that then keeps all of them, or has none, reads rows N-1..2N-2; one
 *    that rejects at K reads instead (sampling mode) the previous call's MASK
 *    row N+K, and never its rows N-1..2N-2, whose proposals a rejection would
 *    discard.  A row holding NaN or +Inf, or only -Inf, fails the sequence
 *    (ISD_ERR_NONFINITE) only if the sequence reads it.
 *  - Randomness: Philox4x32-10 (Salmon et al., SC'11) with key =
 *    (seed low, seed high) and counter = (step low, step high, b, row).
 *    Word 0 gives the acceptance uniform of that row, word 1 the inverse-CDF
 *    uniform of that row; u = (word >> 8) * 2^-24.
 *  - Inverse CDF: the smallest token index i with w_0+...+w_i > u*sum(w).
 *  - Greedy mode (ISD_GREEDY): argmax (lowest index on ties) replaces every
 *    draw; a pending token is kept iff it is the argmax of its anchor row; the
 *    saved q of an argmax proposal is 1.  Temperature is ignored.
 *  - Argmax-proposal mode (ISD_ARGMAX_PROPOSE): the proposals are argmax
 *    (saved q = 1); verification, the replacement after a rejection and the
 *    token after the pending ones are sampled at the temperature.
 *  - The fast path wants V*sizeof(element) to be a multiple of 16 bytes and
 *    16-byte aligned logits; other shapes run a scalar-load path.
 */
#ifndef ISD_B300_ISD_H
#define ISD_B300_ISD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ISD_OK = 0,
    ISD_ERR_INVALID_ARG = -1, /* host-side argument check failed; nothing launched */
    ISD_ERR_CUDA = -2,        /* a CUDA runtime call failed */
    ISD_ERR_NONFINITE = -3,   /* device: a row the step reads holds NaN/+Inf or is all -Inf */
    ISD_ERR_WORKSPACE = -4,   /* workspace missing, misaligned or smaller than isd_workspace_size */
    ISD_ERR_TIMEOUT = -5,     /* device: a bounded wait gave up (~1 s; see isd_debug_set_wait_limit_ns) */
    ISD_ERR_BAD_PENDING = -6, /* device: pending token outside [0,V) or pending q not in (0,inf) */
    ISD_ERR_SCRATCH_LIMIT = -7 /* isd_step_noalloc: the sizes need more than its static scratch */
} isd_status;

typedef enum { ISD_BF16 = 0, ISD_F32 = 1 } isd_dtype;

/* Words of the optional diag array (int32, device).  They accumulate across
 * calls (zero them to start counting) except ISD_DIAG_STATUS, which keeps the
 * first device-side error code seen (0 while none). */
enum {
    ISD_DIAG_STATUS = 0,       /* 0 or a negative isd_status found on the device */
    ISD_DIAG_ACCEPTS = 1,      /* pending tokens accepted */
    ISD_DIAG_TESTS = 2,        /* acceptance tests made */
    ISD_DIAG_NEAR_TIE_ACC = 3, /* tests with |u - p/q| < 1e-6 in the kernel's arithmetic */
    ISD_DIAG_NEAR_TIE_CDF = 4, /* draws within 1e-6 (relative) of a CDF edge */
    ISD_DIAG_RESIDUALS = 5,    /* replacement tokens drawn from the residual */
    ISD_DIAG_RECOVERY = 6,     /* sequences that had no pending tokens */
    ISD_DIAG_EMITTED = 7,      /* tokens emitted (sum of accepted_len) */
    ISD_DIAG_WORDS = 8
};

/* Largest supported stride: N-1 pending tokens are tested by one warp. */
/* Values of the `greedy` argument of the step calls. */
enum {
    ISD_SAMPLE = 0,          /* sampled proposals, sampled verification */
    ISD_GREEDY = 1,          /* argmax everywhere (temperature unused) */
    ISD_ARGMAX_PROPOSE = 2   /* argmax proposals (q = 1) verified by sampling */
};

#define ISD_MAX_N 32

/* Bytes of device workspace isd_step needs for these sizes (0 on bad sizes).
 * The workspace holds per-chunk and per-row statistics that live within one
 * call, the statistics pass's work counter, and a keyed cache that one call
 * leaves for the next (see isd_step, "workspace").  It must be zero-filled once
 * before its first use (isd_workspace_init or cudaMemset), and again when it is
 * used for other sizes; every call leaves its counter at zero again, except
 * after a call that reported ISD_ERR_TIMEOUT, which may leave it anywhere:
 * zero-fill the workspace again before the next call.  One workspace serves
 * one stream at a time. */
size_t isd_workspace_size(int B, int N, int V, int dtype);

/* Zero-fill a workspace on `stream` (asynchronous).  Returns ISD_OK or
 * ISD_ERR_CUDA. */
int isd_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * isd_step -- one verify-and-propose step for B sequences.
 *
 * logits          device, [B][2N-1][V] of `dtype` (ISD_BF16 or ISD_F32).
 * prev_logits     device, the previous step's logits (same shape).  Its MASK
 *                 row N+K gave the q row of a pending token rejected at
 *                 position K, needed by the residual draw.  May be NULL only
 *                 in the ISD_GREEDY and ISD_ARGMAX_PROPOSE modes or when no
 *                 sequence has pending tokens.
 * pending_tokens  device int32, B rows of N-1 tokens at row stride pending_ld;
 *                 pending_tokens[b*pending_ld] < 0 means sequence b has no
 *                 pending tokens (it emits one token from row N-1 and
 *                 proposes afresh).
 * pending_ld      row stride of pending_tokens in elements (>= N-1).  Passing
 *                 the previous call's tokens_out + N with pending_ld = 2N-1
 *                 chains steps without a copy.
 * pending_q       device float [B][N-1]; q(x) saved when each pending token
 *                 was drawn.  Unused in ISD_GREEDY mode.
 * B, N, V         1 <= B, 2 <= N <= ISD_MAX_N, 1 <= V < 2^31 / (2N-1) per sequence.
 * temperature     > 0 unless ISD_GREEDY; applied to p and q alike.
 * greedy          ISD_SAMPLE (0): proposals drawn by sampling, kept with
 *                 min(1, p/q), a rejection resampled from norm(max(0, p - q));
 *                 ISD_GREEDY (1): argmax everywhere;
 *                 ISD_ARGMAX_PROPOSE (2): proposals are the argmax of their MASK
 *                 row (saved q = 1, a point mass), verified by sampling: x is
 *                 kept with probability p(x), and a rejection is resampled from
 *                 p without x (ai.arkapp.pw blog, section "實際部署：SGLang 整合",
 *                 names argmax proposals); prev_logits is not read.  Other
 *                 values are an argument error.
 * philox_seed, step  Philox key and the step half of its counter.
 * accepted_len    device int32 [B]: tokens emitted by sequence b (1..N);
 *                 0 if the sequence hit a device-side error.
 * tokens_out      device int32 [B][2N-1]: entries [0, accepted_len) are the
 *                 emitted tokens, the rest of [0, N) is -1; entries [N, 2N-1)
 *                 are the new pending tokens, or all -1 after a rejection.
 * new_q           device float [B][N-1]: q of each new pending token (0 where
 *                 none; 1 for argmax proposals).
 * p_out           device float [B][N-1] or NULL: anchor p(x_i) of each pending
 *                 token (0 for sequences without pending tokens, and in
 *                 ISD_GREEDY mode).
 * diag            device int32 [ISD_DIAG_WORDS] or NULL (see above).
 * workspace       device, at least isd_workspace_size(B,N,V,dtype) bytes,
 *                 256-byte aligned, zero-filled before its first use.  A
 *                 sampling call leaves in it the
 *                 statistics (max, normaliser) of its MASK rows, keyed by its
 *                 logits pointer, step, B, N, V, dtype and temperature.  The
 *                 next call uses them for the q row of a rejected token when
 *                 its prev_logits is that logits pointer and its step is that
 *                 step + 1 (the sizes and temperature equal); otherwise it
 *                 reads the q row again, with the same result.  So a logits
 *                 buffer must not be rewritten while it may still be passed
 *                 as prev_logits.
 * stream          cudaStream_t or NULL.
 * Outputs must not overlap any input (use two sets of state buffers and
 * alternate them between steps).
 * Returns ISD_OK once the work is enqueued, or a negative isd_status.
 */
int isd_step(const void* logits, const void* prev_logits, int dtype,
             const int32_t* pending_tokens, int pending_ld, const float* pending_q,
             int B, int N, int V, float temperature, int greedy,
             uint64_t philox_seed, uint64_t step,
             int32_t* accepted_len, int32_t* tokens_out, float* new_q,
             float* p_out, int32_t* diag,
             void* workspace, size_t workspace_bytes, void* stream);

/*
 * isd_step_noalloc -- isd_step for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point; it only changes where the
 * scratch memory comes from.  Some callers cannot call cudaMalloc at the point
 * where they run the step: for example a plug-in inside a host runtime that has
 * taken the device memory for its own pool and hands the plug-in nothing but
 * its input and output buffers, or a caller on a latency-critical path where an
 * allocation, which may synchronise the whole device, is not allowed.
 *
 * Arguments are those of isd_step without workspace/workspace_bytes.  The
 * scratch is one array of ISD_STATIC_SCRATCH_BYTES bytes of static device
 * memory inside the library; every GPU that loads the library holds it until
 * the process exits.  Nothing is allocated: no cudaMalloc, cudaFree or
 * allocating library routine is called.
 *  - The first call on a device (made with that device current) looks up the
 *    array's device address; make that first call before any stream capture.
 *  - Sizes whose workspace (isd_workspace_size) exceeds ISD_STATIC_SCRATCH_BYTES
 *    return ISD_ERR_SCRATCH_LIMIT and enqueue nothing.
 *  - Every call shares the one array and it keeps the last calls' contents.
 *    A call reads what an earlier call left only through the keyed cache of
 *    MASK-row statistics that isd_step describes under "workspace"; whatever
 *    must start at zero is cleared by the call (an asynchronous memset on
 *    `stream`).  Calls that may overlap on the GPU (different
 *    streams, or several host threads) race on the array and give wrong
 *    results; serialise them.
 * Returns what isd_step returns, or ISD_ERR_SCRATCH_LIMIT, or ISD_ERR_CUDA.
 */
#define ISD_STATIC_SCRATCH_BYTES (8u << 20)
int isd_step_noalloc(const void* logits, const void* prev_logits, int dtype,
                     const int32_t* pending_tokens, int pending_ld, const float* pending_q,
                     int B, int N, int V, float temperature, int greedy,
                     uint64_t philox_seed, uint64_t step,
                     int32_t* accepted_len, int32_t* tokens_out, float* new_q,
                     float* p_out, int32_t* diag, void* stream);

/*
 * isd_step_fused -- isd_step as one persistent kernel.
 *
 * The pages count launch overhead among the serving costs (ai.arkapp.pw blog,
 * section "實際部署：SGLang 整合": CUDA-graph capture and a stationary batch
 * loop).  isd_step launches two kernels per step, a statistics pass over every
 * row it reads and then a decision pass; this entry point runs the whole step
 * in one launch.  The CTAs stream 4 KB chunks of the rows; a sequence's
 * decisions run, on a few finishing warps, as soon as its anchor rows are
 * summarised, while other rows still stream; a rejection's residual is
 * streamed as two more jobs of the same kernel.  The finishing warps wait for
 * rows that other CTAs stream; every such wait is bounded (about one second,
 * or the limit set by isd_debug_set_wait_limit_ns) and then reports
 * ISD_ERR_TIMEOUT.  The grid is at most one CTA per SM, so all of its CTAs are
 * resident together when nothing else runs on the device; a kernel of another
 * stream that holds SMs delays some of them, and if that lasts past the wait
 * limit the call reports ISD_ERR_TIMEOUT.
 *
 * Arguments, results, the modes, the rows read and the MASK-row statistics
 * kept for the next call are those of isd_step, with one difference: the
 * workspace must hold isd_fused_workspace_size(B, N, V, dtype) bytes.  It is
 * zero-filled before its first use, and again after a call that reported
 * ISD_ERR_TIMEOUT, or before it is used by isd_step instead (the two entry
 * points keep different state in it).  Both compute the same step, but some
 * sums are rounded in a different order (here the residual's sums are formed
 * over half chunks), so a draw whose target lies within rounding of an edge of
 * the CDF may take the neighbouring token in one of them; the tests hold both
 * to the same parity rule against the fp64 oracle.  isd_step is the faster of
 * the two on a B300 at the sizes measured (B=64, N=4, V=151936).
 */
size_t isd_fused_workspace_size(int B, int N, int V, int dtype);
int isd_step_fused(const void* logits, const void* prev_logits, int dtype,
                   const int32_t* pending_tokens, int pending_ld, const float* pending_q,
                   int B, int N, int V, float temperature, int greedy,
                   uint64_t philox_seed, uint64_t step,
                   int32_t* accepted_len, int32_t* tokens_out, float* new_q,
                   float* p_out, int32_t* diag,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * isd_lm_head -- the LM-head projection that turns one forward's final hidden
 * states into the logit rows the step reads ("Introspective Diffusion Language
 * Models", ai.arkapp.pw blog, section "I-DLM 如何解決這些問題": the clean and
 * MASK positions of a sequence are scored by one forward, whose output layer
 * this is).
 *
 * logits[m][v] = bf16_round( sum_k hidden[m][k] * lm_head[v][k] ), the sum
 * accumulated in fp32 on the tensor cores, rounded to nearest-even bf16 once.
 * hidden   device bf16 [M][K], row-major (K contiguous), 16-byte aligned.
 * lm_head  device bf16 [V][K], row-major (the weight as [vocab][hidden]),
 *          16-byte aligned; streamed from memory once per block of 448 rows of
 *          hidden.
 * M, K, V  M >= 1 query rows, K >= 8 and a multiple of 8, V >= 1.
 * logits   device bf16 [M][V], row-major; fully written.  Must not overlap the
 *          inputs.
 * status   device int32 or NULL: if a bounded wait inside the kernel gave up
 *          (about one second), ISD_ERR_TIMEOUT is stored there unless it
 *          already holds a nonzero code; the logits are then incomplete.
 * stream   cudaStream_t or NULL.
 * Returns ISD_OK once enqueued, ISD_ERR_INVALID_ARG on bad sizes or
 * alignment (nothing launched), ISD_ERR_CUDA if a launch or tensor-map
 * encoding failed.
 */
int isd_lm_head(const void* hidden, const void* lm_head, int M, int K, int V,
                void* logits, int32_t* status, void* stream);

/* Kernel launches enqueued by the last isd_lm_head or isd_step_from_hidden
 * (projection and statistics merge; not the step's own) on this process: one
 * projection per block of 448 query rows. */
int isd_lm_head_last_launch_count(void);

/*
 * isd_step_from_hidden -- the LM-head projection and the step, on one stream:
 * the hidden states of one forward in, the step's decisions out.  The
 * projection's epilogue computes the softmax statistics of every logit row from
 * the accumulator (so the step's statistics pass over the logits is skipped);
 * the logits are still stored, because the draws and the residual read whole
 * rows.
 *
 * hidden   device bf16 [B][2N-1][K]: the final hidden state of every clean and
 *          MASK position of the forward, rows in the logits' row order.
 * lm_head  device bf16 [V][K].
 * K        hidden size (a multiple of 8).
 * logits   device bf16 [B][2N-1][V], written by the projection and then read by
 *          the step.  Keep it unchanged until the next step has run: pass it
 *          there as prev_logits (alternate two such buffers).  In the
 *          ISD_GREEDY mode nothing reads whole rows, so the logits are not
 *          stored (the buffer is left as it was).
 * workspace  device, at least isd_from_hidden_workspace_size(B, N, V) bytes,
 *          256-byte aligned, zero-filled before its first use; it holds an
 *          isd_step workspace (with the same carry semantics) and the
 *          projection's per-tile statistics.
 * The remaining arguments are those of isd_step with dtype = ISD_BF16.  A
 * bounded-wait failure of the projection is reported in diag[ISD_DIAG_STATUS]
 * (diag may be NULL, then it is not reported).
 * Returns as isd_lm_head and isd_step.
 */
size_t isd_from_hidden_workspace_size(int B, int N, int V);
int isd_step_from_hidden(const void* hidden, const void* lm_head, int K, void* logits,
                         const void* prev_logits,
                         const int32_t* pending_tokens, int pending_ld, const float* pending_q,
                         int B, int N, int V, float temperature, int greedy,
                         uint64_t philox_seed, uint64_t step,
                         int32_t* accepted_len, int32_t* tokens_out, float* new_q,
                         float* p_out, int32_t* diag,
                         void* workspace, size_t workspace_bytes, void* stream);

/* A short English description of a status code (static storage). */
const char* isd_status_string(int status);

/* Number of kernel launches the last isd_step (or isd_step_fused) on this host
 * thread enqueued. */
int isd_last_launch_count(void);

/*
 * Kernel timing for measurement (not needed to run the step).
 * isd_profile_begin(capacity): from now on, each kernel launch of isd_step
 * and isd_lm_head (up to `capacity` launches) is bracketed by a pair of CUDA timing events
 * on its stream; under stream capture the events become graph nodes and are
 * re-recorded on every replay.  Returns ISD_OK, ISD_ERR_INVALID_ARG or
 * ISD_ERR_CUDA.
 * isd_profile_read(kind, &total_ms, &launches): synchronizes the recorded
 * events and sums the durations of kernels of one kind (0 = the statistics
 * pass of isd_step, 1 = the decision pass of isd_step and isd_step_from_hidden,
 * 2 = the LM-head projection, 3 = the merge of the projection's per-tile
 * statistics, 4 = the kernel of isd_step_fused).  While a session is open the
 * decision pass is not launched as a programmatic dependent, so that each
 * kernel is timed on its own.
 * isd_profile_end(): stops recording and frees the events.
 * Not thread-safe; one profiling session per process at a time.
 */
int isd_profile_begin(int capacity);
int isd_profile_read(int kind, double* total_ms, int* launches);
void isd_profile_end(void);

/*
 * Testing hook (not needed to run the step): how long a bounded device wait of
 * isd_step, isd_step_noalloc and isd_step_fused lasts before it gives up and the
 * call reports
 * ISD_ERR_TIMEOUT in diag (ns; 0 restores the default of about one second).  A
 * test shortens it to make a wait run out on purpose, without faulting or
 * hanging anything: the kernel lets its copies in flight land, leaves, and a
 * later call with the default limit works normally once the workspace has been
 * zero-filled again (isd_workspace_init).  Applies to calls made after it, on
 * every host thread.  Returns ISD_OK.
 */
int isd_debug_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* ISD_B300_ISD_H */
