/*
 * isd_oracle.c -- fp64 CPU oracle for the ISD verify-and-propose step.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline / reference legs load this
 * library.  It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (Introspective Strided Decoding, "Introspective Diffusion
 * Language Models"; the pages describing it):
 *   - one forward gives 2N-1 logit rows per sequence: N-1 clean rows that
 *     verify the N-1 tokens proposed on the previous step, one clean anchor
 *     row for the next token, N-1 MASK rows that propose the next N-1 tokens
 *     (ai.arkapp.pw blog, section "I-DLM 如何解決這些問題" and the compute
 *     efficiency paragraph giving 2N-1 = 7 queries per forward);
 *   - a proposed token x drawn from q is kept with probability
 *     min(1, p(x)/q(x)), p the anchor (clean-position) distribution
 *     (same section; de.news.hada.io, "Inference & ISD");
 *   - N tokens per forward at most (zhuanzhiai.com, introduction; tinai-dev,
 *     "Introspective Strided Decoding (ISD)");
 *   - tokens per forward obeys TPF = (2+p+...+p^(N-2)) / (2-p^(N-1))
 *     (de.news.hada.io, "Speedup Factor Explorer").  That closed form holds
 *     exactly when a rejection emits the accepted prefix plus one
 *     replacement token, discards the pending proposals, and the next
 *     forward emits one token and proposes afresh; this file implements
 *     exactly that schedule.
 * The replacement token is drawn from the normalised residual max(0, p - q),
 * the standard reading that makes the output distribution equal p.
 *
 * Three modes (the `greedy` argument): 0 samples everywhere; 1 takes the
 * argmax everywhere (the lossless greedy invariant); 2 proposes the argmax of
 * each MASK row (ai.arkapp.pw blog, section "實際部署：SGLang 整合", names
 * argmax proposals) with q the point mass at it, so a proposal is kept with
 * probability p(x) and a rejection draws from max(0, p - delta_x), p without x.
 *
 * Everything is plain fp64: bf16 and fp32 inputs convert to double exactly,
 * softmax uses exp() with the row maximum subtracted, sums are sequential.
 *
 * Parity status: every function here is pinned by tests (Philox known-answer
 * vectors, exact enumeration of the emitted-token law, Monte-Carlo tokens per
 * forward against the closed form, the greedy lossless invariant, the
 * argmax-proposal mode's exact law and closed form, and special cases); none
 * is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_DTYPE_BF16 0
#define ORACLE_DTYPE_F32 1

/* per-sequence status codes */
#define ORACLE_SEQ_OK 0
#define ORACLE_SEQ_NONFINITE 1   /* a row the step reads holds NaN/+Inf or is all -Inf */
#define ORACLE_SEQ_BAD_PENDING 2 /* pending token outside [0,V) or pending q not in (0, inf) */

/* ------------------------------------------------------------------------ */
/* Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As   */
/* Easy as 1, 2, 3", SC'11, section 4 (Philox).  Four 32-bit counter words,  */
/* two key words, ten rounds; each round multiplies words 0 and 2 by the two  */
/* Philox constants, XORs the high halves with the other words and the key,  */
/* and the key advances by the two Weyl constants between rounds.            */
/* ------------------------------------------------------------------------ */
static const uint32_t PHILOX_M0 = 0xD2511F53u;
static const uint32_t PHILOX_M1 = 0xCD9E8D57u;
static const uint32_t PHILOX_W0 = 0x9E3779B9u;
static const uint32_t PHILOX_W1 = 0xBB67AE85u;

void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t x[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += PHILOX_W0;
            k1 += PHILOX_W1;
        }
        uint64_t prod0 = (uint64_t)PHILOX_M0 * (uint64_t)x[0];
        uint64_t prod1 = (uint64_t)PHILOX_M1 * (uint64_t)x[2];
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t y0 = hi1 ^ x[1] ^ k0;
        uint32_t y1 = lo1;
        uint32_t y2 = hi0 ^ x[3] ^ k1;
        uint32_t y3 = lo0;
        x[0] = y0; x[1] = y1; x[2] = y2; x[3] = y3;
    }
    out[0] = x[0]; out[1] = x[1]; out[2] = x[2]; out[3] = x[3];
}

/* A uniform in [0, 1 - 2^-24] from one Philox word: its top 24 bits times
 * 2^-24.  Exactly representable in fp32 and fp64. */
double oracle_uniform(uint32_t w)
{
    return ldexp((double)(w >> 8), -24);
}

/* The two uniforms of one logit row: word 0 drives the acceptance test at
 * that row, word 1 drives the inverse-CDF draw at that row.
 * key = (seed low, seed high), counter = (step low, step high, seq, row). */
void oracle_row_uniforms(uint64_t seed, uint64_t step, uint32_t seq, uint32_t row,
                         double* u_accept, double* u_sample)
{
    uint32_t ctr[4] = {(uint32_t)step, (uint32_t)(step >> 32), seq, row};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t w[4];
    oracle_philox4x32_10(ctr, key, w);
    *u_accept = oracle_uniform(w[0]);
    *u_sample = oracle_uniform(w[1]);
}

/* ------------------------------------------------------------------------ */
/* Reading logits exactly.                                                  */
/* ------------------------------------------------------------------------ */
static double logit_at(const void* base, int dtype, size_t idx)
{
    if (dtype == ORACLE_DTYPE_BF16) {
        uint16_t h = ((const uint16_t*)base)[idx];
        uint32_t bits = (uint32_t)h << 16; /* bf16 is the top half of an fp32 */
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float*)base)[idx];
}

/* A row the step reads must hold no NaN, no +Inf, and at least one value
 * above -Inf (otherwise its softmax is undefined). */
static int row_is_finite(const void* base, int dtype, size_t off, int V)
{
    int any_above_neg_inf = 0;
    for (int j = 0; j < V; ++j) {
        double x = logit_at(base, dtype, off + (size_t)j);
        if (isnan(x) || x == INFINITY) return 0;
        if (x > -INFINITY) any_above_neg_inf = 1;
    }
    return any_above_neg_inf;
}

/* Rows r0..r1-1 of the sequence whose rows start at off: all usable. */
static int rows_are_finite(const void* base, int dtype, size_t off, int r0, int r1, int V)
{
    for (int r = r0; r < r1; ++r)
        if (!row_is_finite(base, dtype, off + (size_t)r * V, V)) return 0;
    return 1;
}

/* softmax(row / T) in fp64: subtract the maximum, exponentiate, normalise.
 * Entries equal to -Inf get probability exactly 0. */
static void softmax_row(const void* base, int dtype, size_t off, int V, double T, double* P)
{
    double m = -INFINITY;
    for (int j = 0; j < V; ++j) {
        double z = logit_at(base, dtype, off + (size_t)j) / T;
        if (z > m) m = z;
    }
    double S = 0.0;
    for (int j = 0; j < V; ++j) {
        double z = logit_at(base, dtype, off + (size_t)j) / T;
        P[j] = exp(z - m);
        S += P[j];
    }
    for (int j = 0; j < V; ++j) P[j] /= S;
}

/* Index of the largest logit, lowest index on ties. */
static int argmax_row(const void* base, int dtype, size_t off, int V)
{
    int best = 0;
    double bv = logit_at(base, dtype, off);
    for (int j = 1; j < V; ++j) {
        double x = logit_at(base, dtype, off + (size_t)j);
        if (x > bv) { bv = x; best = j; }
    }
    return best;
}

/* Inverse CDF: the smallest index i with w_0 + ... + w_i > u * sum(w),
 * vocabulary indices taken in ascending order.  *margin receives the
 * distance from u*sum(w) to the nearer edge of the chosen interval, divided
 * by sum(w) (how close the draw came to a neighbouring token).  If rounding
 * leaves no such index, the last index with positive weight is returned and
 * the margin is 0.
 * [*lo, *hi] receives the range of indices with positive weight whose
 * interval [w_0+...+w_{j-1}, w_0+...+w_j) comes within tol*sum(w) of
 * u*sum(w): the tokens a draw could return if no edge of the cumulative sum
 * moved by tol*sum(w) or more (-1, -1 when no weight is positive). */
static int inverse_cdf(const double* w, int V, double u, double tol, double* margin,
                       int32_t* lo, int32_t* hi)
{
    double S = 0.0;
    for (int j = 0; j < V; ++j) S += w[j];
    double target = u * S;
    double C = 0.0;
    int last_positive = -1;
    int pick = -1;
    *margin = 0.0;
    *lo = -1;
    *hi = -1;
    for (int i = 0; i < V; ++i) {
        double C_before = C;
        C += w[i];
        if (w[i] > 0.0) {
            last_positive = i;
            if (*lo < 0 && C > target - tol * S) *lo = i;
            if (C_before <= target + tol * S) *hi = i;
        }
        if (pick < 0 && C > target) {
            double below = target - C_before, above = C - target;
            *margin = (below < above ? below : above) / S;
            pick = i;
        }
    }
    if (pick < 0) pick = last_positive; /* rounding overshoot; margin stays 0 */
    return pick;
}

/* A sequence that cannot be decoded this step: no token, no proposal, no
 * probability and no decision is reported for it. */
static void fail_sequence(int b, int status, int N, int32_t* accepted_len, int32_t* seq_status,
                          int32_t* tok, double* nq, double* pout, double* am, double* cm,
                          int32_t* clo, int32_t* chi)
{
    const int R = 2 * N - 1;
    for (int r = 0; r < R; ++r) { tok[r] = -1; cm[r] = -1.0; clo[r] = -1; chi[r] = -1; }
    for (int i = 0; i < N - 1; ++i) { nq[i] = 0.0; pout[i] = 0.0; am[i] = -1.0; }
    accepted_len[b] = 0;
    seq_status[b] = status;
}

/* ------------------------------------------------------------------------ */
/* One ISD verify-and-propose step with the uniforms given explicitly.      */
/*                                                                          */
/* logits, prev_logits : [B][2N-1][V], row r of sequence b at (b*R + r)*V.  */
/*   rows 0..N-2  : clean rows; row i-1 is the anchor p for pending x_i     */
/*   row  N-1     : clean anchor row for the token after the pending ones   */
/*   rows N..2N-2 : MASK rows; row N-1+j proposes the j-th next token       */
/*   prev_logits is the previous step's forward: its row N+K is the MASK    */
/*   row that proposed the pending token x_{K+1}.  May be NULL if no        */
/*   sequence has pending tokens (or in greedy mode).                       */
/* pending_tokens [B][N-1] : pending_tokens[b][0] < 0 means no pending.     */
/* pending_q      [B][N-1] : q(x) saved when x was drawn.                   */
/* u_accept, u_sample [B][2N-1] : the uniforms of each row.                 */
/* Outputs: accepted_len [B] (1..N, 0 on a bad sequence); tokens_out        */
/* [B][2N-1] (emitted tokens in [0,N), -1 padded; new pending in [N,2N-1)   */
/* or -1); new_q [B][N-1]; p_out [B][N-1] (anchor p of each pending token); */
/* seq_status [B] (a sequence fails, with every output cleared, if a row   */
/* it reads holds NaN or +Inf or is all -Inf: the anchor rows 0..N-2 when  */
/* it has pending tokens; the q row N+K of prev_logits when it rejects at  */
/* K; rows N-1..2N-2 when it proposes, i.e. when all pending tokens are    */
/* kept or it had none -- after a rejection those rows are not read);     */
/* accept_margin [B][N-1] = |u - p/q| of each test made                     */
/* (-1 where none); cdf_margin [B][2N-1] = margin of the inverse-CDF draw   */
/* made at that row (-1 where none); cdf_lo, cdf_hi [B][2N-1] = the range  */
/* of tokens within near_tol*sum(w) of that draw's target (see             */
/* inverse_cdf; -1 where no draw).                                          */
/* greedy: 0 = sampling everywhere; 1 = argmax everywhere (T unused);      */
/* 2 = argmax proposals (q = 1, a point mass) verified by sampling: x is    */
/* kept with probability p(x), and after a rejection the replacement is     */
/* drawn from max(0, p - delta_x) = p without x (no previous row needed).   */
/* Returns 0, or -1 on bad arguments / allocation failure.                  */
/* ------------------------------------------------------------------------ */
int oracle_isd_step_u(const void* logits, const void* prev_logits, int dtype,
                      const int32_t* pending_tokens, const float* pending_q,
                      int B, int N, int V, double temperature, int greedy,
                      const double* u_accept, const double* u_sample,
                      int32_t* accepted_len, int32_t* tokens_out, double* new_q,
                      double* p_out, int32_t* seq_status,
                      double* accept_margin, double* cdf_margin,
                      double near_tol, int32_t* cdf_lo, int32_t* cdf_hi)
{
    if (B < 0 || N < 2 || V < 1 || logits == NULL) return -1;
    if (greedy < 0 || greedy > 2) return -1;
    if (greedy != 1 && !(temperature > 0.0)) return -1;
    const int R = 2 * N - 1;
    double* P = (double*)malloc(sizeof(double) * (size_t)R * (size_t)V);
    double* Q = (double*)malloc(sizeof(double) * (size_t)V);
    double* resid = (double*)malloc(sizeof(double) * (size_t)V);
    if (!P || !Q || !resid) { free(P); free(Q); free(resid); return -1; }

    for (int b = 0; b < B; ++b) {
        const int32_t* pend = pending_tokens + (size_t)b * (N - 1);
        const float* pq = pending_q + (size_t)b * (N - 1);
        int32_t* tok = tokens_out + (size_t)b * R;
        double* nq = new_q + (size_t)b * (N - 1);
        double* pout = p_out + (size_t)b * (N - 1);
        double* am = accept_margin + (size_t)b * (N - 1);
        double* cm = cdf_margin + (size_t)b * R;
        int32_t* clo = cdf_lo + (size_t)b * R;
        int32_t* chi = cdf_hi + (size_t)b * R;
        const double* ua = u_accept + (size_t)b * R;
        const double* us = u_sample + (size_t)b * R;

        for (int r = 0; r < R; ++r) { tok[r] = -1; cm[r] = -1.0; clo[r] = -1; chi[r] = -1; }
        for (int i = 0; i < N - 1; ++i) { nq[i] = 0.0; pout[i] = 0.0; am[i] = -1.0; }
        accepted_len[b] = 0;
        seq_status[b] = ORACLE_SEQ_OK;

        const int has_pending = pend[0] >= 0;
        const size_t seq_off = (size_t)b * R * (size_t)V;

        /* the pending state must be usable */
        if (has_pending) {
            int bad = 0;
            for (int i = 0; i < N - 1; ++i) {
                if (pend[i] < 0 || pend[i] >= V) bad = 1;
                if (greedy != 1 && !(pq[i] > 0.0f && pq[i] < INFINITY)) bad = 1;
            }
            if (bad || (greedy == 0 && prev_logits == NULL)) {
                seq_status[b] = ORACLE_SEQ_BAD_PENDING;
                continue;
            }
        }

        /* 1. the anchor rows of the pending tokens (clean rows 0..N-2) are
         * read by every step that has pending tokens: they must be usable,
         * and P(r) = softmax(row r / T) */
        if (has_pending) {
            if (!rows_are_finite(logits, dtype, seq_off, 0, N - 1, V)) {
                fail_sequence(b, ORACLE_SEQ_NONFINITE, N, accepted_len, seq_status, tok, nq, pout, am, cm, clo, chi);
                continue;
            }
            if (greedy != 1)
                for (int r = 0; r < N - 1; ++r)
                    softmax_row(logits, dtype, seq_off + (size_t)r * V, V, temperature, P + (size_t)r * V);
        }

        int n_emit = 0;
        int propose = 1;

        if (has_pending) {
            /* 2. verify x_1..x_{N-1} in order against the anchor rows */
            if (greedy != 1)
                for (int i = 1; i <= N - 1; ++i)
                    pout[i - 1] = P[(size_t)(i - 1) * V + pend[i - 1]];
            int K = 0;
            for (int i = 1; i <= N - 1; ++i) {
                const int x = pend[i - 1];
                int accept;
                if (greedy == 1) {
                    accept = (x == argmax_row(logits, dtype, seq_off + (size_t)(i - 1) * V, V));
                } else {
                    const double ratio = pout[i - 1] / (double)pq[i - 1];
                    accept = ua[i - 1] < ratio; /* probability min(1, p/q) */
                    am[i - 1] = fabs(ua[i - 1] - ratio);
                }
                if (!accept) break;
                ++K;
            }
            for (int i = 0; i < K; ++i) tok[n_emit++] = pend[i];

            if (K < N - 1) {
                /* 3a. first rejection at x_{K+1}: one replacement token from
                 * the residual max(0, p - q); p is anchor row K, q is the
                 * previous step's MASK row N+K that proposed x_{K+1} */
                int y;
                if (greedy == 1) {
                    y = argmax_row(logits, dtype, seq_off + (size_t)K * V, V);
                } else {
                    if (greedy == 2) {
                        /* an argmax proposal's q is the point mass at it */
                        for (int j = 0; j < V; ++j) Q[j] = 0.0;
                        Q[pend[K]] = 1.0;
                    } else {
                        const size_t qoff = seq_off + (size_t)(N + K) * V;
                        if (!row_is_finite(prev_logits, dtype, qoff, V)) {
                            fail_sequence(b, ORACLE_SEQ_NONFINITE, N, accepted_len, seq_status, tok, nq, pout, am,
                                          cm, clo, chi);
                            continue;
                        }
                        softmax_row(prev_logits, dtype, qoff, V, temperature, Q);
                    }
                    const double* Pk = P + (size_t)K * V;
                    double mass = 0.0;
                    for (int j = 0; j < V; ++j) {
                        double d = Pk[j] - Q[j];
                        resid[j] = d > 0.0 ? d : 0.0;
                        mass += resid[j];
                    }
                    if (mass > 0.0) {
                        y = inverse_cdf(resid, V, us[K], near_tol, &cm[K], &clo[K], &chi[K]);
                    } else {
                        /* only reachable through rounding: fall back to p; any
                         * token of p is then within reach (a window of 2) */
                        y = inverse_cdf(Pk, V, us[K], 2.0, &cm[K], &clo[K], &chi[K]);
                        cm[K] = 0.0;
                    }
                }
                tok[n_emit++] = y;
                propose = 0; /* the proposals rest on x_{K+1}: discard them */
            }
        }

        if (propose) {
            /* 3b. all N-1 accepted, or 4. no pending tokens: the sequence
             * ends the step with a valid prefix, so it reads the anchor row
             * N-1 and the MASK rows: one more token from row N-1, then the
             * proposals.  (A rejecting sequence reads neither: its proposals
             * would be discarded.) */
            if (!rows_are_finite(logits, dtype, seq_off, N - 1, R, V)) {
                fail_sequence(b, ORACLE_SEQ_NONFINITE, N, accepted_len, seq_status, tok, nq, pout, am, cm, clo, chi);
                continue;
            }
            if (greedy != 1)
                for (int r = N - 1; r < R; ++r)
                    softmax_row(logits, dtype, seq_off + (size_t)r * V, V, temperature, P + (size_t)r * V);
            int y;
            if (greedy == 1) {
                y = argmax_row(logits, dtype, seq_off + (size_t)(N - 1) * V, V);
            } else {
                y = inverse_cdf(P + (size_t)(N - 1) * V, V, us[N - 1], near_tol,
                                &cm[N - 1], &clo[N - 1], &chi[N - 1]);
            }
            tok[n_emit++] = y;

            /* 5. proposals for the next step from the MASK rows, with q saved */
            for (int j = 1; j <= N - 1; ++j) {
                const int r = N - 1 + j;
                int x;
                if (greedy >= 1) {
                    x = argmax_row(logits, dtype, seq_off + (size_t)r * V, V);
                    nq[j - 1] = 1.0; /* an argmax proposal is a point mass */
                } else {
                    x = inverse_cdf(P + (size_t)r * V, V, us[r], near_tol, &cm[r], &clo[r], &chi[r]);
                    nq[j - 1] = P[(size_t)r * V + x];
                }
                tok[N - 1 + j] = x;
            }
        }
        accepted_len[b] = n_emit;
    }
    free(P);
    free(Q);
    free(resid);
    return 0;
}

/* The same step with the uniforms drawn from Philox4x32-10 as
 * oracle_row_uniforms defines them. */
int oracle_isd_step(const void* logits, const void* prev_logits, int dtype,
                    const int32_t* pending_tokens, const float* pending_q,
                    int B, int N, int V, double temperature, int greedy,
                    uint64_t seed, uint64_t step,
                    int32_t* accepted_len, int32_t* tokens_out, double* new_q,
                    double* p_out, int32_t* seq_status,
                    double* accept_margin, double* cdf_margin,
                    double near_tol, int32_t* cdf_lo, int32_t* cdf_hi)
{
    if (B < 0 || N < 2) return -1;
    const int R = 2 * N - 1;
    double* ua = (double*)malloc(sizeof(double) * (size_t)(B > 0 ? B : 1) * R);
    double* us = (double*)malloc(sizeof(double) * (size_t)(B > 0 ? B : 1) * R);
    if (!ua || !us) { free(ua); free(us); return -1; }
    for (int b = 0; b < B; ++b)
        for (int r = 0; r < R; ++r)
            oracle_row_uniforms(seed, step, (uint32_t)b, (uint32_t)r,
                                ua + (size_t)b * R + r, us + (size_t)b * R + r);
    int rc = oracle_isd_step_u(logits, prev_logits, dtype, pending_tokens, pending_q,
                               B, N, V, temperature, greedy, ua, us,
                               accepted_len, tokens_out, new_q, p_out, seq_status,
                               accept_margin, cdf_margin, near_tol, cdf_lo, cdf_hi);
    free(ua);
    free(us);
    return rc;
}

/* softmax(row / T)[token] in fp64, for a row of V logits (the probability a
 * proposal drawn at `token` would save as its q). */
double oracle_softmax_prob(const void* row, int dtype, int V, double temperature, int token)
{
    if (V < 1 || token < 0 || token >= V || !(temperature > 0.0)) return -1.0;
    double* P = (double*)malloc(sizeof(double) * (size_t)V);
    if (!P) return -1.0;
    softmax_row(row, dtype, 0, V, temperature, P);
    double p = P[token];
    free(P);
    return p;
}
