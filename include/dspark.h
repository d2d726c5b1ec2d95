/*
 * dspark.h -- C ABI of libdspark.so: the batched, confidence-driven,
 * variable-length verify step of DSpark-style speculative decoding, in
 * hand-written CUDA kernels for sm_103a (GB300).
 *
 * One step is three calls on one CUDA stream:
 *
 *   dspark_score_budget  confidence head + sequential temperature scaling,
 *                        survival curve, per-request budget, batch-wide cap,
 *                        exclusive scans of the verify lengths;
 *   dspark_compact       ragged packing of the rows the target must score;
 *   (the caller's target forward fills target_logits for the packed rows)
 *   dspark_verify        vocab-wide softmax of target and draft rows,
 *                        accept / resample / bonus, commit.
 *
 * dspark_score_compact is the first two calls in one kernel launch, with
 * the same outputs.
 *
 * Variants: dspark_score_entropy scores drafts by the entropy of their
 * distribution instead of the head; dspark_verify_cap_accept is the audit arm
 * that verifies the full block and commits the scheduled window;
 * dspark_verify_noalloc runs dspark_verify on the library's own scratch;
 * dspark_fit_sts_tau calibrates sts_tau offline from logged steps.
 *
 * Sources (page title and section):
 *   [DS] "DFlash to DSpark in SGLang: 4.3x faster decode, and DeepSeek-V4
 *        support": "Background"; "DSpark: a sequential head and a verify
 *        budget"; "The confidence scheduler and verify modes"; "Ragged verify
 *        under full CUDA graphs"; "Zero-overhead scheduling and kernels".
 *   [KC] "SGLang Integrates DSpark: How Confidence-Driven Speculative
 *        Decoding Cracks the High-Concurrency Failure Problem": "The Old
 *        Problem with Speculative Decoding: It Breaks Down at Scale" (the
 *        speculative-sampling rule of Chen et al. 2023); "DSpark's Core Idea:
 *        Only Verify the Parts You're Confident About" (entropy confidence).
 *   [SC11] Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3"
 *        (Philox4x64-10).
 *
 * Conventions for every call:
 *   - Ownership: the caller owns all memory.  Every pointer in dspark_step is
 *     device memory of the current CUDA device unless marked otherwise.  The
 *     library allocates nothing and keeps no pointer after a call returns
 *     (dspark_verify_noalloc's scratch is a fixed array of the library).
 *   - Asynchrony: calls enqueue kernels on `stream` and return; no call
 *     synchronises with the host.  Totals that depend on data (sum of L,
 *     number of packed rows) stay on the device; grids are sized for the
 *     worst case and surplus blocks exit.
 *   - Errors: argument checks run on the host before anything is enqueued
 *     and return a negative dspark_status; nothing is launched then.  A
 *     failed launch returns DSPARK_ECUDA.  dspark_last_error() gives a
 *     thread-local message for the last failing call on this thread.
 *   - Layout: row-major, contiguous.  Index b is the request (0..B-1), i or
 *     k the 0-based draft position (0..gamma-1), y a token id (0..V-1).
 *   - Values: logits and hidden states are finite (dspark_score_entropy
 *     also takes -inf logits as masked ids).
 *   - Alignment: hidden, draft_logits and target_logits start on 16-byte
 *     boundaries and their rows are multiples of 16 bytes (d and V multiples
 *     of 8 for bf16, of 4 for fp32); otherwise DSPARK_EALIGN.
 *   - Workspace: one caller-allocated device buffer of at least
 *     dspark_workspace_size() bytes, 256-byte aligned, zeroed once with
 *     dspark_workspace_init() before its first use.  Every call that runs to
 *     completion leaves it ready for the next call.  Steps that run at the
 *     same time (other streams) need workspaces of their own.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *dspark_stream_t;

typedef enum {
    DSPARK_OK = 0,
    DSPARK_EINVAL = -1,     /* bad shape, scalar, mode combination or NULL pointer */
    DSPARK_EDTYPE = -2,     /* unsupported dtype code */
    DSPARK_EALIGN = -3,     /* a pointer or row size breaks the 16-byte rule */
    DSPARK_ECUDA = -4,      /* a CUDA call or kernel launch failed */
    DSPARK_EWORKSPACE = -5, /* workspace missing, misaligned or too small */
    DSPARK_EDEVICE = -6     /* the current device is not sm_103 */
} dspark_status;

typedef enum {
    DSPARK_F32 = 0,  /* IEEE binary32 */
    DSPARK_BF16 = 1  /* bfloat16 */
} dspark_dtype;

/* Limits checked by every call. */
#define DSPARK_MAX_B 65536
#define DSPARK_MAX_GAMMA 64
#define DSPARK_MAX_V (1 << 24)
#define DSPARK_MAX_D (1 << 20)

/* No batch-wide cap (cap_T).  Any negative value means the same. */
#define DSPARK_NO_CAP (-1)
/* Dynamic budget (fixed_budget).  Any negative value means the same. */
#define DSPARK_DYNAMIC (-1)

typedef struct dspark_step {
    /* ---- shapes ---------------------------------------------------------- */
    int32_t B;            /* requests, 0..DSPARK_MAX_B (0: every call is a no-op) */
    int32_t gamma;        /* draft block size, 1..DSPARK_MAX_GAMMA */
    int32_t V;            /* vocabulary size, 1..DSPARK_MAX_V */
    int32_t d;            /* drafter hidden size, 1..DSPARK_MAX_D */
    int32_t logit_dtype;  /* dspark_dtype of draft_logits and target_logits */
    int32_t hidden_dtype; /* dspark_dtype of hidden */

    /* ---- inputs (device, read only) -------------------------------------- */
    const int32_t *draft_tokens; /* [B, gamma] drafted ids d_1..d_gamma; an id outside
                                    [0, V) is always rejected */
    const void *draft_logits;    /* [B, gamma, V] drafter logits z_q; row (b,k) is read
                                    only when k < L_b and temperature > 0 */
    const void *target_logits;   /* [N_rows, V] target logits z_p in the ragged order
                                    that dspark_compact writes: request b owns rows
                                    row_off[b] .. row_off[b] + L_b (root first) */
    const void *hidden;          /* [B, gamma, d] drafter hidden state per draft */
    const float *head_w;         /* [d] confidence-head weight */
    const float *head_bias;      /* [B] confidence-head bias per request */
    const float *sts_tau;        /* [gamma] STS temperature per position, > 0 */
    const int32_t *last_tokens;  /* [B] root token per request, or NULL (packed id -1) */
    const int32_t *seq_lens_in;  /* [B] cached length = position of the root, or NULL (0) */

    /* ---- scalars (host values) ------------------------------------------- */
    float cost_c;         /* marginal cost c of one more verify token */
    int32_t cap_T;        /* batch-wide cap on sum of L; < 0: no cap */
    int32_t fixed_budget; /* >= 0: every L_b = min(fixed_budget, gamma) and the head
                             is not run; < 0: the confidence-driven budget.  A
                             fixed budget together with cap_T >= 0 is DSPARK_EINVAL */
    float temperature;    /* sampling temperature Tm > 0, or 0 for greedy verify */
    uint64_t seed;        /* Philox key word 0 (word 1 is 0) */

    /* ---- outputs (device, caller-allocated) ------------------------------ */
    float *conf;          /* [B, gamma] sigmoid((w.h + bias_b) / tau_i) */
    float *survival;      /* [B, gamma] S_{b,k} for k = 1..gamma (S_0 = 1 implied) */
    int32_t *L0;          /* [B] pre-cap length max{k : S_k >= c} */
    int32_t *L;           /* [B] verify length after the cap */
    int32_t *draft_off;   /* [B+1] exclusive scan of L; draft_off[B] = sum of L */
    int32_t *row_off;     /* [B+1] exclusive scan of L+1; row_off[B] = N_rows */
    int32_t *packed_ids;  /* [B*(gamma+1)] ragged rows [root, d_1..d_L] per request;
                             -1 past N_rows */
    int32_t *packed_pos;  /* [B*(gamma+1)] seq_len_b + j for row j of request b; 0 past */
    int32_t *row_req;     /* [B*(gamma+1)] request of each packed row; -1 past */
    int32_t *row_k;       /* [B*(gamma+1)] index j of each packed row in its request; -1 past */
    int32_t *accept_len;  /* [B] accepted drafts a_b, 0..L_b */
    int32_t *num_emitted; /* [B] a_b + 1 */
    int32_t *out_tokens;  /* [B, gamma+1] d_1..d_{a_b}, then the resampled or bonus
                             token, then -1 */
    float *p_tok;         /* [B*gamma] p(d_k) at draft_off[b] + k, k < L_b (0 if greedy) */
    float *q_tok;         /* [B*gamma] q(d_k) likewise (0 if greedy) */
    int32_t *seq_lens_commit; /* [B] incremented by num_emitted in place, or NULL */

    /* ---- scratch --------------------------------------------------------- */
    void *workspace;        /* device, see the workspace convention above */
    size_t workspace_bytes; /* its size in bytes */
} dspark_step;

/*
 * Bytes of workspace a step of this shape needs (independent of dtypes).
 * Returns 0 when the shape is outside the limits above.
 */
size_t dspark_workspace_size(int32_t B, int32_t gamma, int32_t V, int32_t d);

/*
 * Zero a workspace (cudaMemsetAsync on `stream`).  Call once after
 * allocating it, and again after any call reported an error.
 */
dspark_status dspark_workspace_init(void *workspace, size_t workspace_bytes,
                                    dspark_stream_t stream);

/*
 * Steps a1-a3 and the scans of a4.  [DS] "DSpark: a sequential head and a
 * verify budget" and "The confidence scheduler and verify modes":
 *   x_{b,i} = (w . h_{b,i} + bias_b) / tau_i,  conf_{b,i} = sigmoid(x_{b,i});
 *   S_{b,0} = 1,  S_{b,k+1} = S_{b,k} * conf_{b,k};
 *   L0_b = max{k in 0..gamma : S_{b,k} >= c}  (0 when no k qualifies).
 * [DS] "Zero-overhead scheduling and kernels" (verify-length top-k): when
 * cap_T >= 0 and sum L0 > cap_T, keep the cap_T largest gains S_{b,k}
 * (1 <= k <= L0_b) in the order (S desc, b asc, k asc); L_b = number kept in
 * request b.  Otherwise L = L0.  With fixed_budget >= 0 only L = min(F, gamma)
 * is written (conf, survival and L0 are untouched).  Then draft_off and
 * row_off are the exclusive scans of L and L + 1.
 * Reads: hidden, head_w, head_bias, sts_tau.  Writes: conf, survival, L0, L,
 * draft_off, row_off.
 */
dspark_status dspark_score_budget(const dspark_step *step, dspark_stream_t stream);

/*
 * Steps a1-a4 in one launch: dspark_score_budget followed by dspark_compact,
 * with the same outputs bit for bit.  The CTA that computes the batch's
 * lengths also writes the packing, so no second kernel and no launch gap
 * sit between the budget and the packed rows.  With fixed_budget >= 0 one
 * thread per packing slot writes L, the offsets (closed form) and the
 * packing.
 * Reads what the two calls read; writes what they write.  Errors: those of
 * dspark_score_budget, and DSPARK_EINVAL for a NULL draft_tokens, packed_ids,
 * packed_pos, row_req or row_k.
 */
dspark_status dspark_score_compact(const dspark_step *step, dspark_stream_t stream);

/*
 * Steps a1-a3 with the entropy-confidence variant of step a1.  [KC] "DSpark's
 * Core Idea: Only Verify the Parts You're Confident About": the lower the
 * entropy of the drafter's output distribution at a position, the more
 * certain the draft and the more a verify of it is worth.  Read here as
 *   q_{b,i} = softmax(z_q[b,i] / theta),  H_{b,i} = -sum_y q ln q  (nats),
 *   conf_{b,i} = exp(-H_{b,i})   (in (1/V, 1]: 1 for a one-hot q, 1/V for a
 *                                 uniform one),
 * computed from the draft logits [B, gamma, V] (logit_dtype; each row needs
 * a finite maximum, -inf entries are masked ids).  The survival curve, L0,
 * the cap and the scans are those of dspark_score_budget.
 * theta: host value, finite and > 0.  Reads draft_logits.  Writes conf,
 * survival, L0, L, draft_off, row_off.  hidden, head_w, head_bias and
 * sts_tau are not read.  fixed_budget >= 0 is DSPARK_EINVAL.
 */
dspark_status dspark_score_entropy(const dspark_step *step, float theta, dspark_stream_t stream);

/*
 * Step a4, ragged packing.  [DS] "Ragged verify under full CUDA graphs": the
 * scheduled rows are front-packed and a cu_seqlens-style offset marks each
 * request's segment.  Request b owns rows row_off[b] + j, j = 0..L_b, holding
 * the root (j = 0) then drafts d_1..d_{L_b}.  Reads L, row_off, draft_tokens,
 * last_tokens, seq_lens_in.  Writes packed_ids, packed_pos, row_req, row_k
 * (all B*(gamma+1) entries; rows past N_rows get the padding values).
 */
dspark_status dspark_compact(const dspark_step *step, dspark_stream_t stream);

/*
 * Steps a5-a6.  [DS] "Background"; [KC] "The Old Problem with Speculative
 * Decoding" (speculative sampling).  For draft k < L_b of request b:
 * p = softmax(z_p[row_off[b]+k] / Tm), q = softmax(z_q[b,k] / Tm),
 * r = min(1, p(d)/q(d)) (1 when q(d) = 0, 0 when d is outside [0, V));
 * accept iff u_{b,k} < r, with (u, u', u'') the top 24 bits / 2^24 of
 * words 0, 1 and 2 of Philox4x64-10 at counter (b, k, 0, 0), key (seed, 0).
 * a_b is the first rejected k (L_b if none).  A rejection draws the emitted token from
 * norm(max(0, p - q)) at row a_b (from p when that mass is 0); otherwise the
 * bonus token is drawn from p at row L_b.  Draws are a two-level inverse
 * CDF over ascending token id: the ids are cut into blocks of 4096; u'
 * (word 1) picks the smallest block whose running mass exceeds u' times the
 * total, and u'' (word 2) the smallest id of that block whose running weight
 * exceeds u'' times the block's mass.  That draws id y with probability
 * weight(y) / total.  Tm = 0 is greedy: accept iff d == argmax z_p (lowest
 * id on ties); the emitted token is that argmax at row a_b.
 * p_tok and q_tok are written for every verified draft k < L_b.  Rows are
 * read only as far as the method needs: the bonus row of a request known to
 * reject may be skipped.
 * Reads draft_tokens, draft_logits, target_logits, L, draft_off, row_off,
 * row_req, row_k.  Writes accept_len, num_emitted, out_tokens, p_tok, q_tok,
 * and seq_lens_commit[b] += a_b + 1 when not NULL.
 */
dspark_status dspark_verify(const dspark_step *step, dspark_stream_t stream);

/*
 * The cap-accept audit arm of steps a5-a6.  [DS] "The confidence scheduler
 * and verify modes": cap-accept verifies the full block like static, so it
 * costs what static costs, but commits only the scheduled window, so its
 * output is compact's; it records what the trim gave up.  [DS] "Scheduling
 * results" quotes utilization against the ceiling from such runs.
 *
 * The step's L, draft_off, row_off and target_logits describe the block
 * that is verified (for the static audit: fixed_budget = gamma in
 * dspark_score_budget, then dspark_compact).  commit_len[b] (device, [B],
 * read only) is the window W_b the scheduler chose (the L of a
 * confidence-driven dspark_score_budget); it is clamped to [0, L_b].
 * Every draft k < L_b is verified as in dspark_verify; with a_b the first
 * rejected k (L_b if none), the committed drafts are min(a_b, W_b):
 *   - a_b < W_b: the residual draw at row a_b, as in dspark_verify;
 *   - a_b >= W_b, W_b < L_b: the window ends inside the accepted run; the
 *     token is drawn from p at row W_b with the uniforms (u', u'') of
 *     position W_b -- the bonus draw compact would make with L_b = W_b
 *     (greedy: the argmax of row W_b);
 *   - a_b = W_b = L_b: the bonus draw at row L_b.
 * accept_len, num_emitted, out_tokens and seq_lens_commit hold the
 * committed result; p_tok and q_tok cover every draft k < L_b of the block.
 *
 * accept_full:  device int32 [B] or NULL; receives a_b, the acceptance of
 *               the full verify (the ceiling).  The call zeroes it on
 *               `stream` before the launch (cudaMemsetAsync), which gives
 *               a_b = 0 to requests with L_b = 0.
 * audit_totals: device int32 [2] or NULL; receives (sum of a_b, sum of
 *               accept_len) over the batch.  Their ratio is the utilization
 *               against the ceiling.
 * Errors as dspark_verify; commit_len NULL with B > 0 is DSPARK_EINVAL.
 */
dspark_status dspark_verify_cap_accept(const dspark_step *step, const int32_t *commit_len,
                                       int32_t *accept_full, int32_t *audit_totals,
                                       dspark_stream_t stream);

/*
 * Offline calibration of the STS temperatures sts_tau from logged steps.
 * [DS] "DSpark: a sequential head and a verify budget": Sequential
 * Temperature Scaling calibrates the survival product to match true
 * acceptance rates.  Read here as: for each position i, tau_i is the
 * maximum-likelihood temperature of conf = sigmoid(x / tau_i) on the logged
 * outcomes.  Logged request-step n (the conf, L and accept_len a step wrote)
 * observes position i when i < L_n and i <= a_n; the outcome is accept
 * (i < a_n) or reject (i = a_n).  The head logit is recovered as
 * x = tau_used_i * logit(conf_{n,i}), conf clamped to [2^-126, 1 - 2^-24].
 * The likelihood is convex in 1/tau; the fit bisects its derivative over
 * [1/tau_max, 1/tau_min] (a bound when the data are separable).  Not a step
 * of the per-step path: run it now and then over accumulated logs.
 *
 * All pointers are device memory.  conf [N, gamma] (the step's conf rows,
 * stacked over logged steps), tau_used [gamma] (the sts_tau that produced
 * them), L [N], accept_len [N]: read only.  tau_out [gamma]: the fitted
 * temperatures (tau_used where a position has no observation).  nll_out
 * [gamma] (the minimised negative log-likelihood, nats) and n_obs [gamma]
 * (observations per position) may be NULL.  N may be 0.
 * Errors: DSPARK_EINVAL for N < 0, gamma outside [1, DSPARK_MAX_GAMMA],
 * bounds not 0 < tau_min <= tau_max < inf, or a NULL required pointer.
 */
dspark_status dspark_fit_sts_tau(int32_t N, int32_t gamma, const float *conf,
                                 const float *tau_used, const int32_t *L,
                                 const int32_t *accept_len, float tau_min, float tau_max,
                                 float *tau_out, float *nll_out, int32_t *n_obs,
                                 dspark_stream_t stream);

/*
 * Blocking read of the workspace's device status word (0 = healthy).  A
 * nonzero value means a kernel gave up on a bounded wait: bit 0 (1) an
 * in-CTA wait on the copy ring, bit 1 (2) a wait on the verify's work
 * (events, residual jobs, the end of the batch).  The workspace must then be
 * re-initialised.  Synchronises `stream`.
 */
dspark_status dspark_read_device_status(const void *workspace, int32_t *status_out,
                                        dspark_stream_t stream);

/*
 * Bytes of the fixed scratch that dspark_verify_noalloc uses instead of a
 * workspace: 8 MiB.  Its last 256 bytes record a shape; the rest holds a
 * step's workspace layout, enough for B = 512 at gamma = 16 and V = 151936.
 */
#define DSPARK_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

/*
 * dspark_verify without a caller workspace.  The pages have no counterpart:
 * this is a calling convention of this library, not a step of the method.
 *
 * For callers that cannot allocate device memory where they call the verify
 * step: a serving runtime whose device memory belongs to its own caching
 * allocator, with no hook to borrow a buffer from it at this call site, or a
 * step loop that must not allocate between its set-up and its steps.  The
 * scratch is one array of DSPARK_NOALLOC_SCRATCH_BYTES in this library's
 * device image, one copy per device, held until the process exits.  No call
 * allocates or frees device memory.
 *
 * Inputs, outputs, errors and results are those of dspark_verify;
 * step->workspace and step->workspace_bytes are ignored.  A shape whose
 * workspace (dspark_workspace_size) exceeds DSPARK_NOALLOC_SCRATCH_BYTES - 256
 * is rejected with DSPARK_EWORKSPACE before anything is enqueued.
 *
 * The first call on a device sets up: with that device current it looks up
 * the device's copy of the array.  Make that first call before any stream
 * capture.  The scratch's counters and queue flags must start at zero, and
 * where they sit depends on (B, gamma, V).  Every call enqueues, before the
 * verify launch, a one-CTA kernel that compares (B, gamma, V) with the shape
 * recorded in the scratch; when they differ it zeroes the first
 * dspark_workspace_size() bytes and records the new shape.  The check runs on
 * the device in stream order, so a captured graph replayed after calls of
 * other shapes zeroes again as needed.  A launch that ends with a zero device
 * status leaves the counters at zero for the next call of that shape.
 *
 * reset:      nonzero zeroes them in any case.  Pass it after a call whose
 *             status was nonzero.
 * status_out: device int32, or NULL.  When set, it receives the scratch's
 *             device status word after the launch (meaning as in
 *             dspark_read_device_status: 0 = healthy).
 *
 * Every call on a device shares the one array and finds the last call's
 * contents in it.  Calls whose kernels may overlap on the GPU (other
 * streams, other host threads) race on it and give wrong results: order
 * them on one stream or synchronise between them.
 */
dspark_status dspark_verify_noalloc(const dspark_step *step, int32_t reset,
                                    int32_t *status_out, dspark_stream_t stream);

/*
 * Bound, in nanoseconds, of every wait inside the kernels launched after this
 * call (process-wide; 0 restores the default of 2 s).  A kernel whose wait
 * runs out sets a nonzero device status (dspark_read_device_status), lets
 * its own copies in flight land, and returns; its outputs are then not
 * valid and the workspace must be re-initialised.  Meant for tests of that
 * error path: a bound of a few microseconds makes ordinary waits give up.
 * Always returns DSPARK_OK.
 */
dspark_status dspark_set_wait_timeout_ns(uint64_t ns);

/* The current bound (see dspark_set_wait_timeout_ns). */
uint64_t dspark_wait_timeout_ns(void);

/* Thread-local message for the last failing call on this thread ("" if none). */
const char *dspark_last_error(void);

/* Library version string. */
const char *dspark_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
