/*
 * specverify.h -- C ABI of the batched draft-verification sampler for
 * speculative decoding (sm_103a, one GPU).
 *
 * What it computes (web pages cited by title and section):
 *
 *  - "Speculative Decoding: Draft, Verify, and Correct" (DVC)
 *      'Name the two distributions at one prefix': accept a draft y ~ q with
 *      probability min(1, p(y)/q(y)); on rejection draw from the normalised
 *      residual [p - q]+.  'Verify several proposed tokens in one target pass':
 *      walk the drafts in order, stop at the first rejection, and add a bonus
 *      token from p when every draft is accepted.  'Speculation needs cache
 *      rollback': cache lengths must agree with the emitted tokens.
 *      'Preserve the distribution you actually intend': p and q are the
 *      post-temperature, post-mask sampling laws.
 *  - "Speculative Decoding: How a Small Model Speeds Up a Big One Without
 *    Changing Its Output" (SMB) 'The Guarantee Behind Rejection Sampling':
 *      the greedy rule (keep the draft iff it is the target argmax, else emit
 *      the argmax); 'Beyond Two Models: The EAGLE Line': draft trees verified
 *      in one pass, the best branch kept.
 *  - "Speculative decoding: why correcting a rejection is not resampling
 *    from the target" (CRS) sections 1-2, 5: the same rule, masks before
 *    correction, one to K+1 tokens per cycle.
 *  - "Margins, Not Windows: Training-Free Per-Step Lossy Speculative
 *    Decoding" (MNW) section 3: promote a mismatched draft when
 *    p_target(draft) / p_target(top1) exceeds kappa.
 *
 * Conventions for every entry point:
 *  - All array pointers are DEVICE pointers owned by the caller; the library
 *    never allocates, never frees and never synchronises the stream.
 *  - Arrays are dense, row-major, with the shapes given in brackets.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously; read results after synchronising.
 *  - Argument errors return a spec_status before anything is enqueued and
 *    write no output.  B == 0 is a valid no-op (pointers may then be NULL).
 *    Data errors in a row (NaN logit, token id out of range, ...) set that
 *    row's row_status; the row's accepted_len becomes -1, num_emitted 0 and
 *    its token outputs -1; other rows are unaffected.
 *  - Workspace: `ws` is caller-owned device memory of at least the size the
 *    matching *_workspace_size() returns, 256-byte aligned.  Its contents
 *    need no initialisation.  The stochastic chain calls keep a small header
 *    in the last 16 bytes of the `ws_bytes` they are given: a work counter,
 *    cleared before every call, and a generation count, advanced before
 *    every call (skipping 0, so zero-filled memory never looks current) and
 *    stamped on every record the call writes, so nothing an earlier call
 *    left behind is ever read, whatever its shapes.  Keep
 *    passing the same `ws_bytes` for the same buffer.  Calls on one stream
 *    may share a workspace; calls that may overlap in time (different
 *    streams) need separate workspaces.
 *  - Each verify call enqueues a streaming kernel (a truncated verify adds
 *    a selection kernel after it) and a small per-row kernel that starts
 *    early and waits for it on the device (programmatic dependent launch);
 *    the stochastic calls first enqueue a one-thread kernel that advances
 *    the workspace's generation count and clears its work counter.  That
 *    kernel is itself a programmatic dependent of whatever precedes it
 *    and waits for it to complete before anything of the call reads its
 *    inputs.  The last kernel of a stochastic chain call lets the kernel
 *    after it start early if that kernel is launched as a programmatic
 *    dependent: such a kernel must wait for its dependency
 *    (cudaGridDependencySynchronize) before it reads this call's outputs,
 *    as programmatic dependent launch requires of every dependent.
 *  - Logits are bf16 (SPEC_BF16) or fp32 (SPEC_F32).  Rows whose byte
 *    length is a multiple of 16 with a 16-byte aligned base take the bulk-
 *    copy (TMA) path; any other V still works, more slowly.
 *  - Apart from the workspace header above, the calls keep no state other
 *    than a per-process cache of device occupancy queries (thread safe).
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes of every entry point. */
typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_NULL = 1,      /* a required pointer is NULL */
  SPEC_ERR_SHAPE = 2,     /* B, K, N or V outside the supported range */
  SPEC_ERR_DTYPE = 3,     /* unknown dtype or mode */
  SPEC_ERR_ALIGN = 4,     /* a pointer is not aligned to its element size */
  SPEC_ERR_ARG = 5,       /* another bad scalar argument (e.g. kappa is NaN) */
  SPEC_ERR_CUDA = 6,      /* a CUDA runtime call failed (no device, launch error) */
  SPEC_ERR_WORKSPACE = 7, /* workspace NULL, misaligned or too small */
  SPEC_ERR_STATIC_LIMIT = 8 /* problem too large for spec_verify_chain_static */
} spec_status;

/* Per-row data status written to row_status[b].  When several problems meet
 * in one row the smallest code is reported. */
enum {
  SPEC_ROW_OK = 0,
  SPEC_ROW_NONFINITE = 1,       /* a logit the row reads is NaN or +inf */
  SPEC_ROW_BAD_TOKEN = 2,       /* a draft / node token outside [0, V) */
  SPEC_ROW_BAD_UNIFORM = 3,     /* a uniform outside [0, 1) */
  SPEC_ROW_BAD_PARENT = 4,      /* tree: parent[0] != -1 or not 0 <= parent[i] < i */
  SPEC_ROW_EMPTY = 5,           /* a logit row that is -inf everywhere */
  SPEC_ROW_TIMEOUT = 6,         /* a bounded on-device wait gave up (see below) */
  SPEC_ROW_BAD_TEMPERATURE = 7  /* temperature used and not finite and > 0 */
};

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;
typedef enum { SPEC_STOCHASTIC = 0, SPEC_GREEDY = 1 } spec_mode;

/* Limits checked by the entry points. */
#define SPEC_MAX_K 1023          /* drafts per chain */
#define SPEC_MAX_TREE_NODES 1024 /* nodes per tree, root included */
#define SPEC_MAX_V 262144        /* vocabulary size */

/* ------------------------------------------------------------------ chain */

typedef struct {
  int32_t B;                 /* rows (>= 0) */
  int32_t K;                 /* drafts per row, 0 <= K <= SPEC_MAX_K */
  int32_t V;                 /* vocabulary size, 1 <= V <= SPEC_MAX_V */
  int32_t dtype;             /* spec_dtype of both logit arrays */
  int32_t mode;              /* spec_mode */
  float margin_kappa;        /* GREEDY only: margin threshold; <= 0 = strict match */
  const void *target_logits; /* [B, K+1, V]: row j is the target's logits for the
                                token at draft position j (row K: bonus) */
  const void *draft_logits;  /* [B, K, V]: the logits the drafter sampled y_j from;
                                masked entries are -inf.  STOCHASTIC only (may be
                                NULL in GREEDY) */
  const int32_t *draft_tokens; /* [B, K] */
  const float *temperature;  /* [B] per-row T > 0 applied to both laws; NULL = 1.
                                GREEDY uses it only inside the margin ratio */
  const float *u_accept;     /* [B, K] uniforms in [0,1) of the acceptance tests
                                (STOCHASTIC only) */
  const float *u_sample;     /* [B, K+1] uniforms in [0,1): u_sample[b,j] draws the
                                correction when position j is the first rejection,
                                u_sample[b,K] draws the bonus (STOCHASTIC only) */
} spec_chain_args;

typedef struct {
  int32_t *accepted_len; /* [B] number of accepted drafts a, 0..K (-1: bad row) */
  int32_t *out_tokens;   /* [B, K+1] y_0..y_{a-1}, then the correction or bonus
                            token, then -1 */
  int32_t *num_emitted;  /* [B] a + 1 (0: bad row) */
  int32_t *row_status;   /* [B] SPEC_ROW_* */
  /* Optional diagnostics (NULL to skip), STOCHASTIC only, unspecified for
   * rows with a nonzero row_status.  p and q are given for every j < K,
   * independently of the walk: */
  float *p_at_draft;     /* [B, K] p_j(y_j) */
  float *q_at_draft;     /* [B, K] q_j(y_j) */
  float *resid_mass;     /* [B, K] sum_v [p_j - q_j]+ at the position where the
                            walk stops on a rejection (the residual that is
                            sampled), 0 at every other position */
} spec_chain_out;

/* Bytes of workspace spec_verify_chain needs for these sizes (any mode and
 * dtype).  0 on invalid sizes. */
size_t spec_verify_chain_workspace_size(int32_t B, int32_t K, int32_t V);

/* Bytes of workspace spec_verify_chain_truncated needs for these sizes (any
 * dtype): the records of spec_verify_chain plus a 2-byte maximum per chunk
 * of logits that the selection of the thresholds reads, about V / 8 bytes
 * per logit row, and 512 bytes per target row for small kept sets (c3:
 * 11.7 MB).  Never less than
 * spec_verify_chain_workspace_size, so one such workspace serves both calls;
 * spec_drift_residuals needs this size too.  0 on invalid sizes. */
size_t spec_verify_chain_truncated_workspace_size(int32_t B, int32_t K, int32_t V);

/*
 * spec_verify_chain -- one verification step of B independent chains.
 *
 * STOCHASTIC (DVC; CRS section 2): p_j = softmax(target_j / T_b),
 * q_j = softmax(draft_j / T_b).  Position j accepts iff
 * p_j(y_j)/q_j(y_j) >= 1 or u_accept[b,j] < p_j(y_j)/q_j(y_j).  The walk
 * stops at the first rejecting j and emits the inverse CDF of [p_j - q_j]+
 * at u_sample[b,j] (the smallest v whose cumulative residual mass, in
 * vocabulary order, exceeds u * total); if the residual is numerically zero
 * it draws from p_j instead.  If all K drafts pass, the bonus is the inverse
 * CDF of p_K at u_sample[b,K].
 *
 * GREEDY (SMB; MNW section 3): position j accepts iff y_j is the lowest-
 * index argmax of target_j, or margin_kappa > 0 and
 * p(y_j)/p(top1) > margin_kappa at temperature T_b (evaluated in fp64 as
 * l(y_j) - l(top1) > T_b * ln(kappa)).  The first failure emits the argmax;
 * if all pass, the bonus is argmax target_K.  draft_logits is not read.
 *
 * Precision: fp32 arithmetic (fp32 accumulation, hardware exp2/log2); the
 * greedy, tree and margin decisions are exact.
 */
spec_status spec_verify_chain(const spec_chain_args *args, const spec_chain_out *out,
                              void *ws, size_t ws_bytes, void *stream);

/*
 * spec_verify_chain_static -- spec_verify_chain with a scratch buffer built
 * into the library instead of one the caller passes.  The pages have no
 * counterpart: this is a convenience of this library, not part of the method.
 *
 * It is meant for callers that cannot allocate device memory where they
 * verify: a plain C host loop that has no device allocator of its own, a
 * serving engine whose memory pool has already claimed the device's free
 * memory for its KV cache, or a decode loop that must not pay the
 * device-wide synchronisation a cudaFree implies.  The call itself never
 * allocates or frees anything.
 *
 * Limit: the built-in buffer holds SPEC_STATIC_WS_BYTES (4 MiB) per device.
 * A problem whose spec_verify_chain_workspace_size(B, K, V) is larger is
 * rejected with SPEC_ERR_STATIC_LIMIT before anything is launched.  4 MiB
 * covers, for example, B = 256 chains of K = 8 drafts over V = 128256.
 *
 * Set-up: the first call on a device (with that device current) looks up
 * the buffer's device address once; that lookup may load the library's
 * kernels onto the device.  Make that first call before any stream capture
 * begins.  The address is kept for the life of the process: it does not
 * survive cudaDeviceReset (or any other teardown of the device's primary
 * context), after which this entry point must not be called again.
 *
 * Concurrency: all calls on one device share the one buffer.  Calls queued
 * on one stream run one after another and are safe; calls whose kernels may
 * overlap on the GPU (other streams, other host threads) race on the buffer.
 * Such a call may return wrong tokens, or stall for up to the wait limit
 * (spec_set_wait_timeout_ns, 1 s by default) because another call advanced
 * the buffer's generation under its readers, and then report its rows as
 * SPEC_ROW_TIMEOUT.  The buffer never needs clearing.
 *
 * Arguments, outputs and status codes are otherwise those of
 * spec_verify_chain.
 */
#define SPEC_STATIC_WS_BYTES ((size_t)4 << 20)
spec_status spec_verify_chain_static(const spec_chain_args *args, const spec_chain_out *out,
                                     void *stream);

/* ------------------------------------------------------------------- tree */

typedef struct {
  int32_t B;                 /* rows (>= 0) */
  int32_t N;                 /* nodes per tree incl. the root, 1..SPEC_MAX_TREE_NODES */
  int32_t V;                 /* vocabulary size */
  int32_t dtype;             /* spec_dtype */
  float margin_kappa;        /* <= 0: strict argmax match */
  const void *target_logits; /* [B, N, V]: row i = target logits after node i
                                (node 0 = root = last committed token) */
  const int32_t *parent;     /* [B, N]: parent[b,0] = -1, 0 <= parent[b,i] < i */
  const int32_t *node_tokens;/* [B, N]: token of node i (entry 0 ignored) */
  const float *temperature;  /* [B] for the margin ratio; NULL = 1 */
} spec_tree_args;

typedef struct {
  int32_t *accepted_len; /* [B] depth d of the kept node (edges from the root) */
  int32_t *path_nodes;   /* [B, N] node ids on the kept root path, root
                            excluded, then -1 (use to compact tree KV entries) */
  int32_t *out_tokens;   /* [B, N] tokens of those nodes, then argmax of the kept
                            node's target row, then -1 */
  int32_t *num_emitted;  /* [B] d + 1 */
  int32_t *row_status;   /* [B] SPEC_ROW_* */
} spec_tree_out;

size_t spec_verify_tree_workspace_size(int32_t B, int32_t N, int32_t V);

/*
 * spec_verify_tree -- greedy (+ margin) verification of one parent-indexed
 * draft tree per row (SMB 'Beyond Two Models'; MNW section 3).  Node i >= 1
 * is accepted iff its parent is accepted and node_tokens[i] is the argmax of
 * target[parent[i]] or the margin rule promotes it.  The kept node is the
 * deepest accepted one (ties: lowest node index).
 */
spec_status spec_verify_tree(const spec_tree_args *args, const spec_tree_out *out,
                             void *ws, size_t ws_bytes, void *stream);

/* --------------------------------------------------------------- rollback */

/*
 * spec_rollback_lengths -- committed KV-cache lengths that agree with the
 * emitted tokens (DVC 'Speculation needs cache rollback'; CRS section 5).
 *
 * kv_len_in [B]: cache entries before the verify pass.  The pass fed the
 * last emitted token and the drafts, so the entries of that token and of the
 * accepted drafts are valid; the new correction/bonus token has none yet.
 * Emission is cut after the first eos_id (kept; eos_id < 0: none) and so the
 * sequence (kv_len_in + 1 tokens before the step) does not exceed max_len[b]
 * (max_len NULL: no limit).  With n tokens kept and a = accepted_len[b]:
 *   committed_kv_len[b] = kv_len_in[b] + 1 + min(n, a),  num_emitted_out[b] = n.
 * Rows with accepted_len < 0 keep kv_len_in and emit 0.
 * out_tokens [B, max_emit] and num_emitted_in [B] are the verify outputs.
 */
spec_status spec_rollback_lengths(int32_t B, int32_t max_emit, const int32_t *kv_len_in,
                                  const int32_t *accepted_len, const int32_t *num_emitted_in,
                                  const int32_t *out_tokens, int32_t eos_id,
                                  const int32_t *max_len, int32_t *committed_kv_len,
                                  int32_t *num_emitted_out, void *stream);

/* ------------------------------------------------------------------ misc */

/*
 * spec_verify_chain_truncated -- spec_verify_chain (STOCHASTIC mode only,
 * else SPEC_ERR_DTYPE) with top-k / top-p truncated target and draft laws
 * ("Speculative Decoding: Draft, Verify, and Correct", 'Preserve the
 * distribution you actually intend': if top-p (or top-k) filtering defines
 * the target sampling law, acceptance and correction both use the truncated
 * p, and q must be the truncated law that actually produced the draft).
 *
 * Per row b, applied to every p_j and q_j after the temperature: top-k
 * (1 <= top_k[b] < V, else off) keeps the tokens whose logit is >= the k-th
 * largest (ties at the boundary kept); then top-p (0 < top_p[b] < 1, else
 * off) keeps, of those, whole groups of equal logits in descending order
 * until their renormalised mass reaches top_p[b].  Everything else of
 * spec_verify_chain holds with p and q replaced by the renormalised
 * truncated laws: a draft outside the kept set of p is rejected, the
 * residual and the bonus are drawn from them.  Either array may be NULL;
 * both NULL is spec_verify_chain.  The top-p boundary is a floating-point
 * decision taken in fp32 (the band rule covers rows whose cumulative mass
 * lands within ~1e-5 of top_p).  The workspace must hold
 * spec_verify_chain_truncated_workspace_size(B, K, V) bytes (when both
 * arrays are NULL, spec_verify_chain's size).
 * After the one-thread generation step, three kernels: the stream of
 * spec_verify_chain, which also keeps, per truncated logit row, the largest
 * logit of every chunk of 32 (bf16) or 16 (fp32) it reads; per truncated
 * logit row the top-k and top-p thresholds, from the logits of the chunks
 * whose maxima can reach them (a row they cannot settle passes over its own
 * logits); then the per-row resolve, which draws from p's kept set when the
 * selection handed it over (at most 64 tokens) and passes over the
 * stopping position's logits otherwise.
 */
typedef struct {
  const int32_t *top_k;  /* [B] device, or NULL */
  const float *top_p;    /* [B] device, or NULL */
} spec_truncation;

spec_status spec_verify_chain_truncated(const spec_chain_args *args, const spec_truncation *trunc,
                                        const spec_chain_out *out, void *ws, size_t ws_bytes,
                                        void *stream);

/*
 * spec_drift_residuals -- the free supervision signal of "Speculative
 * Decoding Under Distribution Shift: DRIFT Recalibration" (the residual
 * paragraph of its method): at every drafted position j < K of row b, the m
 * tokens of highest target probability (ties to the lower token id), in
 * that order, and the target minus the draft log-probability on them, in
 * nats, from the full temperature-scaled distributions (p and q as in
 * spec_verify_chain).  The page's "shared top m tokens" is read as the
 * target's top m.  A masked (-inf) draft logit gives +inf.
 *
 * Reads target_logits, draft_logits, temperature, B, K, V and dtype of
 * `args` (the rest is ignored; draft_tokens may be NULL).  K <= 64,
 * 1 <= m <= 64 and m <= V (else SPEC_ERR_SHAPE / SPEC_ERR_ARG), B <= 65535.
 * support [B, K, m] int32, residual [B, K, m] float32, row_status [B]
 * (device, caller-owned): a row with a non-finite logit, no finite logit or
 * a bad temperature at any drafted position gets its code and support -1,
 * residual NaN.  The workspace must hold
 * spec_verify_chain_truncated_workspace_size(B, K, V) bytes.
 * After the one-thread generation step, three kernels: the stream of
 * spec_verify_chain over positions 0 .. K-1 of both laws, which also keeps
 * the largest logit of every chunk of 32 (bf16) or 16 (fp32) target logits;
 * one CTA per drafted position, which takes the support from the logits of
 * the chunks whose maxima can reach the m-th largest (a row they cannot
 * settle is searched whole) and writes the residuals; then one CTA per row
 * for the row's status.  Residuals carry fp32 rounding: agreement with an exact
 * computation is within about 1e-4 nats for logits of magnitude up to ~50/T.
 */
spec_status spec_drift_residuals(const spec_chain_args *args, int32_t m, int32_t *support,
                                 float *residual, int32_t *row_status, void *ws, size_t ws_bytes,
                                 void *stream);

/* ------------------------------------------------------- after verification */

/*
 * spec_kv_compact_tree -- keep the KV-cache entries of each row's accepted
 * tree path ("Speculative Decoding: Draft, Verify, and Correct", 'Speculation
 * needs cache rollback': keep the cache for the accepted prefix and discard
 * the rest; "Speculative Decoding: How a Small Model Speeds Up a Big One",
 * 'Where Speculative Decoding Disappoints': rejected drafts' keys and values
 * must be rewound).
 *
 * The verify pass wrote tree node i of row b at token slot kv_len_in[b] + i
 * (node 0 is the root, the last committed token).  With a = accepted_len[b]
 * and path_nodes[b][0..a-1] as returned by spec_verify_tree, the entry of
 * path node k moves to slot kv_len_in[b] + 1 + k, in place, in every plane;
 * spec_rollback_lengths then gives the committed length.  A chain needs no
 * move (its accepted drafts already sit in order).
 *
 * Cache layout, all in bytes: the entry of (plane p, row b, slot s) starts at
 * kv + p*plane_stride + b*row_stride + s*tok_stride and is entry_bytes long
 * (for example planes = layers x {K, V}, entry = heads x head_dim x element
 * size).  kv must be 16-byte aligned and entry_bytes and the three strides
 * multiples of 16 (else SPEC_ERR_ALIGN).  The moved entries must not overlap
 * other rows' or planes' entries.
 *
 * row_status[b] (optional, device, [B]): 0, or SPEC_ROW_BAD_PARENT when the
 * path is not strictly increasing within [1, N) or the slots leave
 * [0, S_max); such a row is left untouched.  a <= 0 is a no-op.
 * B, planes <= 65535.  Asynchronous on `stream`; no workspace.
 */
typedef struct {
  int32_t B;              /* rows */
  int32_t N;              /* tree nodes per row, root included: 1..SPEC_MAX_TREE_NODES */
  int32_t planes;         /* independent planes (layer x K/V, ...) */
  int32_t pad;
  int64_t S_max;          /* token slots per row */
  int64_t entry_bytes;    /* bytes of one token's entry in one plane */
  int64_t plane_stride;   /* bytes between planes */
  int64_t row_stride;     /* bytes between rows */
  int64_t tok_stride;     /* bytes between token slots */
  void *kv;               /* device, read and written in place */
  const int32_t *kv_len_in;     /* [B] cache length before the verify pass */
  const int32_t *accepted_len;  /* [B] from spec_verify_tree */
  const int32_t *path_nodes;    /* [B, N] from spec_verify_tree */
} spec_kv_compact_args;

spec_status spec_kv_compact_tree(const spec_kv_compact_args *args, int32_t *row_status,
                                 void *stream);

/*
 * spec_adaptive_tree_policy -- one step of the per-sequence draft-tree shape
 * policy of "Margins, Not Windows: Training-Free Per-Step Lossy Speculative
 * Decoding" ('Method', dynamic draft tree-shaping), for B sequences at once.
 * For each row, with the step's accepted_len, the verified draft depth and
 * the draft's top-1 probability p1 for the next step:
 *   f    = accepted_len / depth, clamped to [0, 1] (0 if depth <= 0)
 *   ema  = alpha * f + (1 - alpha) * ema          (alpha = 0.3 on the page)
 *   zero = accepted_len == 0 ? zero + 1 : 0
 *   zero >= breaker (5 on the page): shape = start, ema = ema0, zero = 0
 *   else dcs = min(1, clamp(p1, 0, 1) * ema / divisor) and
 *        shape[i] = floor(shallow[i] + dcs * (deep[i] - shallow[i]) + 0.5)
 * with shape = (nsteps, top-k, number of draft tokens).  The page's range is
 * shallow (3, 4, 4) <-> deep (7, 1, 8).  The page does not print the score's
 * formula; this product form, saturating through the divisor, is the
 * plainest reading of its description.  All arithmetic in fp64, each
 * operation rounded on its own, so results are reproducible bit for bit.
 * ema [B] (fp64) and zero_run [B] are per-sequence state, read and written;
 * shape [B, 3] is written.  SPEC_ERR_ARG: alpha outside [0, 1], divisor not
 * finite and > 0, ema0 not finite, or breaker < 1.
 */
typedef struct {
  double alpha;       /* weight of the newest step in the moving average */
  double divisor;     /* saturation point of the confidence score */
  double ema0;        /* moving average after a reset */
  int32_t shallow[3]; /* (nsteps, top-k, ndt) at score 0 */
  int32_t deep[3];    /* (nsteps, top-k, ndt) at score 1 */
  int32_t start[3];   /* shape restored by the circuit breaker */
  int32_t breaker;    /* consecutive zero-accept steps that trigger it */
} spec_adaptive_params;

spec_status spec_adaptive_tree_policy(const spec_adaptive_params *params, int32_t B,
                                      const int32_t *accepted_len, const int32_t *depth,
                                      const float *draft_top1, double *ema, int32_t *zero_run,
                                      int32_t *shape, void *stream);

/* Zero-fill a workspace on `stream` (a cudaMemsetAsync).  Optional: the
 * verify calls do not need a zeroed workspace. */
spec_status spec_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* Human-readable name of a spec_status. */
const char *spec_status_string(spec_status s);

/*
 * Bounded on-device waits.  Every wait of the stochastic kernels on an
 * asynchronous copy or on another block's record gives up after this many
 * nanoseconds (default 1e9 = 1 s), marks the rows it served SPEC_ROW_TIMEOUT
 * and lets the kernel finish.  The greedy and tree kernels stream with plain
 * loads and never wait.  Process-wide setting, read at each launch.
 * spec_debug_force_wait_timeout(1) tests the give-up path on a healthy GPU:
 * the bulk-copy stream waits on a barrier that nothing completes, and the
 * truncation and DRIFT kernels withhold their records, so every reader gives
 * up (or finds a record missing) and its rows report SPEC_ROW_TIMEOUT; 0
 * turns it off.
 */
void spec_set_wait_timeout_ns(uint64_t ns);
uint64_t spec_get_wait_timeout_ns(void);
void spec_debug_force_wait_timeout(int on);

#ifdef SV_BOUNDS
/*
 * Bounds-check builds only (the library compiled with -DSV_BOUNDS, e.g.
 * libspecverify_bounds.so; the pages have no counterpart: a test aid that
 * stands in for a memory checker).  Their chain and tree kernels check every
 * computed global or shared-memory index before the access; a bad one is
 * counted, the first one's source line kept, and the access skipped, never
 * trapped (the row's outputs then come out wrong or flagged).
 * spec_debug_bounds writes the count and that line of every kernel launched
 * since its last call, then clears them; it returns the CUDA error of the
 * reads (synchronous).  spec_debug_bounds_selftest enqueues one check that
 * fails by design without touching memory, so the record can be seen to work.
 */
int spec_debug_bounds(unsigned *count, unsigned *line);
int spec_debug_bounds_selftest(void *stream);
#endif

#ifdef __cplusplus
}
#endif
#endif /* SPECVERIFY_H */
