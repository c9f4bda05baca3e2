/*
 * specverify.h - C ABI of libspecverify: the batched target-side verify/sample
 * step of speculative decoding, on one NVIDIA GB300 (sm_103a).
 *
 * The operation (from "11.1 核心原理: Draft + Verify 与 Rejection Sampling",
 * sections 11.1.1-11.1.3 and its code listing 10-1, and from the notes "Fast
 * Inference from Transformers via Speculative Decoding", speculative-sampling
 * paragraph):
 *
 *   A draft proposed gamma tokens d_0..d_{gamma-1}, drawing d_i from its actual
 *   proposal distribution q_i.  One target forward over the context plus the
 *   drafts gave gamma+1 rows of logits; row i predicts the token at draft
 *   position i (it was computed from the prefix ending just before d_i), row
 *   gamma is the distribution after all drafts (section 11.1.1).  The target
 *   distribution of row i is p_i = softmax(logits_i / temperature), optionally
 *   restricted by top-k and then top-p and renormalised (section 11.1.2: the
 *   same transforms the draft applied to q_i).
 *
 *   Sampling (sv_verify_sample): for i = 0, 1, ... accept d_i iff
 *   u_i < a_i = min(1, p_i(d_i) / q_i(d_i)); stop at the first rejection n.
 *   On a rejection draw the next token from the residual
 *   norm(max(p_n - q_n, 0)); if every draft was accepted (n = gamma) draw the
 *   bonus token from p_gamma.  Emit d_0..d_{n-1} followed by that token.
 *
 *   Greedy (sv_verify_greedy): accept while d_i == argmax p_i (ties -> the
 *   lowest index); at the first mismatch n emit argmax p_n; if all match emit
 *   argmax p_gamma.
 *
 * Readings where the pages are silent (fixed by this ABI):
 *   - the caller supplies gamma+1 uniforms per sequence: uniforms[b][i] is the
 *     accept test of position i, uniforms[b][gamma] the one final draw;
 *   - a categorical draw with uniform u from weights r is the inverse CDF in
 *     token-index order: the smallest v with sum_{w<=v} r(w) > u * sum(r);
 *   - truncation order: temperature, then top-k ranked by (logit descending,
 *     index ascending), renormalise, then top-p keeps the shortest prefix of
 *     that ranking whose mass reaches top_p (the crossing token is kept);
 *   - q is used as given: it must already be the draft's actual (truncated,
 *     renormalised) proposal; the step never re-truncates it.
 *
 * Memory and execution conventions (all entry points):
 *   - Every pointer argument is DEVICE memory owned by the caller, contiguous
 *     row-major, left unmodified except outputs and workspace.  The library
 *     allocates nothing.
 *   - logits and q must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Arguments are validated on the host first; a failed
 *     validation returns an error status and launches nothing.  A launch
 *     failure returns SV_ERR_CUDA.
 *   - The workspace must be zero-filled before its first use (for example with
 *     cudaMemsetAsync).  Every call that completes leaves it zero-filled again,
 *     so one workspace can be reused for any sequence of calls on one stream.
 *     Calls that run concurrently must use different workspaces.
 *   - Problems in the DATA never fault or trap: they set bits in the
 *     per-sequence status word (SV_SEQ_*) and the outputs stay in range.
 *   - B = 0 is a valid empty call: nothing is launched.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1,  /* a size, pointer, alignment or parameter is invalid */
  SV_ERR_UNSUPPORTED = 2,  /* valid but not implemented (see sv_verify_sample) */
  SV_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than sv_workspace_bytes() */
  SV_ERR_CUDA = 4,         /* a CUDA launch or runtime call failed */
  SV_ERR_TIMEOUT = 5       /* reserved: a bounded device wait gave up */
} sv_status;

typedef enum {
  SV_DTYPE_F32 = 0,
  SV_DTYPE_BF16 = 1,
  SV_DTYPE_F16 = 2
} sv_dtype;

/* Per-sequence status bits written to out_status[b]. */
#define SV_SEQ_DRAFT_OUT_OF_RANGE 1 /* some d_i outside [0, V): that position is rejected (a_i = 0) */
#define SV_SEQ_Q_NOT_POSITIVE 2     /* some q_i(d_i) <= 0 or NaN: a_i = 1 if p_i(d_i) > 0, else 0 */
#define SV_SEQ_BAD_ROW 4            /* a row holds NaN or +inf, or only -inf: outputs undefined but in range */
#define SV_SEQ_RESIDUAL_ZERO 8      /* rejection with zero residual mass: the token was drawn from p_n */

/* Opaque stream handle, binary-compatible with cudaStream_t. */
typedef struct CUstream_st* sv_stream_t;

/* Limits checked by the entry points. */
#define SV_MAX_GAMMA 64
#define SV_MAX_VOCAB (1 << 24)
#define SV_MAX_TOP_K 1024
#define SV_MAX_STOP_TOKENS 64

/*
 * Bytes of device workspace that sv_verify_sample / sv_verify_greedy need for
 * this problem size (any logits dtype).  top_k = 0 for greedy or for sampling
 * without top-k.  Returns 0 for invalid sizes (B < 0, gamma < 0 or above
 * SV_MAX_GAMMA, V < 1 or above SV_MAX_VOCAB, top_k outside [0, SV_MAX_TOP_K]).
 */
size_t sv_workspace_bytes(int B, int gamma, int V, int top_k);

/*
 * Sampling verify (speculative sampling, section 11.1.2 and listing 10-1).
 *
 *   B, gamma, V      batch size (>= 0), drafts per sequence (0..SV_MAX_GAMMA),
 *                    vocabulary size (1..SV_MAX_VOCAB)
 *   logits           [B][gamma+1][V] of logits_dtype; row i predicts the token
 *                    at draft position i, row gamma the bonus position
 *   q                [B][gamma][V] float32, the draft's actual proposal
 *                    probabilities (non-negative), 16-byte aligned, in device
 *                    memory or in pinned host memory the device reads at the
 *                    same address (sv_pointer_device_readable): the kernels
 *                    read q only at the drafted tokens, at the kept
 *                    candidates (top-k / top-p) and along the residual row
 *                    of a rejected sequence, so host-resident q crosses the
 *                    host link only there; or NULL:
 *                    deterministic drafts (n-gram, prompt lookup), each q_i
 *                    one-hot at d_i.  Then a_i = p_i(d_i) and a rejection at
 *                    i draws from p_i with d_i removed, renormalised; no q
 *                    bytes are read.  (The pages use the draft's actual q,
 *                    section 11.1.2; a one-hot q is that q for such drafts.)
 *   draft_tokens     [B][gamma] int32 drafted ids; may be NULL when gamma = 0
 *   uniforms         [B][gamma+1] float32 in [0, 1)
 *   temperature      > 0 and finite
 *   top_k            0 = off, else 1..SV_MAX_TOP_K
 *   top_p            in (0, 1]; 1 = off.  With top_k = 0 (or top_k >= V) the
 *                    kept set of each row is found by a mass-weighted
 *                    bisection over the logits' order-preserving keys (any
 *                    V; ties at the crossing logit kept in index order), and
 *                    the final draw runs under that mask.
 *   out_tokens       [B][gamma+1] int32: d_0..d_{n-1}, the drawn token, then -1
 *   out_num_accepted [B] int32: n in 0..gamma (n+1 tokens were emitted)
 *   out_accept_prob  [B][gamma] float32 a_i for every position, or NULL
 *   out_status       [B] int32 SV_SEQ_* bits, or NULL
 *   workspace        device scratch of at least sv_workspace_bytes(B, gamma, V, top_k)
 */
sv_status sv_verify_sample(int B, int gamma, int V,
                           const void* logits, sv_dtype logits_dtype,
                           const float* q, const int32_t* draft_tokens,
                           const float* uniforms,
                           float temperature, int top_k, float top_p,
                           int32_t* out_tokens, int32_t* out_num_accepted,
                           float* out_accept_prob, int32_t* out_status,
                           void* workspace, size_t workspace_bytes,
                           sv_stream_t stream);

/*
 * Greedy verify (section 11.1.2, greedy rule).  Arguments as in
 * sv_verify_sample; no q, uniforms, temperature or truncation (they do not move
 * the argmax).  Ties of the argmax go to the lowest index; -0.0 equals +0.0.
 */
sv_status sv_verify_greedy(int B, int gamma, int V,
                           const void* logits, sv_dtype logits_dtype,
                           const int32_t* draft_tokens,
                           int32_t* out_tokens, int32_t* out_num_accepted,
                           int32_t* out_status,
                           void* workspace, size_t workspace_bytes,
                           sv_stream_t stream);

/*
 * Greedy verify for callers that cannot allocate device memory - for example
 * a plugin whose host framework owns every device allocation and passes none
 * down, a runtime that fixes its memory budget before serving, or a loop that
 * must not call cudaMalloc because it can synchronise the device.  (The pages
 * have no counterpart: this is a deployment convenience, not part of the
 * method.)  Same arguments, results and status bits as sv_verify_greedy,
 * without the workspace.
 *
 * Scratch: the library holds one array of SV_NOALLOC_SCRATCH_BYTES (8 MiB)
 * in device memory on every GPU that loads it, until the process exits.  A
 * problem whose sv_workspace_bytes(B, gamma, V, 0) exceeds that size returns
 * SV_ERR_WORKSPACE and launches nothing.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture.  Every call clears the part
 * of the array it uses (cudaMemsetAsync on `stream`) and then runs the greedy
 * kernel on it.  All calls on a device share the one array: calls that can
 * overlap on the GPU (different streams, several host threads) race and must
 * be serialised by the caller.  Allocates nothing: no cudaMalloc / cudaFree.
 */
#define SV_NOALLOC_SCRATCH_BYTES (8u << 20)
sv_status sv_verify_greedy_noalloc(int B, int gamma, int V,
                                   const void* logits, sv_dtype logits_dtype,
                                   const int32_t* draft_tokens,
                                   int32_t* out_tokens, int32_t* out_num_accepted,
                                   int32_t* out_status,
                                   sv_stream_t stream);

/*
 * Ragged rounds (the lmnt.cn blog section 3.2 and the reading notes let the
 * number of drafts change per round; here per sequence).  As sv_verify_sample
 * / sv_verify_greedy, plus
 *
 *   gamma_b   [B] int32 device array, drafts of sequence b in this round, in
 *             [0, gamma] (values outside are clamped).  Sequence b is then
 *             exactly the step with gamma = gamma_b[b] on its first
 *             gamma_b[b] + 1 logit rows, gamma_b[b] q rows and drafts: the
 *             acceptance scan stops at gamma_b[b], the bonus comes from row
 *             gamma_b[b], the final draw uses uniforms[b][gamma_b[b]].  Rows,
 *             q rows and drafts beyond gamma_b[b] are ignored (they may hold
 *             anything; they raise no status bit).  out_tokens is padded with
 *             -1 after the drawn token, out_accept_prob with 0 beyond
 *             gamma_b[b].  NULL gamma_b with B > 0 is SV_ERR_INVALID_ARG.
 * The arrays keep their padded [B][gamma (+1)] shapes.
 */
sv_status sv_verify_sample_ragged(int B, int gamma, int V,
                                  const void* logits, sv_dtype logits_dtype,
                                  const float* q, const int32_t* draft_tokens,
                                  const float* uniforms, const int32_t* gamma_b,
                                  float temperature, int top_k, float top_p,
                                  int32_t* out_tokens, int32_t* out_num_accepted,
                                  float* out_accept_prob, int32_t* out_status,
                                  void* workspace, size_t workspace_bytes,
                                  sv_stream_t stream);
sv_status sv_verify_greedy_ragged(int B, int gamma, int V,
                                  const void* logits, sv_dtype logits_dtype,
                                  const int32_t* draft_tokens, const int32_t* gamma_b,
                                  int32_t* out_tokens, int32_t* out_num_accepted,
                                  int32_t* out_status,
                                  void* workspace, size_t workspace_bytes,
                                  sv_stream_t stream);

/*
 * Sampling verify with the draft's proposal supplied as the draft model's
 * LOGITS ("11.1 核心原理", section 11.1.2: temperature and truncation are
 * applied to the draft's q_i exactly as to the target's p_i, and q_i must be
 * the draft's actual proposal).  As sv_verify_sample, except
 *
 *   q_logits        [B][gamma][V] of q_logits_dtype (float32, bfloat16 or
 *                   float16), 16-byte aligned: the draft's logits at the
 *                   drafted positions; may be NULL when gamma = 0.  q_i =
 *                   softmax(q_logits_i / temperature), truncated as below.
 *                   When q_logits has the logits' dtype and V is a multiple
 *                   of the 16-byte vector width (8 for 16-bit types, 4 for
 *                   float32), the verify kernels stream the draft rows with
 *                   the target rows and form q where they need it (it is
 *                   never written out); otherwise a kernel first writes q in
 *                   float32 into the workspace and the sv_verify_sample
 *                   path runs on it.  A row holding NaN or +inf, or only
 *                   -inf, gives q_i = 0, so testing position i raises
 *                   SV_SEQ_Q_NOT_POSITIVE.
 *   top_k, top_p    as in sv_verify_sample, applied to q_i too: q_i is the
 *                   draft's softmax renormalised over its own top-k then
 *                   top-p set (one CTA per draft row: radix select of the
 *                   k-th largest, ties to the lowest index, sorted top-p
 *                   prefix), zero elsewhere.  Same limits as sv_verify_sample.
 *   workspace       at least sv_qlogits_workspace_bytes(B, gamma, V, top_k)
 *                   bytes: the layout of sv_workspace_bytes(B, gamma, V,
 *                   top_k) first (so the other entry points can share it),
 *                   then the float32 q and the kept-index lists of truncated
 *                   draft rows.  The usual contract covers all of it: zero-
 *                   filled before the first use, left zero-filled by every
 *                   call that completes (truncated q is written only where
 *                   kept, and cleared after the call).
 */
size_t sv_qlogits_workspace_bytes(int B, int gamma, int V, int top_k);
sv_status sv_verify_sample_qlogits(int B, int gamma, int V,
                                   const void* logits, sv_dtype logits_dtype,
                                   const void* q_logits, sv_dtype q_logits_dtype,
                                   const int32_t* draft_tokens, const float* uniforms,
                                   float temperature, int top_k, float top_p,
                                   int32_t* out_tokens, int32_t* out_num_accepted,
                                   float* out_accept_prob, int32_t* out_status,
                                   void* workspace, size_t workspace_bytes,
                                   sv_stream_t stream);

/*
 * Ending a round early ("11.1 核心原理", listing 10-1's comment: an EOS / stop
 * token or max_new_tokens may end the round, and no bonus token is forced).
 * In place on the outputs of a verify call:
 *
 *   tokens          [B][gamma+1] int32 (device), out_tokens of the call;
 *                   rewritten: the emitted tokens tokens[b][0 .. n_b] are
 *                   kept up to and including the first stop token, and at
 *                   most max_new[b] of them; the rest become -1
 *   num_accepted    [B] int32 (device), n_b as the call wrote it (clamped to
 *                   [0, gamma])
 *   stop_tokens     n_stop int32 token ids (device), n_stop in
 *                   [0, SV_MAX_STOP_TOKENS]; may be NULL when n_stop = 0
 *   max_new         [B] int32 (device) token budgets (<= 0 keeps nothing), or
 *                   NULL for no budget
 *   out_num_emitted [B] int32 (device): how many tokens remain
 *
 * Returns SV_ERR_INVALID_ARG for bad sizes or NULL arrays, SV_ERR_CUDA if the
 * launch fails.  Runs on `stream`.
 */
sv_status sv_truncate_emitted(int B, int gamma, int32_t* tokens, const int32_t* num_accepted,
                              const int32_t* stop_tokens, int n_stop, const int32_t* max_new,
                              int32_t* out_num_emitted, sv_stream_t stream);

/* Static description of a status code. */
const char* sv_status_string(sv_status s);

/*
 * Names of the kernels the last sv_verify_sample / sv_verify_greedy call made
 * on this host thread launched, comma-separated in launch order (for example
 * "cluster_kernel", or "stream_dense_kernel,final_draw_kernel");
 * "" before the first call, after
 * a call that launched nothing (B = 0, an argument error) or a launch failure.
 * Static storage owned by the library; thread-local.
 */
const char* sv_last_kernels(void);

/*
 * 1 if the device reads p at the same address: device memory, managed
 * memory, or host memory that is pinned and mapped (cudaHostAlloc under
 * unified addressing); else 0 (pageable host memory, a foreign pointer,
 * NULL).  Launches nothing; clears the CUDA error it may raise.  Callers use
 * it before passing q in host memory (see sv_verify_sample).
 */
int sv_pointer_device_readable(const void* p);

/*
 * Measurement hook (outside the verify computation; used by the benchmark to
 * time each kernel with CUDA events).  Registers n = 3 caller-created CUDA
 * events (cudaEvent_t handles cast to void*) that every later call records on
 * its stream: events[0] before its first kernel, events[1] after the kernel
 * that streams the logits, events[2] after its last kernel.  n = 0 clears the
 * registration.  The record between the two kernels of an untruncated sampling
 * call prevents their overlapped (programmatic) launch, so time headline
 * throughput with the hook cleared.  Process-wide state; not thread-safe.
 * Returns SV_ERR_INVALID_ARG for n other than 0 or 3 or NULL events.
 */
sv_status sv_set_timing_events(void* const* events, int n);

/*
 * Vocabulary-sharded verify.  When a row's logits (and q) are split by token
 * range across processes - the layout a tensor-parallel output layer leaves -
 * each process calls these steps on its own range [v0, v0 + V) of the Vg
 * tokens, and the caller moves a few records between them.  The result is
 * the one sv_verify_sample / sv_verify_greedy gives on the whole rows (same
 * method, section 11.1.2 and listing 10-1): the softmax normaliser of every
 * row and the inverse CDF of the final draw are sums over tokens, so every
 * shard reduces its own range.  Supported: greedy, and sampling without
 * truncation (q dense or NULL).  Per call, every shard in the same order:
 *
 *   1. sv_shard_row_stats           -> stats_local [B][gamma+1][SV_SHARD_STAT_WORDS]
 *   2. all-gather of stats_local    -> stats_all [nshard][B][gamma+1][...],
 *                                      shards in token order (v0 ascending)
 *   3. sv_shard_scan                -> every output; for sampling all but
 *                                      out_tokens[b][n] and out_status
 *      (greedy ends here)
 *   4. sv_shard_draw_sums           -> totals_local [B][SV_SHARD_TOTAL_WORDS]
 *   5. all-gather of totals_local   -> totals_all [nshard][B][...]
 *   6. sv_shard_draw_pick           -> out_tokens[b][n]: the drawn token on
 *                                      the shard whose range holds it, -1 on
 *                                      every other shard; out_status
 *   7. element-wise maximum of out_tokens over the shards (all-reduce MAX).
 *
 * Every shard computes identical outputs in steps 3 and 6 (the merges run in
 * shard order), so only the token of step 6 needs the reduction.  Arguments
 * as in sv_verify_sample, with: V = this shard's token count (>= 1), v0 its
 * first token, Vg the vocabulary (v0 + V <= Vg); logits [B][gamma+1][V] and
 * q [B][gamma][V] are this shard's columns, contiguous; draft_tokens and
 * uniforms hold GLOBAL token ids and are the same on every shard; nshard in
 * 1..SV_MAX_SHARDS, rank = this shard's position in token order.  greedy != 0
 * selects the greedy rule (temperature and q ignored).  The workspace (at
 * least sv_shard_workspace_bytes(B, gamma, V), zero-filled before first use
 * and left zero-filled) carries the state from step 3 to steps 4 and 6; steps
 * 1-6 of one call must run in order on one stream.  Record buffers are
 * device memory, 16-byte aligned.  Status bits as in sv_verify_sample; a draft
 * id outside [0, Vg) sets SV_SEQ_DRAFT_OUT_OF_RANGE.
 */
#define SV_MAX_SHARDS 32
#define SV_SHARD_STAT_WORDS 8   /* 32-bit words per row record */
#define SV_SHARD_TOTAL_WORDS 8  /* 32-bit words per sequence total */
size_t sv_shard_workspace_bytes(int B, int gamma, int V);
sv_status sv_shard_row_stats(int B, int gamma, int V, int v0, int Vg,
                             const void* logits, sv_dtype logits_dtype,
                             const float* q, const int32_t* draft_tokens,
                             float temperature, int greedy,
                             void* stats_local, sv_stream_t stream);
sv_status sv_shard_scan(int nshard, int B, int gamma, int V, int Vg,
                        const void* stats_all, const int32_t* draft_tokens,
                        const float* uniforms, float temperature, int greedy,
                        int32_t* out_tokens, int32_t* out_num_accepted,
                        float* out_accept_prob, int32_t* out_status,
                        void* workspace, size_t workspace_bytes,
                        sv_stream_t stream);
sv_status sv_shard_draw_sums(int B, int gamma, int V, int v0, int Vg,
                             const void* logits, sv_dtype logits_dtype,
                             const float* q, const int32_t* draft_tokens,
                             float temperature, void* totals_local,
                             void* workspace, size_t workspace_bytes,
                             sv_stream_t stream);
sv_status sv_shard_draw_pick(int nshard, int rank, int B, int gamma, int V,
                             int v0, int Vg, const void* logits,
                             sv_dtype logits_dtype, const float* q,
                             const int32_t* draft_tokens,
                             const float* uniforms, float temperature,
                             const void* totals_all, int32_t* out_tokens,
                             int32_t* out_status, void* workspace,
                             size_t workspace_bytes, sv_stream_t stream);

/*
 * Vocabulary shards with truncation (top_k in 1..SV_MAX_TOP_K, then
 * top_p): every token of a row's global top-k is in the top-k of the shard
 * holding it, so the shards' candidate lists hold the whole truncated
 * distribution and the q it needs (section 11.1.2: the transforms of p; q
 * used as given).  Per call, every shard:
 *
 *   1. sv_shard_topk_candidates  -> cand_local [B][gamma+1][top_k+1] entries
 *                                   of SV_SHARD_CAND_BYTES: the row's local
 *                                   top-k by (logit, lowest index) with q of
 *                                   the drafted row at each (one-hot at d_i
 *                                   when q is NULL), after a header entry
 *   2. all-gather of cand_local  -> cand_all [nshard][...], token order
 *   3. sv_shard_topk_finish      -> every output (identical on every shard)
 *
 * Requirements: V a multiple of 8 (16-bit logits) or 4 (float32) (else
 * SV_ERR_UNSUPPORTED); nshard * top_k <= 2048 (else SV_ERR_UNSUPPORTED).
 * The workspace of step 1 is at least sv_workspace_bytes(B, gamma, V, top_k)
 * (zero-filled, left zero-filled); step 3 needs none.  Top-p without top-k
 * is not offered sharded.
 */
#define SV_SHARD_CAND_BYTES 16
sv_status sv_shard_topk_candidates(int B, int gamma, int V, int v0, int Vg,
                                   const void* logits, sv_dtype logits_dtype,
                                   const float* q, const int32_t* draft_tokens,
                                   float temperature, int top_k,
                                   void* cand_local, void* workspace,
                                   size_t workspace_bytes, sv_stream_t stream);
sv_status sv_shard_topk_finish(int nshard, int B, int gamma, int Vg,
                               const void* cand_all,
                               const int32_t* draft_tokens,
                               const float* uniforms, float temperature,
                               int top_k, float top_p, int32_t* out_tokens,
                               int32_t* out_num_accepted,
                               float* out_accept_prob, int32_t* out_status,
                               sv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
