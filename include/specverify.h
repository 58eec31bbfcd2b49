/*
 * specverify.h -- C ABI of the GB300 speculative-decoding verify library
 * (libspecverify.so, CUDA kernels for sm_103a).
 *
 * The verify step compares K drafted tokens with the target model's
 * distributions and emits between 1 and K+1 tokens per sequence:
 *
 *   "Speculative Decoding & Draft Model Topologies: Slashing Enterprise LLM
 *   Latency by 3.5x in 2026", sec. 2 (Mathematical Foundation: Speculative
 *   Verification & Rejection Sampling): accept x with probability
 *   min(1, p(x)/q(x)) using u ~ U(0,1); on rejection discard x and every later
 *   draft and resample from max(0, p - q) / sum max(0, p - q).
 *   "Speculative Decoding for LLM Inference: How Draft-and-Verify Accelerates
 *   Token Generation", sections "The draft-and-verify loop" (longest accepted
 *   prefix, one resampled token, one bonus token when every draft is accepted)
 *   and "The correctness guarantee".
 *   "Speculative Decoding at Scale: Latency Reduction in Distributed LLM
 *   Serving", sequence diagram (greedy form: accept matching tokens, reject the
 *   first mismatch, plus one bonus token) and sec. 1 (relu(P - Q) residual).
 *   "Speculative Decoding in Production: How Small Draft Models & Medusa Heads
 *   Deliver 2x-3x LLM Speedups Without Accuracy Loss", sec. 2 (P_accept) and
 *   sec. 4 (SpecInfer candidate trees verified under a 2D causal mask).
 *
 * Conventions shared by every entry point
 *   - All array arguments are DEVICE pointers to contiguous row-major memory
 *     owned by the caller.  The library keeps no reference after the call.
 *   - Calls are asynchronous and ordered on `stream` (0 = legacy default
 *     stream).  Per-call scratch memory comes from a library-owned,
 *     stream-ordered CUDA memory pool on the current device and is returned on
 *     the same stream (spec_verify_bf16_static_scratch alone uses a fixed
 *     buffer instead).
 *   - bf16 logits are passed as their raw 16-bit patterns (uint16_t).
 *   - Logits may be -inf (masked vocabulary).  A row containing NaN or +inf,
 *     a row with no finite entry, a drafted token outside [0, V), or a tree
 *     parent index outside [-1, i) is bad data: that sequence's count is -1,
 *     every one of its output tokens is -1 (tree: mask words 0), and bit
 *     SPEC_FLAG_BAD_DATA is set in the device status word (spec_get_status).
 *     The call itself still returns SPEC_OK and never traps.
 *   - Return codes: SPEC_OK, or a negative SPEC_ERR_* from host-side checks
 *     (nothing is launched) or from the CUDA runtime.
 *   - Results are deterministic: the same inputs and seed give bit-identical
 *     outputs on every run.
 *   - Calls may be captured into a CUDA graph on `stream` (the scratch then
 *     comes from graph memory nodes of the library's pool and is initialised
 *     on the captured stream).  Make one call on the device before the first
 *     capture: it creates the library's device state and pool, which a
 *     capture in global mode would not allow.  Calls may also come from
 *     several host threads at once, each on its own stream.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_OK 0
#define SPEC_ERR_NULL (-1)        /* a required pointer is NULL */
#define SPEC_ERR_SHAPE (-2)       /* B < 0, K outside [0, 255], V < 1, N outside [0, 1024], or size overflow */
#define SPEC_ERR_TEMPERATURE (-3) /* temperature NaN, negative, or in (0, 1e-30) */
#define SPEC_ERR_CUDA (-4)        /* CUDA runtime error; spec_status_string(-4) gives the message */
#define SPEC_ERR_SCRATCH (-5)     /* spec_verify_bf16_static_scratch: the problem needs more than
                                     SPEC_STATIC_SCRATCH_BYTES of scratch */
#define SPEC_ERR_HINT (-6)        /* spec_verify_khint_*: k_min < 0, k_max > 255, k_min > k_max,
                                     a NaN threshold or h_lo > h_hi */

/* Size of the fixed per-device scratch buffer of spec_verify_bf16_static_scratch. */
#define SPEC_STATIC_SCRATCH_BYTES ((size_t)8 << 20)

#define SPEC_FLAG_BAD_DATA 1u     /* some sequence had bad data (see above) */
#define SPEC_FLAG_TIMEOUT 2u      /* an internal bounded wait ran out; outputs of that call are invalid */

/*
 * Speculative-sampling verification of B independent sequences.
 *
 *   target_logits  [B, K+1, V]  target row i scores draft position i; row K is
 *                               the bonus row.
 *   draft_logits   [B, K, V]    draft row i is the distribution x_i was drawn
 *                               from.  May be NULL when temperature == 0 or K == 0.
 *   draft_tokens   [B, K]       int32 drafted ids x_i.  May be NULL when K == 0.
 *   temperature    tau > 0: p = softmax(target / tau), q = softmax(draft / tau)
 *                  (the same tau divides both).  tau == 0 selects greedy
 *                  verification: x_i is accepted while it equals the lowest-id
 *                  argmax g_i of target row i; the token after the accepted
 *                  prefix is g_n; draft_logits is not read.
 *   seed           64-bit Philox-4x64-10 key word.  Position i's acceptance
 *                  uniform uses counter (b, i, 0, 0), the resampling uniform
 *                  counter (b, n, 1, 0); key (seed, 0x5350454356455249).  The
 *                  first output word r gives u = (2 (r >> 12) + 1) 2^-53, an
 *                  odd multiple of 2^-53 in (0, 1).
 *   out_tokens     [B, K+1] int32: x_0 .. x_{n-1}, then the resampled (n < K)
 *                  or bonus (n == K) token, then -1 padding.
 *   out_n_accepted [B] int32: n in [0, K], or -1 for bad data.
 *
 * Acceptance: x_i is kept iff q_i(x_i) == 0 or u_i < p_i(x_i) / q_i(x_i).
 * n is the first rejected position (K if none).  The emitted token at n is the
 * smallest id j whose running sum (vocabulary order) of the weights exceeds
 * w * (total weight), w the resampling uniform; the weights are
 * max(0, p_n - q_n) when n < K and p_K when n == K (p_n when a rejection left
 * no positive residual through rounding).
 * B == 0 is a no-op.  Sizes: K <= 255, (K+1) * V and B * (K+1) * V must fit in
 * 62 bits.
 */
int spec_verify_f32(const float *target_logits, const float *draft_logits,
                    const int32_t *draft_tokens, int B, int K, int V, float temperature,
                    uint64_t seed, int32_t *out_tokens, int32_t *out_n_accepted,
                    cudaStream_t stream);
int spec_verify_bf16(const uint16_t *target_logits, const uint16_t *draft_logits,
                     const int32_t *draft_tokens, int B, int K, int V, float temperature,
                     uint64_t seed, int32_t *out_tokens, int32_t *out_n_accepted,
                     cudaStream_t stream);

/*
 * spec_verify with early exit: the same arguments, layouts and outputs, but
 * only the rows the result depends on are read -- the target and draft rows
 * of positions 0..n (n the first rejection) and target row K when all K
 * drafts are accepted.  A sequence is decided as soon as its positions 0..n
 * are resolved, and the statistics slices of its later rows that have not
 * started by then are skipped, so far fewer logits are read when drafts are
 * rejected early ([P2] "The draft-and-verify loop": the tokens after the
 * first rejection are discarded, so their rows cannot change the result).
 * Tokens and counts equal spec_verify's on every sequence whose inputs are
 * valid.  Bad data is checked, in position order, only on what is used: a
 * NaN / +inf logit or an empty row among target/draft rows 0..n, a drafted
 * token x_0..x_n outside [0, V), or a bad target row K when n == K; then
 * n = -1, the sequence's outputs are -1 and SPEC_FLAG_BAD_DATA is set.  Bad
 * data after the first rejection is not reported (spec_verify reports it).
 * With K > 31 every row is read (the sequence is decided once all positions
 * are resolved).
 * Temperature 0 (draft_logits may be NULL): the greedy verify of spec_verify
 * with the same early exit -- target rows are read by position and a row
 * after a decided sequence's first mismatch n is skipped.  Bad data is
 * checked in position order on what is used: target row i (NaN, +inf, no
 * finite maximum), then x_i outside [0, V), for i = 0..n, and target row K
 * when all K drafts match.  (1 <= K <= 31; otherwise every row is read, as in
 * spec_verify.)
 */
int spec_verify_early_exit_f32(const float *target_logits, const float *draft_logits,
                               const int32_t *draft_tokens, int B, int K, int V, float temperature,
                               uint64_t seed, int32_t *out_tokens, int32_t *out_n_accepted,
                               cudaStream_t stream);
int spec_verify_early_exit_bf16(const uint16_t *target_logits, const uint16_t *draft_logits,
                                const int32_t *draft_tokens, int B, int K, int V, float temperature,
                                uint64_t seed, int32_t *out_tokens, int32_t *out_n_accepted,
                                cudaStream_t stream);

/*
 * spec_verify_bf16 without any device allocation.  The pages describe the
 * verify step only; they have no counterpart of this entry point, which exists
 * for callers that cannot let the library allocate: a serving process that
 * reserved nearly all device memory up front, a latency-critical loop that
 * must not enter the allocator, or a device without stream-ordered memory
 * pools.
 *
 * Arguments, layouts, outputs, temperature == 0 (greedy) and results are
 * exactly those of spec_verify_bf16: the same kernels run and give
 * bit-identical outputs.  The difference is the scratch memory: instead of
 * the stream-ordered pool, every call uses one fixed buffer of
 * SPEC_STATIC_SCRATCH_BYTES per device that is part of the library image
 * (a static __device__ array, created when the module is loaded); the call
 * only clears parts of it with cudaMemsetAsync on `stream` and makes no
 * cudaMalloc/cudaFree or other allocating call.
 *   - A problem whose scratch exceeds SPEC_STATIC_SCRATCH_BYTES returns
 *     SPEC_ERR_SCRATCH and launches nothing (for K = 8, V = 152064, B = 256
 *     needs about 1.7 MB).
 *   - The buffer's address is looked up on the first call on each device
 *     (cudaGetSymbolAddress, which may load the module): make that first call
 *     before any stream capture on that device.
 *   - One buffer serves every call on a device, so calls that overlap in time
 *     (different streams or host threads on the same device) race on it and
 *     produce garbage; calls issued in order on one stream are safe.
 */
int spec_verify_bf16_static_scratch(const uint16_t *target_logits,
                                    const uint16_t *draft_logits,
                                    const int32_t *draft_tokens, int B, int K, int V,
                                    float temperature, uint64_t seed, int32_t *out_tokens,
                                    int32_t *out_n_accepted, cudaStream_t stream);

/*
 * spec_verify_* plus the verify step's intermediate probabilities, for
 * checking against a reference.  Same arguments, then (each may be NULL):
 *   out_row_stats  [B, 2K+1, 2] float: for target rows 0..K then draft rows
 *                  0..K-1, max_v z_v / tau and sum_v exp(z_v / tau - max).
 *                  (tau == 0: not written.)
 *   out_pq         [B, K, 2] float: p_i(x_i), q_i(x_i) for every position.
 *   out_resid_mass [B] float: total mass of the distribution the token at n
 *                  was drawn from (sum max(0, p_n - q_n), or about 1 for the
 *                  bonus row).
 *   out_row_entropy [B, 2K+1] float: entropy in nats, -sum_v p(v) ln p(v), of
 *                  each row's softmax(z / tau), rows in the order of
 *                  out_row_stats, computed in the same streaming pass ([P3]
 *                  sec. 3 "Engineering Recommendations": choose the
 *                  speculation depth from how uncertain the distribution is).
 *                  Unspecified for the rows of a sequence flagged bad.
 * With temperature == 0 the extra outputs are not written (the greedy argmax
 * of every target row comes from spec_verify_greedy_argmax_*).
 */
int spec_verify_stats_f32(const float *target_logits, const float *draft_logits,
                          const int32_t *draft_tokens, int B, int K, int V, float temperature,
                          uint64_t seed, int32_t *out_tokens, int32_t *out_n_accepted,
                          float *out_row_stats, float *out_pq, float *out_resid_mass,
                          float *out_row_entropy, cudaStream_t stream);
int spec_verify_stats_bf16(const uint16_t *target_logits, const uint16_t *draft_logits,
                           const int32_t *draft_tokens, int B, int K, int V, float temperature,
                           uint64_t seed, int32_t *out_tokens, int32_t *out_n_accepted,
                           float *out_row_stats, float *out_pq, float *out_resid_mass,
                           float *out_row_entropy, cudaStream_t stream);

/*
 * spec_verify_* plus a suggested draft length for each sequence's next
 * iteration, from the same streaming pass ([P3] sec. 3 "Engineering
 * Recommendations": a shorter draft where the target is uncertain, a longer
 * one where it is predictable; [P2] "How much speedup to expect": the draft
 * length trades tokens per iteration against work wasted on rejections).
 * The pages give no formula.  Here
 *   Hbar_b = mean over target rows i = 0..n_b of H(softmax(z_i / tau)) (nats),
 * the rows whose verdicts made this call's tokens, and
 *   out_k_next[b] = clamp(K + 1, k_min, k_max) if Hbar_b < h_lo,
 *                   clamp(K - 1, k_min, k_max) if Hbar_b > h_hi,
 *                   clamp(K,     k_min, k_max) otherwise,
 * or -1 for a sequence flagged bad.  The mean is the fp64 sum of the rows'
 * fp32 entropies over n_b + 1, compared in fp64.
 *   temperature   must be > 0 (else SPEC_ERR_TEMPERATURE).
 *   h_lo, h_hi    thresholds in nats, h_lo <= h_hi; k_min, k_max in [0, 255],
 *                 k_min <= k_max (else SPEC_ERR_HINT).
 *   out_k_next    [B] int32, required.
 *   out_mean_entropy [B] float, may be NULL: Hbar_b (NaN for a bad sequence).
 * Tokens and n_accepted are those of spec_verify_* with the same seed.
 */
int spec_verify_khint_f32(const float *target_logits, const float *draft_logits,
                          const int32_t *draft_tokens, int B, int K, int V, float temperature,
                          uint64_t seed, double h_lo, double h_hi, int k_min, int k_max,
                          int32_t *out_tokens, int32_t *out_n_accepted, int32_t *out_k_next,
                          float *out_mean_entropy, cudaStream_t stream);
int spec_verify_khint_bf16(const uint16_t *target_logits, const uint16_t *draft_logits,
                           const int32_t *draft_tokens, int B, int K, int V, float temperature,
                           uint64_t seed, double h_lo, double h_hi, int k_min, int k_max,
                           int32_t *out_tokens, int32_t *out_n_accepted, int32_t *out_k_next,
                           float *out_mean_entropy, cudaStream_t stream);

/*
 * Greedy verification (temperature 0) that also writes the lowest-id argmax of
 * every target row: out_row_argmax [B, K+1] int32 (-1 for an unusable row).
 */
int spec_verify_greedy_argmax_f32(const float *target_logits, const int32_t *draft_tokens,
                                  int B, int K, int V, int32_t *out_tokens,
                                  int32_t *out_n_accepted, int32_t *out_row_argmax,
                                  cudaStream_t stream);
int spec_verify_greedy_argmax_bf16(const uint16_t *target_logits, const int32_t *draft_tokens,
                                   int B, int K, int V, int32_t *out_tokens,
                                   int32_t *out_n_accepted, int32_t *out_row_argmax,
                                   cudaStream_t stream);

/*
 * Greedy verification of a candidate tree per sequence (SpecInfer-style).
 *
 *   target_logits [B, N+1, V]  row 0: the root's next-token row; row i+1: node i.
 *   tree_tokens   [B, N] int32 the candidate token of node i.
 *   parent_idx    [B, N] int32 parent of node i, -1 for a child of the root;
 *                              parents precede children (parent_idx[i] < i).
 *   out_path      [B, N+1] int32: tokens of the accepted path from the root's
 *                 child down to the deepest accepted node, then the bonus
 *                 token (argmax of that node's row; of row 0 when no node is
 *                 accepted), then -1 padding.
 *   out_len       [B] int32: path length + 1, or -1 for bad data.
 *   out_mask      [B, N, ceil(N/32)] uint32: bit j of word j/32 in row i is set
 *                 iff j == i or node j is an ancestor of node i (the 2D tree
 *                 attention mask; it depends only on parent_idx).
 * Node i is accepted iff its parent is accepted (the root always is) and its
 * token equals the lowest-id argmax of its parent's row; the deepest accepted
 * node wins, the lowest node index on ties.  N <= 1024.  N == 0 emits the
 * bonus token of row 0 only.
 */
int spec_tree_verify_greedy_f32(const float *target_logits, const int32_t *tree_tokens,
                                const int32_t *parent_idx, int B, int N, int V,
                                int32_t *out_path, int32_t *out_len, uint32_t *out_mask,
                                cudaStream_t stream);
int spec_tree_verify_greedy_bf16(const uint16_t *target_logits, const int32_t *tree_tokens,
                                 const int32_t *parent_idx, int B, int N, int V,
                                 int32_t *out_path, int32_t *out_len, uint32_t *out_mask,
                                 cudaStream_t stream);

/*
 * spec_tree_verify_greedy with early exit: the same arguments, layouts and
 * outputs, but a node's row is read only while the node may still be
 * accepted.  A node's row serves only to judge its children and as the bonus
 * row ([P1] sec. 4: the longest accepted path is kept), so the rows under a
 * rejected node cannot change the result.  Rows are streamed by node index;
 * a row of a node already known to be rejected is skipped.  Path, length and
 * mask equal spec_tree_verify_greedy's on valid inputs.  Bad data is checked
 * on what is used: every parent index (the mask needs all of them), the
 * root's row, the rows of accepted nodes and the tokens of nodes whose parent
 * is accepted; bad data under a rejected node is not reported.  For
 * 1 <= N <= 32 (one warp holds a sequence's nodes); larger trees read every
 * row, as spec_tree_verify_greedy does.
 */
int spec_tree_verify_greedy_early_exit_f32(const float *target_logits, const int32_t *tree_tokens,
                                           const int32_t *parent_idx, int B, int N, int V,
                                           int32_t *out_path, int32_t *out_len, uint32_t *out_mask,
                                           cudaStream_t stream);
int spec_tree_verify_greedy_early_exit_bf16(const uint16_t *target_logits, const int32_t *tree_tokens,
                                            const int32_t *parent_idx, int B, int N, int V,
                                            int32_t *out_path, int32_t *out_len, uint32_t *out_mask,
                                            cudaStream_t stream);

/*
 * Stochastic verification of a candidate tree per sequence (temperature > 0).
 * The tree of "Speculative Decoding in Production: How Small Draft Models &
 * Medusa Heads Deliver 2x-3x LLM Speedups Without Accuracy Loss", sec. 4,
 * checked with the acceptance rule and residual of "Speculative Decoding &
 * Draft Model Topologies: Slashing Enterprise LLM Latency by 3.5x in 2026",
 * sec. 2, one node at a time.
 *
 *   target_logits [B, N+1, V]  row 0: the root; row i+1: node i.
 *   draft_logits  [B, N+1, V]  row u+1: the draft distribution the children
 *                              of node u (row 0: of the root) were drawn from.
 *   tree_tokens, parent_idx    as for spec_tree_verify_greedy_*.
 *   temperature   > 0: p = softmax(target / T), q = softmax(draft / T).
 *   seed          Philox-4x64-10 key word as for spec_verify_*: node c's
 *                 acceptance uniform uses counter (b, c, 0, 0); the final
 *                 draw at node u uses counter (b, u + 1, 1, 0).
 *   out_path      [B, N+1] int32: the accepted tokens from the root down, then
 *                 the token drawn at the last accepted node, then -1 padding.
 *   out_len       [B] int32: accepted nodes + 1, or -1 for bad data.
 * At the current node (the root first) with current distribution P = p of its
 * row, the children are tried in node-index order: child x is accepted with
 * probability min(1, P(x) / q(x)) (always when q(x) == 0) and becomes the
 * current node; a rejected child replaces P by norm(max(0, P - q)) for the
 * next sibling.  When no child is accepted, or the node is a leaf, one token
 * is drawn from the current P by inverse CDF in vocabulary order.  Each
 * emitted token is then distributed exactly as p at its position.  Every row
 * of both inputs is checked for bad data, leaves' draft rows included.
 * N <= 1024.  temperature 0 is SPEC_ERR_TEMPERATURE here (the greedy tree is
 * spec_tree_verify_greedy_*).  Two kernels run on `stream`: the row
 * statistics, then the walk, launched with programmatic stream serialisation
 * (capturable into a CUDA graph); scratch comes from the library's
 * stream-ordered pool.  Asynchronous on `stream`.
 */
int spec_tree_verify_sampling_f32(const float *target_logits, const float *draft_logits,
                                  const int32_t *tree_tokens, const int32_t *parent_idx, int B,
                                  int N, int V, float temperature, uint64_t seed,
                                  int32_t *out_path, int32_t *out_len, cudaStream_t stream);
int spec_tree_verify_sampling_bf16(const uint16_t *target_logits, const uint16_t *draft_logits,
                                   const int32_t *tree_tokens, const int32_t *parent_idx, int B,
                                   int N, int V, float temperature, uint64_t seed,
                                   int32_t *out_path, int32_t *out_len, cudaStream_t stream);

/*
 * Acceptance statistics of a batch of verify outputs ([P2] "How much speedup
 * to expect": the per-position acceptance rate and the expected tokens per
 * iteration, measured instead of predicted).
 *
 *   n_accepted       [B] int32 counts as written by spec_verify (-1 = bad
 *                    sequence).  For tree outputs pass out_len - 1.
 *   K                drafts per sequence, 0 <= K <= 1024.
 *   out_hist         [K+2] uint64 (required): out_hist[j] = #(n == j) for
 *                    j = 0..K; out_hist[K+1] counts every other value.
 *   out_alpha        [K] double or NULL: #(n > i) / #(n >= i), the fraction of
 *                    sequences whose position i was tested that accepted it
 *                    (NaN if none reached position i).
 *   out_mean_tokens  [1] double or NULL: mean of n + 1 over the counted
 *                    sequences (NaN if none).
 * All pointers are device pointers; counts are exact.  Returns SPEC_OK,
 * SPEC_ERR_NULL (out_hist NULL, or n_accepted NULL with B > 0),
 * SPEC_ERR_SHAPE (B < 0, K outside [0, 1024]) or SPEC_ERR_CUDA.
 */
int spec_acceptance_stats(const int32_t *n_accepted, int B, int K, uint64_t *out_hist,
                          double *out_alpha, double *out_mean_tokens, cudaStream_t stream);

/*
 * N-gram (prompt-lookup) drafting: for every sequence, draft up to K tokens by
 * copying what followed an earlier occurrence of the history's last tokens
 * ([P2] "Speculative Decoding for LLM Inference: How Draft-and-Verify
 * Accelerates Token Generation", sections "The variant landscape" and
 * "Support in production systems", FAQ "Do all variants require a separate
 * draft model?": candidates copied from the prompt or prior output through an
 * n-gram lookup, no drafter weights).
 *   tokens        [B, stride] int32, device: row b holds the history of
 *                 sequence b (prompt and output so far) in its first
 *                 lengths[b] entries; the rest is never read.
 *   lengths       [B] int32, device.
 *   n_min, n_max  match lengths tried, longest first: 1 <= n_min <= n_max <= 32.
 *   K             drafts per sequence, 0 <= K <= 4096.
 *   out_drafts    [B, K] int32, device: the drafts, -1 past the last one.
 *   out_n_drafts  [B] int32, device: the number of drafts (0 when nothing
 *                 matches).
 *   out_match_len [B] int32, device (may be NULL): the match length m used (0
 *                 when nothing matches).
 * Rule: the longest m in [n_min, n_max] whose last-m-token suffix occurred
 * earlier wins; of its occurrences the latest one with at least one token
 * after it (end e <= L - 1) is copied: drafts = h[e .. e + d - 1],
 * d = min(K, L - e).  Token values are compared and copied as given.
 * Bad data: a length outside [0, stride] gives n_drafts = match_len = -1 and
 * -1 drafts for that sequence and sets SPEC_FLAG_BAD_DATA.
 * Each history token is read from device memory once; scratch (8 bytes per
 * 4096 positions of every row, plus 256 bytes) comes from the library's
 * stream-ordered pool.  Two kernels run on `stream`, the second with
 * programmatic stream serialisation (capturable into a CUDA graph).  A
 * bounded wait that ran out sets SPEC_FLAG_TIMEOUT; the outputs are then in
 * range (drafts copied from the history or -1) but may miss the best match.
 * Returns SPEC_OK, SPEC_ERR_NULL (an output, or tokens / lengths with B > 0,
 * is NULL), SPEC_ERR_SHAPE (B < 0, stride < 1 or above 2^30, bad n_min /
 * n_max / K, or B * ceil(stride / 4096) >= 2^31 - 2^20) or SPEC_ERR_CUDA.
 * Asynchronous on `stream`.
 */
int spec_ngram_draft(const int32_t *tokens, const int32_t *lengths, int B, int stride, int n_min,
                     int n_max, int K, int32_t *out_drafts, int32_t *out_n_drafts,
                     int32_t *out_match_len, cudaStream_t stream);

/*
 * Test hook, for fault-injection tests: the next n scratch allocations from
 * the library's pool (any device, any entry point that allocates) fail as if
 * the pool were exhausted.  The call then returns SPEC_ERR_CUDA before
 * launching anything, and spec_status_string(SPEC_ERR_CUDA) says so.  n <= 0
 * clears it.  Returns the count that was pending.  The pages have no
 * counterpart; it exists so that the error path can be tested without a real
 * allocation failure.
 */
int spec_test_fail_allocations(int n);

/*
 * Test hook, for failure-detection tests: every bounded wait inside the
 * kernels of later calls on the current device gives up after `iterations`
 * polls (0 restores the default, about half a second).  A wait that gives up
 * sets SPEC_FLAG_TIMEOUT, the kernel returns without faulting, and that call's
 * outputs are invalid; the device stays usable.  Synchronises the device
 * first.  Returns SPEC_OK or SPEC_ERR_CUDA.  The pages have no counterpart; it
 * exists so that the timeout path can be exercised without a real stall.
 */
int spec_test_spin_limit(uint32_t iterations);

/*
 * Test hook, for failure-detection tests: runs each of the library's seven
 * bounded-wait helpers once on a slot that nothing writes and once on a slot
 * already written, under the limit spec_test_spin_limit set (synchronous; its
 * own status words, not the device status word).  out_flags (host, 2 words):
 * [0] bit k set when helper k gave up on the unwritten slot and flagged
 * SPEC_FLAG_TIMEOUT (the decision read also returns "no decision");
 * [1] bit k set when helper k flagged the written slot.  A correct library
 * returns {0x7f, 0}.  Returns SPEC_OK, SPEC_ERR_NULL or SPEC_ERR_CUDA.  With
 * the default limit each unwritten wait lasts about half a second or more.
 */
int spec_test_wait_probe(uint32_t* out_flags);

/*
 * Synchronises `stream`, then returns in *flags_out (may be NULL) the device
 * status word of the current device (an OR of SPEC_FLAG_* set by every call
 * since the last read) and clears it.  Returns SPEC_OK or SPEC_ERR_CUDA.
 */
int spec_get_status(cudaStream_t stream, uint32_t *flags_out);

/* Static description of a return code; for SPEC_ERR_CUDA the message of the
 * calling thread's most recent CUDA error. */
const char *spec_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
