/*
 * specdec.h -- C ABI of the GB300 (sm_103a) verify step of speculative decoding.
 *
 * The operation (source: "Chapter 15: Decoding acceleration", LLM edge
 * inference notes, section 15.1.2 "mathematical framework of speculative
 * decoding", speculative sampling steps 2-4 and the theorem after them):
 *
 *   for one request with gamma drafted tokens x~_0 .. x~_{gamma-1}, the target
 *   model's logits over gamma+1 positions and the draft's stored
 *   distributions q_0 .. q_{gamma-1}:
 *     p_i      = softmax(logits_i / T)              (T = 0: one-hot argmax)
 *     accept x~_i iff u_i <= min(1, p_i(x~_i) / q_i(x~_i)), i = 0, 1, ...,
 *              stopping at the first rejection k;
 *     if k < gamma: final token ~ max(0, p_k - q_k) / Z        (correction)
 *     else:         final token ~ p_gamma                      (bonus token)
 *   The emitted tokens are x~_0 .. x~_{k-1} followed by the final token; their
 *   law is the target model's (the section's theorem).
 *
 *   The token-tree form generalises the chain: a node's children were drawn
 *   i.i.d. from that node's draft distribution; they are tried in ascending
 *   node index and each rejection replaces the current target distribution P
 *   by max(0, P - q) / sum (recursive rejection over siblings).  Accepting a
 *   child descends; a leaf draws a bonus token from its own target row; a node
 *   whose children are all rejected draws from the renormalised residual.
 *
 * Conventions (all functions):
 *   - every array pointer is a DEVICE pointer owned by the caller (the
 *     *_host calls take host arrays and a device staging buffer); row-major;
 *   - logits and q hold float32 (SPECDEC_F32) or bfloat16 bits (SPECDEC_BF16),
 *     both in the same dtype;
 *   - every device array starts on a multiple of its element size: 4 bytes
 *     for float32 data and for the int32 / float32 arrays, 2 for bfloat16
 *     data; a call given a misaligned device array returns
 *     SPECDEC_ERR_INVALID_ARG and launches nothing (rows need not be 16-byte
 *     aligned: such rows are read through aligned vectors and shifts);
 *   - uniforms are float32 values in (0, 1) that the caller draws (e.g. from a
 *     counter-based generator); the library draws no random numbers;
 *   - the library allocates nothing; scratch lives in a caller-provided
 *     workspace of at least specdec_workspace_size(...) bytes (no
 *     initialisation needed: every call writes what it later reads).  Calls
 *     that share a workspace must not overlap on the GPU;
 *   - `stream` is a cudaStream_t (NULL = legacy default stream); work is
 *     asynchronous and stream-ordered; inputs are read only; outputs are
 *     overwritten entirely;
 *   - the return value reports synchronous argument checks and launch errors
 *     (SPECDEC_ERR_*); data errors inside a request are reported per request
 *     through row_status[b] (SPECDEC_ROW_* bits) and never trap the device;
 *     a request with a nonzero status gets n_accepted = 0, is_bonus = 0 and
 *     -1 in every token output (one exception: when a tree walk's exchange
 *     between the CTAs of a request's cluster runs out of time, the status
 *     gets SPECDEC_ROW_INTERNAL and the other outputs are not to be used);
 *   - B = 0 is a no-op that returns SPECDEC_OK.
 *
 * Numerics: target probabilities are computed in float32 with base-2
 * exponentials (exp(z) = 2^(z log2 e)) and compared in float64; the final
 * draw sums its weights in float32 over short runs of consecutive elements
 * (one 16-byte vector, or 16 or 32 elements, depending on the kernel) and in
 * 64-bit fixed point with 40 fraction bits above that, so the crossing index
 * of the inverse CDF is exact for the weights the kernel computes.
 */
#ifndef SPECDEC_H
#define SPECDEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPECDEC_ABI_VERSION 1

/* element types of logits and q */
#define SPECDEC_F32 0
#define SPECDEC_BF16 1

/* return codes */
#define SPECDEC_OK 0
#define SPECDEC_ERR_INVALID_ARG 1 /* null pointer, bad size or dtype */
#define SPECDEC_ERR_UNSUPPORTED 2 /* sizes beyond the documented limits */
#define SPECDEC_ERR_WORKSPACE 3   /* workspace missing or too small */
#define SPECDEC_ERR_CUDA 4        /* a CUDA runtime call or launch failed */
#define SPECDEC_ERR_STATIC_LIMIT 5 /* sizes need more scratch than specdec_verify_linear_static has */

/* per-request status bits written to row_status[b] */
#define SPECDEC_ROW_OK 0
#define SPECDEC_ROW_BAD_TOKEN 1  /* a drafted token is outside [0, V) */
#define SPECDEC_ROW_BAD_Q 2      /* q at a drafted token is <= 0, NaN or inf */
#define SPECDEC_ROW_NONFINITE 4  /* a target row holds NaN or +inf, no finite value, or a max > 2^100 */
#define SPECDEC_ROW_BAD_TEMP 8   /* temperature not 0 and not in [2^-20, 2^20] */
#define SPECDEC_ROW_BAD_TREE 16  /* parent[0] != -1, parent[n] not in [0, n), or depth > max_depth */
#define SPECDEC_ROW_INTERNAL 32  /* a kernel's bounded wait ran out: for a copy of its own, or (tree walk)
                                    for another CTA of the request's cluster */

/* Limits. */
#define SPECDEC_MAX_GAMMA 32       /* linear: drafted positions per request */
#define SPECDEC_MAX_TREE_NODES 1024
#define SPECDEC_MAX_TREE_DEPTH 64
#define SPECDEC_MAX_V (1 << 21)
#define SPECDEC_MAX_UNIFORMS (1ll << 40) /* words per specdec_philox_uniforms call */
#define SPECDEC_MAX_TOPK 1024            /* candidates of specdec_verify_linear_topk */

/* ABI version of the loaded library (SPECDEC_ABI_VERSION at build time). */
int specdec_abi_version(void);

/* Static, human-readable text of a return code or of one SPECDEC_ROW_* bit. */
const char *specdec_status_string(int code);

/* Bytes of workspace a call with these sizes needs (rows_per_request is
 * gamma+1 for the linear form and N for the tree form).  Depends only on its
 * arguments, not on the device.  Returns 0 for invalid sizes. */
size_t specdec_workspace_size(int B, int rows_per_request, int V, int dtype);

/*
 * Linear verify (section 15.1.2, steps 2-4; bonus draw per section 15.1.3).
 *
 *   logits        [B, gamma+1, V]  target logits; row i scores draft i, row gamma
 *                                  is the bonus row
 *   q             [B, gamma, V]    draft probabilities (as stored, no renormalisation)
 *   draft_tokens  int32 [B, gamma]
 *   temperature   float32 [B]      0 = greedy (argmax accept test, lowest index on ties)
 *   uniforms      float32 [B, gamma+1]  slot i: test of draft i; slot gamma: final draw
 *   n_accepted    int32 [B]        k in [0, gamma]
 *   out_tokens    int32 [B, gamma+1]  x~_0..x~_{k-1}, final token, then -1
 *   final_token   int32 [B]        correction or bonus token
 *   is_bonus      uint8 [B]        1 iff every draft was accepted
 *   row_status    int32 [B]        SPECDEC_ROW_* bits
 *   p_draft       float32 [B, gamma] or NULL: p_i(x~_i) for every position
 *                                  (greedy rows: 1 if x~_i is the argmax, else 0)
 *   workspace     >= specdec_workspace_size(B, gamma+1, V, dtype) bytes
 * Limits: 1 <= gamma <= SPECDEC_MAX_GAMMA, 1 <= V <= SPECDEC_MAX_V.
 */
int specdec_verify_linear(const void *logits, const void *q, int dtype,
                          const int32_t *draft_tokens, const float *temperature,
                          const float *uniforms, int B, int gamma, int V,
                          int32_t *n_accepted, int32_t *out_tokens, int32_t *final_token,
                          uint8_t *is_bonus, int32_t *row_status, float *p_draft,
                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * The normaliser of each request's final draw in the last verify call on
 * `workspace` ("Chapter 15: Decoding acceleration", section 15.1.2 step 4:
 * after a rejection the correction is drawn from max(0, p - q) / Z), a
 * diagnostic for checking the draw against a reference:
 *   mass[b] = Z = sum_v max(0, p_k(v) - q_k(v)) after a rejection at row k
 *             (the linear form), or the sum of the bonus row's p (1 up to
 *             rounding); in the tree form the mass of max(0, p - c q) at the
 *             final node after its rejected siblings (the product of the
 *             renormalisations), 1 up to rounding without one; in the top-k
 *             mode the residual's mass on the k candidates; NaN for greedy
 *             and malformed requests (nothing is drawn).
 * The value comes from the draw's own fixed-point total over the row's merged
 * sum, so it carries the draw's arithmetic.  B, rows_per_request, V, dtype as
 * in that call; mass: device float32 [B].  Asynchronous on `stream`.
 */
int specdec_final_mass(const void *workspace, size_t workspace_bytes, int B,
                       int rows_per_request, int V, int dtype, float *mass, void *stream);

/*
 * Which path specdec_verify_linear takes for these arguments (host only):
 *   SPECDEC_PATH_SMALL_ONE_LAUNCH  a small batch: one cluster of C CTAs per
 *       request (C the largest of 16, 8, 4, 2 of which the device holds B
 *       clusters at once, one CTA per SM) holding its rows in shared memory;
 *       needs rows, logits and q 16-byte aligned and each CTA's 1/C share of
 *       the request's gamma + 1 target rows (plus the gamma q rows, or else
 *       of one q row) fitting its shared memory;
 *   SPECDEC_PATH_TWO_LAUNCHES      the stats pass, then the draw.
 * Every path gives the same outputs and leaves the same workspace.
 * SPECDEC_PATH_NONE for B = 0, -1 for invalid sizes.
 */
#define SPECDEC_PATH_NONE 0
#define SPECDEC_PATH_SMALL_ONE_LAUNCH 1
#define SPECDEC_PATH_TWO_LAUNCHES 3
int specdec_verify_linear_path(int B, int gamma, int V, int dtype, const void *logits,
                               const void *q);

/*
 * How many kernels specdec_verify_linear launches for these arguments: 1 on
 * either one-launch path, 2 on the two-launch path (see
 * specdec_verify_linear_path).  0 for B = 0, -1 for invalid sizes.  Host only.
 */
int specdec_verify_linear_launches(int B, int gamma, int V, int dtype, const void *logits,
                                   const void *q);

/*
 * Phase 1 of either form, callable alone: per-row softmax statistics
 * (section 15.1.2 step 2) of B*rows_per_request rows of V logits, written
 * into the workspace as per-stage partials (max, base-2 exponential sum,
 * first arg-max position).  One streaming pass over the logits.
 *   logits        [B, rows_per_request, V], temperature float32 [B]
 *   q, draft_tokens  linear form: [B, gamma, V] and int32 [B, gamma] with
 *                 gamma = rows_per_request - 1; the pass then also gathers
 *                 each drafted token's logit and q value for phase 2.  Both
 *                 NULL for the tree form or for the statistics alone; one
 *                 without the other is SPECDEC_ERR_INVALID_ARG.
 *   flags         0, or SPECDEC_STATS_ENTROPY to keep per stage the sum of
 *                 p-weighted logit offsets that specdec_row_entropy reads (about
 *                 one extra fused multiply-add per element; the verify calls
 *                 run without it).  Other bits: SPECDEC_ERR_INVALID_ARG.
 */
#define SPECDEC_STATS_ENTROPY 1u /* flag: also the sums specdec_row_entropy needs */
int specdec_row_stats(const void *logits, const void *q, int dtype, const int32_t *draft_tokens,
                      const float *temperature, int B, int rows_per_request, int V,
                      unsigned flags, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Phase 2 of the linear form: the accept test with early stop (section
 * 15.1.2 step 3), the correction / bonus draw (step 4) and every output.
 * Same arguments as specdec_verify_linear; the workspace must hold phase 1's
 * result for the same logits, q, draft_tokens, temperature, B, gamma, V
 * (phase 1 called in its linear form).  Phase 2 leaves that result intact, so
 * it may run again on it (with other uniforms, for instance).
 */
int specdec_linear_finalize(const void *logits, const void *q, int dtype,
                            const int32_t *draft_tokens, const float *temperature,
                            const float *uniforms, int B, int gamma, int V,
                            int32_t *n_accepted, int32_t *out_tokens, int32_t *final_token,
                            uint8_t *is_bonus, int32_t *row_status, float *p_draft,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * Token-tree verify (the chain form above with several i.i.d. siblings per
 * node; siblings tried in ascending node index, residual renormalised after
 * each rejected sibling; candidate-tree notation of section 15.4.1).
 *
 *   logits       [B, N, V]  row n: target distribution after the path to node n
 *   q            [B, N, V]  row n: draft distribution node n's children were drawn from
 *   node_tokens  int32 [B, N]  token of node n (entry 0, the root, is ignored)
 *   parent       int32 [B, N]  parent[0] = -1, 0 <= parent[n] < n
 *   temperature  float32 [B]
 *   uniforms     float32 [B, N]  slot 0: final draw; slot n: test of node n
 *   max_depth    deepest node depth allowed (root = 0)
 *   n_accepted   int32 [B]      accepted nodes on the path (root excluded)
 *   path_nodes   int32 [B, max_depth+1]  0, accepted node ids, then -1
 *   out_tokens   int32 [B, max_depth+1]  accepted tokens, final token, then -1
 *   final_token, is_bonus, row_status  as in the linear form
 *   p_node       float32 [B, N] or NULL: p_parent(token of n) before any
 *                renormalisation (entry 0: 0)
 *   workspace    >= specdec_workspace_size(B, N, V, dtype) bytes
 * Limits: 1 <= N <= SPECDEC_MAX_TREE_NODES, 0 <= max_depth <= SPECDEC_MAX_TREE_DEPTH.
 */
int specdec_verify_tree(const void *logits, const void *q, int dtype,
                        const int32_t *node_tokens, const int32_t *parent,
                        const float *temperature, const float *uniforms, int B, int N, int V,
                        int max_depth, int32_t *n_accepted, int32_t *path_nodes,
                        int32_t *out_tokens, int32_t *final_token, uint8_t *is_bonus,
                        int32_t *row_status, float *p_node, void *workspace,
                        size_t workspace_bytes, void *stream);

/*
 * Linear verify that allocates nothing and takes no workspace.
 *
 * No counterpart in the method description: an addition of this library for
 * callers that cannot allocate device memory for a workspace -- for example a
 * host runtime that forbids allocation after start-up, or a plug-in interface
 * whose calls carry only the inputs and outputs.  The scratch lives in a fixed
 * device array inside the library, SPECDEC_STATIC_SCRATCH_BYTES long, which
 * every GPU that loads the library holds until the process exits.
 *
 * Same arguments and outputs as specdec_verify_linear, without the workspace.
 * Returns SPECDEC_ERR_STATIC_LIMIT, launching nothing, when
 * specdec_workspace_size(B, gamma+1, V, dtype) exceeds the array.
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before capturing a stream into a
 * graph.  All calls share the one array: calls whose work overlaps on the GPU
 * (different streams without ordering, or different host threads) race and
 * corrupt each other's results; serialise them.  Nothing in the array needs
 * to start at zero.  The looked-up address lives as long as the device's
 * context: do not call this entry point after cudaDeviceReset of that device
 * in the same process.
 */
#define SPECDEC_STATIC_SCRATCH_BYTES (4u << 20)
int specdec_verify_linear_static(const void *logits, const void *q, int dtype,
                                 const int32_t *draft_tokens, const float *temperature,
                                 const float *uniforms, int B, int gamma, int V,
                                 int32_t *n_accepted, int32_t *out_tokens, int32_t *final_token,
                                 uint8_t *is_bonus, int32_t *row_status, float *p_draft,
                                 void *stream);

/*
 * Host-buffer forms of the two verify calls.
 *
 * No counterpart in the method description: an addition of this library for
 * callers whose inputs and results live in host memory (one request at a
 * time, the latency case).  Here every array argument is a HOST pointer;
 * only `staging` is device memory.  One call enqueues on `stream`:
 *   1. one host-to-device copy per input array into `staging`;
 *   2. the device call (specdec_verify_linear / specdec_verify_tree) on those
 *      copies, with its workspace inside `staging`;
 *   3. one device-to-host copy per output array (p_draft / p_node skipped
 *      when NULL).
 * It returns once they are enqueued: synchronise `stream` (or an event
 * recorded after the call) before reading the outputs or reusing the input
 * buffers.  Page-locked host memory (cudaHostAlloc, cudaHostRegister) keeps
 * the copies asynchronous; pageable memory works, but the runtime then copies
 * synchronously with respect to the host, and cannot be captured into a CUDA
 * graph.  Arguments, layouts, outputs and return codes as in the device
 * calls, with the staging buffer in place of the workspace:
 *   staging   device memory, 16-byte aligned, at least
 *             specdec_linear_staging_size(B, gamma, V, dtype) /
 *             specdec_tree_staging_size(B, N, V, max_depth, dtype) bytes;
 *             SPECDEC_ERR_WORKSPACE if smaller, unaligned or NULL.  Calls that
 *             share a staging buffer must not overlap on the GPU.
 * The size functions return 0 for invalid sizes and for B = 0.  A CUDA error
 * while enqueuing (SPECDEC_ERR_CUDA) may leave earlier copies enqueued.
 */
size_t specdec_linear_staging_size(int B, int gamma, int V, int dtype);
size_t specdec_tree_staging_size(int B, int N, int V, int max_depth, int dtype);
int specdec_verify_linear_host(const void *logits, const void *q, int dtype,
                               const int32_t *draft_tokens, const float *temperature,
                               const float *uniforms, int B, int gamma, int V,
                               int32_t *n_accepted, int32_t *out_tokens, int32_t *final_token,
                               uint8_t *is_bonus, int32_t *row_status, float *p_draft,
                               void *staging, size_t staging_bytes, void *stream);
int specdec_verify_tree_host(const void *logits, const void *q, int dtype,
                             const int32_t *node_tokens, const int32_t *parent,
                             const float *temperature, const float *uniforms, int B, int N,
                             int V, int max_depth, int32_t *n_accepted, int32_t *path_nodes,
                             int32_t *out_tokens, int32_t *final_token, uint8_t *is_bonus,
                             int32_t *row_status, float *p_node, void *staging,
                             size_t staging_bytes, void *stream);

/* Phase 2 of the tree form (phase 1 is specdec_row_stats with rows_per_request = N). */
int specdec_tree_finalize(const void *logits, const void *q, int dtype,
                          const int32_t *node_tokens, const int32_t *parent,
                          const float *temperature, const float *uniforms, int B, int N,
                          int V, int max_depth, int32_t *n_accepted, int32_t *path_nodes,
                          int32_t *out_tokens, int32_t *final_token, uint8_t *is_bonus,
                          int32_t *row_status, float *p_node, void *workspace,
                          size_t workspace_bytes, void *stream);

/*
 * The linear step with the top-k residual: an APPROXIMATION of step 4 after
 * the implementation note of section 15.1.2 (precompute the residual
 * probabilities of the top-k candidates instead of the whole vocabulary).
 * At a rejection at row k the correction token is drawn from max(0, p - q)
 * restricted to the topk tokens of largest p_k (ties to the lower index) and
 * renormalised; if that mass is 0, from p_k restricted to the candidates.
 * The q row is then read at topk tokens only.  The law of the emitted token
 * is no longer exactly p: its total-variation distance from the exact step's
 * law is the residual mass outside the candidates over the residual mass
 * (the oracle reports it per request).  The accept test, the bonus draw and
 * the greedy rows are exact.  Same arguments and outputs as
 * specdec_verify_linear plus topk in [1, SPECDEC_MAX_TOPK] (values above V
 * act as V, which is the exact step); same workspace size.
 */
int specdec_verify_linear_topk(const void *logits, const void *q, int dtype,
                               const int32_t *draft_tokens, const float *temperature,
                               const float *uniforms, int B, int gamma, int V, int topk,
                               int32_t *n_accepted, int32_t *out_tokens, int32_t *final_token,
                               uint8_t *is_bonus, int32_t *row_status, float *p_draft,
                               void *workspace, size_t workspace_bytes, void *stream);

/*
 * Entropy -sum_v p ln p (natural log) of every target row, for policies that
 * set the draft length from the target's confidence (the adaptive draft
 * length of the multi-token-prediction section: entropy = -sum p(x) log p(x)).
 * Reads the workspace of a specdec_row_stats call made with
 * SPECDEC_STATS_ENTROPY (then phase 2 may run as usual) for the same B,
 * rows_per_request, V, dtype; temperature float32 [B].
 *   entropy  float32 [B, rows_per_request]; 0 for greedy rows (T = 0),
 *            NaN for an invalid temperature, an unusable row, or a workspace
 *            whose statistics were taken without the flag.
 * One small launch; the logits are not read again.
 */
int specdec_row_entropy(const void *workspace, size_t workspace_bytes, int dtype,
                        const float *temperature, int B, int rows_per_request, int V,
                        float *entropy, void *stream);

/*
 * Log-probability under the target of the path a verify step emitted (the
 * path-probability passage of the tree section: log P(path) = sum_i log
 * p(x_i | prefix_i)):
 *     logprob[b] = sum_{j = 0 .. n_accepted[b]} ln p_{row_j}(out_tokens[b, j])
 * with row_j = j for the linear form (path_nodes NULL) and
 * row_j = path_nodes[b, j] for the tree form; out_tokens and path_nodes have
 * rows of path_len entries (gamma + 1, or max_depth + 1), as the verify calls
 * write them.  Greedy requests: 0 along arg-maxima, -inf otherwise.  NaN for
 * a request with a nonzero row_status (row_status may be NULL), an invalid
 * temperature, an unusable row, or a token or node out of range.  Needs the
 * logits and the workspace of the same verify call.
 */
int specdec_path_logprob(const void *logits, int dtype, const float *temperature,
                         const int32_t *out_tokens, const int32_t *n_accepted,
                         const int32_t *path_nodes, const int32_t *row_status, int B,
                         int rows_per_request, int V, int path_len, const void *workspace,
                         size_t workspace_bytes, float *logprob, void *stream);

/*
 * Acceptance rate of every drafted position: alpha[b, i] = sum_v
 * min(p_i(v), q_i(v)), the probability that the test of section 15.1.2
 * accepts one token drawn from q_i (the first term of Lemma 1; the chapter's
 * sliding-window draft length averages these rates).  p_i as in the verify
 * step (greedy rows: one-hot at the first arg-max, so alpha = min(1,
 * q_i(argmax))); q_i as stored.  Reads the logits and q of a linear verify
 * call and the workspace of its specdec_row_stats pass (any flags) for the
 * same B, gamma, V, dtype; a second pass over the drafted logits and q rows
 * (2 * B * gamma * V * elem bytes), so opt-in.
 *   logits [B, gamma+1, V], q [B, gamma, V], temperature float32 [B]
 *   alpha  float32 [B, gamma]; NaN for an invalid temperature or an
 *          unusable target row
 */
int specdec_row_alpha(const void *logits, const void *q, int dtype, const float *temperature,
                      int B, int gamma, int V, const void *workspace, size_t workspace_bytes,
                      float *alpha, void *stream);

/*
 * Uniforms on the device for the accept tests and the final draw (section
 * 15.1.2 step 3 draws u ~ U(0,1); the other entry points take them as an
 * input).  Generator: Philox4x64-10 ("Parallel random numbers: as easy as
 * 1, 2, 3", Salmon, Moraes, Dror, Shaw, SC'11).  Word i of the stream that
 * starts from `counter` is word i mod 4 of the block for counter
 * counter + floor(i/4) + 1 under `key` (the counter advances before each
 * block, as NumPy's Philox bit generator does, so a stream started from that
 * generator's state continues it word for word); the call writes
 *     out[j] = ((w_{first_word + j} >> 41) + 0.5) * 2^-23,   j in [0, n),
 * exact float32 values strictly inside (0, 1).
 *   key      host pointer, 2 words;  counter  host pointer, 4 words (little-endian)
 *   out      device pointer, n floats
 * Returns SPECDEC_ERR_INVALID_ARG for a null pointer, n < 0, or a word range
 * beyond 2^64; SPECDEC_ERR_UNSUPPORTED for n > SPECDEC_MAX_UNIFORMS.  n = 0 is a
 * no-op.  Asynchronous on `stream`; key and counter are read before return.
 */
int specdec_philox_uniforms(const uint64_t *key, const uint64_t *counter,
                            unsigned long long first_word, long long n, float *out,
                            void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECDEC_H */
