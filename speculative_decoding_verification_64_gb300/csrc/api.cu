// C ABI of the verify step: argument checks, workspace sizing and launches.
// Every entry point is asynchronous on the caller's stream and allocates
// nothing; see include/specdec.h for the contract of each call.
#include <climits>
#include <cstdlib>
#include <cstring>
#include <initializer_list>

#include "common.cuh"

namespace specdec {
// row_extras.cu: sum_v min(p_i, q_i) of every drafted row
cudaError_t launch_row_alpha(const void *logits, const void *q, int dtype, const RowPartial *part,
                             const float *temperature, int B, int gamma, int V, int spr,
                             float *alpha, cudaStream_t stream);
// finalize_linear.cu: the draw launched right after this call's stats pass
cudaError_t launch_linear_finalize_after_stats(const LinearFinalizeParams &p, cudaStream_t stream);
// small_verify.cu: the linear step of a small batch in one launch
bool small_verify_applies(int B, int gamma, int V, int dtype, const void *logits, const void *q);
cudaError_t launch_small_verify(const LinearFinalizeParams &p, cudaStream_t stream);
}  // namespace specdec

using namespace specdec;

namespace {

int elem_bytes(int dtype) { return dtype == SPECDEC_F32 ? 4 : 2; }

bool dtype_ok(int dtype) { return dtype == SPECDEC_F32 || dtype == SPECDEC_BF16; }

// Workspace regions, each 256-byte aligned: the stage partials of the stats
// pass; for the linear form the gathered (logit, q) of every drafted token,
// p_i(x~_i), one decision record per request, the fixed-point chunk totals of
// the draw and two ticket counters per request (zero between calls).
size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct WsLayout {
  size_t gather, chunk, draw_cnt, mass, total;
};

// Stage partials first, then the linear form's gathered values, draw chunk
// totals and tickets, then the normaliser of every request's final draw
// (both forms).
WsLayout workspace_layout(long long B, int R, int V, int dtype) {
  const long long rows = B * (long long)R;
  WsLayout w;
  w.gather = align256((size_t)rows * (size_t)stages_per_row(V, elem_bytes(dtype)) *
                      sizeof(RowPartial));
  w.chunk = w.gather + align256((size_t)rows * sizeof(float2));
  w.draw_cnt = w.chunk + align256((size_t)B * draw_total_slots(V, elem_bytes(dtype)) *
                                  sizeof(unsigned long long));
  w.mass = w.draw_cnt + align256((size_t)B * sizeof(unsigned int));
  w.total = w.mass + align256((size_t)B * sizeof(float));
  return w;
}

LinearWs linear_ws(void *workspace, long long B, int R, int V, int dtype) {
  const WsLayout w = workspace_layout(B, R, V, dtype);
  uint8_t *base = reinterpret_cast<uint8_t *>(workspace);
  LinearWs ws;
  ws.gather = reinterpret_cast<float2 *>(base + w.gather);
  ws.chunk_tot = reinterpret_cast<unsigned long long *>(base + w.chunk);
  ws.draw_cnt = reinterpret_cast<unsigned int *>(base + w.draw_cnt);
  ws.mass = reinterpret_cast<float *>(base + w.mass);
  return ws;
}

size_t workspace_bytes_for(long long B, int R, int V, int dtype) {
  if (B <= 0) return 0;  // no requests, no scratch
  return workspace_layout(B, R, V, dtype).total;
}

int check_sizes(int B, int R, int V, int dtype) {
  if (!dtype_ok(dtype) || B < 0 || R < 1 || V < 1) return SPECDEC_ERR_INVALID_ARG;
  if (V > SPECDEC_MAX_V) return SPECDEC_ERR_UNSUPPORTED;
  if ((long long)B * 8 > INT_MAX || (long long)B * R > INT_MAX) return SPECDEC_ERR_UNSUPPORTED;
  return SPECDEC_OK;
}

int check_workspace(const void *ws, size_t ws_bytes, int B, int R, int V, int dtype) {
  const size_t need = workspace_bytes_for(B, R, V, dtype);
  if (need == 0) return SPECDEC_OK;
  if (ws == nullptr || ws_bytes < need) return SPECDEC_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 15) != 0) return SPECDEC_ERR_WORKSPACE;
  return SPECDEC_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? SPECDEC_OK : SPECDEC_ERR_CUDA; }

// An array must start on a multiple of its element size: a misaligned
// element load or store faults the device, so such pointers are refused here.
bool misaligned(const void *ptr, uintptr_t elem) {
  return (reinterpret_cast<uintptr_t>(ptr) & (elem - 1)) != 0;
}

// logits and q in their dtype; every other array holds 4-byte elements
bool arrays_misaligned(int dtype, const void *logits, const void *q,
                       std::initializer_list<const void *> words) {
  const uintptr_t es = (uintptr_t)elem_bytes(dtype);
  if (misaligned(logits, es) || misaligned(q, es)) return true;
  for (const void *w : words)
    if (misaligned(w, 4)) return true;
  return false;
}

RowStatsParams stats_params(const void *logits, const void *q, int dtype, const int32_t *tokens,
                           const float *temperature, int B, int R, int V, void *workspace,
                           bool entropy) {
  const long long rows = (long long)B * R;
  const int spr = stages_per_row(V, elem_bytes(dtype));
  RowStatsParams p;
  p.logits = logits;
  p.temperature = temperature;
  p.part = reinterpret_cast<RowPartial *>(workspace);
  p.stages = rows * spr;
  p.dtype = dtype;
  p.R = R;
  p.V = V;
  p.spr = spr;
  p.B = B;
  p.entropy = entropy ? 1 : 0;
  p.tokens = tokens;
  p.q = q;
  p.ws = linear_ws(workspace, B, R, V, dtype);
  return p;
}

int launch_stats(const void *logits, const void *q, int dtype, const int32_t *tokens,
                 const float *temperature, int B, int R, int V, void *workspace,
                 cudaStream_t stream, bool entropy = false) {
  return cuda_status(launch_row_stats(
      stats_params(logits, q, dtype, tokens, temperature, B, R, V, workspace, entropy), stream));
}

}  // namespace

extern "C" {

int specdec_abi_version(void) { return SPECDEC_ABI_VERSION; }

const char *specdec_status_string(int code) {
  switch (code) {
    case SPECDEC_OK: return "ok";
    case SPECDEC_ERR_INVALID_ARG: return "invalid argument (null pointer, size or dtype)";
    case SPECDEC_ERR_UNSUPPORTED: return "sizes beyond the supported limits";
    case SPECDEC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SPECDEC_ERR_CUDA: return "CUDA runtime or launch error";
    case SPECDEC_ERR_STATIC_LIMIT:
      return "sizes need more scratch than the fixed array of specdec_verify_linear_static";
    default: break;
  }
  return "unknown status";
}

size_t specdec_workspace_size(int B, int rows_per_request, int V, int dtype) {
  if (check_sizes(B, rows_per_request, V, dtype) != SPECDEC_OK) return 0;
  return workspace_bytes_for(B, rows_per_request, V, dtype);
}

int specdec_row_stats(const void *logits, const void *q, int dtype, const int32_t *draft_tokens,
                      const float *temperature, int B, int rows_per_request, int V,
                      unsigned flags, void *workspace, size_t workspace_bytes, void *stream) {
  if (flags & ~(unsigned)SPECDEC_STATS_ENTROPY) return SPECDEC_ERR_INVALID_ARG;
  int st = check_sizes(B, rows_per_request, V, dtype);
  if (st != SPECDEC_OK) return st;
  if (B == 0) return SPECDEC_OK;
  if (!logits || !temperature) return SPECDEC_ERR_INVALID_ARG;
  const int linear = (q != nullptr) + (draft_tokens != nullptr);
  if (linear == 1) return SPECDEC_ERR_INVALID_ARG;
  if (linear && (rows_per_request < 2 || rows_per_request - 1 > SPECDEC_MAX_GAMMA))
    return SPECDEC_ERR_INVALID_ARG;
  if (arrays_misaligned(dtype, logits, q, {draft_tokens, temperature}))
    return SPECDEC_ERR_INVALID_ARG;
  st = check_workspace(workspace, workspace_bytes, B, rows_per_request, V, dtype);
  if (st != SPECDEC_OK) return st;
  return launch_stats(logits, linear ? q : nullptr, dtype, linear ? draft_tokens : nullptr,
                      temperature, B, rows_per_request, V, workspace,
                      static_cast<cudaStream_t>(stream), (flags & SPECDEC_STATS_ENTROPY) != 0);
}

}  // extern "C"

// Size checks of every linear entry point (also the no-workspace one), in the
// order that decides which code a bad call gets.
int specdec::linear_size_status(int B, int gamma, int V, int dtype) {
  if (gamma < 1) return SPECDEC_ERR_INVALID_ARG;
  if (gamma > SPECDEC_MAX_GAMMA) return SPECDEC_ERR_UNSUPPORTED;
  return check_sizes(B, gamma + 1, V, dtype);
}

extern "C" {

static int linear_checks(const void *logits, const void *q, int dtype, const int32_t *tokens,
                         const float *temperature, const float *uniforms, int B, int gamma,
                         int V, int32_t *n_accepted, int32_t *out_tokens, int32_t *final_token,
                         uint8_t *is_bonus, int32_t *row_status, const float *p_draft,
                         void *workspace, size_t workspace_bytes) {
  const int st = linear_size_status(B, gamma, V, dtype);
  if (st != SPECDEC_OK) return st;
  if (B == 0) return SPECDEC_OK;
  if (!logits || !q || !tokens || !temperature || !uniforms || !n_accepted || !out_tokens ||
      !final_token || !is_bonus || !row_status)
    return SPECDEC_ERR_INVALID_ARG;
  if (arrays_misaligned(dtype, logits, q,
                        {tokens, temperature, uniforms, n_accepted, out_tokens, final_token,
                         row_status, p_draft}))
    return SPECDEC_ERR_INVALID_ARG;
  return check_workspace(workspace, workspace_bytes, B, gamma + 1, V, dtype);
}

static LinearFinalizeParams linear_params(const void *logits, const void *q, int dtype,
                                          const int32_t *tokens, const float *temperature,
                                          const float *uniforms, int B, int gamma, int V,
                                          int32_t *n_accepted, int32_t *out_tokens,
                                          int32_t *final_token, uint8_t *is_bonus,
                                          int32_t *row_status, float *p_draft, void *workspace) {
  LinearFinalizeParams p;
  p.logits = logits;
  p.q = q;
  p.tokens = tokens;
  p.temperature = temperature;
  p.uniforms = uniforms;
  p.part = reinterpret_cast<const RowPartial *>(workspace);
  p.n_accepted = n_accepted;
  p.out_tokens = out_tokens;
  p.final_token = final_token;
  p.is_bonus = is_bonus;
  p.row_status = row_status;
  p.p_draft = p_draft;
  p.ws = linear_ws(workspace, B, gamma + 1, V, dtype);
  p.dtype = dtype;
  p.B = B;
  p.gamma = gamma;
  p.V = V;
  p.spr = stages_per_row(V, elem_bytes(dtype));
  p.nchunk = draw_chunks(V);
  p.ntot = draw_total_slots(V, elem_bytes(dtype));
  return p;
}

static int linear_finalize_launch(const void *logits, const void *q, int dtype,
                                  const int32_t *tokens, const float *temperature,
                                  const float *uniforms, int B, int gamma, int V,
                                  int32_t *n_accepted, int32_t *out_tokens,
                                  int32_t *final_token, uint8_t *is_bonus, int32_t *row_status,
                                  float *p_draft, void *workspace, cudaStream_t stream,
                                  bool after_stats = false) {
  const LinearFinalizeParams p =
      linear_params(logits, q, dtype, tokens, temperature, uniforms, B, gamma, V, n_accepted,
                    out_tokens, final_token, is_bonus, row_status, p_draft, workspace);
  return cuda_status(after_stats ? launch_linear_finalize_after_stats(p, stream)
                                 : launch_linear_finalize(p, stream));
}

int specdec_linear_finalize(const void *logits, const void *q, int dtype,
                            const int32_t *draft_tokens, const float *temperature,
                            const float *uniforms, int B, int gamma, int V,
                            int32_t *n_accepted, int32_t *out_tokens, int32_t *final_token,
                            uint8_t *is_bonus, int32_t *row_status, float *p_draft,
                            void *workspace, size_t workspace_bytes, void *stream) {
  const int st = linear_checks(logits, q, dtype, draft_tokens, temperature, uniforms, B, gamma,
                               V, n_accepted, out_tokens, final_token, is_bonus, row_status,
                               p_draft, workspace, workspace_bytes);
  if (st != SPECDEC_OK || B == 0) return st;
  return linear_finalize_launch(logits, q, dtype, draft_tokens, temperature, uniforms, B, gamma,
                                V, n_accepted, out_tokens, final_token, is_bonus, row_status,
                                p_draft, workspace, static_cast<cudaStream_t>(stream));
}

int specdec_verify_linear(const void *logits, const void *q, int dtype,
                          const int32_t *draft_tokens, const float *temperature,
                          const float *uniforms, int B, int gamma, int V,
                          int32_t *n_accepted, int32_t *out_tokens, int32_t *final_token,
                          uint8_t *is_bonus, int32_t *row_status, float *p_draft,
                          void *workspace, size_t workspace_bytes, void *stream) {
  int st = linear_checks(logits, q, dtype, draft_tokens, temperature, uniforms, B, gamma, V,
                         n_accepted, out_tokens, final_token, is_bonus, row_status, p_draft,
                         workspace, workspace_bytes);
  if (st != SPECDEC_OK || B == 0) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (small_verify_applies(B, gamma, V, dtype, logits, q)) {
    // a small batch: both phases in one launch, leaving the same workspace
    const LinearFinalizeParams p =
        linear_params(logits, q, dtype, draft_tokens, temperature, uniforms, B, gamma, V,
                      n_accepted, out_tokens, final_token, is_bonus, row_status, p_draft, workspace);
    return cuda_status(launch_small_verify(p, s));
  }
  st = launch_stats(logits, q, dtype, draft_tokens, temperature, B, gamma + 1, V, workspace, s);
  if (st != SPECDEC_OK) return st;
  return linear_finalize_launch(logits, q, dtype, draft_tokens, temperature, uniforms, B, gamma,
                                V, n_accepted, out_tokens, final_token, is_bonus, row_status,
                                p_draft, workspace, s, /*after_stats=*/true);
}

int specdec_verify_linear_path(int B, int gamma, int V, int dtype, const void *logits,
                               const void *q) {
  if (B <= 0) return SPECDEC_PATH_NONE;
  if (linear_size_status(B, gamma, V, dtype) != SPECDEC_OK) return -1;
  if (small_verify_applies(B, gamma, V, dtype, logits, q)) return SPECDEC_PATH_SMALL_ONE_LAUNCH;
  return SPECDEC_PATH_TWO_LAUNCHES;
}

int specdec_verify_linear_launches(int B, int gamma, int V, int dtype, const void *logits,
                                   const void *q) {
  const int path = specdec_verify_linear_path(B, gamma, V, dtype, logits, q);
  if (path <= 0) return path;
  return path == SPECDEC_PATH_TWO_LAUNCHES ? 2 : 1;
}

static int tree_checks(const void *logits, const void *q, int dtype, const int32_t *tokens,
                       const int32_t *parent, const float *temperature, const float *uniforms,
                       int B, int N, int V, int max_depth, int32_t *n_accepted,
                       int32_t *path_nodes, int32_t *out_tokens, int32_t *final_token,
                       uint8_t *is_bonus, int32_t *row_status, const float *p_node,
                       void *workspace, size_t workspace_bytes) {
  if (N < 1 || max_depth < 0) return SPECDEC_ERR_INVALID_ARG;
  if (N > SPECDEC_MAX_TREE_NODES || max_depth > SPECDEC_MAX_TREE_DEPTH)
    return SPECDEC_ERR_UNSUPPORTED;
  int st = check_sizes(B, N, V, dtype);
  if (st != SPECDEC_OK) return st;
  if (B == 0) return SPECDEC_OK;
  if (!logits || !q || !tokens || !parent || !temperature || !uniforms || !n_accepted ||
      !path_nodes || !out_tokens || !final_token || !is_bonus || !row_status)
    return SPECDEC_ERR_INVALID_ARG;
  if (arrays_misaligned(dtype, logits, q,
                        {tokens, parent, temperature, uniforms, n_accepted, path_nodes,
                         out_tokens, final_token, row_status, p_node}))
    return SPECDEC_ERR_INVALID_ARG;
  return check_workspace(workspace, workspace_bytes, B, N, V, dtype);
}

static int tree_finalize_launch(const void *logits, const void *q, int dtype,
                                const int32_t *tokens, const int32_t *parent,
                                const float *temperature, const float *uniforms, int B, int N,
                                int V, int max_depth, int32_t *n_accepted, int32_t *path_nodes,
                                int32_t *out_tokens, int32_t *final_token, uint8_t *is_bonus,
                                int32_t *row_status, float *p_node, void *workspace,
                                cudaStream_t stream) {
  TreeFinalizeParams p;
  p.logits = logits;
  p.q = q;
  p.tokens = tokens;
  p.parent = parent;
  p.temperature = temperature;
  p.uniforms = uniforms;
  p.part = reinterpret_cast<const RowPartial *>(workspace);
  p.n_accepted = n_accepted;
  p.path_nodes = path_nodes;
  p.out_tokens = out_tokens;
  p.final_token = final_token;
  p.is_bonus = is_bonus;
  p.row_status = row_status;
  p.p_node = p_node;
  p.mass = linear_ws(workspace, B, N, V, dtype).mass;
  p.dtype = dtype;
  p.B = B;
  p.N = N;
  p.V = V;
  p.spr = stages_per_row(V, elem_bytes(dtype));
  p.max_depth = max_depth;
  return cuda_status(launch_tree_finalize(p, stream));
}

int specdec_tree_finalize(const void *logits, const void *q, int dtype,
                          const int32_t *node_tokens, const int32_t *parent,
                          const float *temperature, const float *uniforms, int B, int N, int V,
                          int max_depth, int32_t *n_accepted, int32_t *path_nodes,
                          int32_t *out_tokens, int32_t *final_token, uint8_t *is_bonus,
                          int32_t *row_status, float *p_node, void *workspace,
                          size_t workspace_bytes, void *stream) {
  const int st = tree_checks(logits, q, dtype, node_tokens, parent, temperature, uniforms, B, N,
                             V, max_depth, n_accepted, path_nodes, out_tokens, final_token,
                             is_bonus, row_status, p_node, workspace, workspace_bytes);
  if (st != SPECDEC_OK || B == 0) return st;
  return tree_finalize_launch(logits, q, dtype, node_tokens, parent, temperature, uniforms, B, N,
                              V, max_depth, n_accepted, path_nodes, out_tokens, final_token,
                              is_bonus, row_status, p_node, workspace,
                              static_cast<cudaStream_t>(stream));
}

int specdec_verify_tree(const void *logits, const void *q, int dtype, const int32_t *node_tokens,
                        const int32_t *parent, const float *temperature, const float *uniforms,
                        int B, int N, int V, int max_depth, int32_t *n_accepted,
                        int32_t *path_nodes, int32_t *out_tokens, int32_t *final_token,
                        uint8_t *is_bonus, int32_t *row_status, float *p_node, void *workspace,
                        size_t workspace_bytes, void *stream) {
  int st = tree_checks(logits, q, dtype, node_tokens, parent, temperature, uniforms, B, N, V,
                       max_depth, n_accepted, path_nodes, out_tokens, final_token, is_bonus,
                       row_status, p_node, workspace, workspace_bytes);
  if (st != SPECDEC_OK || B == 0) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = launch_stats(logits, nullptr, dtype, nullptr, temperature, B, N, V, workspace, s);
  if (st != SPECDEC_OK) return st;
  return tree_finalize_launch(logits, q, dtype, node_tokens, parent, temperature, uniforms, B, N,
                              V, max_depth, n_accepted, path_nodes, out_tokens, final_token,
                              is_bonus, row_status, p_node, workspace, s);
}


int specdec_final_mass(const void *workspace, size_t workspace_bytes, int B,
                       int rows_per_request, int V, int dtype, float *mass, void *stream) {
  int st = check_sizes(B, rows_per_request, V, dtype);
  if (st != SPECDEC_OK) return st;
  if (B == 0) return SPECDEC_OK;
  if (!mass || misaligned(mass, 4)) return SPECDEC_ERR_INVALID_ARG;
  st = check_workspace(workspace, workspace_bytes, B, rows_per_request, V, dtype);
  if (st != SPECDEC_OK) return st;
  const LinearWs ws = linear_ws(const_cast<void *>(workspace), B, rows_per_request, V, dtype);
  return cuda_status(cudaMemcpyAsync(mass, ws.mass, (size_t)B * sizeof(float),
                                     cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream)));
}

int specdec_philox_uniforms(const uint64_t *key, const uint64_t *counter,
                            unsigned long long first_word, long long n, float *out,
                            void *stream) {
  if (n < 0) return SPECDEC_ERR_INVALID_ARG;
  if (n == 0) return SPECDEC_OK;
  if (!key || !counter || !out) return SPECDEC_ERR_INVALID_ARG;
  if (misaligned(out, 4)) return SPECDEC_ERR_INVALID_ARG;
  if (n > SPECDEC_MAX_UNIFORMS) return SPECDEC_ERR_UNSUPPORTED;
  if (first_word > ~0ull - (unsigned long long)(n - 1)) return SPECDEC_ERR_INVALID_ARG;
  PhiloxParams p;
  p.key[0] = key[0];
  p.key[1] = key[1];
  for (int i = 0; i < 4; ++i) p.counter[i] = counter[i];
  p.first = first_word;
  p.n = n;
  p.out = out;
  return cuda_status(launch_philox_uniforms(p, static_cast<cudaStream_t>(stream)));
}

int specdec_row_entropy(const void *workspace, size_t workspace_bytes, int dtype,
                        const float *temperature, int B, int rows_per_request, int V,
                        float *entropy, void *stream) {
  int st = check_sizes(B, rows_per_request, V, dtype);
  if (st != SPECDEC_OK) return st;
  if (B == 0) return SPECDEC_OK;
  if (!temperature || !entropy) return SPECDEC_ERR_INVALID_ARG;
  if (misaligned(temperature, 4) || misaligned(entropy, 4)) return SPECDEC_ERR_INVALID_ARG;
  st = check_workspace(workspace, workspace_bytes, B, rows_per_request, V, dtype);
  if (st != SPECDEC_OK) return st;
  return cuda_status(launch_row_entropy(reinterpret_cast<const RowPartial *>(workspace),
                                        temperature, B, rows_per_request,
                                        stages_per_row(V, elem_bytes(dtype)), entropy,
                                        static_cast<cudaStream_t>(stream)));
}

int specdec_row_alpha(const void *logits, const void *q, int dtype, const float *temperature,
                      int B, int gamma, int V, const void *workspace, size_t workspace_bytes,
                      float *alpha, void *stream) {
  if (gamma < 1 || gamma > SPECDEC_MAX_GAMMA) return SPECDEC_ERR_INVALID_ARG;
  int st = check_sizes(B, gamma + 1, V, dtype);
  if (st != SPECDEC_OK) return st;
  if (B == 0) return SPECDEC_OK;
  if (!logits || !q || !temperature || !alpha) return SPECDEC_ERR_INVALID_ARG;
  if (arrays_misaligned(dtype, logits, q, {temperature, alpha})) return SPECDEC_ERR_INVALID_ARG;
  st = check_workspace(workspace, workspace_bytes, B, gamma + 1, V, dtype);
  if (st != SPECDEC_OK) return st;
  return cuda_status(launch_row_alpha(logits, q, dtype, reinterpret_cast<const RowPartial *>(workspace),
                                      temperature, B, gamma, V, stages_per_row(V, elem_bytes(dtype)),
                                      alpha, static_cast<cudaStream_t>(stream)));
}

int specdec_path_logprob(const void *logits, int dtype, const float *temperature,
                         const int32_t *out_tokens, const int32_t *n_accepted,
                         const int32_t *path_nodes, const int32_t *row_status, int B,
                         int rows_per_request, int V, int path_len, const void *workspace,
                         size_t workspace_bytes, float *logprob, void *stream) {
  int st = check_sizes(B, rows_per_request, V, dtype);
  if (st != SPECDEC_OK) return st;
  if (B == 0) return SPECDEC_OK;
  if (!logits || !temperature || !out_tokens || !n_accepted || !logprob || path_len < 1)
    return SPECDEC_ERR_INVALID_ARG;
  if (arrays_misaligned(dtype, logits, nullptr,
                        {temperature, out_tokens, n_accepted, path_nodes, row_status, logprob}))
    return SPECDEC_ERR_INVALID_ARG;
  st = check_workspace(workspace, workspace_bytes, B, rows_per_request, V, dtype);
  if (st != SPECDEC_OK) return st;
  PathLogprobParams p;
  p.logits = logits;
  p.part = reinterpret_cast<const RowPartial *>(workspace);
  p.temperature = temperature;
  p.out_tokens = out_tokens;
  p.n_accepted = n_accepted;
  p.path_nodes = path_nodes;
  p.row_status = row_status;
  p.logprob = logprob;
  p.dtype = dtype;
  p.B = B;
  p.R = rows_per_request;
  p.V = V;
  p.spr = stages_per_row(V, elem_bytes(dtype));
  p.path_len = path_len;
  return cuda_status(launch_path_logprob(p, static_cast<cudaStream_t>(stream)));
}

int specdec_verify_linear_topk(const void *logits, const void *q, int dtype,
                               const int32_t *draft_tokens, const float *temperature,
                               const float *uniforms, int B, int gamma, int V, int topk,
                               int32_t *n_accepted, int32_t *out_tokens, int32_t *final_token,
                               uint8_t *is_bonus, int32_t *row_status, float *p_draft,
                               void *workspace, size_t workspace_bytes, void *stream) {
  if (topk < 1) return SPECDEC_ERR_INVALID_ARG;
  if (topk > SPECDEC_MAX_TOPK) return SPECDEC_ERR_UNSUPPORTED;
  int st = linear_checks(logits, q, dtype, draft_tokens, temperature, uniforms, B, gamma, V,
                         n_accepted, out_tokens, final_token, is_bonus, row_status, p_draft,
                         workspace, workspace_bytes);
  if (st != SPECDEC_OK || B == 0) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = launch_stats(logits, q, dtype, draft_tokens, temperature, B, gamma + 1, V, workspace, s);
  if (st != SPECDEC_OK) return st;
  const LinearFinalizeParams p =
      linear_params(logits, q, dtype, draft_tokens, temperature, uniforms, B, gamma, V,
                    n_accepted, out_tokens, final_token, is_bonus, row_status, p_draft, workspace);
  return cuda_status(launch_linear_topk(p, topk, s));
}

}  // extern "C"
