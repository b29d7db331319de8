// Host-buffer forms of the verify calls (see include/specdec.h): the inputs
// are copied from host memory into one caller-provided device staging
// buffer, the device call runs on them, and the outputs are copied back into
// host memory -- every step enqueued on the caller's stream, so a host-side
// caller (a request at a time, the B = 1 latency case) pays one library call
// per verify step instead of a dozen runtime calls of its own.
//
// Staging layout: the input arrays, then the output arrays, then the
// workspace of the device call, each region 256-byte aligned.  The library
// still allocates nothing.
#include "common.cuh"

namespace {

size_t a256(size_t x) { return (x + 255) / 256 * 256; }

// Offsets of n regions of the given sizes, one after the other, then the
// workspace; returns the total.
template <int N>
size_t place(const size_t (&bytes)[N], size_t ws_bytes, size_t (&off)[N + 1]) {
  size_t at = 0;
  for (int i = 0; i < N; ++i) {
    off[i] = at;
    at += a256(bytes[i]);
  }
  off[N] = at;
  return at + ws_bytes;
}

int h2d(void *dst, const void *src, size_t n, cudaStream_t s) {
  if (n == 0) return SPECDEC_OK;
  return cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, s) == cudaSuccess
             ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

int d2h(void *dst, const void *src, size_t n, cudaStream_t s) {
  if (n == 0 || dst == nullptr) return SPECDEC_OK;
  return cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, s) == cudaSuccess
             ? SPECDEC_OK : SPECDEC_ERR_CUDA;
}

// ---- linear form -------------------------------------------------------------
// regions: logits, q, draft_tokens, temperature, uniforms | n_accepted,
// out_tokens, final_token, row_status, p_draft, is_bonus
constexpr int kLin = 11;

struct LinearStaging {
  size_t bytes[kLin];
  size_t off[kLin + 1];
  size_t ws_bytes, total;
};

// 0 for invalid sizes (and for B = 0)
LinearStaging linear_staging(int B, int gamma, int V, int dtype) {
  LinearStaging st{};
  if (gamma < 1 || gamma > SPECDEC_MAX_GAMMA) return st;
  st.ws_bytes = specdec_workspace_size(B, gamma + 1, V, dtype);
  if (st.ws_bytes == 0) return st;
  const size_t b = (size_t)B, R = (size_t)gamma + 1, g = (size_t)gamma;
  const size_t es = (dtype == SPECDEC_F32) ? 4 : 2;
  const size_t sizes[kLin] = {b * R * V * es, b * g * V * es, b * g * 4, b * 4, b * R * 4,
                              b * 4, b * R * 4, b * 4, b * 4, b * g * 4, b};
  for (int i = 0; i < kLin; ++i) st.bytes[i] = sizes[i];
  st.total = place(st.bytes, st.ws_bytes, st.off);
  return st;
}

// ---- tree form -----------------------------------------------------------------
// regions: logits, q, node_tokens, parent, temperature, uniforms | n_accepted,
// path_nodes, out_tokens, final_token, row_status, p_node, is_bonus
constexpr int kTree = 13;

struct TreeStaging {
  size_t bytes[kTree];
  size_t off[kTree + 1];
  size_t ws_bytes, total;
};

TreeStaging tree_staging(int B, int N, int V, int max_depth, int dtype) {
  TreeStaging st{};
  if (N < 1 || N > SPECDEC_MAX_TREE_NODES || max_depth < 0 ||
      max_depth > SPECDEC_MAX_TREE_DEPTH)
    return st;
  st.ws_bytes = specdec_workspace_size(B, N, V, dtype);
  if (st.ws_bytes == 0) return st;
  const size_t b = (size_t)B, n = (size_t)N, D1 = (size_t)max_depth + 1;
  const size_t es = (dtype == SPECDEC_F32) ? 4 : 2;
  const size_t sizes[kTree] = {b * n * V * es, b * n * V * es, b * n * 4, b * n * 4, b * 4,
                               b * n * 4, b * 4, b * D1 * 4, b * D1 * 4, b * 4, b * 4,
                               b * n * 4, b};
  for (int i = 0; i < kTree; ++i) st.bytes[i] = sizes[i];
  st.total = place(st.bytes, st.ws_bytes, st.off);
  return st;
}

// the size checks of the device calls, for the status a bad size gets
int size_status(int B, int rows, int V, int dtype) {
  if (dtype != SPECDEC_F32 && dtype != SPECDEC_BF16) return SPECDEC_ERR_INVALID_ARG;
  if (B < 0 || rows < 1 || V < 1) return SPECDEC_ERR_INVALID_ARG;
  if (V > SPECDEC_MAX_V) return SPECDEC_ERR_UNSUPPORTED;
  return SPECDEC_ERR_UNSUPPORTED;  // sizes the workspace cannot be counted for
}

}  // namespace

extern "C" {

size_t specdec_linear_staging_size(int B, int gamma, int V, int dtype) {
  return linear_staging(B, gamma, V, dtype).total;
}

size_t specdec_tree_staging_size(int B, int N, int V, int max_depth, int dtype) {
  return tree_staging(B, N, V, max_depth, dtype).total;
}

int specdec_verify_linear_host(const void *logits, const void *q, int dtype,
                               const int32_t *draft_tokens, const float *temperature,
                               const float *uniforms, int B, int gamma, int V,
                               int32_t *n_accepted, int32_t *out_tokens, int32_t *final_token,
                               uint8_t *is_bonus, int32_t *row_status, float *p_draft,
                               void *staging, size_t staging_bytes, void *stream) {
  if (gamma < 1) return SPECDEC_ERR_INVALID_ARG;
  if (gamma > SPECDEC_MAX_GAMMA) return SPECDEC_ERR_UNSUPPORTED;
  if (B == 0)  // the device call's size checks; nothing to copy
    return specdec_verify_linear(nullptr, nullptr, dtype, nullptr, nullptr, nullptr, 0, gamma, V,
                                 nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 0,
                                 stream);
  const LinearStaging st = linear_staging(B, gamma, V, dtype);
  if (st.total == 0) return size_status(B, gamma + 1, V, dtype);
  if (!logits || !q || !draft_tokens || !temperature || !uniforms || !n_accepted ||
      !out_tokens || !final_token || !is_bonus || !row_status)
    return SPECDEC_ERR_INVALID_ARG;
  if (!staging || staging_bytes < st.total || (reinterpret_cast<uintptr_t>(staging) & 15))
    return SPECDEC_ERR_WORKSPACE;
  uint8_t *base = static_cast<uint8_t *>(staging);
  void *d[kLin];
  for (int i = 0; i < kLin; ++i) d[i] = base + st.off[i];
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void *in[5] = {logits, q, draft_tokens, temperature, uniforms};
  for (int i = 0; i < 5; ++i) {
    const int rc = h2d(d[i], in[i], st.bytes[i], s);
    if (rc != SPECDEC_OK) return rc;
  }
  const int rc = specdec_verify_linear(
      d[0], d[1], dtype, static_cast<const int32_t *>(d[2]), static_cast<const float *>(d[3]),
      static_cast<const float *>(d[4]), B, gamma, V, static_cast<int32_t *>(d[5]),
      static_cast<int32_t *>(d[6]), static_cast<int32_t *>(d[7]), static_cast<uint8_t *>(d[10]),
      static_cast<int32_t *>(d[8]), p_draft ? static_cast<float *>(d[9]) : nullptr,
      base + st.off[kLin], st.ws_bytes, stream);
  if (rc != SPECDEC_OK) return rc;
  void *out[6] = {n_accepted, out_tokens, final_token, row_status, p_draft, is_bonus};
  for (int i = 0; i < 6; ++i) {
    const int r = d2h(out[i], d[5 + i], st.bytes[5 + i], s);
    if (r != SPECDEC_OK) return r;
  }
  return SPECDEC_OK;
}

int specdec_verify_tree_host(const void *logits, const void *q, int dtype,
                             const int32_t *node_tokens, const int32_t *parent,
                             const float *temperature, const float *uniforms, int B, int N,
                             int V, int max_depth, int32_t *n_accepted, int32_t *path_nodes,
                             int32_t *out_tokens, int32_t *final_token, uint8_t *is_bonus,
                             int32_t *row_status, float *p_node, void *staging,
                             size_t staging_bytes, void *stream) {
  if (N < 1 || max_depth < 0) return SPECDEC_ERR_INVALID_ARG;
  if (N > SPECDEC_MAX_TREE_NODES || max_depth > SPECDEC_MAX_TREE_DEPTH)
    return SPECDEC_ERR_UNSUPPORTED;
  if (B == 0)
    return specdec_verify_tree(nullptr, nullptr, dtype, nullptr, nullptr, nullptr, nullptr, 0, N,
                               V, max_depth, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                               nullptr, nullptr, 0, stream);
  const TreeStaging st = tree_staging(B, N, V, max_depth, dtype);
  if (st.total == 0) return size_status(B, N, V, dtype);
  if (!logits || !q || !node_tokens || !parent || !temperature || !uniforms || !n_accepted ||
      !path_nodes || !out_tokens || !final_token || !is_bonus || !row_status)
    return SPECDEC_ERR_INVALID_ARG;
  if (!staging || staging_bytes < st.total || (reinterpret_cast<uintptr_t>(staging) & 15))
    return SPECDEC_ERR_WORKSPACE;
  uint8_t *base = static_cast<uint8_t *>(staging);
  void *d[kTree];
  for (int i = 0; i < kTree; ++i) d[i] = base + st.off[i];
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void *in[6] = {logits, q, node_tokens, parent, temperature, uniforms};
  for (int i = 0; i < 6; ++i) {
    const int rc = h2d(d[i], in[i], st.bytes[i], s);
    if (rc != SPECDEC_OK) return rc;
  }
  const int rc = specdec_verify_tree(
      d[0], d[1], dtype, static_cast<const int32_t *>(d[2]), static_cast<const int32_t *>(d[3]),
      static_cast<const float *>(d[4]), static_cast<const float *>(d[5]), B, N, V, max_depth,
      static_cast<int32_t *>(d[6]), static_cast<int32_t *>(d[7]), static_cast<int32_t *>(d[8]),
      static_cast<int32_t *>(d[9]), static_cast<uint8_t *>(d[12]), static_cast<int32_t *>(d[10]),
      p_node ? static_cast<float *>(d[11]) : nullptr, base + st.off[kTree], st.ws_bytes, stream);
  if (rc != SPECDEC_OK) return rc;
  void *out[7] = {n_accepted, path_nodes, out_tokens, final_token, row_status, p_node, is_bonus};
  for (int i = 0; i < 7; ++i) {
    const int r = d2h(out[i], d[6 + i], st.bytes[6 + i], s);
    if (r != SPECDEC_OK) return r;
  }
  return SPECDEC_OK;
}

}  // extern "C"
