// specdec_verify_linear_static: the linear verify step for callers that
// cannot allocate device memory for a workspace (see include/specdec.h).
//
// The scratch the kernels need (stage partials, gathered drafted values,
// decision records, draw chunk totals) lives in a fixed __device__ array of
// this translation unit instead of a caller workspace.  Host code cannot use
// the array's name as a device address, so the address is looked up with
// cudaGetSymbolAddress once per device, with that device current, on the
// first call there, and then handed to the same launches as
// specdec_verify_linear.  Nothing in the array needs to start at zero: every
// entry a kernel reads was written earlier in the same call.
#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[SPECDEC_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];

// Device address of the array on the current device, looked up once.
cudaError_t static_scratch(void **ptr) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    err = cudaGetSymbolAddress(&p, g_static_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int specdec_verify_linear_static(const void *logits, const void *q, int dtype,
                                            const int32_t *draft_tokens,
                                            const float *temperature, const float *uniforms,
                                            int B, int gamma, int V, int32_t *n_accepted,
                                            int32_t *out_tokens, int32_t *final_token,
                                            uint8_t *is_bonus, int32_t *row_status,
                                            float *p_draft, void *stream) {
  if (B == 0) return SPECDEC_OK;
  const size_t need = specdec_workspace_size(B, gamma + 1, V, dtype);
  if (need == 0) return (gamma > SPECDEC_MAX_GAMMA || V > SPECDEC_MAX_V)
                            ? SPECDEC_ERR_UNSUPPORTED : SPECDEC_ERR_INVALID_ARG;
  if (need > (size_t)SPECDEC_STATIC_SCRATCH_BYTES) return SPECDEC_ERR_STATIC_LIMIT;
  void *scratch = nullptr;
  if (static_scratch(&scratch) != cudaSuccess) return SPECDEC_ERR_CUDA;
  return specdec_verify_linear(logits, q, dtype, draft_tokens, temperature, uniforms, B, gamma,
                               V, n_accepted, out_tokens, final_token, is_bonus, row_status,
                               p_draft, scratch, (size_t)SPECDEC_STATIC_SCRATCH_BYTES, stream);
}
