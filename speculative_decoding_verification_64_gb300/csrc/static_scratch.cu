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

specdec::DeviceOnce g_scratch_once;
void *g_scratch_ptr[specdec::kMaxCachedDevices];  // written under g_scratch_once

// Device address of the array on the current device, looked up once (first
// calls from several host threads serialise inside device_once).
cudaError_t static_scratch(void **ptr) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= specdec::kMaxCachedDevices) return cudaErrorInvalidDevice;
  err = specdec::device_once(g_scratch_once, [](int d) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e == cudaSuccess) g_scratch_ptr[d] = p;
    return e;
  });
  if (err != cudaSuccess) return err;
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
  // the size checks of specdec_verify_linear first, so that both entry points
  // return the same code for the same sizes (B = 0 included)
  const int st = specdec::linear_size_status(B, gamma, V, dtype);
  if (st != SPECDEC_OK || B == 0) return st;
  const size_t need = specdec_workspace_size(B, gamma + 1, V, dtype);
  if (need > (size_t)SPECDEC_STATIC_SCRATCH_BYTES) return SPECDEC_ERR_STATIC_LIMIT;
  void *scratch = nullptr;
  if (static_scratch(&scratch) != cudaSuccess) return SPECDEC_ERR_CUDA;
  return specdec_verify_linear(logits, q, dtype, draft_tokens, temperature, uniforms, B, gamma,
                               V, n_accepted, out_tokens, final_token, is_bonus, row_status,
                               p_draft, scratch, (size_t)SPECDEC_STATIC_SCRATCH_BYTES, stream);
}
