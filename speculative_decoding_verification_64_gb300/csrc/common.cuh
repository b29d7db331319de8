// Shared device helpers and launch-side structures of the verify-step kernels.
// sm_103a only: 1-D bulk TMA copies (cp.async.bulk) completing on shared-memory
// mbarriers, thread-block clusters with distributed shared memory.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>
#include <mutex>

#include "specdec.h"

namespace specdec {

// ---------------------------------------------------------------------------
// workspace layout: one partial per (row, stage) written by the row-stats pass
// ---------------------------------------------------------------------------
struct RowPartial {
  float m;        // max of the raw logits in the stage (NaN if one is NaN, -inf if none finite)
  float s;        // sum over the stage of 2^((l - m) c), c = log2(e) / T
  int32_t arg;    // greedy rows: first index holding m; other rows: INT_MAX, or (stats
                  // pass with SPECDEC_STATS_ENTROPY) the float bits of the stage's
                  // sum of 2^((l - m) c) (l - m), for the row entropy
  int32_t flags;  // SPECDEC_ROW_INTERNAL when a bounded wait ran out
};
static_assert(sizeof(RowPartial) == 16, "RowPartial is 16 bytes");

// Every row is cut into stages of kStageBytes of its 16-byte aligned interior;
// a pure function of the sizes, so the workspace size needs no device.
#ifndef SPECDEC_STAGE_BYTES
#define SPECDEC_STAGE_BYTES 8192
#endif
constexpr int kStageBytes = SPECDEC_STAGE_BYTES;

// Elements per chunk of the linear draw over rows that are not 16-byte aligned.
#define SPECDEC_DRAW_CHUNK 8192

inline int draw_chunks(int V) { return (V + SPECDEC_DRAW_CHUNK - 1) / SPECDEC_DRAW_CHUNK; }

// Bytes of the final row per consumer stage of the linear draw over aligned
// rows (bulk copies), and the stage count of a row.
#define SPECDEC_DRAW_STAGE_BYTES 4096

inline int draw_stages(int V, int elem_bytes) {
  const long long b = (long long)V * elem_bytes;
  return (int)((b + SPECDEC_DRAW_STAGE_BYTES - 1) / SPECDEC_DRAW_STAGE_BYTES);
}

// Fixed-point totals kept per request by either form of the draw.
inline int draw_total_slots(int V, int elem_bytes) {
  const int a = draw_chunks(V), b = draw_stages(V, elem_bytes);
  return a > b ? a : b;
}

inline int stages_per_row(int V, int elem_bytes) {
  const long long b = (long long)V * elem_bytes;
  return (int)((b + kStageBytes - 1) / kStageBytes);
}

// ---------------------------------------------------------------------------
// kernel parameter blocks
// ---------------------------------------------------------------------------
// The outcome of one request's accept test, built in shared memory by every
// CTA of the draw kernel from the stats pass's partials.
struct LinearDecision {
  int32_t k;       // first rejected position (gamma: all accepted)
  int32_t status;  // SPECDEC_ROW_* bits; nonzero: nothing to draw
  int32_t greedy;  // T == 0: the final token is `arg`
  int32_t arg;     // first arg-max of the final row (greedy requests)
  float M;         // max of the final row
  float S;         // sum of 2^((l - M) c) over the final row
  float c;         // log2(e) / T
  int32_t pad;
};

// Linear-form workspace records shared by the two phases (device pointers
// into the caller's workspace).
struct LinearWs {
  float2 *gather;                // [B*R] (l_i(x~_i), q_i(x~_i)) of row i < gamma
  unsigned long long *chunk_tot; // [B, draw_total_slots] fixed-point chunk / stage sums of the draw
  unsigned int *draw_cnt;        // [B] chunks done (ticket of the draw); the stats pass zeroes it
  float *mass;                   // [B] normaliser of each request's final draw (below)
};

// The normaliser of a request's final draw, in target-probability units, as
// specdec_final_mass reports it: the draw's fixed-point weight total (units
// of the row maximum: weights 2^((l - M) c) or their residual) over the
// row's merged sum S.  NaN when nothing was drawn.
__device__ __forceinline__ float draw_mass(unsigned long long Z, float S) {
  return __ull2float_rn(Z) * 0x1p-40f / S;
}
constexpr float kNoMass = __builtin_nanf("");

struct RowStatsParams {
  const void *logits;
  const float *temperature;
  RowPartial *part;
  long long stages;  // rows * spr
  int dtype;
  int R, V, spr;     // rows per request, vocabulary, stages per row
  int B;
  int entropy;       // also the entropy sums of non-greedy rows (in RowPartial::arg)
  // Linear form only (tokens == nullptr otherwise): row i < R - 1 of request b
  // scores draft token tokens[b * (R - 1) + i].  The pass gathers that token's
  // logit and q value and zeroes the draw kernel's tickets.
  const int32_t *tokens;
  const void *q;
  LinearWs ws;
};

struct LinearFinalizeParams {
  const void *logits;
  const void *q;
  const int32_t *tokens;
  const float *temperature;
  const float *uniforms;
  const RowPartial *part;
  int32_t *n_accepted;
  int32_t *out_tokens;
  int32_t *final_token;
  uint8_t *is_bonus;
  int32_t *row_status;
  float *p_draft;
  LinearWs ws;
  int dtype, B, gamma, V, spr, nchunk;
  int ntot;  // draw_total_slots(V, element bytes): row stride of ws.chunk_tot
};

struct TreeFinalizeParams {
  const void *logits;
  const void *q;
  const int32_t *tokens;
  const int32_t *parent;
  const float *temperature;
  const float *uniforms;
  const RowPartial *part;
  int32_t *n_accepted;
  int32_t *path_nodes;
  int32_t *out_tokens;
  int32_t *final_token;
  uint8_t *is_bonus;
  int32_t *row_status;
  float *p_node;
  float *mass;  // [B] normaliser of the final draw (workspace), as in LinearWs
  int dtype, B, N, V, spr, max_depth;
};

// host launchers (defined in the .cu files)
// Philox4x64-10 uniforms: words [first, first + n) of the stream (key, counter).
struct PhiloxParams {
  uint64_t key[2];
  uint64_t counter[4];
  uint64_t first;
  long long n;
  float *out;
};

// Path log-probability of a verify step's outputs (see row_extras.cu).
struct PathLogprobParams {
  const void *logits;
  const RowPartial *part;
  const float *temperature;
  const int32_t *out_tokens;   // [B, path_len]
  const int32_t *n_accepted;   // [B]
  const int32_t *path_nodes;   // [B, path_len] (tree form) or NULL (linear form: row j = j)
  const int32_t *row_status;   // [B] or NULL
  float *logprob;              // [B]
  int dtype, B, R, V, spr, path_len;
};

// Per-device set-up done once per process: a device is marked only after the
// set-up succeeded on it; first calls from several host threads serialise on
// the mutex, later calls read one atomic flag.  Devices past the table redo
// the set-up on every call.
constexpr int kMaxCachedDevices = 64;
struct DeviceOnce {
  std::mutex mu;
  std::atomic<bool> done[kMaxCachedDevices]{};
};

template <typename F>
inline cudaError_t device_once(DeviceOnce &o, F &&setup) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxCachedDevices) return setup(dev);
  if (o.done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(o.mu);
  if (o.done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  err = setup(dev);
  if (err == cudaSuccess) o.done[dev].store(true, std::memory_order_release);
  return err;
}

// The dynamic shared-memory opt-in of `kernel`, once per device.
template <typename K>
inline cudaError_t smem_opt_in_once(DeviceOnce &o, K kernel, int bytes) {
  return device_once(o, [&](int) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  });
}

// Multiprocessor count of the current device (looked up once per device).
int device_sm_count();
// Status of the sizes of a linear verify call (gamma, B, V, dtype), as every
// linear entry point reports them.
int linear_size_status(int B, int gamma, int V, int dtype);
cudaError_t launch_row_stats(const RowStatsParams &p, cudaStream_t stream);
cudaError_t launch_linear_finalize(const LinearFinalizeParams &p, cudaStream_t stream);
cudaError_t launch_linear_topk(const LinearFinalizeParams &p, int topk, cudaStream_t stream);


cudaError_t launch_tree_finalize(const TreeFinalizeParams &p, cudaStream_t stream);
cudaError_t launch_philox_uniforms(const PhiloxParams &p, cudaStream_t stream);
cudaError_t launch_row_entropy(const RowPartial *part, const float *temperature, int B, int R,
                               int spr, float *entropy, cudaStream_t stream);
cudaError_t launch_path_logprob(const PathLogprobParams &p, cudaStream_t stream);

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

constexpr float kLog2e = 1.4426950408889634f;

// Temperature check shared by both phases (0 = greedy, else [2^-20, 2^20]).
__device__ __forceinline__ bool temperature_valid(float T) {
  return T == 0.0f || (T >= 0x1p-20f && T <= 0x1p20f);
}

// Exponent scale c such that exp(l / T) = 2^(l * c), in float32 (one IEEE
// division; the same value in every kernel).  Greedy rows and invalid
// temperatures use T = 1: their sums only serve the finiteness check.
__device__ __forceinline__ float temperature_scale(float T) {
  if (T > 0.0f && temperature_valid(T)) return __fdiv_rn(kLog2e, T);
  return kLog2e;
}

// The low part of log2(e)/T beyond temperature_scale(T), for the draws that
// need the exponent argument to float precision (computed once per CTA).
__device__ __forceinline__ float temperature_scale_lo(float T, float c_hi) {
  if (!(T > 0.0f && temperature_valid(T))) return 0.0f;
  return (float)(1.4426950408889634 / (double)T - (double)c_hi);
}

// Largest logit a usable row may hold: with T >= 2^-20, (l - M) c stays finite.
constexpr float kMaxLogit = 0x1p100f;

__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// Merged statistics of one row.
struct RowStat {
  float M;    // row max of the raw logits (NaN if the row holds a NaN)
  float S;    // sum of 2^((l - M) c)
  int arg;    // first index holding M (greedy rows)
  int flags;
};

__device__ __forceinline__ float ex2_approx(float x);

// Merge of two stage partials (each sum is taken relative to its own max).
__device__ __forceinline__ void merge2(float &m, float &s, int &a, float m2, float s2, int a2,
                                       float c);

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void merge2(float &m, float &s, int &a, float m2, float s2, int a2,
                                       float c) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    a = a2;
    return;
  }
  const float M = fmax_nan(m, m2);
  const float f1 = ex2_approx((m - M) * c);
  const float f2 = ex2_approx((m2 - M) * c);
  a = (m > m2) ? a : (m2 > m) ? a2 : min(a, a2);
  s = s * f1 + s2 * f2;
  m = M;
}

// A usable row: finite max within the logit bound and a finite positive sum.
__device__ __forceinline__ bool row_usable(const RowStat &r) {
  return r.M > -INFINITY && r.M <= kMaxLogit && r.S > 0.0f && r.S < INFINITY;
}

// Merge of all stage partials of one row by one warp: lane j takes partials
// j, j + 32, ..., then a butterfly merge.  merge2 is symmetric in its operands,
// so every lane ends with the same, bit-identical result.
__device__ __forceinline__ RowStat warp_merge_row(const RowPartial *part, long long row, int spr,
                                                  float c, int lane) {
  const float4 *pr = reinterpret_cast<const float4 *>(part + row * (long long)spr);
  float m = -INFINITY, s = 0.0f;
  int a = 0x7FFFFFFF, fl = 0;
  for (int j = lane; j < spr; j += 32) {
    const float4 x = pr[j];
    fl |= __float_as_int(x.w);
    merge2(m, s, a, x.x, x.y, __float_as_int(x.z), c);
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, d);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, d);
    const int a2 = __shfl_xor_sync(0xffffffffu, a, d);
    merge2(m, s, a, m2, s2, a2, c);
  }
  RowStat r;
  r.M = m;
  r.S = s;
  r.arg = a;
  r.flags = __reduce_or_sync(0xffffffffu, fl);
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float load_elem(const void *base, int dtype, long long idx) {
  if (dtype == SPECDEC_F32) return __ldg(reinterpret_cast<const float *>(base) + idx);
  const unsigned short h = __ldg(reinterpret_cast<const unsigned short *>(base) + idx);
  return __uint_as_float(((uint32_t)h) << 16);
}

// Exact floor(w * 2^40) for a finite w >= 0 (weights in units of the row
// maximum, w <= 2^20).
__device__ __forceinline__ unsigned long long to_fixed40(float w) {
  const uint32_t b = __float_as_uint(w);
  const int e = (int)(b >> 23) & 0xFF;
  if (e == 0 || (b >> 31)) return 0ull;
  const unsigned long long m = (unsigned long long)((b & 0x7FFFFFu) | 0x800000u);
  const int s = e - 110;  // w * 2^40 = m * 2^(e - 127 - 23 + 40)
  if (s >= 0) return m << s;
  if (s <= -24) return 0ull;
  return m >> (-s);
}

// floor(U * Z) for U in (0, 1) given as float32 and an integer Z:
// exact 88-bit product of U's significand with Z, then the exponent shift.
__device__ __forceinline__ unsigned long long uniform_target(float U, unsigned long long Z) {
  if (!(U > 0.0f)) return 0ull;
  if (!(U < 1.0f)) return Z ? Z - 1 : 0ull;
  const uint32_t ub = __float_as_uint(U);
  const int e = (int)(ub >> 23) & 0xFF;
  const unsigned long long mant = (ub & 0x7FFFFFu) | (e ? 0x800000u : 0u);
  const int sh = (e ? 150 - e : 149);  // U = mant * 2^-sh, sh >= 24
  const unsigned long long lo = mant * Z;
  const unsigned long long hi = __umul64hi(mant, Z);
  if (sh >= 128) return 0ull;
  if (sh >= 64) return hi >> (sh - 64);
  return (lo >> sh) | (hi << (64 - sh));
}

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int m) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)v, m);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(v >> 32), m);
  return ((unsigned long long)hi << 32) | lo;
}

__device__ __forceinline__ unsigned long long shfl_up_u64(unsigned long long v, int d) {
  const uint32_t lo = __shfl_up_sync(0xffffffffu, (uint32_t)v, d);
  const uint32_t hi = __shfl_up_sync(0xffffffffu, (uint32_t)(v >> 32), d);
  return ((unsigned long long)hi << 32) | lo;
}

// --- mbarrier / bulk-copy wrappers (PTX ISA 8.x, sm_90 and later) ----------

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Programmatic dependent launch.  A phase-2 kernel is launched so that its
// CTAs may start while the kernel before it on the stream is finishing;
// pdl_wait() (every thread, before its first global-memory access) blocks
// until that kernel has completed and its writes are visible.  The stats pass
// lets its dependents launch as soon as all of its CTAs are running.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: gives up after ~2 s of wall time (returns false).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
// The limit of a consumer's wait for a copy it is about to read.  A test
// build sets it to 0 (SPECDEC_CONSUMER_WAIT_NS): those waits then give up
// without looking, every time, so that the give-up paths run; the waits that
// keep a CTA until its copies have landed (the producers' and the drains')
// keep kWaitLimitNs.
#ifndef SPECDEC_CONSUMER_WAIT_NS
#define SPECDEC_CONSUMER_WAIT_NS 2000000000ull
#endif
constexpr unsigned long long kConsumerWaitNs = SPECDEC_CONSUMER_WAIT_NS;

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  unsigned long long limit = kWaitLimitNs) {
  if (limit == 0) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit) return false;
  }
}

// ---- distributed shared memory: asynchronous remote stores ----------------
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

// 8 bytes into another CTA's shared memory, completing bytes on its barrier
__device__ __forceinline__ void st_async_u64(uint32_t addr, unsigned long long v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u64 [%0], %1, [%2];" ::"r"(addr),
               "l"(v), "r"(bar)
               : "memory");
}

// 4 bytes into another CTA's shared memory, completing bytes on its barrier
__device__ __forceinline__ void st_async_u32(uint32_t addr, uint32_t v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(addr),
               "r"(v), "r"(bar)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on a barrier that other CTAs' asynchronous stores complete.
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Block (bounded) until every bulk copy issued into a ring of `slots` "full"
// barriers has landed, so that a CTA whose consumers stopped waiting (after
// some wait gave up) never exits while a copy still writes its shared memory.  Units 0 .. n_issued-1 were
// issued in order, unit n into slot n % slots; a slot's phases complete in
// order, so waiting for its last issued phase covers the earlier ones.
__device__ __forceinline__ void drain_ring(uint64_t *full, int slots, long long n_issued) {
  for (int s = 0; s < slots && s < n_issued; ++s) {
    const long long last = s + (long long)slots * ((n_issued - 1 - s) / slots);
    mbar_wait_bounded(&full[s], (uint32_t)((last / slots) & 1));
  }
}

// 1-D bulk copy global -> shared, completing `bytes` of transaction count on
// `bar`.  Source and destination 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void *dst_smem, const void *src_gmem,
                                              uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

#endif  // __CUDACC__

}  // namespace specdec
