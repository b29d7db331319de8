// Row statistics of the target logits: the "parallel verification" step of
// speculative sampling ("Chapter 15: Decoding acceleration", section 15.1.2,
// step 2), which scores every drafted position in one pass.  Every row is cut
// into 8 KB stages of its 16-byte aligned interior; for each stage the kernel
// produces
//     m = max_v l_v,   s = sum_v 2^((l_v - m) c),   c = log2(e)/T,
// and, for greedy rows (T = 0), the first index holding m.  A merge over the
// stages of a row gives p(x) = 2^((l_x - M) c) / S.  This pass
// reads every logit exactly once and carries almost all of the verify step's
// HBM traffic.
//
// Structure (GB300): a persistent grid of one CTA per SM.  Rows are moved in
// units of two consecutive 8 KB stages (16 KB: one 1-D bulk TMA copy,
// cp.async.bulk, per unit, since the copy engine's cost is per operation);
// unit g goes to CTA g mod grid, so at any moment the CTAs sweep neighbouring
// units and a request's rows are read close together in time.  In each CTA
// one producer thread streams its units into a ring of 12 shared-memory slots
// whose "full" mbarriers the copies complete.  Fifteen consumer warps take the
// stages round robin: a warp reads a whole stage with 128-bit shared loads
// (16 vectors per lane), arrives on the unit's "empty" barrier, takes the
// stage max with NaN-propagating packed bf16 max, then forms the exponent
// arguments (l - m) c with packed fp32x2 add and multiply (l - m is exact for
// bf16 inputs), one ex2 per element and packed adds,
// reduces over the warp with shuffles and writes the stage's partial.
// Consumer warps never wait on each other.  In the linear form the warp whose
// stage holds a row's drafted token also records that token's logit and q
// value, so that the accept test needs no second look at the rows.  The unaligned edge
// elements of a row (< 16 bytes at each end) are read with plain loads by the
// warp of the row's first stage.  Every wait is bounded in time.
#include <cfloat>

#include "stats_role.cuh"

namespace specdec {
namespace {

using namespace stage;


// kA: also the entropy sums of non-greedy rows (SPECDEC_STATS_ENTROPY).
template <int DT, bool kA>
__global__ void __launch_bounds__(kThreads, 1) row_stats_kernel(const RowStatsParams p) {
  // Launched programmatically dependent on the kernel before it on the stream:
  // wait for that kernel's completion before anything else, so only the
  // launch itself overlaps it; then let phase 2 launch (it waits for this
  // grid's completion itself).
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ __align__(128) uint8_t smem_raw[];
  StatsSmem &sm = *reinterpret_cast<StatsSmem *>(smem_raw);
  stats_role<DT, kA>(p, sm, (long long)blockIdx.x, (long long)gridDim.x);
}

template <int DT, bool kA>
cudaError_t launch_dt(const RowStatsParams &p, cudaStream_t stream) {
  static DeviceOnce once;
  const int smem = (int)sizeof(StatsSmem);
  const cudaError_t err = smem_opt_in_once(once, row_stats_kernel<DT, kA>, smem);
  if (err != cudaSuccess) return err;
  const long long units = p.stages / p.spr * ((p.spr + kUnit - 1) / kUnit);
  long long grid = device_sm_count();
  if (grid > units) grid = units;
  return launch_pdl(row_stats_kernel<DT, kA>, dim3((unsigned)grid), dim3(kThreads), (size_t)smem,
                    stream, p);
}

}  // namespace

cudaError_t launch_row_stats(const RowStatsParams &p, cudaStream_t stream) {
  if (p.stages <= 0) return cudaSuccess;
  if (p.entropy)
    return p.dtype == SPECDEC_F32 ? launch_dt<SPECDEC_F32, true>(p, stream)
                                  : launch_dt<SPECDEC_BF16, true>(p, stream);
  return p.dtype == SPECDEC_F32 ? launch_dt<SPECDEC_F32, false>(p, stream)
                                : launch_dt<SPECDEC_BF16, false>(p, stream);
}

namespace {
std::atomic<int> g_sm_count[kMaxCachedDevices]{};
}  // namespace

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  int n = (dev < kMaxCachedDevices) ? g_sm_count[dev].load(std::memory_order_relaxed) : 0;
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    if (dev < kMaxCachedDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace specdec
