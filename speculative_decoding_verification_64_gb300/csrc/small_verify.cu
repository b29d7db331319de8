// Linear verify of a small batch in one launch ("Chapter 15: Decoding
// acceleration", section 15.1.2 steps 2-4): the B = 1 latency case and
// batches up to a few dozen requests.
//
// The two-kernel step (stats pass, then the draw) pays two launches and
// several dependent memory round trips in each; with few requests the data is
// small enough to stay on chip instead.  One cluster of C CTAs per request
// (C = 16, 8, 4 or 2: the largest of which the device holds all B clusters at
// once, one CTA per SM):
//
// * CTA r bulk-copies its share of every target row of the request -- stages
//   r*n .. r*n + n - 1 (8 KB each) of the gamma+1 rows -- into shared memory,
//   once, and the same share of the gamma q rows when they fit as well;
// * each warp reduces whole stages exactly as the stats pass does (the same
//   stage routines on the same 8 KB stages), so the partials it writes to the
//   workspace are the stats pass's, bit for bit; rank 0 also writes the
//   gathered (logit, q) of the drafted tokens and zeroes the request's ticket,
//   so the workspace ends as the two-kernel step leaves it;
// * the partials (and rank 0's gathered logit and q values) also go to every
//   CTA's shared memory by asynchronous remote stores on an mbarrier; every
//   CTA then merges them and runs the accept test with the draw kernels' own
//   routine (same merge order, same decision);
// * when the q rows are not resident and draft k was rejected, each CTA copies
//   its share of q row k into the slot of the bonus row, which is no longer
//   needed (k < gamma);
// * the draw reads row k's slices from shared memory: per-vector weights in
//   40-bit fixed point summed per thread, a scan over the CTA and one over the
//   cluster (distributed shared memory), then the thread whose range holds
//   U * Z finds the token -- the vector-ordered CDF of the bulk draw, so the
//   token is the two-kernel step's.
//
// Every CTA of a cluster runs the same sequence of cluster barriers and
// exchanges (the branches between them depend only on the decision, which all
// CTAs compute alike); the waits on memory (the bulk copies, the exchanges)
// are bounded.  Remote shared memory is only written, by asynchronous stores
// that complete on the receiver's barrier (each slot once per launch), never
// read.
#include <cfloat>

#include <cooperative_groups.h>

#include "linear_decision.cuh"
#include "stats_stage.cuh"

namespace specdec {
namespace {

namespace cg = cooperative_groups;
using namespace drawc;

// CTAs per request at most: 16, a cluster size beyond the portable 8 that
// the kernel opts into (taken only where the device can hold such a cluster)
#ifndef SPECDEC_SMALL_MAX_C
#define SPECDEC_SMALL_MAX_C 16
#endif
constexpr int kMaxC = SPECDEC_SMALL_MAX_C;
constexpr int kT = 512;                    // threads per CTA (a warp per stage at B = 1)
constexpr int kW = kT / 32;
constexpr int kVecPerStage = kStageBytes / 16;
constexpr int kMaxDynSmem = 200 * 1024;    // row slices plus the header
// stage partials of a request: (gamma + 1) * ceil(spr / C) stage slots fit in
// kMaxDynSmem, so R * spr <= 25 C
constexpr int kMaxPart = (kMaxDynSmem / kStageBytes) * kMaxC;

struct Head {
  alignas(8) uint64_t full;                // completes when this CTA's slices have landed
  alignas(8) uint64_t pbar;                // every CTA's stage partials and rank 0's gathers have arrived
  alignas(16) RowPartial part[kMaxPart];   // the request's stage partials [R][spr], pushed by their CTAs
  float2 gath[SPECDEC_MAX_GAMMA];          // the drafted tokens' (logit, q), pushed by rank 0
  lindec::DecisionSmem dec;
  unsigned long long red[kW];
  unsigned long long tot[2][kMaxC];        // every CTA's draw weight, stored by that CTA; by attempt
  alignas(8) uint64_t xbar[2];             // the exchange's arrivals, by attempt
  int abort_flag;                          // 1 + the parity of the copy wait that gave up, or 0
  int abort_any;                           // some CTA's q-row wait (or an exchange wait) gave up
};
// A CTA total carrying this bit reports a q-row wait that gave up (totals stay
// below it: at most 2^21 weights <= 1 with 40 fraction bits).
constexpr unsigned long long kAbortBit = 1ull << 63;
constexpr int kHeadBytes = (int)((sizeof(Head) + 127) / 128 * 128);

__device__ __forceinline__ unsigned long long cta_exscan_u64(unsigned long long v,
                                                             unsigned long long *red,
                                                             unsigned long long &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const unsigned long long y = shfl_up_u64(inc, d);
    if (lane >= d) inc += y;
  }
  if (lane == 31) red[warp] = inc;
  __syncthreads();
  unsigned long long pre = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < kW; ++i) {
    if (i < warp) pre += red[i];
    tot += red[i];
  }
  __syncthreads();  // red is reused by the next scan
  total = tot;
  return pre + inc - v;
}

// 16 bytes into another CTA's shared memory, completing bytes on its barrier
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint4 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::
                   "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(bar)
               : "memory");
}

// The stats results of the request as the decision reads them: the copies
// pushed into this CTA's shared memory.
struct CopySrc {
  const RowPartial *part;  // [R][spr]
  const float2 *gath;
  int spr, R;
  long long b;
  __device__ __forceinline__ float4 partial(long long row, int j) const {
    return *reinterpret_cast<const float4 *>(part + (row - b * R) * spr + j);
  }
  __device__ __forceinline__ float2 gather(long long, int i) const { return gath[i]; }
};

// kC: CTAs per request (the launch's cluster size); qres: the q rows are
// resident too, else q row k is copied in after the decision.
template <int DT>
__global__ void __launch_bounds__(kT, 1)
    small_verify_kernel(const LinearFinalizeParams p, const int kC, const bool qres) {
  // launched programmatically dependent on the kernel before it: only the
  // launch overlaps that kernel (wait for it first); a next call's kernels
  // wait for this grid's completion themselves
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Head &h = *reinterpret_cast<Head *>(smem_raw);
  uint8_t *slices = smem_raw + kHeadBytes;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const long long b = blockIdx.x / kC;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int es = (DT == SPECDEC_F32) ? 4 : 2;
  constexpr int kN = 16 / es;
  const int gamma = p.gamma, R = gamma + 1, V = p.V, spr = p.spr;
  const int rowbytes = V * es;
  const int nst = (spr + kC - 1) / kC;          // stage slots per CTA
  const int j0 = rank * nst;                    // this CTA's first stage
  const int nj = max(0, min(spr - j0, nst));    // stages it holds
  uint8_t *lsl = slices;                        // [R][nst][kStageBytes]
  uint8_t *qsl = slices + (size_t)R * nst * kStageBytes;  // [gamma][nst][kStageBytes] if qres
  const uint8_t *qg = reinterpret_cast<const uint8_t *>(p.q) + (size_t)b * gamma * rowbytes;
  auto stage_bytes = [&](int j) { return min(kStageBytes, rowbytes - j * kStageBytes); };

  if (tid == 0) {
    mbar_init(&h.full, 1);
    mbar_init(&h.pbar, 1);     // initialised before the cluster arrival below,
    mbar_init(&h.xbar[0], 1);  // so before any remote store completes on them
    mbar_init(&h.xbar[1], 1);
    h.abort_flag = 0;
    h.abort_any = 0;
    fence_mbar_init();
    mbar_arrive_expect_tx(&h.pbar, (uint32_t)(R * spr * sizeof(RowPartial) + gamma * sizeof(float2)));
  }
  __syncthreads();
  // every CTA of the cluster is running with its barriers initialised before
  // any stores into its shared memory (arrive now, wait before the first)
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  // ---- this CTA's slices of the request's rows, one bulk copy per stage ----
  if (tid == 0) {
    const int qrows = qres ? gamma : 0;
    uint32_t total = 0;
    for (int t = 0; t < nj; ++t) total += (uint32_t)stage_bytes(j0 + t) * (uint32_t)(R + qrows);
    mbar_arrive_expect_tx(&h.full, total);
    const uint8_t *lg = reinterpret_cast<const uint8_t *>(p.logits) + (size_t)b * R * rowbytes;
    for (int r = 0; r < R; ++r)
      for (int t = 0; t < nj; ++t)
        bulk_copy_g2s(lsl + ((size_t)r * nst + t) * kStageBytes,
                      lg + (size_t)r * rowbytes + (size_t)(j0 + t) * kStageBytes,
                      (uint32_t)stage_bytes(j0 + t), &h.full);
    for (int r = 0; r < qrows; ++r)
      for (int t = 0; t < nj; ++t)
        bulk_copy_g2s(qsl + ((size_t)r * nst + t) * kStageBytes,
                      qg + (size_t)r * rowbytes + (size_t)(j0 + t) * kStageBytes,
                      (uint32_t)stage_bytes(j0 + t), &h.full);
  }
  // ---- the gathered (logit, q) of the drafted tokens, and the ticket ----------
  float2 gx = make_float2(0.0f, 1.0f);  // (pushed to every CTA below; unused for a bad token)
  if (rank == 0 && tid < gamma) {
    const int x = __ldg(p.tokens + b * gamma + tid);
    if (x >= 0 && x < V) {
      const float lx = load_elem(p.logits, DT, (b * R + tid) * (long long)V + x);
      const float qx = load_elem(p.q, DT, (b * gamma + tid) * (long long)V + x);
      gx = make_float2(lx, qx);
      p.ws.gather[b * R + tid] = gx;
    }
  }
  if (rank == 0 && tid == 0) p.ws.draw_cnt[b] = 0u;
  // ---- stage statistics, as the stats pass computes them --------------------
  // one outcome for the whole CTA (the threads could see the wait give up
  // differently, and the stage reductions below are warp-synchronous)
  const bool ok = __syncthreads_and(mbar_wait_bounded(&h.full, 0, kConsumerWaitNs)) != 0;
  if (!ok) h.abort_flag = 1;  // the partials carry SPECDEC_ROW_INTERNAL: no draw follows
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  // the request's partials and gathers go to every CTA of the cluster by
  // asynchronous remote stores completing on its barrier pbar (the decision
  // then reads them from shared memory: no cluster barrier, no L2 round trip)
  const uint32_t pbar_a = smem_addr(&h.pbar);
  if (rank == 0 && tid < gamma) {
    // (x in the low word, y in the high: the float2's bytes)
    const unsigned long long g =
        ((unsigned long long)__float_as_uint(gx.y) << 32) | __float_as_uint(gx.x);
    for (int r = 0; r < kC; ++r)
      st_async_u64(cluster_addr(smem_addr(&h.gath[tid]), (uint32_t)r), g,
                   cluster_addr(pbar_a, (uint32_t)r));
  }
  const float T = __ldg(p.temperature + b);
  const float c = temperature_scale(T);
  for (int item = warp; item < R * nj; item += kW) {
    const int r = item / nj, t = item - r * nj;
    const int j = j0 + t;
    stage::LaneData<DT> d;
    d.edge = -INFINITY;
    d.edge_idx = 0x7FFFFFFF;
    RowPartial part;
    part.flags = ok ? 0 : SPECDEC_ROW_INTERNAL;
    part.arg = 0x7FFFFFFF;
    part.m = -INFINITY;
    part.s = 0.0f;
    if (ok) {
      stage::load_lane<DT>(d, lsl + ((size_t)r * nst + t) * kStageBytes, stage_bytes(j) / 16, lane);
      const float wm = stage::warp_max_nan(stage::lane_max<DT>(d));
      part.m = wm;
      if (T == 0.0f) {
        const int first_idx = (wm == wm && wm != -INFINITY)
                                  ? stage::lane_first<DT>(d, wm, j * (kStageBytes / es), lane)
                                  : 0x7FFFFFFF;
        part.arg = stage::warp_min(first_idx);
        part.s = (wm == -INFINITY) ? 0.0f : 1.0f;
      } else if (wm != -INFINITY) {
        part.s = stage::warp_sum(stage::lane_sum<DT>(d, c, wm));
      }
    }
    // the workspace's partials (read-only for the draw kernels, written here)
    if (lane == 0) const_cast<RowPartial *>(p.part)[(b * R + r) * (long long)spr + j] = part;
    if (lane < kC)  // and every CTA's copy, lane r storing into CTA r
      st_async_v4(cluster_addr(smem_addr(&h.part[r * spr + j]), (uint32_t)lane),
                  make_uint4(__float_as_uint(part.m), __float_as_uint(part.s), (uint32_t)part.arg,
                             (uint32_t)part.flags),
                  cluster_addr(pbar_a, (uint32_t)lane));
  }
  // every CTA's partials and the gathers here (one outcome for the CTA)
  const bool got = __syncthreads_and(mbar_wait_cluster_bounded(&h.pbar, 0)) != 0;
  // ---- the accept test: every CTA alike, rank 0 writes the outputs ----------
  LinearDecision d;
  if (got) {
    d = lindec::request_decision_from<DT, kT>(p, b, rank == 0, h.dec, CopySrc{h.part, h.gath, spr, R, b});
  } else {
    // another CTA's results never arrived: the request gets SPECDEC_ROW_INTERNAL
    d.status = SPECDEC_ROW_INTERNAL;
    d.greedy = false;
    if (rank == 0) {
      if (tid < R) p.out_tokens[b * R + tid] = -1;
      if (tid < gamma && p.p_draft) p.p_draft[b * gamma + tid] = __int_as_float(0x7fc00000);
      if (tid == 0) {
        p.n_accepted[b] = 0;
        p.is_bonus[b] = 0;
        p.row_status[b] = SPECDEC_ROW_INTERNAL;
        p.final_token[b] = -1;
        p.ws.mass[b] = kNoMass;
      }
    }
  }
  if (!(d.status || d.greedy)) {
    // ---- the draw over row k: this CTA's vectors, in index order -------------
    const int k = d.k;
    bool use_q = k < gamma;
    const int nvec = (nj > 0) ? (nj - 1) * kVecPerStage + stage_bytes(j0 + nj - 1) / 16 : 0;
    const uint4 *lk = reinterpret_cast<const uint4 *>(lsl + (size_t)k * nst * kStageBytes);
    const uint4 *qk = reinterpret_cast<const uint4 *>(qsl + (size_t)(use_q ? k : 0) * nst * kStageBytes);
    if (!qres && use_q) {
      // q row k into the bonus row's slot (k < gamma; every read of that slot,
      // by the stage statistics, was before the CTA barriers above), second
      // phase of the copy barrier
      uint8_t *slot = lsl + (size_t)gamma * nst * kStageBytes;
      if (tid == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        uint32_t total = 0;
        for (int t = 0; t < nj; ++t) total += (uint32_t)stage_bytes(j0 + t);
        mbar_arrive_expect_tx(&h.full, total);
        for (int t = 0; t < nj; ++t)
          bulk_copy_g2s(slot + (size_t)t * kStageBytes,
                        qg + (size_t)k * rowbytes + (size_t)(j0 + t) * kStageBytes,
                        (uint32_t)stage_bytes(j0 + t), &h.full);
      }
      qk = reinterpret_cast<const uint4 *>(slot);
      // one outcome for the CTA: a thread that saw the wait give up while
      // thread 0 did not must not let junk sums pass as a draw
      if (!__syncthreads_and(mbar_wait_bounded(&h.full, 1, kConsumerWaitNs))) {
        // this CTA's share never landed: the request gets SPECDEC_ROW_INTERNAL
        // (told to every CTA with the first exchange); its sums are junk
        if (tid == 0) h.abort_flag = 2;
      }
    }
    const int per = (nvec + kT - 1) / kT;
    const int v0 = min(nvec, tid * per), v1 = min(nvec, v0 + per);
    const uint4 none = make_uint4(0u, 0u, 0u, 0u);
    unsigned long long mine = 0, pre = 0, Z = 0, cta_pre = 0;
    for (int attempt = 0; attempt < 2; ++attempt) {
      mine = 0;
      for (int v = v0; v < v1; ++v) mine += to_fixed40(vec_sum<DT>(lk[v], use_q ? qk[v] : none, d, use_q));
      unsigned long long tot;
      pre = cta_exscan_u64(mine, h.red, tot);
      // this CTA's total (with the abort bit if its q-row wait gave up) into
      // slot [attempt][rank] of every CTA by asynchronous remote stores that
      // complete on that CTA's barrier xbar[attempt]; then the kC totals here
      if (tid == 0) {
        uint64_t *bar = &h.xbar[attempt];
        mbar_arrive_expect_tx(bar, (uint32_t)(kC * sizeof(unsigned long long)));
        const uint32_t slot = smem_addr(&h.tot[attempt][rank]), ba = smem_addr(bar);
        const unsigned long long v = tot | (h.abort_flag == 2 ? kAbortBit : 0ull);
        for (int r = 0; r < kC; ++r) st_async_u64(cluster_addr(slot, (uint32_t)r), v, cluster_addr(ba, (uint32_t)r));
        bool any = !mbar_wait_cluster_bounded(bar, 0);
        for (int r = 0; r < kC; ++r) any |= (h.tot[attempt][r] & kAbortBit) != 0;
        h.abort_any = any;
      }
      __syncthreads();
      if (h.abort_any) break;  // uniform: every CTA sees every total's abort bit
      cta_pre = 0;
      Z = 0;
      for (int r = 0; r < kC; ++r) {
        const unsigned long long x = h.tot[attempt][r];
        if (r < rank) cta_pre += x;
        Z += x;
      }
      if (!(Z == 0 && use_q)) break;
      use_q = false;   // residual mass 0 (only by rounding): draw from p, as the other draws do
    }
    const unsigned long long target = uniform_target(__ldg(p.uniforms + b * R + gamma), Z);
    const unsigned long long lo = cta_pre + pre;
    if (rank == 0 && tid == 0) p.ws.mass[b] = h.abort_any ? kNoMass : draw_mass(Z, d.S);
    if (h.abort_any) {
      // the malformed-request outputs, over what the decision wrote (same threads)
      if (rank == 0) {
        if (tid < R) p.out_tokens[b * R + tid] = -1;
        if (tid == 0) {
          p.n_accepted[b] = 0;
          p.is_bonus[b] = 0;
          p.row_status[b] = SPECDEC_ROW_INTERNAL;
          p.final_token[b] = -1;
        }
      }
    } else if (lo <= target && target - lo < mine) {
      unsigned long long run = lo;
      for (int v = v0; v < v1; ++v) {
        const uint4 lv = lk[v], qv = use_q ? qk[v] : none;
        const unsigned long long f = to_fixed40(vec_sum<DT>(lv, qv, d, use_q));
        if (run + f > target) {
          const int e = vec_find<DT>(lv, qv, d, use_q, run, target);
          const int tok = ((j0 * kVecPerStage) + v) * kN + e;
          p.final_token[b] = tok;
          p.out_tokens[b * R + k] = tok;
          break;
        }
        run += f;
      }
    }
  }
  // Every store into this CTA's shared memory has landed once its last
  // exchange wait completed, and none follows (no remote store at all on the
  // other paths), so a CTA may leave now.  Copies of a
  // CTA whose wait gave up are waited for (bounded) before it exits.
  if (h.abort_flag && tid == 0) mbar_wait_bounded(&h.full, (uint32_t)(h.abort_flag - 1));
}

// The cluster size and residency a call takes, or false for the two kernels.
struct Plan {
  int C;
  bool qres;
};

// How many clusters of C CTAs (C = 16, 8, 4 or 2) the device holds at once
// with one CTA of this kernel per SM, once per device and size: the count
// depends on how the SMs fall into GPCs, so it can be below SMs / C, and a
// batch of more clusters runs in two waves.  16 needs the non-portable
// cluster size opt-in.  -1 when the query is not answered (no device).
constexpr int kSizes = 4;  // C = 16 >> i
std::atomic<int> g_capacity[kMaxCachedDevices][kSizes]{};  // count + 2; 0: not asked yet

int cluster_capacity(int C) {
  const int i = (C == 16) ? 0 : (C == 8) ? 1 : (C == 4) ? 2 : 3;
  int dev = 0;
  if (C > kMaxC || cudaGetDevice(&dev) != cudaSuccess || dev < 0) return -1;
  int c = (dev < kMaxCachedDevices) ? g_capacity[dev][i].load(std::memory_order_relaxed) : 0;
  if (c != 0) return c - 2;
  int n = -1;
  const int smem = kHeadBytes + kMaxDynSmem;
  auto kernel = small_verify_kernel<SPECDEC_BF16>;
  bool ok = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess;
  if (ok && C > 8)
    ok = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
         cudaFuncSetAttribute(small_verify_kernel<SPECDEC_F32>,
                              cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
  if (ok) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)C);
    cfg.blockDim = dim3(kT);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute a[1];
    a[0].id = cudaLaunchAttributeClusterDimension;
    a[0].val.clusterDim.x = (unsigned)C;
    a[0].val.clusterDim.y = 1;
    a[0].val.clusterDim.z = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
    int m = 0;
    if (cudaOccupancyMaxActiveClusters(&m, kernel, &cfg) == cudaSuccess) n = m;
    else ok = false;
  }
  if (!ok) (void)cudaGetLastError();  // a refused query leaves no error behind
  if (dev < kMaxCachedDevices) g_capacity[dev][i].store(n + 2, std::memory_order_relaxed);
  return n;
}

bool plan_for(int B, int gamma, int V, int dtype, const void *logits, const void *q, Plan &pl) {
  const int es = (dtype == SPECDEC_F32) ? 4 : 2;
  const long long rowbytes = (long long)V * es;
  if (B < 1 || rowbytes % 16 != 0) return false;
  if ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(q)) & 15) return false;
  // the largest cluster size whose B clusters the device holds at once (one
  // CTA per SM); without an answer from the device, B C no more than its SMs
  // and at most 8
  const long long sms = device_sm_count();
  int C = kMaxC;
  for (; C >= 2; C /= 2) {
    const int cap = cluster_capacity(C);
    if (cap >= 0 ? B <= cap : (C <= 8 && (long long)B * C <= sms)) break;
  }
  if (C < 2) return false;
  const int spr = stages_per_row(V, es);
  if ((long long)(gamma + 1) * spr > kMaxPart) return false;  // (implied by the fit below)
  const long long slot = (long long)((spr + C - 1) / C) * kStageBytes;  // one row's share
  pl.C = C;
  if ((long long)(2 * gamma + 1) * slot <= kMaxDynSmem) {
    pl.qres = true;
    return true;
  }
  pl.qres = false;
  return (long long)(gamma + 1) * slot <= kMaxDynSmem;
}

template <int DT>
cudaError_t launch_dt(const LinearFinalizeParams &p, const Plan &pl, cudaStream_t stream) {
  static DeviceOnce once;
  cudaError_t err = smem_opt_in_once(once, small_verify_kernel<DT>, kHeadBytes + kMaxDynSmem);
  if (err != cudaSuccess) return err;
  const int es = (DT == SPECDEC_F32) ? 4 : 2;
  const int spr = stages_per_row(p.V, es);
  const int nst = (spr + pl.C - 1) / pl.C;
  const int rows = pl.qres ? 2 * p.gamma + 1 : p.gamma + 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * pl.C));
  cfg.blockDim = dim3(kT);
  cfg.dynamicSmemBytes = (size_t)kHeadBytes + (size_t)rows * nst * kStageBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)pl.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, small_verify_kernel<DT>, p, pl.C, pl.qres);
}

}  // namespace

bool small_verify_applies(int B, int gamma, int V, int dtype, const void *logits, const void *q) {
  Plan pl;
  return plan_for(B, gamma, V, dtype, logits, q, pl);
}

cudaError_t launch_small_verify(const LinearFinalizeParams &p, cudaStream_t stream) {
  if (p.B <= 0) return cudaSuccess;
  Plan pl;
  if (!plan_for(p.B, p.gamma, p.V, p.dtype, p.logits, p.q, pl)) return cudaErrorInvalidValue;
  return (p.dtype == SPECDEC_F32) ? launch_dt<SPECDEC_F32>(p, pl, stream)
                                  : launch_dt<SPECDEC_BF16>(p, pl, stream);
}

}  // namespace specdec
