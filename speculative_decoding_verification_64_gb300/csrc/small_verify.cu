// Linear verify of a small batch in one launch ("Chapter 15: Decoding
// acceleration", section 15.1.2 steps 2-4): the B = 1 latency case.
//
// The two-kernel step (stats pass, then the draw) pays two launches and
// several dependent memory round trips in each; with a handful of requests
// the data is small enough to stay on chip instead.  One 8-CTA cluster per
// request:
//
// * CTA r bulk-copies its share of every row of the request -- stages r*n ..
//   r*n + n - 1 (8 KB each) of the gamma+1 target rows and of the gamma q
//   rows -- into shared memory, once;
// * each warp reduces whole stages exactly as the stats pass does (the same
//   stage routines on the same 8 KB stages), so the partials it writes to the
//   workspace are the stats pass's, bit for bit; rank 0 also writes the
//   gathered (logit, q) of the drafted tokens and zeroes the request's ticket,
//   so the workspace ends as the two-kernel step leaves it;
// * after a cluster barrier every CTA merges the partials and runs the accept
//   test with the draw kernels' own routine (same merge order, same decision);
// * the draw reads row k's slices from shared memory: per-vector weights in
//   40-bit fixed point summed per thread, a scan over the CTA and one over the
//   cluster (distributed shared memory), then the thread whose range holds
//   U * Z finds the token -- the vector-ordered CDF of the bulk draw, so the
//   token is the two-kernel step's.
//
// Every CTA of a cluster runs the same sequence of cluster barriers (the
// branches between them depend only on the decision, which all CTAs compute
// alike); the one wait on memory (the bulk copies) is bounded.  Remote shared
// memory is only written (each slot once per launch) before a cluster barrier,
// never read.
#include <cfloat>

#include <cooperative_groups.h>

#include "linear_decision.cuh"
#include "stats_stage.cuh"

namespace specdec {
namespace {

namespace cg = cooperative_groups;
using namespace drawc;

constexpr int kC = 8;                      // CTAs per request: one portable cluster
constexpr int kT = 512;                    // threads per CTA (a warp per stage at B = 1)
constexpr int kW = kT / 32;
constexpr int kVecPerStage = kStageBytes / 16;
constexpr int kMaxDynSmem = 200 * 1024;    // row slices plus the header

struct Head {
  alignas(8) uint64_t full;                // completes when this CTA's slices have landed
  lindec::DecisionSmem dec;
  unsigned long long red[kW];
  unsigned long long tot[2][kC];           // every CTA's draw weight, stored by that CTA; by attempt
  int abort_flag;
};
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

template <int DT>
__global__ void __cluster_dims__(kC, 1, 1) __launch_bounds__(kT, 1)
    small_verify_kernel(const LinearFinalizeParams p) {
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
  uint8_t *qsl = slices + (size_t)R * nst * kStageBytes;  // [gamma][nst][kStageBytes]
  auto stage_bytes = [&](int j) { return min(kStageBytes, rowbytes - j * kStageBytes); };

  if (tid == 0) {
    mbar_init(&h.full, 1);
    h.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // ---- this CTA's slices of the request's rows, one bulk copy per stage ----
  if (tid == 0) {
    uint32_t total = 0;
    for (int t = 0; t < nj; ++t) total += (uint32_t)stage_bytes(j0 + t) * (uint32_t)(R + gamma);
    mbar_arrive_expect_tx(&h.full, total);
    const uint8_t *lg = reinterpret_cast<const uint8_t *>(p.logits) + (size_t)b * R * rowbytes;
    const uint8_t *qg = reinterpret_cast<const uint8_t *>(p.q) + (size_t)b * gamma * rowbytes;
    for (int r = 0; r < R; ++r)
      for (int t = 0; t < nj; ++t)
        bulk_copy_g2s(lsl + ((size_t)r * nst + t) * kStageBytes,
                      lg + (size_t)r * rowbytes + (size_t)(j0 + t) * kStageBytes,
                      (uint32_t)stage_bytes(j0 + t), &h.full);
    for (int r = 0; r < gamma; ++r)
      for (int t = 0; t < nj; ++t)
        bulk_copy_g2s(qsl + ((size_t)r * nst + t) * kStageBytes,
                      qg + (size_t)r * rowbytes + (size_t)(j0 + t) * kStageBytes,
                      (uint32_t)stage_bytes(j0 + t), &h.full);
  }
  // ---- the gathered (logit, q) of the drafted tokens, and the ticket ----------
  if (rank == 0 && tid < gamma) {
    const int x = __ldg(p.tokens + b * gamma + tid);
    if (x >= 0 && x < V) {
      const float lx = load_elem(p.logits, DT, (b * R + tid) * (long long)V + x);
      const float qx = load_elem(p.q, DT, (b * gamma + tid) * (long long)V + x);
      p.ws.gather[b * R + tid] = make_float2(lx, qx);
    }
  }
  if (rank == 0 && tid == 0) p.ws.draw_cnt[b] = 0u;
  // ---- stage statistics, as the stats pass computes them --------------------
  const bool ok = mbar_wait_bounded(&h.full, 0);
  if (!ok) h.abort_flag = 1;
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
  }
  // A cluster barrier with release (arrive) and acquire (wait) semantics at
  // cluster scope orders global memory as well: the partials and gathers
  // written above are visible to every CTA of the cluster after it, with no
  // GPU-scope fence.
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
  // ---- the accept test: every CTA alike, rank 0 writes the outputs ----------
  const LinearDecision d = lindec::request_decision<DT, kT>(p, b, rank == 0, h.dec);
  if (!(d.status || d.greedy)) {
    // ---- the draw over row k: this CTA's vectors, in index order -------------
    const int k = d.k;
    bool use_q = k < gamma;
    const int nvec = (nj > 0) ? (nj - 1) * kVecPerStage + stage_bytes(j0 + nj - 1) / 16 : 0;
    const uint4 *lk = reinterpret_cast<const uint4 *>(lsl + (size_t)k * nst * kStageBytes);
    const uint4 *qk = reinterpret_cast<const uint4 *>(qsl + (size_t)(use_q ? k : 0) * nst * kStageBytes);
    const int per = (nvec + kT - 1) / kT;
    const int v0 = min(nvec, tid * per), v1 = min(nvec, v0 + per);
    const uint4 none = make_uint4(0u, 0u, 0u, 0u);
    unsigned long long mine = 0, pre = 0, Z = 0, cta_pre = 0;
    for (int attempt = 0; attempt < 2; ++attempt) {
      mine = 0;
      for (int v = v0; v < v1; ++v) mine += to_fixed40(vec_sum<DT>(lk[v], use_q ? qk[v] : none, d, use_q));
      unsigned long long tot;
      pre = cta_exscan_u64(mine, h.red, tot);
      // this CTA's total into slot [attempt][rank] of every CTA (remote stores,
      // visible after the barrier; a slot is written once per launch)
      if (tid == 0)
        for (int r = 0; r < kC; ++r) cluster.map_shared_rank(&h, r)->tot[attempt][rank] = tot;
      cluster.sync();
      cta_pre = 0;
      Z = 0;
#pragma unroll
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
    if (lo <= target && target - lo < mine) {
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
  // No CTA touches another's shared memory after the draw's last cluster
  // barrier (the totals are stored before it; none at all on the other
  // paths), so a CTA may leave now.  Copies of a
  // CTA whose wait gave up are waited for (bounded) before it exits.
  if (h.abort_flag && tid == 0) mbar_wait_bounded(&h.full, 0);
}

template <int DT>
cudaError_t launch_dt(const LinearFinalizeParams &p, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    err = cudaFuncSetAttribute(small_verify_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kHeadBytes + kMaxDynSmem);
    if (err != cudaSuccess) return err;
    attr_set[dev] = true;
  }
  const int es = (DT == SPECDEC_F32) ? 4 : 2;
  const int spr = stages_per_row(p.V, es);
  const int nst = (spr + kC - 1) / kC;
  const size_t smem = (size_t)kHeadBytes + (size_t)(2 * p.gamma + 1) * nst * kStageBytes;
  small_verify_kernel<DT><<<(unsigned)(p.B * kC), kT, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool small_verify_applies(int B, int gamma, int V, int dtype, const void *logits, const void *q) {
  const int es = (dtype == SPECDEC_F32) ? 4 : 2;
  const long long rowbytes = (long long)V * es;
  if (B < 1 || rowbytes % 16 != 0) return false;
  if ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(q)) & 15) return false;
  if ((long long)B * kC > device_sm_count()) return false;  // one CTA per SM, one wave
  const int spr = stages_per_row(V, es);
  const int nst = (spr + kC - 1) / kC;
  return (long long)(2 * gamma + 1) * nst * kStageBytes <= kMaxDynSmem;
}

cudaError_t launch_small_verify(const LinearFinalizeParams &p, cudaStream_t stream) {
  if (p.B <= 0) return cudaSuccess;
  return (p.dtype == SPECDEC_F32) ? launch_dt<SPECDEC_F32>(p, stream)
                                  : launch_dt<SPECDEC_BF16>(p, stream);
}

}  // namespace specdec
