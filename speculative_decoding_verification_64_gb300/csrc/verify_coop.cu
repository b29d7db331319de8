// Linear verify of a large batch in one cooperative launch ("Chapter 15:
// Decoding acceleration", section 15.1.2: step 2 scores every drafted
// position in one pass over the target logits; steps 3 and 4 accept drafts
// while u_i <= min(1, p_i/q_i) and draw the correction from max(0, p - q) / Z,
// or the bonus token from the last row when every draft is accepted).
//
// The same arithmetic as the two-launch step (the stats kernel, then the bulk
// draw), arranged as one persistent launch of one CTA per SM:
//
// 1. the stats pass's own loop (stats_role.cuh) on every CTA;
// 2. a grid barrier (every CTA is resident: a cooperative launch);
// 3. CTA i decides requests [B i / G, B (i + 1) / G): the draw kernels' row
//    merges and accept test, every output but a drawn token, and the
//    decision record of each request in the workspace behind a ready flag;
// 4. the draw's (request, 16 KB unit) pairs are dealt round robin, unit u to
//    CTA u mod G, the way the stats pass deals its units: every CTA gets the
//    same mix of rejected requests (logits and q rows), bonus requests
//    (logits only) and greedy ones (nothing), and at any moment the CTAs read
//    neighbouring units.  A CTA loads the records of its units' requests,
//    then a producer thread bulk-copies the units into a ring of shared-
//    memory slots and fifteen consumer warps sum each 4 KB stage's draw
//    weights in 40-bit fixed point;
// 5. per unit, the CTA adds the unit's stage count to its request's ticket;
//    the CTA that completes a ticket finds the token (search_warp).
//
// Against the two launches this removes the launch boundary, and the draw's
// stream ends with every CTA at about the same time (contiguous runs gave
// some CTAs twice the bytes of others).  Every routine is the two-launch
// step's on the same data, so the outputs and the workspace are the same bit
// for bit.  Every wait is bounded; a request whose wait gave up is reported
// as SPECDEC_ROW_INTERNAL.
#include <cfloat>

#include <cooperative_groups.h>

#include "linear_decision.cuh"
#include "stats_role.cuh"

namespace specdec {
namespace {

namespace cg = cooperative_groups;
using namespace drawc;

constexpr int kT = stage::kThreads;                 // 512: the stats pass's CTA
constexpr int kWarpsT = kT / 32;                    // 16
constexpr int kUnitStages = 4;                      // 4 KB draw stages per bulk copy
constexpr int kUnitBytes = kStage * kUnitStages;    // 16 KB of logits (+ 16 KB of q)
constexpr int kSlots = 6;
constexpr int kConsumers = kWarpsT - 1;             // the last warp produces
constexpr int kMaxReq = kWarpsT;                    // requests one CTA decides (a warp each)
constexpr int kMaxLocal = 256;                      // draw units of one CTA
constexpr unsigned kAbort = 1u << 24;               // ticket increment of a CTA whose wait ran out
static_assert(kConsumers <= kSlots * kUnitStages, "no more consumer warps than ring stages");

struct DrawSmem {
  alignas(128) uint8_t l[kSlots][kUnitBytes];
  alignas(128) uint8_t q[kSlots][kUnitBytes];
  alignas(8) uint64_t full[kSlots];
  alignas(8) uint64_t empty[kSlots];
  RowStat rs[kMaxReq][SPECDEC_MAX_GAMMA + 1];
  LinearDecision dec[kMaxLocal];  // the decision of each local unit's request
  unsigned char search[kMaxLocal];  // 1: this CTA completed the unit's ticket; 2: so, but a wait ran out
  volatile int abort_flag;
};

constexpr size_t kSmemBytes = (sizeof(stage::StatsSmem) > sizeof(DrawSmem))
                                  ? sizeof(stage::StatsSmem) : sizeof(DrawSmem);
static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM");

struct CoopParams {
  RowStatsParams st;
  LinearFinalizeParams p;
};

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned *a) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u32(unsigned *a, unsigned v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

template <int DT>
__device__ __forceinline__ Req req_of(const LinearFinalizeParams &p, long long b, int k) {
  constexpr int es = (DT == SPECDEC_F32) ? 4 : 2;
  Req r;
  r.b = b;
  const int R = p.gamma + 1;
  r.rowbytes = p.V * es;
  r.nst = (r.rowbytes + kStage - 1) / kStage;
  r.lrow = reinterpret_cast<const uint8_t *>(p.logits) + (size_t)(b * R + k) * r.rowbytes;
  r.qrow = (k < p.gamma)
               ? reinterpret_cast<const uint8_t *>(p.q) + (size_t)(b * p.gamma + k) * r.rowbytes
               : r.lrow;
  return r;
}

// Phase 3: the accept decisions of requests [b0, b0 + nreq) (warp j for
// request b0 + j), their outputs but a drawn token, and their records.
template <int DT>
__device__ __forceinline__ void decide_phase(const LinearFinalizeParams &p, DrawSmem &sm,
                                             long long b0, int nreq) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = p.gamma + 1;
  DraftIn din;
  float Tj = 0.0f;
  if (warp < nreq) {
    Tj = __ldg(p.temperature + b0 + warp);
    din = load_draft(p, b0 + warp, lane);
  }
  const int pairs = nreq * R;
  for (int base = 0; base < pairs; base += kT / kSeg) {
    if (base + warp * (32 / kSeg) >= pairs) continue;  // both segments of this warp idle
    const int pr = base + tid / kSeg;
    const bool active = pr < pairs;
    const int j = active ? pr / R : 0, r = active ? pr - j * R : 0;
    const float c = temperature_scale(__ldg(p.temperature + b0 + j));
    const RowStat st = segment_merge_row(p.part, (b0 + j) * R + r, active, p.spr, c, tid % kSeg);
    if (active && tid % kSeg == 0) sm.rs[j][r] = st;
  }
  __syncthreads();
  if (warp < nreq) {
    const long long b = b0 + warp;
    float pd;
    const LinearDecision d = decide(p, din, Tj, temperature_scale(Tj), sm.rs[warp], lane, pd);
    write_outputs_warp(p, b, d, pd, lane);
    if (lane == 0) {
      p.ws.dec[b] = d;
      __threadfence();  // the record before its flag
      st_relaxed_u32(p.ws.dec_ready + b, 1u);
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(kT, 1) verify_coop_kernel(const CoopParams cp) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const LinearFinalizeParams &p = cp.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long G = gridDim.x, i = blockIdx.x;
  cg::grid_group grid = cg::this_grid();

  // ---- the ready flags of the decision records start at zero (ordered
  // before any flag is set by the grid barrier below) ----
  for (long long b = i * kT + tid; b < p.B; b += G * kT) p.ws.dec_ready[b] = 0u;

  // ---- phase 1: the stats pass ----
  stage::StatsSmem &ss = *reinterpret_cast<stage::StatsSmem *>(smem_raw);
  stage::stats_role<DT, false>(cp.st, ss, i, G);
  __syncthreads();
  if (tid == 0) {  // the stats ring's barriers are done with: their memory is reused
    for (int s = 0; s < stage::kSlots; ++s) {
      mbar_inval(&ss.full[s]);
      mbar_inval(&ss.empty[s]);
    }
  }
  grid.sync();  // every partial, gather and zeroed ticket is visible

  DrawSmem &sm = *reinterpret_cast<DrawSmem *>(smem_raw);
  constexpr int es = (DT == SPECDEC_F32) ? 4 : 2;
  const int gamma = p.gamma;
  const int rowbytes = p.V * es;
  const int nst = (rowbytes + kStage - 1) / kStage;
  const int upr = (nst + kUnitStages - 1) / kUnitStages;  // draw units per row
  const long long units = (long long)p.B * upr;
  const int n_local = (units > i) ? (int)((units - i + G - 1) / G) : 0;  // <= kMaxLocal (host)

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kUnitStages);  // one arrival per stage of the unit
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }

  // ---- phase 3: this CTA's decisions ----
  {
    const long long b0 = (long long)p.B * i / G, b1 = (long long)p.B * (i + 1) / G;
    decide_phase<DT>(p, sm, b0, (int)(b1 - b0));
  }

  // ---- phase 4: the records of this CTA's draw units ----
  for (int t = tid; t < n_local; t += kT) {
    const long long b = (i + (long long)t * G) / upr;
    const unsigned *flag = p.ws.dec_ready + b;
    bool ok = ld_relaxed_u32(flag) != 0u;
    if (!ok) {
      const unsigned long long t0 = global_timer_ns();
      while (!(ok = ld_relaxed_u32(flag) != 0u) && global_timer_ns() - t0 < kWaitLimitNs) {
      }
    }
    LinearDecision d;
    if (ok) {
      __threadfence();  // acquire: the record is the one its flag announced
      const int4 *src = reinterpret_cast<const int4 *>(p.ws.dec + b);
      union {
        int4 v[2];
        LinearDecision d;
      } rec;
      rec.v[0] = __ldcg(src);
      rec.v[1] = __ldcg(src + 1);
      d = rec.d;
    } else {
      d.k = 0;
      d.status = SPECDEC_ROW_INTERNAL;  // nothing drawn; the ticket reports it
      d.greedy = 0;
      sm.abort_flag = 1;
    }
    sm.dec[t] = d;
  }
  __syncthreads();

  long long n_issued = 0;  // producer: units issued
  if (warp == kConsumers) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      uint32_t slot = 0, use = 0;
      for (int t = 0; t < n_local; ++t) {
        if (use > 0 && !mbar_wait_bounded(&sm.empty[slot], (use - 1) & 1)) {
          sm.abort_flag = 1;
          break;
        }
        if (sm.abort_flag) break;
        const long long u = i + (long long)t * G;
        const long long b = u / upr;
        const int ju = (int)(u - b * upr);
        const LinearDecision d = sm.dec[t];
        if (d.status || d.greedy) {
          mbar_arrive(&sm.full[slot]);  // nothing to draw: an empty unit
        } else {
          const Req rq = req_of<DT>(p, b, d.k);
          const bool use_q = d.k < gamma;
          const int bytes = min(kUnitBytes, rowbytes - ju * kUnitBytes);
          mbar_arrive_expect_tx(&sm.full[slot], (uint32_t)(bytes * (use_q ? 2 : 1)));
          bulk_copy_g2s(sm.l[slot], rq.lrow + (size_t)ju * kUnitBytes, (uint32_t)bytes,
                        &sm.full[slot]);
          if (use_q)
            bulk_copy_g2s(sm.q[slot], rq.qrow + (size_t)ju * kUnitBytes, (uint32_t)bytes,
                          &sm.full[slot]);
        }
        ++n_issued;
        if (++slot == kSlots) {
          slot = 0;
          ++use;
        }
      }
    }
  } else {
    // ------------------------------ consumers -----------------------------
    // local stage c = 4 t + ts (stage ts of local unit t) belongs to warp c % 15
    const int n_stages_local = n_local * kUnitStages;
    for (int c = warp; c < n_stages_local; c += kConsumers) {
      const int t = c / kUnitStages, ts = c - t * kUnitStages;
      const long long u = i + (long long)t * G;
      const long long b = u / upr;
      const int ju = (int)(u - b * upr);
      const uint32_t slot = (uint32_t)(t % kSlots), use = (uint32_t)(t / kSlots);
      const LinearDecision d = sm.dec[t];
      const int s = ju * kUnitStages + ts;  // stage within the row
      const bool real = !(d.status || d.greedy) && s < nst;
      const bool use_q = d.k < gamma;
      // the slot's previous use released first (a parity wait tells only two
      // phases apart, and copies land in any order), then this use's copy;
      // one outcome for the whole warp
      const bool ok = __all_sync(0xffffffffu,
                                 !sm.abort_flag &&
                                     (use == 0 || mbar_wait_bounded(&sm.empty[slot], (use - 1) & 1)) &&
                                     mbar_wait_bounded(&sm.full[slot], use & 1));
      if (!ok) sm.abort_flag = 1;
      uint4 lv[kVec], qv[kVec];
      const int sbytes = (ok && real) ? min(kStage, rowbytes - s * kStage) : 0;
      load_stage<DT>(lv, qv, sm.l[slot] + ts * kStage, sm.q[slot] + ts * kStage, sbytes, use_q,
                     lane, false);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[slot]);  // this stage is in registers now
      if (!real || !ok) continue;
      unsigned long long acc = 0;
#pragma unroll
      for (int k = 0; k < kVec; ++k) acc += to_fixed40(vec_sum<DT>(lv[k], qv[k], d, use_q));
      acc = warp_sum_u64(acc);
      if (lane == 0) p.ws.chunk_tot[b * p.ntot + s] = acc;
    }
  }
  __syncthreads();
  // after any wait of the CTA gave up, consumers stopped waiting for copies:
  // the CTA stays until every copy the producer issued has landed
  if (sm.abort_flag && warp == kConsumers && lane == 0) drain_ring(sm.full, kSlots, n_issued);

  // ---- phase 5: tickets (a thread per unit), then the searches ----
  for (int t = tid; t < n_local; t += kT) {
    sm.search[t] = 0;
    const LinearDecision d = sm.dec[t];
    if (d.status || d.greedy) continue;
    const long long u = i + (long long)t * G;
    const long long b = u / upr;
    const int ju = (int)(u - b * upr);
    __threadfence();  // this CTA's stage totals before its ticket
    const unsigned add = (unsigned)min(kUnitStages, nst - ju * kUnitStages) +
                         (sm.abort_flag ? kAbort : 0u);
    const unsigned now = atomicAdd(p.ws.draw_cnt + b, add) + add;
    if ((now & (kAbort - 1)) == (unsigned)nst) sm.search[t] = (now >= kAbort) ? 2 : 1;
  }
  __syncthreads();
  for (int t = warp; t < n_local; t += kWarpsT) {
    if (!sm.search[t]) continue;
    __threadfence();  // acquire: every CTA's totals of the request
    const LinearDecision d = sm.dec[t];
    const long long b = (i + (long long)t * G) / upr;
    const Req rq = req_of<DT>(p, b, d.k);
    if (lane == 0) p.ws.draw_cnt[b] = 0;  // phase 2 may run again on the same phase-1 result
    search_warp<DT>(p, rq, d, sm.search[t] == 2, lane,
                    GlobalTotals{p.ws.chunk_tot + b * p.ntot});
  }
}

}  // namespace

// The cooperative step needs 16-byte aligned rows (bulk copies), at most one
// request per warp to decide in each CTA and the records of its draw units in
// shared memory.
bool coop_verify_applies(const LinearFinalizeParams &p) {
  const int es = (p.dtype == SPECDEC_F32) ? 4 : 2;
  const long long rowbytes = (long long)p.V * es;
  if (rowbytes % 16 != 0) return false;
  if ((reinterpret_cast<uintptr_t>(p.logits) & 15) || (reinterpret_cast<uintptr_t>(p.q) & 15))
    return false;
  const long long G = device_sm_count();
  const long long nst = (rowbytes + kStage - 1) / kStage;
  const long long upr = (nst + kUnitStages - 1) / kUnitStages;
  if ((long long)p.B > G * kMaxReq) return false;
  if (((long long)p.B * upr + G - 1) / G > kMaxLocal) return false;
  return p.B >= G / 2;  // smaller batches: the other paths
}

cudaError_t launch_coop_verify(const RowStatsParams &st, const LinearFinalizeParams &p,
                               cudaStream_t stream) {
  static DeviceOnce once;
  const cudaError_t err = (p.dtype == SPECDEC_F32)
                              ? smem_opt_in_once(once, verify_coop_kernel<SPECDEC_F32>, (int)kSmemBytes)
                              : smem_opt_in_once(once, verify_coop_kernel<SPECDEC_BF16>, (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  CoopParams cp;
  cp.st = st;
  cp.p = p;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)device_sm_count());
  cfg.blockDim = dim3(kT);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: the grid barrier
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.dtype == SPECDEC_F32) return cudaLaunchKernelEx(&cfg, verify_coop_kernel<SPECDEC_F32>, cp);
  return cudaLaunchKernelEx(&cfg, verify_coop_kernel<SPECDEC_BF16>, cp);
}

}  // namespace specdec
