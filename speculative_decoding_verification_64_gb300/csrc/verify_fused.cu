// Linear verify of a large batch in one launch ("Chapter 15: Decoding
// acceleration", section 15.1.2: step 2 scores every drafted position in one
// pass over the target logits, steps 3 and 4 accept drafts while
// u_i <= min(1, p_i/q_i) and draw the correction from max(0, p - q) / Z, or
// the bonus token from the last row when every draft is accepted).
//
// The two-launch step runs the stats pass over all B (gamma+1) rows, then the
// draw, which starts only when the whole pass is done and reads each
// request's final logits row a second time from HBM, plus its q row after a
// rejection.  Here one persistent launch (one CTA per SM, all resident: a
// cooperative launch) splits the SMs by role:
//
// * the first S CTAs run the stats pass's own loop (stats_role.cuh) over the
//   requests in ascending order, cut into waves of Wr requests.  After every
//   stage a consumer warp counts it against its wave in shared memory; the
//   warp that completes the CTA's share of a wave fences and stores the
//   launch's epoch into the wave's flag of this CTA;
// * the other D CTAs draw.  Draw CTA d takes requests d, d + D, d + 2D, ...
//   A decider warp waits for the S flags of the request's wave, merges the
//   request's row partials (the draw kernels' merge order), runs the accept
//   test (their routine) and writes every output but the drawn token; then a
//   producer thread bulk-copies the final logits row -- read by the stats
//   pass moments before, so an L2 hit -- and, after a rejection, its q row
//   into a ring of shared-memory slots; thirteen consumer warps sum each 4 KB
//   stage's draw weights in 40-bit fixed point (the bulk draw's arithmetic:
//   the same totals); a searcher warp finds the token from the totals held in
//   shared memory.  Up to four requests are in flight in a CTA: the decider
//   runs ahead, the searcher behind the stream.
//
// So the draws of early waves overlap the stats pass of later ones: the q
// rows share HBM with the stats stream instead of following it, the final
// logits rows come from L2, and only the last wave's draws follow the pass.
// Every value is computed by the same routines on the same data as in the
// two-launch step (stage partials, gathers, decisions, stage totals), so the
// outputs and the workspace it leaves are the same bit for bit.
//
// Cross-CTA waits use a per-launch epoch instead of counters that would need
// zeroing (FusedSync in common.cuh): every CTA reads the epoch of the last
// completed launch when it starts and uses the next value; the last CTA to
// exit stores it.  Every wait is bounded in time; a request whose wait gave
// up is reported as SPECDEC_ROW_INTERNAL.
#include <cfloat>

#include "linear_decision.cuh"
#include "stats_role.cuh"

namespace specdec {
namespace {

using namespace drawc;

constexpr int kT = stage::kThreads;                 // 512: the stats pass's CTA
constexpr int kWarpsT = kT / 32;
constexpr int kUnitStages = 4;                      // 4 KB draw stages per bulk copy
constexpr int kUnitBytes = kStage * kUnitStages;    // 16 KB of logits (+ 16 KB of q)
constexpr int kSlots = 6;
constexpr int kDecider = 0, kProducer = 1, kSearcher = 2, kFirstConsumer = 3;
constexpr int kConsumers = kWarpsT - kFirstConsumer;  // 13
constexpr int kQ = 4;                               // requests in flight in a draw CTA
constexpr int kMaxStages = 128;                     // draw stages of a row held in shared memory
constexpr int kMinStages = 16;                      // shorter rows take the two-launch step
static_assert(kConsumers <= kSlots * kUnitStages, "no more consumer warps than ring stages");

struct ReqSlot {
  LinearDecision dec;
  long long b;
  unsigned int nsum;  // stages summed by the consumers
  unsigned int pad;
  unsigned long long tot[kMaxStages];
};

struct DrawSmem {
  alignas(128) uint8_t l[kSlots][kUnitBytes];
  alignas(128) uint8_t q[kSlots][kUnitBytes];
  alignas(8) uint64_t full[kSlots];
  alignas(8) uint64_t empty[kSlots];
  ReqSlot rq[kQ];
  RowStat rs[SPECDEC_MAX_GAMMA + 1];
  volatile int armed;        // requests handed to the producer, consumers and searcher
  volatile int last;         // the CTA's count of drawn requests, once known (else INT_MAX)
  volatile int freed;        // requests the searcher finished
  volatile int abort_flag;
  volatile long long issued;  // units the producer issued, once it stopped (else -1)
};

struct StatsExtra {
  unsigned int cnt[8];                         // stages done, per wave (mod 8)
  unsigned int need[SPECDEC_FUSED_MAX_WAVES];  // stages of this CTA in each wave
};

struct FusedParams {
  RowStatsParams st;
  LinearFinalizeParams p;
  int S;        // stats CTAs (the first S of the grid); the others draw
  int Wr;       // requests per wave
  int n_waves;
  int rpw;      // rows per wave: Wr * (gamma + 1)
};

constexpr size_t kStatsBytes = (sizeof(stage::StatsSmem) + 127) / 128 * 128;
constexpr size_t kSmemBytes =
    (kStatsBytes + sizeof(StatsExtra) > sizeof(DrawSmem)) ? kStatsBytes + sizeof(StatsExtra)
                                                          : sizeof(DrawSmem);
static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM");

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned *p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u32(unsigned *p, unsigned v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void mbar_arrive_cnt(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// ---------------------------------------------------------------------------
// stats CTAs: the wave hook
// ---------------------------------------------------------------------------
// Called by every consumer warp after each of its stages (lane 0 stored the
// partial).  The warp completing the CTA's share of a wave releases the
// partials and gathers of the whole CTA (they were ordered before each warp's
// count by a CTA-scope fence) with a GPU-scope fence, then stores the flag.
struct WaveHook {
  unsigned int *flags;  // this CTA's flag of wave 0; wave w at flags[w * S]
  StatsExtra *ex;
  int S, rpw;
  unsigned int epoch;
  __device__ __forceinline__ void operator()(int row, int lane) const {
    if (lane != 0) return;
    const int w = row / rpw;
    __threadfence_block();
    const unsigned old = atomicAdd(&ex->cnt[w & 7], 1u);
    if (old + 1 == ex->need[w]) {
      ex->cnt[w & 7] = 0;  // free for wave w + 8 (at most three waves are ever open)
      __threadfence();
      st_relaxed_u32(flags + (size_t)w * S, epoch);
    }
  }
};

// Stages (kUnit per unit, padding stages included) of stats CTA `first` in
// wave w: units g in [w upw, min((w+1) upw, units)) with g = first mod S.
__device__ __forceinline__ unsigned wave_need(long long upw, long long units, int first, int S,
                                              int w) {
  auto below = [&](long long x) -> long long {  // units g < x of this CTA
    return x > first ? (x - first + S - 1) / S : 0;
  };
  const long long lo = (long long)w * upw;
  const long long hi = min(units, lo + upw);
  return (unsigned)(stage::kUnit * (below(hi) - below(lo)));
}

template <int DT>
__device__ __forceinline__ void stats_cta(const FusedParams &fp, uint8_t *smem, unsigned epoch) {
  stage::StatsSmem &ss = *reinterpret_cast<stage::StatsSmem *>(smem);
  StatsExtra &ex = *reinterpret_cast<StatsExtra *>(smem + kStatsBytes);
  const int first = blockIdx.x, S = fp.S;
  const RowStatsParams &st = fp.st;
  const int upr = (st.spr + stage::kUnit - 1) / stage::kUnit;
  const long long units = st.stages / st.spr * upr;
  const long long upw = (long long)fp.rpw * upr;
  const int tid = threadIdx.x;
  if (tid < 8) ex.cnt[tid] = 0;
  for (int w = tid; w < fp.n_waves; w += kT) ex.need[w] = wave_need(upw, units, first, S, w);
  // (stats_role starts with a barrier after its own set-up: these are visible)
  unsigned int *flags = st.ws.sync->flags + first;
  WaveHook hook{flags, &ex, S, fp.rpw, epoch};
  stage::stats_role<DT, false>(st, ss, (long long)first, (long long)S, hook);
  __syncthreads();
  // waves without a stage of this CTA (only the last, short wave can have none)
  if (tid == 0) {
    __threadfence();
    for (int w = 0; w < fp.n_waves; ++w)
      if (ex.need[w] == 0) st_relaxed_u32(flags + (size_t)w * S, epoch);
  }
}

// ---------------------------------------------------------------------------
// draw CTAs
// ---------------------------------------------------------------------------

// Bounded wait until request `it` of this CTA is armed: true when it is,
// false when the CTA has no such request (or a wait of the CTA gave up).
// One thread; a warp uses warp_wait_armed.
__device__ __forceinline__ bool wait_armed(DrawSmem &sm, int it) {
  unsigned long long t0 = 0;
  for (;;) {
    if (sm.armed > it) {
      __threadfence_block();
      return true;
    }
    if (sm.last <= it || sm.abort_flag) return false;
    const unsigned long long t = global_timer_ns();
    if (t0 == 0) {
      t0 = t;
    } else if (t - t0 > kWaitLimitNs) {
      sm.abort_flag = 1;
      return false;
    }
    __nanosleep(64);
  }
}

// wait_armed by lane 0, its outcome broadcast: one outcome per warp.
__device__ __forceinline__ bool warp_wait_armed(DrawSmem &sm, int it, int lane) {
  int r = 0;
  if (lane == 0) r = wait_armed(sm, it);
  r = __shfl_sync(0xffffffffu, r, 0);
  __threadfence_block();
  return r != 0;
}

// Bounded wait by lane 0 until *word >= want (a counter of this CTA), the
// outcome broadcast to the warp; false when a wait of the CTA gave up.
__device__ __forceinline__ bool warp_wait_count(DrawSmem &sm, volatile const unsigned *word,
                                                unsigned want, int lane) {
  int r = 1;
  if (lane == 0) {
    unsigned long long t0 = 0;
    while (*word < want) {
      if (sm.abort_flag) {
        r = 0;
        break;
      }
      const unsigned long long t = global_timer_ns();
      if (t0 == 0) {
        t0 = t;
      } else if (t - t0 > kWaitLimitNs) {
        sm.abort_flag = 1;
        r = 0;
        break;
      }
      __nanosleep(32);
    }
  }
  r = __shfl_sync(0xffffffffu, r, 0);
  __threadfence_block();
  return r != 0;
}

// Bounded wait until every stats CTA flagged wave w with this launch's epoch.
// The whole warp calls it; every decision to stop is a warp vote.
__device__ __forceinline__ bool wait_wave(const unsigned *flags, int S, unsigned epoch, int lane,
                                          DrawSmem &sm) {
  unsigned long long t0 = 0;
  unsigned seen = 0;  // bit i: flag lane + 32 i already carries the epoch
  for (;;) {
    bool all = true;
#pragma unroll
    for (int i = 0; i < SPECDEC_FUSED_MAX_STATS_CTAS / 32; ++i) {
      const int c = lane + 32 * i;
      if (c < S && !(seen >> i & 1u)) {
        if (ld_relaxed_u32(flags + c) == epoch) seen |= 1u << i;
        else all = false;
      }
    }
    if (__all_sync(0xffffffffu, all)) {
      __threadfence();  // acquire: the partials and gathers of the wave are visible
      return true;
    }
    bool stop = sm.abort_flag;
    const unsigned long long t = global_timer_ns();
    if (t0 == 0) {
      t0 = t;
    } else if (t - t0 > kWaitLimitNs) {
      stop = true;
    }
    if (__any_sync(0xffffffffu, stop)) return false;
  }
}

// Outputs of a request whose wait gave up: status SPECDEC_ROW_INTERNAL, nothing drawn.
__device__ __forceinline__ void write_internal(const LinearFinalizeParams &p, long long b,
                                               int lane) {
  const int R = p.gamma + 1;
  for (int i = lane; i < R; i += 32) p.out_tokens[b * R + i] = -1;
  if (p.p_draft)
    for (int i = lane; i < p.gamma; i += 32) p.p_draft[b * p.gamma + i] = __int_as_float(0x7fc00000);
  if (lane == 0) {
    p.row_status[b] = SPECDEC_ROW_INTERNAL;
    p.n_accepted[b] = 0;
    p.is_bonus[b] = 0;
    p.final_token[b] = -1;
  }
}

// The merged statistics of rows [0, R) of request b into rs[], by one warp:
// 16-lane segments merge two rows at a time in the order of segment_merge_row
// (so M, S and the arg-max are those of the draw kernels bit for bit); the
// first two partials of up to eight rows are loaded before any arithmetic.
__device__ __forceinline__ void merge_rows(const LinearFinalizeParams &p, long long b, float c,
                                           RowStat *rs, int lane) {
  const int R = p.gamma + 1, spr = p.spr, sl = lane % kSeg, half = lane / kSeg;
  for (int r0 = 0; r0 < R; r0 += 8) {
    float4 x0[4], x1[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = r0 + 2 * i + half;
      const bool active = r < R;
      const float4 *pr = reinterpret_cast<const float4 *>(p.part + (b * R + (active ? r : 0)) *
                                                                       (long long)spr);
      x0[i] = load_partial(pr, sl, spr, active);
      x1[i] = load_partial(pr, sl + kSeg, spr, active);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = r0 + 2 * i + half;
      if (r0 + 2 * i >= R) break;  // both segments idle (warp-uniform)
      const bool active = r < R;
      const float4 *pr = reinterpret_cast<const float4 *>(p.part + (b * R + (active ? r : 0)) *
                                                                       (long long)spr);
      float m = -INFINITY, s = 0.0f;
      int a = 0x7FFFFFFF;
      int fl = __float_as_int(x0[i].w) | __float_as_int(x1[i].w);
      merge2(m, s, a, x0[i].x, x0[i].y, __float_as_int(x0[i].z), c);
      merge2(m, s, a, x1[i].x, x1[i].y, __float_as_int(x1[i].z), c);
      if (active) {
        for (int j = sl + 2 * kSeg; j < spr; j += kSeg) {  // rows of more than 32 stages
          const float4 x = __ldcg(pr + j);
          fl |= __float_as_int(x.w);
          merge2(m, s, a, x.x, x.y, __float_as_int(x.z), c);
        }
      }
#pragma unroll
      for (int d = kSeg / 2; d >= 1; d >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, d);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, d);
        const int a2 = __shfl_xor_sync(0xffffffffu, a, d);
        fl |= __shfl_xor_sync(0xffffffffu, fl, d);
        merge2(m, s, a, m2, s2, a2, c);
      }
      if (active && sl == 0) {
        RowStat st;
        st.M = m;
        st.S = s;
        st.arg = a;
        st.flags = fl;
        rs[r] = st;
      }
    }
  }
  __syncwarp();
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

template <int DT>
__device__ __forceinline__ void draw_cta(const FusedParams &fp, uint8_t *smem, unsigned epoch) {
  DrawSmem &sm = *reinterpret_cast<DrawSmem *>(smem);
  const LinearFinalizeParams &p = fp.p;
  constexpr int es = (DT == SPECDEC_F32) ? 4 : 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int D = gridDim.x - fp.S, d0 = blockIdx.x - fp.S;
  const int gamma = p.gamma;
  const int rowbytes = p.V * es;
  const int nst = (rowbytes + kStage - 1) / kStage;
  const int upr = (nst + kUnitStages - 1) / kUnitStages;

  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], kUnitStages);  // one arrival per stage (the last real one
                                             // of a short unit arrives for the rest)
    }
    sm.armed = 0;
    sm.last = 0x7FFFFFFF;
    sm.freed = 0;
    sm.abort_flag = 0;
    sm.issued = -1;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kDecider) {
    // ------------------------------ decider -------------------------------
    int it = 0;
    for (long long b = d0; b < p.B; b += D) {
      const float T = __ldg(p.temperature + b);
      DraftIn din = load_draft_inputs(p, b, lane);  // the call's own inputs: before the wait
      const int w = (int)(b / fp.Wr);
      if (__any_sync(0xffffffffu, sm.abort_flag) ||
          !wait_wave(p.ws.sync->flags + (size_t)w * fp.S, fp.S, epoch, lane, sm)) {
        sm.abort_flag = 1;
        write_internal(p, b, lane);
        continue;
      }
      load_draft_gather(p, b, lane, din);
      const float c = temperature_scale(T);
      merge_rows(p, b, c, sm.rs, lane);
      float pd;
      const LinearDecision d = decide(p, din, T, c, sm.rs, lane, pd);
      write_outputs_warp(p, b, d, pd, lane);
      if (d.status || d.greedy) continue;  // nothing to draw
      // the request's slot is free once the searcher finished request it - kQ
      if (it >= kQ &&
          !warp_wait_count(sm, (volatile const unsigned *)&sm.freed, (unsigned)(it - kQ + 1), lane)) {
        write_internal(p, b, lane);
        continue;
      }
      if (lane == 0) {
        ReqSlot &rq = sm.rq[it % kQ];
        rq.dec = d;
        rq.b = b;
        rq.nsum = 0;
        __threadfence_block();
        sm.armed = it + 1;
      }
      __syncwarp();
      ++it;
    }
    if (lane == 0) {
      __threadfence_block();
      sm.last = it;
    }
  } else if (warp == kProducer) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      long long n = 0;
      uint32_t slot = 0, use = 0;
      for (int it = 0; wait_armed(sm, it); ++it) {
        const ReqSlot &rq = sm.rq[it % kQ];
        const LinearDecision d = rq.dec;
        const Req r = req_of<DT>(p, rq.b, d.k);
        const bool use_q = d.k < gamma;
        bool stop = false;
        for (int ju = 0; ju < upr; ++ju) {
          if (use > 0 && !mbar_wait_bounded(&sm.empty[slot], (use - 1) & 1)) {
            sm.abort_flag = 1;
            stop = true;
            break;
          }
          if (sm.abort_flag) {
            stop = true;
            break;
          }
          const int bytes = min(kUnitBytes, rowbytes - ju * kUnitBytes);
          mbar_arrive_expect_tx(&sm.full[slot], (uint32_t)(bytes * (use_q ? 2 : 1)));
          bulk_copy_g2s(sm.l[slot], r.lrow + (size_t)ju * kUnitBytes, (uint32_t)bytes,
                        &sm.full[slot]);
          if (use_q)
            bulk_copy_g2s(sm.q[slot], r.qrow + (size_t)ju * kUnitBytes, (uint32_t)bytes,
                          &sm.full[slot]);
          ++n;
          if (++slot == kSlots) {
            slot = 0;
            ++use;
          }
        }
        if (stop) break;
      }
      sm.issued = n;
    }
  } else if (warp == kSearcher) {
    // ------------------------------ searcher ------------------------------
    for (int it = 0; warp_wait_armed(sm, it, lane); ++it) {
      ReqSlot &rq = sm.rq[it % kQ];
      if (!warp_wait_count(sm, (volatile const unsigned *)&rq.nsum, (unsigned)nst, lane)) break;
      const LinearDecision d = rq.dec;
      const Req r = req_of<DT>(p, rq.b, d.k);
      search_warp<DT>(p, r, d, false, lane,
                      SharedTotals{rq.tot, p.ws.chunk_tot + rq.b * p.ntot});
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        sm.freed = it + 1;
      }
      __syncwarp();
    }
  } else {
    // ------------------------------ consumers -----------------------------
    // real stage c of the CTA's drawn requests (request c / nst, stage
    // c % nst of its final row) belongs to consumer warp c % kConsumers
    const int cw = warp - kFirstConsumer;
    for (long long c = cw;; c += kConsumers) {
      const int it = (int)(c / nst);
      const int s = (int)(c - (long long)it * nst);
      if (!warp_wait_armed(sm, it, lane)) break;
      ReqSlot &rq = sm.rq[it % kQ];
      const LinearDecision d = rq.dec;
      const long long b = rq.b;
      const bool use_q = d.k < gamma;
      const int ju = s / kUnitStages, t = s - ju * kUnitStages;
      const long long n = (long long)it * upr + ju;
      const uint32_t slot = (uint32_t)(n % kSlots), use = (uint32_t)(n / kSlots);
      // the slot's previous use released first (a parity wait tells only two
      // phases apart, and copies land in any order), then this use's copy
      const bool ok = __all_sync(0xffffffffu,  // one outcome for the whole warp
                                 !sm.abort_flag &&
                                     (use == 0 || mbar_wait_bounded(&sm.empty[slot], (use - 1) & 1)) &&
                                     mbar_wait_bounded(&sm.full[slot], use & 1));
      if (!ok) sm.abort_flag = 1;
      uint4 lv[kVec], qv[kVec];
      const int sbytes = ok ? min(kStage, rowbytes - s * kStage) : 0;
      load_stage<DT>(lv, qv, sm.l[slot] + t * kStage, sm.q[slot] + t * kStage, sbytes, use_q,
                     lane, false);
      __syncwarp();
      if (lane == 0) {
        // the last real stage of a short unit also arrives for the stages it lacks
        const int in_unit = min(kUnitStages, nst - ju * kUnitStages);
        mbar_arrive_cnt(&sm.empty[slot], (t == in_unit - 1) ? (uint32_t)(kUnitStages - t) : 1u);
      }
      if (!ok) break;
      unsigned long long acc = 0;
#pragma unroll
      for (int k = 0; k < kVec; ++k) acc += to_fixed40(vec_sum<DT>(lv[k], qv[k], d, use_q));
      acc = warp_sum_u64(acc);
      if (lane == 0) {
        rq.tot[s] = acc;
        p.ws.chunk_tot[b * p.ntot + s] = acc;
        __threadfence_block();
        atomicAdd(&rq.nsum, 1u);
      }
    }
  }
  __syncthreads();
  if (sm.abort_flag) {
    // requests handed over but not searched: report them; and keep the CTA
    // until every copy the producer issued has landed
    if (warp == 0) {
      for (int it = sm.freed; it < sm.armed; ++it) write_internal(p, sm.rq[it % kQ].b, lane);
    }
    if (tid == 32) {
      const unsigned long long t0 = global_timer_ns();
      while (sm.issued < 0 && global_timer_ns() - t0 < kWaitLimitNs) {
      }
      if (sm.issued >= 0) drain_ring(sm.full, kSlots, sm.issued);
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(kT, 1) verify_fused_kernel(const FusedParams fp) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __shared__ unsigned s_epoch;
  FusedSync *sync = fp.p.ws.sync;
  if (threadIdx.x == 0) s_epoch = ld_relaxed_u32(&sync->epoch) + 1u;
  __syncthreads();
  const unsigned epoch = s_epoch;
  if ((int)blockIdx.x < fp.S) {
    stats_cta<DT>(fp, smem_raw, epoch);
  } else {
    draw_cta<DT>(fp, smem_raw, epoch);
  }
  __syncthreads();
  // the last CTA to exit publishes the epoch for the next launch (every CTA
  // read the old one before counting itself here)
  if (threadIdx.x == 0) {
    unsigned long long old = *(volatile unsigned long long *)&sync->exits;
    for (;;) {
      const unsigned long long cnt = ((unsigned)(old >> 32) == epoch) ? (old & 0xffffffffull) : 0;
      const unsigned long long want = ((unsigned long long)epoch << 32) | (cnt + 1);
      const unsigned long long seen = atomicCAS(&sync->exits, old, want);
      if (seen == old) {
        if (cnt + 1 == gridDim.x) st_relaxed_u32(&sync->epoch, epoch);
        break;
      }
      old = seen;
    }
  }
}

struct Plan {
  int S, D, Wr, n_waves;
};

// The split of the grid and the waves for these sizes (false: not this path).
bool make_plan(const LinearFinalizeParams &p, int sms, Plan &pl) {
  const int es = (p.dtype == SPECDEC_F32) ? 4 : 2;
  const long long rowbytes = (long long)p.V * es;
  if (rowbytes % 16 != 0) return false;
  if ((reinterpret_cast<uintptr_t>(p.logits) & 15) || (reinterpret_cast<uintptr_t>(p.q) & 15))
    return false;
  const long long nst = (rowbytes + kStage - 1) / kStage;
  if (nst < kMinStages || nst > kMaxStages) return false;
  const int R = p.gamma + 1;
  const long long upr = (p.spr + stage::kUnit - 1) / stage::kUnit;
  if ((long long)p.B * R * upr >= (1ll << 31)) return false;
  // draw CTAs: the draws' share of the bytes (a final logits row and a q row
  // per request, against the R rows of the stats pass)
  int D = (int)(2.0 * sms / (R + 2.0) + 0.5);
  static const int env_d = [] {
    const char *e = getenv("SPECDEC_FUSED_DRAW_CTAS");
    return e ? atoi(e) : 0;
  }();
  if (env_d > 0) D = env_d;
  D = max(4, min(D, sms / 2));
  const int S = sms - D;
  if (S < 1 || S > SPECDEC_FUSED_MAX_STATS_CTAS) return false;
  if (p.B < 2 * D) return false;  // small batches: the other paths
  // waves: each stats CTA holds at least 16 units of every wave but the last
  // (so at most two waves are open in a CTA at once), at most the flag table
  const long long units_per_req = R * upr;
  long long Wr = (16ll * S + units_per_req - 1) / units_per_req;
  Wr = max(Wr, (long long)((p.B + SPECDEC_FUSED_MAX_WAVES - 1) / SPECDEC_FUSED_MAX_WAVES));
  Wr = max(1ll, min(Wr, (long long)p.B));
  pl.S = S;
  pl.D = D;
  pl.Wr = (int)Wr;
  pl.n_waves = (int)((p.B + Wr - 1) / Wr);
  return pl.n_waves <= SPECDEC_FUSED_MAX_WAVES;
}

template <int DT>
cudaError_t launch_dt(const FusedParams &fp, int grid, cudaStream_t stream) {
  static DeviceOnce once;
  const cudaError_t err = smem_opt_in_once(once, verify_fused_kernel<DT>, (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kT);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: the waits end
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_fused_kernel<DT>, fp);
}

}  // namespace

bool fused_verify_applies(const LinearFinalizeParams &p) {
  Plan pl;
  return make_plan(p, device_sm_count(), pl);
}

cudaError_t launch_fused_verify(const RowStatsParams &st, const LinearFinalizeParams &p,
                                cudaStream_t stream) {
  const int sms = device_sm_count();
  Plan pl;
  if (!make_plan(p, sms, pl)) return cudaErrorInvalidValue;
  FusedParams fp;
  fp.st = st;
  fp.p = p;
  fp.S = pl.S;
  fp.Wr = pl.Wr;
  fp.n_waves = pl.n_waves;
  fp.rpw = pl.Wr * (p.gamma + 1);
  return (p.dtype == SPECDEC_F32) ? launch_dt<SPECDEC_F32>(fp, sms, stream)
                                  : launch_dt<SPECDEC_BF16>(fp, sms, stream);
}

}  // namespace specdec
