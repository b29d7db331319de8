// The stats pass's loop as a device function of one CTA: the producer thread
// streaming 16 KB units into the shared-memory ring and the consumer warps
// reducing 8 KB stages into row partials ("Chapter 15: Decoding
// acceleration", section 15.1.2 step 2).  The stats kernel (row_stats.cu)
// runs it on every CTA of its grid.
#pragma once

#include "stats_stage.cuh"

namespace specdec {
namespace stage {

struct StatsSmem {
  alignas(128) uint8_t stage[kSlots][kUnitBytes];
  alignas(8) uint64_t full[kSlots];
  alignas(8) uint64_t empty[kSlots];
  volatile long long issued;  // units the producer issued, once it is done (else -1)
  volatile int abort_flag;
};

// The stats pass of one CTA over units first, first + stride, ... of the
// row-major unit sequence (see row_stats.cu for the structure).  Every thread
// of the CTA (kThreads) calls it; it returns once the CTA's stages are
// reduced and, after a wait that gave up, its copies have landed.
// kA: also the entropy sums of non-greedy rows (SPECDEC_STATS_ENTROPY).
template <int DT, bool kA>
__device__ __forceinline__ void stats_role(const RowStatsParams &p, StatsSmem &sm,
                                           long long first, long long stride) {
  constexpr int es = (DT == SPECDEC_F32) ? 4 : 2;
  constexpr int kPerVec = 16 / es;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int upr = (p.spr + kUnit - 1) / kUnit;  // units per row
  const long long units = p.stages / p.spr * upr;
  const long long n_local = (units > first) ? (units - first + stride - 1) / stride : 0;

  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], kUnit);  // one arrival per stage of the unit
    }
    sm.abort_flag = 0;
    sm.issued = -1;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      UnitCursor cur;
      cur.init(first, stride, upr);
      uint32_t slot = 0, use = 0;
      long long i = 0;
      for (; i < n_local; ++i) {
        if (use > 0 && !mbar_wait_bounded(&sm.empty[slot], (use - 1) & 1)) {
          sm.abort_flag = 1;
          break;
        }
        if (sm.abort_flag) break;
        const UnitGeom g = unit_geometry(p.logits, p.V, p.spr, cur.row, cur.ju, es);
        cur.advance(upr);
        if (g.bytes > 0) {
          mbar_arrive_expect_tx(&sm.full[slot], (uint32_t)g.bytes);
          bulk_copy_g2s(sm.stage[slot], g.src, (uint32_t)g.bytes, &sm.full[slot]);
        } else {
          mbar_arrive(&sm.full[slot]);
        }
        if (++slot == kSlots) {
          slot = 0;
          ++use;
        }
      }
      sm.issued = i;
      if (sm.abort_flag) drain_ring(sm.full, kSlots, i);  // units 0 .. i-1 were issued
    } else if (p.tokens != nullptr) {
      // idle lanes: zero the draw kernel's per-request tickets, which that
      // kernel (launched after this one) counts up from zero
      for (long long b = first * 31 + (lane - 1); b < p.B; b += stride * 31)
        p.ws.draw_cnt[b] = 0u;
    }
    return;
  }

  // ------------------------------ consumers -------------------------------
  // Local stage c = i * kUnit + t (stage t of local unit i) belongs to warp
  // c % W.  Every warp assigned to a unit waits for the unit's copy, takes its
  // stage into registers and arrives once on the unit's "empty" barrier (also
  // for stages past the end of a row, which hold no data), so the barrier
  // completes exactly when all kUnit stages of the unit have been read.  The
  // temperature of the warp's next stage is loaded one iteration ahead.
  const long long n_stages_local = n_local * kUnit;
  const int gamma = p.R - 1;
  auto unit_row = [&](long long c) -> int {
    const long long g = first + (c / kUnit) * stride;
    return (int)(g / upr);
  };
  // temperature and drafted token of a row, loaded one iteration ahead
  auto row_token = [&](int row) -> int {
    if (p.tokens == nullptr) return -1;
    const int b = row / p.R, i = row - b * p.R;
    return (i < gamma) ? __ldg(p.tokens + (long long)b * gamma + i) : -1;
  };
  int row_next = (warp < n_stages_local) ? unit_row(warp) : 0;
  float T_next = (warp < n_stages_local) ? __ldg(p.temperature + row_next / p.R) : 0.0f;
  int x_next = (warp < n_stages_local) ? row_token(row_next) : -1;
  for (long long c = warp; c < n_stages_local; c += kConsumerWarps) {
    const long long i = c / kUnit;
    const int t = (int)(c - i * kUnit);
    const long long g = first + i * stride;
    const int row = (int)(g / upr);
    const UnitGeom u = unit_geometry(p.logits, p.V, p.spr, row, (int)(g - (long long)row * upr), es);
    const uint32_t slot = (uint32_t)(i % kSlots);
    const uint32_t use = (uint32_t)(i / kSlots);
    const float T = T_next;
    const int x = x_next;
    if (c + kConsumerWarps < n_stages_local) {
      row_next = unit_row(c + kConsumerWarps);
      T_next = __ldg(p.temperature + row_next / p.R);
      x_next = row_token(row_next);
    }
    const bool real = t < u.nst;

    LaneData<DT> d;
    d.edge = -INFINITY;
    d.edge_idx = 0x7FFFFFFF;
    if (real && u.j0 + t == 0) {
      const int n_head = u.head_end, n_tail = p.V - u.tail_begin;
      int e = -1;
      if (lane < n_head) e = lane;
      else if (lane < n_head + n_tail) e = u.tail_begin + (lane - n_head);
      if (e >= 0) {
        d.edge = load_elem(p.logits, DT, (long long)row * p.V + e);
        d.edge_idx = e;
      }
    }

    // A parity wait tells only two phases apart.  This warp did not consume
    // the slot's previous use (another warp's stages were there), and copies
    // land in any order, so that use may still be in flight: the full
    // barrier would then read as complete.  Wait first until the previous use
    // has been released (which implies it landed); then the full barrier is
    // at most one phase from the one awaited.
    // (one vote: the lanes of a warp could see a wait give up differently, and
    // everything after it is warp-synchronous)
    const bool ok = __all_sync(0xffffffffu,
                               !sm.abort_flag &&
                                   (use == 0 || mbar_wait_bounded(&sm.empty[slot], (use - 1) & 1,
                                                                  kConsumerWaitNs)) &&
                                   mbar_wait_bounded(&sm.full[slot], use & 1, kConsumerWaitNs));
    if (!ok) sm.abort_flag = 1;
    const int sbytes = max(0, min(kStageBytes, u.bytes - t * kStageBytes));
    if (ok && real) load_lane<DT>(d, sm.stage[slot] + t * kStageBytes, sbytes / 16, lane);
    if (ok && real && lane == 0 && x >= 0 && x < p.V) {
      // gather the drafted token's logit (from this stage, or from global for
      // an edge element) and its q value
      const int se0 = u.elem0 + t * (kStageBytes / es);
      const int sel = sbytes / es;
      const bool in_stage = x >= se0 && x < se0 + sel;
      const bool in_edge = (u.j0 + t == 0) && (x < u.head_end || x >= u.tail_begin);
      if (in_stage || in_edge) {
        const long long roff = (long long)row * p.V;
        float lx;
        if (in_stage) {
          const uint8_t *src = sm.stage[slot] + t * kStageBytes + (size_t)(x - se0) * es;
          lx = (DT == SPECDEC_F32) ? *reinterpret_cast<const float *>(src)
                                   : __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t *>(src)) << 16);
        } else {
          lx = load_elem(p.logits, DT, roff + x);
        }
        const int b = row / p.R, ri = row - b * p.R;
        const float qx = load_elem(p.q, DT, ((long long)b * gamma + ri) * p.V + x);
        p.ws.gather[row] = make_float2(lx, qx);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[slot]);  // this stage is in registers now
    if (!real) continue;

    RowPartial r;
    r.flags = ok ? 0 : SPECDEC_ROW_INTERNAL;
    r.arg = 0x7FFFFFFF;
    r.m = -INFINITY;
    r.s = 0.0f;
    if (ok) {
      const float wm = warp_max_nan(lane_max<DT>(d));
      r.m = wm;
      if (T == 0.0f) {
        // greedy row: only the maximum and its first index are needed
        const int first_idx =
            (wm == wm && wm != -INFINITY)
                ? lane_first<DT>(d, wm, u.elem0 + t * (kStageBytes / es), lane)
                : 0x7FFFFFFF;
        r.arg = warp_min(first_idx);
        r.s = (wm == -INFINITY) ? 0.0f : 1.0f;
      } else if (wm != -INFINITY) {
        if (kA) {
          float a;
          r.s = warp_sum(lane_sum_a<DT>(d, temperature_scale(T), wm, a));
          r.arg = __float_as_int(warp_sum(a));  // sum of e (l - m); arg is for greedy rows only
        } else {
          r.s = warp_sum(lane_sum<DT>(d, temperature_scale(T), wm));
        }
      }
    }
    if (lane == 0) p.part[(long long)row * p.spr + u.j0 + t] = r;
  }
  // After any wait of the CTA gave up, the consumers stop waiting for copies:
  // keep the CTA until every copy the producer issued has landed.
  if (sm.abort_flag && lane == 0) {
    const unsigned long long t0 = global_timer_ns();
    while (sm.issued < 0 && global_timer_ns() - t0 < kWaitLimitNs) {
    }
    if (sm.issued >= 0) drain_ring(sm.full, kSlots, sm.issued);
  }
  (void)kPerVec;
}

}  // namespace stage
}  // namespace specdec
