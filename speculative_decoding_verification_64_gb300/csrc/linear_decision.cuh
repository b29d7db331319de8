// The accept decision of one linear-verify request, shared by the draw
// kernels ("Chapter 15: Decoding acceleration", section 15.1.2 step 3):
// merge the stats pass's stage partials of the request's rows, test the
// drafts in order and stop at the first rejection.
#pragma once

#include "draw_common.cuh"

namespace specdec {
namespace lindec {

using namespace drawc;

// shared-memory record of a decision
struct DecisionSmem {
  RowStat rs[SPECDEC_MAX_GAMMA + 1];
  LinearDecision dec;
};

// Where a decision reads the stats pass's results (stage partials, gathered
// logit and q of the drafted tokens): the workspace.
struct WorkspaceSrc {
  const LinearFinalizeParams &p;
  __device__ __forceinline__ float4 partial(long long row, int j) const {
    return __ldcg(reinterpret_cast<const float4 *>(p.part + row * (long long)p.spr) + j);
  }
  __device__ __forceinline__ float2 gather(long long b, int i) const {
    return __ldcg(p.ws.gather + b * (p.gamma + 1) + i);
  }
};

// The accept test of request b by a whole CTA of kT threads (rows merged by
// 16-lane segments, the test in warp 0); the owner of chunk 0 also writes
// every output but a drawn token.  Two barriers; the result is CTA-uniform.
// S holds RowStat rs[SPECDEC_MAX_GAMMA + 1] and LinearDecision dec; src gives
// the stats pass's results (WorkspaceSrc, or a copy of them).
template <int DT, int kT, typename S, typename Src>
__device__ __forceinline__ LinearDecision request_decision_from(const LinearFinalizeParams &p,
                                                                long long b, bool owns_chunk0,
                                                                S &sm, const Src &src) {
  constexpr int kRowsPerRound = kT / kSeg;
  const int tid = threadIdx.x;
  const int gamma = p.gamma, R = gamma + 1;
  const float T = __ldg(p.temperature + b);
  DraftIn din = load_draft_inputs(p, b, tid);
  if (tid < gamma) din.g = src.gather(b, tid);  // (read for valid tokens only)
  const float c = temperature_scale(T);
  for (int r0 = 0; r0 < R; r0 += kRowsPerRound) {
    const int r = r0 + tid / kSeg;
    if (r0 + (tid / 32) * (32 / kSeg) >= R) continue;  // both segments of this warp idle
    const long long row = b * R + r;
    const RowStat st =
        segment_merge([&](int j) { return src.partial(row, j); }, r < R, p.spr, c, tid % kSeg);
    if (r < R && tid % kSeg == 0) sm.rs[r] = st;
  }
  __syncthreads();
  if (tid < 32) {
    float pd;
    const LinearDecision dd = decide(p, din, T, c, sm.rs, tid, pd);
    if (tid == 0) sm.dec = dd;
    if (owns_chunk0 && p.p_draft && tid < gamma) p.p_draft[b * gamma + tid] = pd;
  }
  __syncthreads();
  const LinearDecision d = sm.dec;
  if (owns_chunk0) {
    const int k = d.k;
    if (tid < R) {
      int t = -1;
      if (!d.status) {
        if (tid < k) t = __ldg(p.tokens + b * gamma + tid);
        else if (tid == k) t = d.arg;  // greedy; a drawn token is written by the search
      }
      if (d.status || tid != k || d.greedy) p.out_tokens[b * R + tid] = t;
    }
    if (tid == 0) {
      p.n_accepted[b] = d.status ? 0 : k;
      p.is_bonus[b] = (uint8_t)(!d.status && k == gamma);
      p.row_status[b] = d.status;
      if (d.status) p.final_token[b] = -1;
      else if (d.greedy) p.final_token[b] = d.arg;
      if (d.status || d.greedy) p.ws.mass[b] = kNoMass;  // nothing drawn
    }
  }
  return d;
}

template <int DT, int kT, typename S>
__device__ __forceinline__ LinearDecision request_decision(const LinearFinalizeParams &p,
                                                           long long b, bool owns_chunk0, S &sm) {
  return request_decision_from<DT, kT>(p, b, owns_chunk0, sm, WorkspaceSrc{p});
}

}  // namespace lindec
}  // namespace specdec
