// Pieces of the linear draw shared by its kernels ("Chapter 15: Decoding
// acceleration", section 15.1.2 steps 3 and 4):
//   * merging a row's stage partials with a 16-lane segment of a warp;
//   * the accept test of one request by one warp, lane i testing draft i with
//     the logit and q value gathered by the stats pass, the first rejection
//     found by a ballot;
//   * draw weights of one 16-byte vector -- 2^((l - M) c), or max(0, that -
//     S q) after a rejection -- summed in float32 in index order, and the
//     search of one request by one warp over 4 KB stages of its final row:
//     stage totals, then vector sums in index order as 40-bit fixed point,
//     then the element.
#pragma once

#include <cfloat>

#include "common.cuh"

namespace specdec {
namespace drawc {

constexpr int kStage = SPECDEC_DRAW_STAGE_BYTES;    // bytes of the final row per draw stage
constexpr int kVec = kStage / 16 / 32;              // 16-byte vectors per lane per draw stage

constexpr int kSeg = 16;                     // lanes merging one row


// Merge of one row's partials by a 16-lane segment of a warp (both segments of
// the warp take part in every shuffle; an idle segment merges nothing).
// part(j) gives partial j < spr of the row.  The first three partials of each
// lane are loaded before any arithmetic, so that rows of up to 48 stages
// (bf16 rows up to 196608 elements) cost one memory round trip.
template <typename Part>
__device__ __forceinline__ RowStat segment_merge(const Part &part, bool active, int spr, float c,
                                                 int sl) {
  const float4 none = make_float4(-INFINITY, 0.0f, __int_as_float(0x7FFFFFFF), 0.0f);
  const float4 x0 = (active && sl < spr) ? part(sl) : none;
  const float4 x1 = (active && sl + kSeg < spr) ? part(sl + kSeg) : none;
  const float4 x2 = (active && sl + 2 * kSeg < spr) ? part(sl + 2 * kSeg) : none;
  float m = -INFINITY, s = 0.0f;
  int a = 0x7FFFFFFF;
  int fl = __float_as_int(x0.w) | __float_as_int(x1.w) | __float_as_int(x2.w);
  merge2(m, s, a, x0.x, x0.y, __float_as_int(x0.z), c);
  merge2(m, s, a, x1.x, x1.y, __float_as_int(x1.z), c);
  merge2(m, s, a, x2.x, x2.y, __float_as_int(x2.z), c);
  if (active) {
    for (int j = sl + 3 * kSeg; j < spr; j += kSeg) {  // rows of more than 48 stages
      const float4 x = part(j);
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
  RowStat r;
  r.M = m;
  r.S = s;
  r.arg = a;
  r.flags = fl;
  return r;
}

// The same from the workspace (L2 loads: the partials may have been written
// by other CTAs of the running kernel).
__device__ __forceinline__ RowStat segment_merge_row(const RowPartial *part, long long row,
                                                     bool active, int spr, float c, int sl) {
  const float4 *pr = reinterpret_cast<const float4 *>(part + row * (long long)spr);
  return segment_merge([&](int j) { return __ldcg(pr + j); }, active, spr, c, sl);
}

// Inputs of one lane's accept test: draft x~_i, its uniform, and the logit
// and q value the stats pass gathered for it.
struct DraftIn {
  int x;
  float u;
  float2 g;
};

// The call's own inputs (draft token, uniform): a kernel launched dependent on
// the stats pass may read them before waiting for it.
__device__ __forceinline__ DraftIn load_draft_inputs(const LinearFinalizeParams &p, long long b,
                                                     int lane) {
  DraftIn in;
  in.x = -1;
  in.u = 0.0f;
  in.g = make_float2(0.0f, 1.0f);
  if (lane < p.gamma) {
    in.x = __ldg(p.tokens + b * p.gamma + lane);
    in.u = __ldg(p.uniforms + b * (p.gamma + 1) + lane);
  }
  return in;
}

// The (logit, q) pair the stats pass gathered: only after waiting for it.
__device__ __forceinline__ void load_draft_gather(const LinearFinalizeParams &p, long long b,
                                                  int lane, DraftIn &in) {
  if (lane < p.gamma) in.g = __ldcg(p.ws.gather + b * (p.gamma + 1) + lane);  // valid x only
}


// The accept test of request b by warp 0 from the merged rows rs[0, R):
// lane i < gamma tests draft i, a ballot gives the first rejection.  Lane
// i's p_i(x~_i) is returned in pd (NaN for a malformed request).
__device__ __forceinline__ LinearDecision decide(const LinearFinalizeParams &p, const DraftIn &in,
                                                 float T, float c, const RowStat *rs, int lane,
                                                 float &pd) {
  const int gamma = p.gamma, R = gamma + 1, V = p.V;
  const bool greedy = (T == 0.0f);
  RowStat r0, r1;
  r0.M = r1.M = -INFINITY;
  r0.S = r1.S = 0.0f;
  r0.arg = r1.arg = 0x7FFFFFFF;
  r0.flags = r1.flags = 0;
  if (lane < R) r0 = rs[lane];
  if (lane + 32 < R) r1 = rs[lane + 32];
  int status = temperature_valid(T) ? 0 : SPECDEC_ROW_BAD_TEMP;
  if (lane < R) status |= r0.flags | (row_usable(r0) ? 0 : SPECDEC_ROW_NONFINITE);
  if (lane + 32 < R) status |= r1.flags | (row_usable(r1) ? 0 : SPECDEC_ROW_NONFINITE);
  bool acc = true;
  pd = 0.0f;
  if (lane < gamma) {
    if (in.x < 0 || in.x >= V) {
      status |= SPECDEC_ROW_BAD_TOKEN;
    } else {
      if (!(in.g.y > 0.0f) || in.g.y == INFINITY) status |= SPECDEC_ROW_BAD_Q;
      if (greedy) {
        acc = (in.x == r0.arg);
        pd = acc ? 1.0f : 0.0f;
      } else {
        pd = exp2f((in.g.x - r0.M) * c) / r0.S;
        // u <= min(1, p/q)  <=>  u q <= p  for q > 0, u < 1 (exact products in float64)
        acc = ((double)in.u * (double)in.g.y <= (double)pd);
      }
    }
  }
  status = __reduce_or_sync(0xffffffffu, status);
  if (status) pd = __int_as_float(0x7fc00000);
  const unsigned rej = __ballot_sync(0xffffffffu, lane < gamma && !acc);
  const int k = rej ? (__ffs(rej) - 1) : gamma;
  const bool hi = k >= 32;  // statistics of the final row k, from the lane holding it
  LinearDecision d;
  d.k = k;
  d.status = status;
  d.greedy = greedy;
  d.arg = __shfl_sync(0xffffffffu, hi ? r1.arg : r0.arg, k & 31);
  d.M = __shfl_sync(0xffffffffu, hi ? r1.M : r0.M, k & 31);
  d.S = __shfl_sync(0xffffffffu, hi ? r1.S : r0.S, k & 31);
  d.c = c;
  d.pad = 0;
  return d;
}


// Weight of element i of a 16-byte vector: 2^((l - M) c), or max(0, that - S q)
// after a rejection (the same arithmetic as the other form of the draw).
template <int DT>
__device__ __forceinline__ float vec_weight(const uint4 &lv, const uint4 &qv, int i,
                                            const LinearDecision &d, bool use_q) {
  float l, q;
  if (DT == SPECDEC_F32) {
    const uint32_t lw = (i == 0) ? lv.x : (i == 1) ? lv.y : (i == 2) ? lv.z : lv.w;
    const uint32_t qw = (i == 0) ? qv.x : (i == 1) ? qv.y : (i == 2) ? qv.z : qv.w;
    l = __uint_as_float(lw);
    q = __uint_as_float(qw);
  } else {
    const int j = i >> 1;
    const uint32_t lw = (j == 0) ? lv.x : (j == 1) ? lv.y : (j == 2) ? lv.z : lv.w;
    const uint32_t qw = (j == 0) ? qv.x : (j == 1) ? qv.y : (j == 2) ? qv.z : qv.w;
    l = (i & 1) ? bf16_hi(lw) : bf16_lo(lw);
    q = (i & 1) ? bf16_hi(qw) : bf16_lo(qw);
  }
  const float ev = ex2_approx((l - d.M) * d.c);
  return use_q ? fmaxf(fmaf(-d.S, q, ev), 0.0f) : ev;
}

template <int DT>
__host__ __device__ constexpr int vec_elems() { return (DT == SPECDEC_F32) ? 4 : 8; }

// float32 sum, in index order, of the weights of one vector
template <int DT>
__device__ __forceinline__ float vec_sum(const uint4 &lv, const uint4 &qv, const LinearDecision &d,
                                         bool use_q) {
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < vec_elems<DT>(); ++i) s += vec_weight<DT>(lv, qv, i, d, use_q);
  return s;
}

// the element of a vector at which base + (running sum, as in vec_sum) first exceeds target
template <int DT>
__device__ __forceinline__ int vec_find(const uint4 &lv, const uint4 &qv, const LinearDecision &d,
                                        bool use_q, unsigned long long base,
                                        unsigned long long target) {
  float run = 0.0f;
#pragma unroll
  for (int i = 0; i < vec_elems<DT>(); ++i) {
    run += vec_weight<DT>(lv, qv, i, d, use_q);
    if (base + to_fixed40(run) > target) return i;
  }
  return vec_elems<DT>() - 1;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v += shfl_xor_u64(v, d);
  return v;
}

__device__ __forceinline__ unsigned long long warp_incl_scan_u64(unsigned long long v, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const unsigned long long y = shfl_up_u64(v, d);
    if (lane >= d) v += y;
  }
  return v;
}

__host__ __device__ constexpr uint32_t kNegInfBits(int dt) { return dt == SPECDEC_F32 ? 0xFF800000u : 0xFF80FF80u; }

// Vectors lane + 32 k of a stage of sbytes bytes (from shared or global
// memory): -inf logits and zero q past the end, which weigh 0.
template <int DT>
__device__ __forceinline__ void load_stage(uint4 (&lv)[kVec], uint4 (&qv)[kVec], const uint8_t *l,
                                           const uint8_t *q, int sbytes, bool use_q, int lane,
                                           bool global) {
  const uint32_t ninf = kNegInfBits(DT);
#pragma unroll
  for (int k = 0; k < kVec; ++k) {
    const int off = (lane + 32 * k) * 16;
    const bool in = off < sbytes;
    if (global) {
      lv[k] = in ? __ldg(reinterpret_cast<const uint4 *>(l + off)) : make_uint4(ninf, ninf, ninf, ninf);
      qv[k] = (in && use_q) ? __ldg(reinterpret_cast<const uint4 *>(q + off)) : make_uint4(0u, 0u, 0u, 0u);
    } else {
      lv[k] = in ? *reinterpret_cast<const uint4 *>(l + off) : make_uint4(ninf, ninf, ninf, ninf);
      qv[k] = (in && use_q) ? *reinterpret_cast<const uint4 *>(q + off) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// Per-request view of the run: the request's index b, its row pointers and sizes.
struct Req {
  long long b;
  const uint8_t *lrow, *qrow;
  int rowbytes, nst;
};

template <int DT>
__device__ __forceinline__ Req make_req(const LinearFinalizeParams &p, long long rb, int k) {
  constexpr int es = (DT == SPECDEC_F32) ? 4 : 2;
  Req r;
  r.b = (long long)p.B - 1 - rb;
  const int R = p.gamma + 1;
  r.rowbytes = p.V * es;
  r.nst = (r.rowbytes + kStage - 1) / kStage;
  r.lrow = reinterpret_cast<const uint8_t *>(p.logits) + (size_t)(r.b * R + k) * r.rowbytes;
  r.qrow = (k < p.gamma)
               ? reinterpret_cast<const uint8_t *>(p.q) + (size_t)(r.b * p.gamma + k) * r.rowbytes
               : r.lrow;
  return r;
}

// Outputs of request b but a drawn token, by one warp.
__device__ __forceinline__ void write_outputs_warp(const LinearFinalizeParams &p, long long b,
                                                   const LinearDecision &d, float pd, int lane) {
  const int gamma = p.gamma, R = gamma + 1, k = d.k;
  if (p.p_draft && lane < gamma) p.p_draft[b * gamma + lane] = pd;
  for (int i = lane; i < R; i += 32) {
    int t = -1;
    if (!d.status) {
      if (i < k) t = __ldg(p.tokens + b * gamma + i);
      else if (i == k) t = d.arg;
    }
    if (d.status || i != k || d.greedy) p.out_tokens[b * R + i] = t;
  }
  if (lane == 0) {
    p.n_accepted[b] = d.status ? 0 : k;
    p.is_bonus[b] = (uint8_t)(!d.status && k == gamma);
    p.row_status[b] = d.status;
    if (d.status) p.final_token[b] = -1;
    else if (d.greedy) p.final_token[b] = d.arg;
    if (d.status || d.greedy) p.ws.mass[b] = kNoMass;  // nothing drawn
  }
}

// Where a request's fixed-point stage totals live: in the workspace (written
// by other CTAs of the running kernel: L2 loads), or in this CTA's shared
// memory with a copy in the workspace.
struct GlobalTotals {
  unsigned long long *g;
  static constexpr bool kRegCache = true;  // keep up to 64 totals in registers
  __device__ __forceinline__ unsigned long long get(int s) const { return __ldcg(g + s); }
  __device__ __forceinline__ void set(int s, unsigned long long v) const { g[s] = v; }
};
struct SharedTotals {
  unsigned long long *sm, *g;
  static constexpr bool kRegCache = false;
  __device__ __forceinline__ unsigned long long get(int s) const { return sm[s]; }
  __device__ __forceinline__ void set(int s, unsigned long long v) const {
    sm[s] = v;
    g[s] = v;
  }
};

// The search of one request by one warp (see the header of this section).
template <int DT, typename Tot>
__device__ __forceinline__ void search_warp(const LinearFinalizeParams &p, const Req &rq,
                                            LinearDecision d, bool aborted, int lane,
                                            const Tot &tot) {
  constexpr int es = (DT == SPECDEC_F32) ? 4 : 2;
  const int gamma = p.gamma, R = gamma + 1;
  const long long b = rq.b;
  if (aborted) {
    // a bounded wait ran out in some CTA of this request: report, draw nothing
    for (int i = lane; i < R; i += 32) p.out_tokens[b * R + i] = -1;
    if (lane == 0) {
      p.row_status[b] = SPECDEC_ROW_INTERNAL;
      p.n_accepted[b] = 0;
      p.is_bonus[b] = 0;
      p.final_token[b] = -1;
      p.ws.mass[b] = kNoMass;
    }
    return;
  }
  bool use_q = d.k < gamma;
  const float U = __ldg(p.uniforms + b * R + gamma);
  // rows of at most 128 stages keep their stage totals in registers (four per
  // lane, loaded together: one round trip)
  const bool cached = Tot::kRegCache && rq.nst <= 128;
  unsigned long long c[4] = {0, 0, 0, 0}, Z = 0;
  if (cached) {
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = (lane + 32 * i < rq.nst) ? tot.get(lane + 32 * i) : 0ull;
    Z = c[0] + c[1] + c[2] + c[3];
  } else {
    for (int s = lane; s < rq.nst; s += 32) Z += tot.get(s);
  }
  Z = warp_sum_u64(Z);
  if (Z == 0 && use_q) {
    // residual mass 0 (only by rounding): draw from p itself
    use_q = false;
    for (int s = 0; s < rq.nst; ++s) {
      uint4 lv[kVec], qv[kVec];
      load_stage<DT>(lv, qv, rq.lrow + (size_t)s * kStage, rq.qrow + (size_t)s * kStage,
                     min(kStage, rq.rowbytes - s * kStage), false, lane, true);
      unsigned long long acc = 0;
#pragma unroll
      for (int k = 0; k < kVec; ++k) acc += to_fixed40(vec_sum<DT>(lv[k], qv[k], d, false));
      acc = warp_sum_u64(acc);
      if (lane == 0) tot.set(s, acc);
      Z += acc;
    }
    __syncwarp();
    if (cached) {
#pragma unroll
      for (int i = 0; i < 4; ++i) c[i] = (lane + 32 * i < rq.nst) ? tot.get(lane + 32 * i) : 0ull;
    }
  }
  const unsigned long long target = uniform_target(U, Z);
  if (lane == 0) p.ws.mass[b] = draw_mass(Z, d.S);
  // the stage holding the crossing
  unsigned long long base = 0;
  int st = -1;
  for (int s0 = 0; s0 < rq.nst && st < 0; s0 += 32) {
    const int i = s0 >> 5;
    const unsigned long long v = cached ? (i == 0 ? c[0] : i == 1 ? c[1] : i == 2 ? c[2] : c[3])
                                        : ((s0 + lane < rq.nst) ? tot.get(s0 + lane) : 0ull);
    const unsigned long long incl = warp_incl_scan_u64(v, lane);
    const unsigned m = __ballot_sync(0xffffffffu, target < base + incl);
    if (m) {
      const int ls = __ffs(m) - 1;
      st = s0 + ls;
      base += __shfl_sync(0xffffffffu, incl - v, ls);
    } else {
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  if (st < 0) return;  // no weight at all: unreachable for a usable row
  // the vector, in index order, then the element: lane L takes the stage's
  // vectors 8L .. 8L + 7, so one warp scan of the lane totals orders them all
  uint4 lv[kVec], qv[kVec];
  const int off = st * kStage;
  {
    const int sb = min(kStage, rq.rowbytes - off);
    const uint32_t ninf = kNegInfBits(DT);
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int o = (lane * kVec + k) * 16;
      const bool in = o < sb;
      lv[k] = in ? __ldg(reinterpret_cast<const uint4 *>(rq.lrow + off + o))
                 : make_uint4(ninf, ninf, ninf, ninf);
      qv[k] = (in && use_q) ? __ldg(reinterpret_cast<const uint4 *>(rq.qrow + off + o))
                            : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  unsigned long long xs[kVec], lt = 0;
#pragma unroll
  for (int k = 0; k < kVec; ++k) {
    xs[k] = to_fixed40(vec_sum<DT>(lv[k], qv[k], d, use_q));
    lt += xs[k];
  }
  const unsigned long long incl = warp_incl_scan_u64(lt, lane);
  const unsigned m = __ballot_sync(0xffffffffu, target < base + incl);
  if (!m) return;
  const int lx = __ffs(m) - 1;
  if (lane != lx) return;
  unsigned long long vbase = base + incl - lt;
  int kx = kVec - 1;
#pragma unroll
  for (int k = kVec - 1; k >= 0; --k) {
    // the first vector of this lane whose running sum passes the target
    unsigned long long pre = vbase;
#pragma unroll
    for (int j = 0; j < k; ++j) pre += xs[j];
    if (target < pre + xs[k]) kx = k;
  }
  uint4 ls = lv[0], qs = qv[0];
#pragma unroll
  for (int k = 0; k < kVec; ++k) {
    if (k == kx) {
      ls = lv[k];
      qs = qv[k];
    }
  }
#pragma unroll
  for (int j = 0; j < kVec; ++j)
    if (j < kx) vbase += xs[j];
  const int e = vec_find<DT>(ls, qs, d, use_q, vbase, target);
  const int v = off / es + (lane * kVec + kx) * vec_elems<DT>() + e;
  p.final_token[b] = v;
  p.out_tokens[b * R + d.k] = v;
}

}  // namespace drawc
}  // namespace specdec
