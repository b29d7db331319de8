// Row-statistics stage math of the stats pass: the geometry of a 16 KB unit
// of a row (its 16-byte aligned interior and the edge elements read with
// plain loads), and one consumer warp's reduction of an 8 KB stage held in
// registers -- NaN-propagating max
// (packed bf16x2), sum of 2^((l - m) c) with packed fp32x2 arithmetic, and the
// first index of the maximum for greedy rows ("Chapter 15: Decoding
// acceleration", section 15.1.2 step 2).
#pragma once

#include <cfloat>

#include "common.cuh"

namespace specdec {
namespace stage {

// Defaults measured on GB300 (B=256, V=128256 bf16): 16 KB copies, 12 slots
// (192 KB in flight per SM); 8 KB copies are limited by the per-copy cost.
// The consumers are latency-bound (fixed-latency dependency stalls), so more
// warps help: 12 / 14 / 15 consumer warps take 98.8 / 91.6 / 88.6 us
// (15 warps: 120 registers, no spills; 16 would spill).
#ifndef SPECDEC_K1_WARPS
#define SPECDEC_K1_WARPS 15
#endif
#ifndef SPECDEC_K1_SLOTS
#define SPECDEC_K1_SLOTS 12
#endif
#ifndef SPECDEC_K1_UNIT
#define SPECDEC_K1_UNIT 2
#endif
constexpr int kConsumerWarps = SPECDEC_K1_WARPS;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kSlots = SPECDEC_K1_SLOTS;             // units in flight per CTA
constexpr int kUnit = SPECDEC_K1_UNIT;               // stages moved by one bulk copy
constexpr int kUnitBytes = kUnit * kStageBytes;
constexpr int kVecPerLane = kStageBytes / 16 / 32;   // 16-byte vectors per lane per stage
static_assert(kVecPerLane * 32 * 16 == kStageBytes, "a stage is a whole number of warp loads");
static_assert(kSlots * kUnitBytes <= 200 * 1024, "stage ring fits in shared memory");
// a warp's next stage lies at most one ring ahead of its last one (the
// consumers' two-barrier wait relies on it)
static_assert(kConsumerWarps <= kSlots * kUnit, "no more consumer warps than ring stages");

struct UnitGeom {
  int row;
  int j0;               // first stage of the unit within the row
  int nst;              // stages in the unit (<= kUnit)
  const uint8_t *src;   // 16-byte aligned start of the unit's bytes
  int bytes;            // 0 .. kUnitBytes, a multiple of 16
  int elem0;            // row index of the unit's first element
  int head_end;         // row elements [0, head_end) and [tail_begin, V)
  int tail_begin;       // are read with plain loads by stage 0's warp
};

// (row, unit) of a unit index, advanced by a fixed step without divisions.
struct UnitCursor {
  int row;  // B * R < 2^31 (checked by the host)
  int ju;
  int drow;
  int dj;
  __device__ __forceinline__ void init(long long g, long long step, int upr) {
    row = (int)(g / upr);
    ju = (int)(g - (long long)row * upr);
    drow = (int)(step / upr);
    dj = (int)(step - (long long)drow * upr);
  }
  __device__ __forceinline__ void advance(int upr) {
    row += drow;
    ju += dj;
    if (ju >= upr) {
      ju -= upr;
      ++row;
    }
  }
};

__device__ __forceinline__ UnitGeom unit_geometry(const void *logits, int V, int spr, int row, int ju,
                                                 int es) {
  UnitGeom s;
  s.row = row;
  s.j0 = ju * kUnit;
  s.nst = min(kUnit, spr - s.j0);
  const uintptr_t a = reinterpret_cast<uintptr_t>(logits) + (uintptr_t)row * V * es;
  const uintptr_t e = a + (uintptr_t)V * es;
  const uintptr_t i0 = (a + 15) & ~(uintptr_t)15;
  uintptr_t i1 = e & ~(uintptr_t)15;
  if (i1 < i0) i1 = i0;
  const uintptr_t s0 = i0 + (uintptr_t)s.j0 * kStageBytes;
  const uintptr_t s1 = (s0 + kUnitBytes < i1) ? s0 + kUnitBytes : i1;
  s.src = reinterpret_cast<const uint8_t *>(s0);
  s.bytes = (s1 > s0) ? (int)(s1 - s0) : 0;
  s.elem0 = (int)((s0 - a) / es);
  s.head_end = min(V, (int)((i0 - a) / es));
  s.tail_begin = max(s.head_end, (int)((i1 - a) / es));
  return s;
}

__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v = fmax_nan(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

__device__ __forceinline__ int warp_min(int v) { return __reduce_min_sync(0xffffffffu, v); }

// Elements held by one lane for one stage: kVecPerLane 16-byte vectors of the
// stage (vector k is the stage's vector lane + 32 k) plus at most one edge
// element of the row.
template <int DT>
struct LaneData {
  uint4 v[kVecPerLane];
  float edge;      // -inf when the lane has no edge element
  int edge_idx;
};

template <int DT>
__device__ __forceinline__ void load_lane(LaneData<DT> &d, const uint8_t *stage, int nvec, int lane) {
  const uint32_t ninf = (DT == SPECDEC_F32) ? 0xFF800000u : 0xFF80FF80u;
  if (nvec == kStageBytes / 16) {
#pragma unroll
    for (int k = 0; k < kVecPerLane; ++k)
      d.v[k] = *reinterpret_cast<const uint4 *>(stage + (size_t)(lane + 32 * k) * 16);
  } else {
#pragma unroll
    for (int k = 0; k < kVecPerLane; ++k) {
      const int j = lane + 32 * k;
      d.v[k] = (j < nvec) ? *reinterpret_cast<const uint4 *>(stage + (size_t)j * 16)
                          : make_uint4(ninf, ninf, ninf, ninf);
    }
  }
}

template <int DT>
__device__ __forceinline__ float lane_max(const LaneData<DT> &d) {
  float m;
  if (DT == SPECDEC_F32) {
    m = d.edge;
#pragma unroll
    for (int k = 0; k < kVecPerLane; ++k) {
      m = fmax_nan(m, fmax_nan(fmax_nan(__uint_as_float(d.v[k].x), __uint_as_float(d.v[k].y)),
                               fmax_nan(__uint_as_float(d.v[k].z), __uint_as_float(d.v[k].w))));
    }
  } else {
    uint32_t a = bf16x2_max_nan(d.v[0].x, d.v[0].y), b = bf16x2_max_nan(d.v[0].z, d.v[0].w);
#pragma unroll
    for (int k = 1; k < kVecPerLane; ++k) {
      a = bf16x2_max_nan(a, bf16x2_max_nan(d.v[k].x, d.v[k].y));
      b = bf16x2_max_nan(b, bf16x2_max_nan(d.v[k].z, d.v[k].w));
    }
    a = bf16x2_max_nan(a, b);
    m = fmax_nan(fmax_nan(bf16_lo(a), bf16_hi(a)), d.edge);
  }
  return m;
}

// Sum of 2^((l - m) c) over the lane's elements (packed fp32x2 math).
template <int DT>
__device__ __forceinline__ float lane_sum(const LaneData<DT> &d, float c, float m) {
  const float2 cc = make_float2(c, c);
  const float2 nm = make_float2(-m, -m);
  float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0, acc2 = acc0, acc3 = acc0;
#pragma unroll
  for (int k = 0; k < kVecPerLane; ++k) {
    const uint4 w = d.v[k];
    float2 x0, x1, x2, x3;
    if (DT == SPECDEC_F32) {
      x0 = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
      x1 = make_float2(__uint_as_float(w.z), __uint_as_float(w.w));
      x0 = __fmul2_rn(__fadd2_rn(x0, nm), cc);
      x1 = __fmul2_rn(__fadd2_rn(x1, nm), cc);
      x0.x = ex2_approx(x0.x);
      x0.y = ex2_approx(x0.y);
      x1.x = ex2_approx(x1.x);
      x1.y = ex2_approx(x1.y);
      if (k & 1) {
        acc2 = __fadd2_rn(acc2, x0);
        acc3 = __fadd2_rn(acc3, x1);
      } else {
        acc0 = __fadd2_rn(acc0, x0);
        acc1 = __fadd2_rn(acc1, x1);
      }
    } else {
      x0 = __fmul2_rn(__fadd2_rn(make_float2(bf16_lo(w.x), bf16_hi(w.x)), nm), cc);
      x1 = __fmul2_rn(__fadd2_rn(make_float2(bf16_lo(w.y), bf16_hi(w.y)), nm), cc);
      x2 = __fmul2_rn(__fadd2_rn(make_float2(bf16_lo(w.z), bf16_hi(w.z)), nm), cc);
      x3 = __fmul2_rn(__fadd2_rn(make_float2(bf16_lo(w.w), bf16_hi(w.w)), nm), cc);
      x0.x = ex2_approx(x0.x);
      x0.y = ex2_approx(x0.y);
      x1.x = ex2_approx(x1.x);
      x1.y = ex2_approx(x1.y);
      x2.x = ex2_approx(x2.x);
      x2.y = ex2_approx(x2.y);
      x3.x = ex2_approx(x3.x);
      x3.y = ex2_approx(x3.y);
      acc0 = __fadd2_rn(acc0, x0);
      acc1 = __fadd2_rn(acc1, x1);
      acc2 = __fadd2_rn(acc2, x2);
      acc3 = __fadd2_rn(acc3, x3);
    }
  }
  acc0 = __fadd2_rn(acc0, acc1);
  acc2 = __fadd2_rn(acc2, acc3);
  acc0 = __fadd2_rn(acc0, acc2);
  const float e = ex2_approx((d.edge - m) * c);  // -inf edge -> 0
  return (acc0.x + acc0.y) + e;
}

// -inf logits (masked tokens) become the most negative finite value before the
// sums below: their weight is 0 either way, and 0 * (l - m) stays 0.
__device__ __forceinline__ uint32_t bf16x2_floor_finite(uint32_t w) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(w), "r"(0xFF7FFF7Fu));
  return r;
}

// Over the lane's elements (packed fp32x2 math): the sum of e = 2^((l - m) c),
// returned, and in `a` the sum of e (l - m) (every term <= 0), from which the
// row's entropy follows: H = ln S - A / (T S) for the merged S and A.
template <int DT>
__device__ __forceinline__ float lane_sum_a(const LaneData<DT> &d, float c, float m, float &a) {
  const float2 cc = make_float2(c, c);
  const float2 nm = make_float2(-m, -m);
  float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0, acc2 = acc0, acc3 = acc0;
  float2 aa0 = acc0, aa1 = acc0;
#pragma unroll
  for (int k = 0; k < kVecPerLane; ++k) {
    const uint4 w = d.v[k];
    if (DT == SPECDEC_F32) {
      const float2 d0 = __fadd2_rn(make_float2(fmaxf(__uint_as_float(w.x), -FLT_MAX),
                                               fmaxf(__uint_as_float(w.y), -FLT_MAX)), nm);
      const float2 d1 = __fadd2_rn(make_float2(fmaxf(__uint_as_float(w.z), -FLT_MAX),
                                               fmaxf(__uint_as_float(w.w), -FLT_MAX)), nm);
      float2 x0 = __fmul2_rn(d0, cc), x1 = __fmul2_rn(d1, cc);
      x0.x = ex2_approx(x0.x);
      x0.y = ex2_approx(x0.y);
      x1.x = ex2_approx(x1.x);
      x1.y = ex2_approx(x1.y);
      if (k & 1) {
        acc2 = __fadd2_rn(acc2, x0);
        acc3 = __fadd2_rn(acc3, x1);
      } else {
        acc0 = __fadd2_rn(acc0, x0);
        acc1 = __fadd2_rn(acc1, x1);
      }
      aa0 = __ffma2_rn(x0, d0, aa0);
      aa1 = __ffma2_rn(x1, d1, aa1);
    } else {
      const uint32_t wx = bf16x2_floor_finite(w.x), wy = bf16x2_floor_finite(w.y);
      const uint32_t wz = bf16x2_floor_finite(w.z), ww = bf16x2_floor_finite(w.w);
      const float2 d0 = __fadd2_rn(make_float2(bf16_lo(wx), bf16_hi(wx)), nm);
      const float2 d1 = __fadd2_rn(make_float2(bf16_lo(wy), bf16_hi(wy)), nm);
      const float2 d2 = __fadd2_rn(make_float2(bf16_lo(wz), bf16_hi(wz)), nm);
      const float2 d3 = __fadd2_rn(make_float2(bf16_lo(ww), bf16_hi(ww)), nm);
      float2 x0 = __fmul2_rn(d0, cc), x1 = __fmul2_rn(d1, cc);
      float2 x2 = __fmul2_rn(d2, cc), x3 = __fmul2_rn(d3, cc);
      x0.x = ex2_approx(x0.x);
      x0.y = ex2_approx(x0.y);
      x1.x = ex2_approx(x1.x);
      x1.y = ex2_approx(x1.y);
      x2.x = ex2_approx(x2.x);
      x2.y = ex2_approx(x2.y);
      x3.x = ex2_approx(x3.x);
      x3.y = ex2_approx(x3.y);
      acc0 = __fadd2_rn(acc0, x0);
      acc1 = __fadd2_rn(acc1, x1);
      acc2 = __fadd2_rn(acc2, x2);
      acc3 = __fadd2_rn(acc3, x3);
      aa0 = __ffma2_rn(x0, d0, aa0);
      aa1 = __ffma2_rn(x1, d1, aa1);
      aa0 = __ffma2_rn(x2, d2, aa0);
      aa1 = __ffma2_rn(x3, d3, aa1);
    }
  }
  acc0 = __fadd2_rn(acc0, acc1);
  acc2 = __fadd2_rn(acc2, acc3);
  acc0 = __fadd2_rn(acc0, acc2);
  aa0 = __fadd2_rn(aa0, aa1);
  float e = 0.0f, ae = 0.0f;
  if (d.edge != -INFINITY) {
    const float de = d.edge - m;
    e = ex2_approx(de * c);
    ae = e * de;
  }
  a = (aa0.x + aa0.y) + ae;
  return (acc0.x + acc0.y) + e;
}

// First index (in the row) of a lane element equal to wm, INT_MAX if none.
// Fully unrolled so the stage stays in registers.
template <int DT>
__device__ __forceinline__ int lane_first(const LaneData<DT> &d, float wm, int elem0, int lane) {
  constexpr int kPerVec = (DT == SPECDEC_F32) ? 4 : 8;
  int best = 0x7FFFFFFF;
#pragma unroll
  for (int k = kVecPerLane - 1; k >= 0; --k) {
    const uint32_t w[4] = {d.v[k].x, d.v[k].y, d.v[k].z, d.v[k].w};
#pragma unroll
    for (int t = kPerVec - 1; t >= 0; --t) {
      const float x = (DT == SPECDEC_F32) ? __uint_as_float(w[t])
                                          : ((t & 1) ? bf16_hi(w[t >> 1]) : bf16_lo(w[t >> 1]));
      if (x == wm) best = elem0 + (lane + 32 * k) * kPerVec + t;
    }
  }
  if (d.edge == wm) best = min(best, d.edge_idx);
  return best;
}

}  // namespace stage
}  // namespace specdec
