// Pieces shared by the linear and tree finalize kernels: merging the split
// partials of a row, the exact first arg-max, and the cluster-wide
// inverse-CDF draw over one vocabulary row.
#pragma once

#include <cfloat>
#include <cooperative_groups.h>

#include "common.cuh"

namespace specdec {
namespace fin {

namespace cg = cooperative_groups;

constexpr int kG = 8;                 // CTAs per cluster: one cluster per request
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPerThread = 16;        // contiguous elements per thread in a tile
constexpr int kTile = kThreads * kPerThread;
constexpr int kMaxTilesPerCta = (SPECDEC_MAX_V + kTile * kG - 1) / (kTile * kG);

struct RowStat {
  float M;    // row max of the raw logits
  float S;    // sum of 2^((l - M) c)
  int arg;    // start of the 16-byte group holding the first maximum
  int flags;
};

// Merge the P split partials of one row (same rule as inside the stats pass).
__device__ __forceinline__ RowStat merge_row(const RowPartial *part, long long row, int P,
                                             float c) {
  const RowPartial *pr = part + row * (long long)P;
  RowStat r;
  r.M = -INFINITY;
  r.S = 0.0f;
  r.arg = 0x7FFFFFFF;
  r.flags = 0;
  for (int j = 0; j < P; ++j) {
    const RowPartial x = pr[j];
    r.flags |= x.flags;
    const float M = fmaxf(r.M, x.m);
    const float Mref = fmaxf(M, -FLT_MAX);
    const float f1 = ex2_approx((fmaxf(r.M, -FLT_MAX) - Mref) * c);
    const float f2 = ex2_approx((fmaxf(x.m, -FLT_MAX) - Mref) * c);
    r.arg = (r.M > x.m) ? r.arg : (x.m > r.M) ? x.arg : min(r.arg, x.arg);
    r.S = r.S * f1 + x.s * f2;
    r.M = M;
  }
  return r;
}

__device__ __forceinline__ bool row_usable(const RowStat &r) {
  return r.M > -INFINITY && r.M < INFINITY && r.S > 0.0f && r.S < INFINITY;
}

// First index holding the row maximum: it lies in the 16-byte group that
// starts at r.arg (or is r.arg itself for an unaligned edge element).
__device__ __forceinline__ int exact_argmax(const void *logits, int dtype, long long row_off,
                                            int V, const RowStat &r) {
  const int span = (dtype == SPECDEC_F32) ? 4 : 8;
  const int a0 = max(0, min(r.arg, V - 1));
  const int a1 = min(V, a0 + span);
  for (int e = a0; e < a1; ++e)
    if (load_elem(logits, dtype, row_off + e) == r.M) return e;
  return a0;  // unreachable for a usable row
}

// Draw weights of one row, 16 contiguous elements starting at e:
//   w_v = max(0, 2^((l_v - M) c) / S - cq * q_v)     (cq = 0: the target row itself)
// Elements at or beyond V get weight 0.
__device__ __forceinline__ void row_weights16(const void *lrow, const void *qrow, int dtype,
                                              int V, int e, float M, float c, float invS,
                                              float cq, bool vec_ok, float w[kPerThread]) {
  float l[kPerThread], qv[kPerThread];
  const bool full = vec_ok && (e + kPerThread <= V);
  if (full && dtype == SPECDEC_BF16) {
    const uint4 *lp = reinterpret_cast<const uint4 *>(
        reinterpret_cast<const uint16_t *>(lrow) + e);
    const uint4 a = __ldg(lp), bb = __ldg(lp + 1);
    const uint32_t wd[8] = {a.x, a.y, a.z, a.w, bb.x, bb.y, bb.z, bb.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      l[2 * k] = bf16_lo(wd[k]);
      l[2 * k + 1] = bf16_hi(wd[k]);
    }
    if (cq != 0.0f) {
      const uint4 *qp = reinterpret_cast<const uint4 *>(
          reinterpret_cast<const uint16_t *>(qrow) + e);
      const uint4 x = __ldg(qp), y = __ldg(qp + 1);
      const uint32_t qd[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        qv[2 * k] = bf16_lo(qd[k]);
        qv[2 * k + 1] = bf16_hi(qd[k]);
      }
    }
  } else if (full) {
    const float4 *lp = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(lrow) + e);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 t = __ldg(lp + k);
      l[4 * k] = t.x;
      l[4 * k + 1] = t.y;
      l[4 * k + 2] = t.z;
      l[4 * k + 3] = t.w;
    }
    if (cq != 0.0f) {
      const float4 *qp =
          reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(qrow) + e);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 t = __ldg(qp + k);
        qv[4 * k] = t.x;
        qv[4 * k + 1] = t.y;
        qv[4 * k + 2] = t.z;
        qv[4 * k + 3] = t.w;
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
      const int v = e + k;
      l[k] = (v < V) ? load_elem(lrow, dtype, v) : -INFINITY;
      qv[k] = (v < V && cq != 0.0f) ? load_elem(qrow, dtype, v) : 0.0f;
    }
  }
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    const float pv = ex2_approx((l[k] - M) * c) * invS;
    const float x = (cq != 0.0f) ? pv - cq * qv[k] : pv;
    w[k] = (e + k < V) ? fmaxf(x, 0.0f) : 0.0f;
  }
}

// fp32 sum of the 16 weights in index order, then to 52-bit fixed point.
__device__ __forceinline__ unsigned long long fixed_sum16(const float w[kPerThread]) {
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) s += w[k];
  return to_fixed52(s);
}

struct DrawSmem {
  unsigned long long warp_tile[kMaxTilesPerCta][kWarps];
  unsigned long long tile_tot[kMaxTilesPerCta];
  unsigned long long cta_total;     // this pass's CTA total
  unsigned long long shared_total[2];  // read by the other CTAs; double-buffered by pass
  unsigned long long prefix, Z, base;
  unsigned long long scan_warp[kWarps];
  int tile;
  int found;
};

struct DrawRow {
  const void *lrow;
  const void *qrow;  // may be null when cq == 0
  int dtype, V;
  float M, c, invS, cq;
  bool vec_ok;
};

// Pass over this CTA's tiles of the row: per-tile fixed-point totals in smem
// and the CTA total (published in slot `pass & 1` for the other CTAs).
__device__ __forceinline__ void draw_sums(DrawSmem &ds, const DrawRow &r, int t0, int t1,
                                          int pass) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int t = t0; t < t1; ++t) {
    float w[kPerThread];
    row_weights16(r.lrow, r.qrow, r.dtype, r.V, t * kTile + tid * kPerThread, r.M, r.c, r.invS,
                  r.cq, r.vec_ok, w);
    unsigned long long f = fixed_sum16(w);
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) f += shfl_xor_u64(f, d);
    if (lane == 0) ds.warp_tile[t - t0][warp] = f;
  }
  __syncthreads();
  for (int i = tid; i < t1 - t0; i += kThreads) {
    unsigned long long s = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += ds.warp_tile[i][w];
    ds.tile_tot[i] = s;
  }
  __syncthreads();
  if (tid == 0) {
    unsigned long long s = 0;
    for (int i = 0; i < t1 - t0; ++i) s += ds.tile_tot[i];
    ds.cta_total = s;
    ds.shared_total[pass & 1] = s;
  }
}

// Cluster-wide exclusive prefix of the CTA totals (all CTAs call it).  A
// slot is rewritten two passes later, after every CTA has passed the cluster
// barrier of the pass in between, so no reader can see a later value.
__device__ __forceinline__ void draw_exchange(DrawSmem &ds, cg::cluster_group &cluster,
                                              int pass) {
  cluster.sync();
  if (threadIdx.x == 0) {
    const unsigned rank = cluster.block_rank();
    unsigned long long pre = 0, tot = 0;
    for (unsigned r = 0; r < (unsigned)kG; ++r) {
      const DrawSmem *other = cluster.map_shared_rank(&ds, r);
      const unsigned long long x = other->shared_total[pass & 1];
      if (r < rank) pre += x;
      tot += x;
    }
    ds.prefix = pre;
    ds.Z = tot;
  }
  __syncthreads();
}

// If the crossing of `target` lies in this CTA, find the smallest v with
// C_v > target and return it (in thread 0 of the CTA: -1 otherwise).
__device__ __forceinline__ int draw_search(DrawSmem &ds, const DrawRow &r, int t0, int t1,
                                           unsigned long long target) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned long long pre = ds.prefix;
  const bool mine = (pre <= target) && (target - pre < ds.cta_total);
  if (!mine) return -1;  // uniform across the CTA
  if (tid == 0) {
    unsigned long long run = pre;
    int tile = t1 - 1;
    for (int i = 0; i < t1 - t0; ++i) {
      if (target - run < ds.tile_tot[i]) {
        tile = t0 + i;
        break;
      }
      run += ds.tile_tot[i];
    }
    ds.tile = tile;
    ds.base = run;
    ds.found = -1;
  }
  __syncthreads();
  const int e = ds.tile * kTile + tid * kPerThread;
  float w[kPerThread];
  row_weights16(r.lrow, r.qrow, r.dtype, r.V, e, r.M, r.c, r.invS, r.cq, r.vec_ok, w);
  const unsigned long long f = fixed_sum16(w);
  // block exclusive scan of f
  unsigned long long inc = f;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const unsigned long long y = shfl_up_u64(inc, d);
    if (lane >= d) inc += y;
  }
  if (lane == 31) ds.scan_warp[warp] = inc;
  __syncthreads();
  unsigned long long wpre = 0;
  for (int k = 0; k < warp; ++k) wpre += ds.scan_warp[k];
  const unsigned long long excl = ds.base + wpre + inc - f;
  if (excl <= target && target - excl < f) {
    float run = 0.0f;
    int v = e + kPerThread - 1;
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
      run += w[k];
      if (excl + to_fixed52(run) > target) {
        v = e + k;
        break;
      }
    }
    ds.found = v;
  }
  __syncthreads();
  return ds.found;
}

}  // namespace fin
}  // namespace specdec
