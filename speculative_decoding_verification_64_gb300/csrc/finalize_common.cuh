// Pieces of the tree finalize kernel: the cluster-wide inverse-CDF draw over
// one vocabulary row.
//
// Draw weights are kept in units of the row maximum: with
//     e_v = 2^((l_v - M) c),  c = log2(e) / T    (e_v <= 1, e = 1 at the maximum),
// computed exactly as the stats pass computes its terms, the target row is
// p = e / S with S the merged sum of the stats pass, and every weight the
// method draws from is w_v = max(0, e_v - K q_v) for a scalar K >= 0
// (K = 0: the target row itself; K = S: the residual max(0, p - q) times S;
// tree walk: K = S c_j after j rejected siblings).  Each thread sums 16
// contiguous weights in float32, and everything above that is summed in
// 40-bit fixed point (exact, associative integer adds), so the search for the
// crossing sees exactly the prefix sums that the totals were made of.
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
// tiles whose loads are in flight together: 4 of bf16 (64 registers of raw
// data a thread), 2 of float32 (the same bytes), within the 128-register cap
template <int DT>
__host__ __device__ constexpr int batch_tiles() { return (DT == SPECDEC_F32) ? 2 : 4; }
constexpr int kMaxTilesPerCta = ((SPECDEC_MAX_V + kG - 1) / kG + 15 + kTile - 1) / kTile;
constexpr double kFixedUnit = 0x1p-40;  // value of one unit of the fixed-point sums

// p(x) from the merged row statistics (accept tests and the p outputs).
__device__ __forceinline__ float target_prob(float lx, const RowStat &r, float c) {
  return exp2f((lx - r.M) * c) / r.S;
}

// One CTA's share of a draw: the slice [v0, v1) of the row, read through
// lrow/qrow (element v at byte v * es; the pointers may point at a copy of
// the slice in shared memory, offset so that the same indexing holds).
struct DrawRow {
  const uint8_t *lrow;  // logits row
  const uint8_t *qrow;  // q row (read only when use_q)
  int v0, v1;           // the slice
  float M, c;           // e_v = 2^((l - M) c)
  float K;              // w_v = max(0, e_v - K q_v)
  bool use_q;
  bool vec_ok;          // 16-byte aligned rows: vector loads
};

__device__ __forceinline__ float elem_e(const DrawRow &r, float l) { return ex2_approx((l - r.M) * r.c); }

__device__ __forceinline__ float elem_w(const DrawRow &r, float e, float q) {
  return r.use_q ? fmaxf(fmaf(-r.K, q, e), 0.0f) : e;
}

// Plain (generic) element load: the row may live in global or shared memory.
template <int DT>
__device__ __forceinline__ uint32_t load_bits(const uint8_t *row, int v) {
  if (DT == SPECDEC_F32) return *reinterpret_cast<const uint32_t *>(row + (size_t)v * 4);
  return *reinterpret_cast<const uint16_t *>(row + (size_t)v * 2);
}

// 16 contiguous elements of a tile as raw 16-byte vectors (bf16: 2 vectors per
// row, float32: 4), so several tiles' loads can be in flight at once.
template <int DT>
struct Raw16 {
  uint4 l[DT == SPECDEC_F32 ? 4 : 2];
  uint4 q[DT == SPECDEC_F32 ? 4 : 2];
};

template <int DT>
__device__ __forceinline__ void load_raw(const DrawRow &r, int e, Raw16<DT> &x) {
  constexpr int n = (DT == SPECDEC_F32) ? 4 : 2;
  constexpr int es = (DT == SPECDEC_F32) ? 4 : 2;
  if (r.vec_ok && e + kPerThread <= r.v1) {
    const uint4 *lp = reinterpret_cast<const uint4 *>(r.lrow + (size_t)e * es);
#pragma unroll
    for (int k = 0; k < n; ++k) x.l[k] = lp[k];
    if (r.use_q) {
      const uint4 *qp = reinterpret_cast<const uint4 *>(r.qrow + (size_t)e * es);
#pragma unroll
      for (int k = 0; k < n; ++k) x.q[k] = qp[k];
    }
  } else {
    // ragged or unaligned: element by element; past the slice the logit is -inf (weight 0)
    uint32_t lw[4 * n], qw[4 * n];
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
      const int v = e + k;
      const bool in = v < r.v1;
      const uint32_t lb = in ? load_bits<DT>(r.lrow, v) : (DT == SPECDEC_F32 ? 0xFF800000u : 0xFF80u);
      const uint32_t qb = (in && r.use_q) ? load_bits<DT>(r.qrow, v) : 0u;
      if (DT == SPECDEC_F32) {
        lw[k] = lb;
        qw[k] = qb;
      } else if (k & 1) {
        lw[k >> 1] |= lb << 16;
        qw[k >> 1] |= qb << 16;
      } else {
        lw[k >> 1] = lb;
        qw[k >> 1] = qb;
      }
    }
#pragma unroll
    for (int k = 0; k < n; ++k) {
      x.l[k] = make_uint4(lw[4 * k], lw[4 * k + 1], lw[4 * k + 2], lw[4 * k + 3]);
      x.q[k] = make_uint4(qw[4 * k], qw[4 * k + 1], qw[4 * k + 2], qw[4 * k + 3]);
    }
  }
}

template <int DT>
__device__ __forceinline__ float raw_elem(const uint4 *v, int k) {
  if (DT == SPECDEC_F32) {
    const uint4 t = v[k >> 2];
    const uint32_t w = (k & 3) == 0 ? t.x : (k & 3) == 1 ? t.y : (k & 3) == 2 ? t.z : t.w;
    return __uint_as_float(w);
  }
  const uint4 t = v[k >> 3];
  const int j = (k >> 1) & 3;
  const uint32_t w = j == 0 ? t.x : j == 1 ? t.y : j == 2 ? t.z : t.w;
  return (k & 1) ? bf16_hi(w) : bf16_lo(w);
}

// Weights of 16 elements and their float32 sum in index order, as fixed point.
template <int DT>
__device__ __forceinline__ unsigned long long weights16(const DrawRow &r, const Raw16<DT> &x, int e,
                                                        float w[kPerThread]) {
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < kPerThread; ++k) {
    const float q = r.use_q ? raw_elem<DT>(x.q, k) : 0.0f;
    w[k] = (e + k < r.v1) ? elem_w(r, elem_e(r, raw_elem<DT>(x.l, k)), q) : 0.0f;
    s += w[k];
  }
  return to_fixed40(s);
}

struct DrawSmem {
  unsigned long long warp_tile[kMaxTilesPerCta][kWarps];
  unsigned long long tile_tot[kMaxTilesPerCta];
  unsigned long long cta_total;        // this pass's CTA total
  unsigned long long totals[2][kG];    // every CTA's total, written by that CTA; by pass parity
  unsigned long long prefix, Z, base;
  float Zf;  // Z as a float, in units of the row maximum
  unsigned long long scan_warp[kWarps];
  alignas(8) uint64_t xbar[2];         // the exchange's arrivals, by pass parity
  int tile;
  int found;
  int lost;                            // an exchange wait of this CTA gave up
};

// Before the first exchange, by thread 0 of every CTA, ahead of a cluster
// barrier (the other CTAs' stores complete on these barriers).
__device__ __forceinline__ void exchange_init(DrawSmem &ds) {
  mbar_init(&ds.xbar[0], 1);
  mbar_init(&ds.xbar[1], 1);
  ds.lost = 0;
  fence_mbar_init();
}


__device__ __forceinline__ int slice_tiles(const DrawRow &r) { return (r.v1 - r.v0 + kTile - 1) / kTile; }

// One pass over this CTA's slice: per-tile fixed-point totals in smem and the
// CTA total, published in slot `pass & 1`.
template <int DT>
__device__ __forceinline__ void draw_sums(DrawSmem &ds, const DrawRow &r, int pass) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nt = slice_tiles(r);
  constexpr int kBatch = batch_tiles<DT>();
  for (int tb = 0; tb < nt; tb += kBatch) {
    Raw16<DT> x[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      if (tb + u < nt) load_raw<DT>(r, r.v0 + (tb + u) * kTile + tid * kPerThread, x[u]);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (tb + u < nt) {
        float w[kPerThread];
        unsigned long long f = weights16<DT>(r, x[u], r.v0 + (tb + u) * kTile + tid * kPerThread, w);
#pragma unroll
        for (int d = 16; d >= 1; d >>= 1) f += shfl_xor_u64(f, d);
        if (lane == 0) ds.warp_tile[tb + u][warp] = f;
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < nt; i += kThreads) {
    unsigned long long s = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += ds.warp_tile[i][w];
    ds.tile_tot[i] = s;
  }
  __syncthreads();
  if (tid == 0) {
    unsigned long long s = 0;
    for (int i = 0; i < nt; ++i) s += ds.tile_tot[i];
    ds.cta_total = s;
  }
}

// Cluster-wide exclusive prefix of the CTA totals (all CTAs call it).  Thread
// 0 of each CTA stores its total into slot [pass & 1][rank] of every CTA's
// shared memory with an asynchronous remote store that completes 8 bytes on
// that CTA's barrier xbar[pass & 1]; it expects kG * 8 bytes on its own and
// waits (bounded) for them, then reads its own copy: no cluster-wide barrier
// and no remote load on the path.  A slot and its barrier are used again two
// passes later: a CTA reaches that pass only after every CTA's store of the
// pass in between, which each CTA makes only after reading this pass's slots.
// A wait that gives up marks the CTA lost (its sums are not to be trusted).
__device__ __forceinline__ void draw_exchange(DrawSmem &ds, cg::cluster_group &cluster,
                                              int pass) {
  if (threadIdx.x == 0) {
    const unsigned rank = cluster.block_rank();
    uint64_t *bar = &ds.xbar[pass & 1];
    mbar_arrive_expect_tx(bar, (uint32_t)(kG * sizeof(unsigned long long)));
    const uint32_t slot = smem_addr(&ds.totals[pass & 1][rank]);
    const uint32_t b = smem_addr(bar);
    const unsigned long long s = ds.cta_total;
#pragma unroll
    for (unsigned r = 0; r < (unsigned)kG; ++r)
      st_async_u64(cluster_addr(slot, r), s, cluster_addr(b, r));
    if (!mbar_wait_cluster_bounded(bar, (uint32_t)((pass >> 1) & 1))) ds.lost = 1;
    unsigned long long pre = 0, tot = 0;
#pragma unroll
    for (unsigned r = 0; r < (unsigned)kG; ++r) {
      const unsigned long long x = ds.totals[pass & 1][r];
      if (r < rank) pre += x;
      tot += x;
    }
    ds.prefix = pre;
    ds.Z = tot;
    ds.Zf = __ull2float_rn(tot) * (float)kFixedUnit;
  }
  __syncthreads();
}

// If the crossing of `target` lies in this CTA's slice, find the smallest v
// with C_v > target (C: prefix sums of the last pass's weights).  Returns v
// in every thread of that CTA, -1 elsewhere.
template <int DT>
__device__ __forceinline__ int draw_search(DrawSmem &ds, const DrawRow &r,
                                           unsigned long long target) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nt = slice_tiles(r);
  const unsigned long long pre = ds.prefix;
  const bool mine = (pre <= target) && (target - pre < ds.cta_total);
  if (!mine) return -1;  // uniform across the CTA
  if (tid == 0) {
    unsigned long long run = pre;
    int tile = nt - 1;
    for (int i = 0; i < nt; ++i) {
      if (target - run < ds.tile_tot[i]) {
        tile = i;
        break;
      }
      run += ds.tile_tot[i];
    }
    ds.tile = tile;
    ds.base = run;
    ds.found = -1;
  }
  __syncthreads();
  const int e = r.v0 + ds.tile * kTile + tid * kPerThread;
  Raw16<DT> x;
  float w[kPerThread];
  load_raw<DT>(r, e, x);
  const unsigned long long f = weights16<DT>(r, x, e, w);
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
      if (excl + to_fixed40(run) > target) {
        v = e + k;
        break;
      }
    }
    ds.found = v;
  }
  __syncthreads();
  return ds.found;
}

// This cluster rank's slice of a row of V elements: a multiple of 16 elements
// long (so every slice starts 32-byte aligned relative to the row).
__device__ __forceinline__ void cta_slice(int V, int rank, int &v0, int &v1) {
  int L = (V + kG - 1) / kG;
  L = (L + 15) & ~15;
  v0 = min(V, rank * L);
  v1 = min(V, v0 + L);
}

__host__ __device__ inline int slice_capacity(int V) {
  int L = (V + kG - 1) / kG;
  return (L + 15) & ~15;
}

}  // namespace fin
}  // namespace specdec
