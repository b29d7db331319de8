// Row statistics of the target logits: the "parallel verification" step of
// speculative sampling ("Chapter 15: Decoding acceleration", section 15.1.2,
// step 2), which scores every drafted position in one pass.  For each row and
// each split of the vocabulary the kernel produces
//     m = max_v l_v,   s = sum_v 2^((l_v - m) c),   c = log2(e) / T,
// and the position of the first maximum, so that p(x) = 2^((l_x - M) c) / S
// after a merge over splits.  This pass reads every logit exactly once and is
// the HBM-bound part of the verify step.
//
// Structure (GB300): a persistent grid of 2 CTAs per SM walks the (row, split)
// work items round robin.  In each CTA one producer thread streams the 16-byte
// aligned interior of each split into a ring of 6 x 16 KB shared-memory
// stages with 1-D bulk TMA copies (cp.async.bulk) that complete on "full"
// mbarriers; 8 consumer warps read the stages with 128-bit shared loads,
// update an online (max, sum) per thread and release each stage on an "empty"
// mbarrier.  The few unaligned elements at the ends of a split are read with
// plain loads.  Every wait is bounded in time.
#include <cfloat>

#include "common.cuh"

namespace specdec {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kStageBytes = 16384;
constexpr int kStages = 6;
constexpr int kVecPerThread = kStageBytes / 16 / kConsumers;  // 4
static_assert(kVecPerThread * kConsumers * 16 == kStageBytes, "stage split");

struct StatsSmem {
  alignas(128) uint8_t stage[kStages][kStageBytes];
  alignas(8) uint64_t full[kStages];
  alignas(8) uint64_t empty[kStages];
  float red_m[2][kConsumerWarps];
  float red_s[2][kConsumerWarps];
  int red_a[2][kConsumerWarps];
  volatile int abort_flag;
};

struct ItemGeom {
  long long row;
  int e0, e1;            // element range of the split
  int head_end;          // elements [e0, head_end) read with plain loads
  int tail_begin;        // elements [tail_begin, e1) read with plain loads
  const uint8_t *i0;     // 16-byte aligned interior [i0, i1) moved by TMA
  long long ibytes;
};

__device__ __forceinline__ ItemGeom item_geometry(const RowStatsParams &p, long long item,
                                                  int es) {
  ItemGeom g;
  g.row = item / p.P;
  const int split = (int)(item - g.row * p.P);
  g.e0 = split * p.chunk_elems;
  g.e1 = min(p.V, g.e0 + p.chunk_elems);
  const uint8_t *row_base =
      reinterpret_cast<const uint8_t *>(p.logits) + (size_t)g.row * (size_t)p.V * es;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(row_base) + (uintptr_t)g.e0 * es;
  const uintptr_t a1 = reinterpret_cast<uintptr_t>(row_base) + (uintptr_t)g.e1 * es;
  const uintptr_t i0 = (a0 + 15) & ~(uintptr_t)15;
  const uintptr_t i1 = a1 & ~(uintptr_t)15;
  if (i1 > i0) {
    g.i0 = reinterpret_cast<const uint8_t *>(i0);
    g.ibytes = (long long)(i1 - i0);
    g.head_end = g.e0 + (int)((i0 - a0) / es);
    g.tail_begin = g.e0 + (int)((i1 - a0) / es);
  } else {
    g.i0 = nullptr;
    g.ibytes = 0;
    g.head_end = g.e1;
    g.tail_begin = g.e1;
  }
  return g;
}

// ---- per-thread online statistics ----------------------------------------

struct Stat {
  float m;     // running max (never NaN)
  float mref;  // max(m, -FLT_MAX): exponent reference that keeps -inf - -inf out
  float s;
  int arg;
};

__device__ __forceinline__ void stat_raise(Stat &st, float vmax, float c, int arg) {
  // rescale the running sum to the new maximum
  st.s = st.s * ex2_approx((st.mref - vmax) * c);
  st.m = vmax;
  st.mref = fmaxf(vmax, -FLT_MAX);
  st.arg = arg;
}

__device__ __forceinline__ void stat_scalar(Stat &st, float x, float c, int idx) {
  if (x > st.m) stat_raise(st, x, c, idx);
  st.s += ex2_approx((x - st.mref) * c);
}

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ float vec_max_bf16(const uint4 &v) {
  const uint32_t m = bf16x2_max(bf16x2_max(v.x, v.y), bf16x2_max(v.z, v.w));
  return fmaxf(bf16_lo(m), bf16_hi(m));
}

__device__ __forceinline__ float vec_max_f32(const uint4 &v) {
  return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
               fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
}

__device__ __forceinline__ float vec_sum_bf16(const uint4 &v, float mref, float c) {
  const float e0 = ex2_approx((bf16_lo(v.x) - mref) * c);
  const float e1 = ex2_approx((bf16_hi(v.x) - mref) * c);
  const float e2 = ex2_approx((bf16_lo(v.y) - mref) * c);
  const float e3 = ex2_approx((bf16_hi(v.y) - mref) * c);
  const float e4 = ex2_approx((bf16_lo(v.z) - mref) * c);
  const float e5 = ex2_approx((bf16_hi(v.z) - mref) * c);
  const float e6 = ex2_approx((bf16_lo(v.w) - mref) * c);
  const float e7 = ex2_approx((bf16_hi(v.w) - mref) * c);
  return ((e0 + e1) + (e2 + e3)) + ((e4 + e5) + (e6 + e7));
}

__device__ __forceinline__ float vec_sum_f32(const uint4 &v, float mref, float c) {
  const float e0 = ex2_approx((__uint_as_float(v.x) - mref) * c);
  const float e1 = ex2_approx((__uint_as_float(v.y) - mref) * c);
  const float e2 = ex2_approx((__uint_as_float(v.z) - mref) * c);
  const float e3 = ex2_approx((__uint_as_float(v.w) - mref) * c);
  return (e0 + e1) + (e2 + e3);
}

// One stage: this thread's (up to) four 16-byte vectors.
template <int DT>
__device__ __forceinline__ void stat_stage(Stat &st, const uint8_t *stage, int nvec,
                                           int first_elem, float c, int tid) {
  constexpr int kElemsPerVec = (DT == SPECDEC_F32) ? 4 : 8;
  uint4 v[kVecPerThread];
  float vm[kVecPerThread];
  float smax = -INFINITY;
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const int j = tid + k * kConsumers;
    if (j < nvec) {
      v[k] = *reinterpret_cast<const uint4 *>(stage + (size_t)j * 16);
      vm[k] = (DT == SPECDEC_F32) ? vec_max_f32(v[k]) : vec_max_bf16(v[k]);
    } else {
      v[k] = make_uint4(0, 0, 0, 0);
      vm[k] = -INFINITY;
    }
    smax = fmaxf(smax, vm[k]);
  }
  if (smax > st.m) {
    int first = 0;
#pragma unroll
    for (int k = kVecPerThread - 1; k >= 0; --k)
      if (vm[k] == smax) first = k;
    stat_raise(st, smax, c, first_elem + (tid + first * kConsumers) * kElemsPerVec);
  }
  float acc = 0.0f;
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const int j = tid + k * kConsumers;
    if (j < nvec)
      acc += (DT == SPECDEC_F32) ? vec_sum_f32(v[k], st.mref, c) : vec_sum_bf16(v[k], st.mref, c);
  }
  st.s += acc;
}

// merge two partial statistics of the same row
__device__ __forceinline__ void stat_merge(float &m, float &s, int &a, float m2, float s2, int a2,
                                           float c) {
  const float M = fmaxf(m, m2);
  const float Mref = fmaxf(M, -FLT_MAX);
  const float f1 = ex2_approx((fmaxf(m, -FLT_MAX) - Mref) * c);
  const float f2 = ex2_approx((fmaxf(m2, -FLT_MAX) - Mref) * c);
  const int an = (m > m2) ? a : (m2 > m) ? a2 : min(a, a2);
  s = s * f1 + s2 * f2;
  m = M;
  a = an;
}

__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 2) row_stats_kernel(const RowStatsParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  StatsSmem &sm = *reinterpret_cast<StatsSmem *>(smem_raw);
  constexpr int es = (DT == SPECDEC_F32) ? 4 : 2;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], kConsumerWarps);
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      uint32_t gstage = 0;
      for (long long item = blockIdx.x; item < p.items; item += gridDim.x) {
        const ItemGeom g = item_geometry(p, item, es);
        for (long long off = 0; off < g.ibytes; off += kStageBytes) {
          const uint32_t bytes = (uint32_t)min((long long)kStageBytes, g.ibytes - off);
          const uint32_t slot = gstage % kStages;
          const uint32_t use = gstage / kStages;
          if (use > 0 && !mbar_wait_bounded(&sm.empty[slot], (use - 1) & 1)) {
            sm.abort_flag = 1;
            return;
          }
          if (sm.abort_flag) return;
          mbar_arrive_expect_tx(&sm.full[slot], bytes);
          bulk_copy_g2s(sm.stage[slot], g.i0 + off, bytes, &sm.full[slot]);
          ++gstage;
        }
      }
    }
    return;
  }

  // ------------------------------ consumers -------------------------------
  uint32_t gstage = 0;
  int par = 0;
  for (long long item = blockIdx.x; item < p.items; item += gridDim.x) {
    const ItemGeom g = item_geometry(p, item, es);
    const long long b = g.row / p.R;
    const float c = temperature_scale(__ldg(p.temperature + b));
    Stat st;
    st.m = -INFINITY;
    st.mref = -FLT_MAX;
    st.s = 0.0f;
    st.arg = 0x7FFFFFFF;
    const long long row_off = g.row * (long long)p.V;

    for (int e = g.e0 + tid; e < g.head_end; e += kConsumers)
      stat_scalar(st, load_elem(p.logits, DT, row_off + e), c, e);

    for (long long off = 0; off < g.ibytes; off += kStageBytes) {
      const int bytes = (int)min((long long)kStageBytes, g.ibytes - off);
      const uint32_t slot = gstage % kStages;
      const uint32_t use = gstage / kStages;
      bool ok = !sm.abort_flag && mbar_wait_bounded(&sm.full[slot], use & 1);
      if (!ok) sm.abort_flag = 1;
      if (ok) stat_stage<DT>(st, sm.stage[slot], bytes / 16, g.head_end + (int)(off / es), c, tid);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[slot]);
      ++gstage;
    }

    for (int e = g.tail_begin + tid; e < g.e1; e += kConsumers)
      stat_scalar(st, load_elem(p.logits, DT, row_off + e), c, e);

    // block merge of the per-thread statistics
    float m = st.m, s = st.s;
    int a = st.arg;
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, d);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, d);
      const int a2 = __shfl_xor_sync(0xffffffffu, a, d);
      stat_merge(m, s, a, m2, s2, a2, c);
    }
    if (lane == 0) {
      sm.red_m[par][warp] = m;
      sm.red_s[par][warp] = s;
      sm.red_a[par][warp] = a;
    }
    consumer_bar();
    if (warp == 0) {
      if (lane < kConsumerWarps) {
        m = sm.red_m[par][lane];
        s = sm.red_s[par][lane];
        a = sm.red_a[par][lane];
      } else {
        m = -INFINITY;
        s = 0.0f;
        a = 0x7FFFFFFF;
      }
#pragma unroll
      for (int d = kConsumerWarps / 2; d >= 1; d >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, d);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, d);
        const int a2 = __shfl_xor_sync(0xffffffffu, a, d);
        stat_merge(m, s, a, m2, s2, a2, c);
      }
      if (lane == 0) {
        RowPartial r;
        r.m = m;
        r.s = s;
        r.arg = a;
        r.flags = sm.abort_flag ? SPECDEC_ROW_INTERNAL : 0;
        p.part[item] = r;
      }
    }
    par ^= 1;
  }
}

int g_sm_count[64];

int sm_count_of_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

template <int DT>
cudaError_t launch_dt(const RowStatsParams &p, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const int smem = (int)sizeof(StatsSmem);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    err = cudaFuncSetAttribute(row_stats_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               smem);
    if (err != cudaSuccess) return err;
    attr_set[dev] = true;
  }
  long long grid = 2LL * sm_count_of_current_device();
  if (grid > p.items) grid = p.items;
  row_stats_kernel<DT><<<(unsigned)grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_row_stats(const RowStatsParams &p, cudaStream_t stream) {
  if (p.items <= 0) return cudaSuccess;
  return p.dtype == SPECDEC_F32 ? launch_dt<SPECDEC_F32>(p, stream)
                                : launch_dt<SPECDEC_BF16>(p, stream);
}

}  // namespace specdec
