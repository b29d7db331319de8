// Linear verify, phase 2: accept test with early stop and the final draw
// ("Chapter 15: Decoding acceleration", section 15.1.2 steps 3 and 4; the
// bonus draw from the last target row follows section 15.1.3's expected
// count (1 - a^(g+1)) / (1 - a) of emitted tokens per step).
//
// Three short kernels, each fully parallel, so that no request waits on a
// long chain of dependent steps:
//
// decide: one CTA per request.  Its warps merge the stage partials of the
//   request's rows in parallel; warp 0 takes the drafted tokens' logits and q
//   values the stats pass gathered, runs the accept test, finds the first
//   rejection k with a ballot and find-first-set, writes the accepted tokens
//   and counts, and leaves a decision record (k, M, S of the final row).
//   Greedy requests (T = 0) get their final token (the first arg-max) here.
//
// draw sums: one CTA per (request, 8192-element chunk of its final row).  With
//   e_v = 2^((l_v - M) c), the weights are max(0, e_v - S q_v) = S max(0, p - q)
//   after a rejection and e_v = S p for the bonus draw; each thread sums its 32
//   contiguous weights in float32, and the CTA adds the thread sums in 40-bit
//   fixed point into the chunk total.  Requests are taken in reverse order so
//   the rows the stats pass read last, still in L2, come first.
//
// draw search: one CTA per request.  An exclusive scan of the chunk totals
//   gives Z and the chunk holding U * Z; the CTA recomputes that chunk's thread
//   sums (the same arithmetic, the same order), scans them, and the thread
//   holding the crossing finds the token among its 32 weights.  Integer sums
//   make the crossing exact for the weights the kernels compute.
#include <cfloat>

#include "common.cuh"

namespace specdec {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPerT = 32;                  // contiguous elements per thread
constexpr int kChunk = kThreads * kPerT;   // elements per chunk (8192)
constexpr int kMaxRows = SPECDEC_MAX_GAMMA + 1;
static_assert(kChunk == SPECDEC_DRAW_CHUNK, "chunk size shared with the workspace layout");

struct RowStat {
  float M, S;
  int arg, flags;
};

// Merge of two stage partials (each sum is taken relative to its own max).
__device__ __forceinline__ void merge2(float &m, float &s, int &a, float m2, float s2, int a2,
                                       float c) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    a = a2;
    return;
  }
  const float M = fmax_nan(m, m2);
  const float f1 = ex2_approx((m - M) * c);
  const float f2 = ex2_approx((m2 - M) * c);
  a = (m > m2) ? a : (m2 > m) ? a2 : min(a, a2);
  s = s * f1 + s2 * f2;
  m = M;
}

__device__ __forceinline__ RowStat warp_merge_row(const RowPartial *part, long long row, int spr,
                                                  float c, int lane) {
  const RowPartial *pr = part + row * (long long)spr;
  float m = -INFINITY, s = 0.0f;
  int a = 0x7FFFFFFF, fl = 0;
  for (int j = lane; j < spr; j += 32) {
    const RowPartial x = pr[j];
    fl |= x.flags;
    merge2(m, s, a, x.m, x.s, x.arg, c);
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, d);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, d);
    const int a2 = __shfl_xor_sync(0xffffffffu, a, d);
    merge2(m, s, a, m2, s2, a2, c);
  }
  RowStat r;
  r.M = m;
  r.S = s;
  r.arg = a;
  r.flags = __reduce_or_sync(0xffffffffu, fl);
  return r;
}

__device__ __forceinline__ bool row_usable(const RowStat &r) {
  return r.M > -INFINITY && r.M <= kMaxLogit && r.S > 0.0f && r.S < INFINITY;
}

template <int DT>
__global__ void __launch_bounds__(kThreads) linear_decide_kernel(const LinearFinalizeParams p) {
  __shared__ RowStat rows[kMaxRows];
  const long long b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gamma = p.gamma, R = gamma + 1, V = p.V;

  const float T = __ldg(p.temperature + b);
  const bool greedy = (T == 0.0f);
  const float c = temperature_scale(T);

  int x = -1;
  float u = 0.0f;
  float2 g = make_float2(0.0f, 1.0f);
  if (warp == 0 && lane < gamma) {
    x = __ldg(p.tokens + b * gamma + lane);
    u = __ldg(p.uniforms + b * R + lane);
    if (x >= 0 && x < V) g = p.gather[b * R + lane];
  }
  for (int i = warp; i < R; i += kWarps) {
    const RowStat r = warp_merge_row(p.part, b * R + i, p.spr, c, lane);
    if (lane == 0) rows[i] = r;
  }
  __syncthreads();
  if (warp != 0) return;

  int status = temperature_valid(T) ? 0 : SPECDEC_ROW_BAD_TEMP;
  for (int i = lane; i < R; i += 32) {
    status |= rows[i].flags;
    if (!row_usable(rows[i])) status |= SPECDEC_ROW_NONFINITE;
  }
  bool acc = true;
  float pd = 0.0f;
  if (lane < gamma) {
    if (x < 0 || x >= V) {
      status |= SPECDEC_ROW_BAD_TOKEN;
    } else {
      const float lx = g.x, qx = g.y;
      if (!(qx > 0.0f) || qx == INFINITY) status |= SPECDEC_ROW_BAD_Q;
      if (greedy) {
        acc = (x == rows[lane].arg);
        pd = acc ? 1.0f : 0.0f;
      } else {
        pd = exp2f((lx - rows[lane].M) * c) / rows[lane].S;
        // u <= min(1, p/q)  <=>  u q <= p  for q > 0, u < 1 (exact products in float64)
        acc = ((double)u * (double)qx <= (double)pd);
      }
    }
  }
  status = __reduce_or_sync(0xffffffffu, status);
  const unsigned rej = __ballot_sync(0xffffffffu, lane < gamma && !acc);
  const int k = rej ? (__ffs(rej) - 1) : gamma;
  if (status) {
    for (int j = lane; j < R; j += 32) p.out_tokens[b * R + j] = -1;
    if (p.p_draft && lane < gamma) p.p_draft[b * gamma + lane] = __int_as_float(0x7fc00000);
  } else {
    for (int j = lane; j < R; j += 32) {
      if (j < k) p.out_tokens[b * R + j] = __ldg(p.tokens + b * gamma + j);
      else if (j > k) p.out_tokens[b * R + j] = -1;
    }
    if (p.p_draft && lane < gamma) p.p_draft[b * gamma + lane] = pd;
  }
  if (lane == 0) {
    p.n_accepted[b] = status ? 0 : k;
    p.is_bonus[b] = (uint8_t)(!status && k == gamma);
    p.row_status[b] = status;
    if (status) {
      p.final_token[b] = -1;
    } else if (greedy) {
      p.final_token[b] = rows[k].arg;
      p.out_tokens[b * R + k] = rows[k].arg;
    }
    LinearDecision d;
    d.k = k;
    d.status = status;
    d.greedy = greedy;
    d.M = rows[k].M;
    d.S = rows[k].S;
    d.c = c;
    d.pad[0] = d.pad[1] = 0;
    p.dec[b] = d;
  }
}

// ---------------------------------------------------------------------------
// the draw
// ---------------------------------------------------------------------------

struct Draw {
  const uint8_t *lrow, *qrow;
  float M, c, K;  // w_v = max(0, e_v - K q_v) (use_q) or e_v, e_v = 2^((l_v - M) c)
  int V;
  bool use_q, vec_ok;
};

template <int DT>
__device__ __forceinline__ Draw make_draw(const LinearFinalizeParams &p, long long b,
                                          const LinearDecision &d) {
  constexpr int es = (DT == SPECDEC_F32) ? 4 : 2;
  const int R = p.gamma + 1;
  Draw w;
  w.lrow = reinterpret_cast<const uint8_t *>(p.logits) + (size_t)(b * R + d.k) * p.V * es;
  w.qrow = (d.k < p.gamma)
               ? reinterpret_cast<const uint8_t *>(p.q) + (size_t)(b * p.gamma + d.k) * p.V * es
               : w.lrow;
  w.M = d.M;
  w.c = d.c;
  w.K = d.S;
  w.V = p.V;
  w.use_q = d.k < p.gamma;
  w.vec_ok = ((reinterpret_cast<uintptr_t>(w.lrow) & 15) == 0) &&
             ((reinterpret_cast<uintptr_t>(w.qrow) & 15) == 0);
  return w;
}

template <int DT>
__device__ __forceinline__ float bits_to_f(uint32_t v) {
  return (DT == SPECDEC_F32) ? __uint_as_float(v) : __uint_as_float(v << 16);
}

// The 32 weights of the elements [e, e + 32) (zero at and beyond V) and their
// float32 sum in index order, as 40-bit fixed point.
template <int DT>
__device__ __forceinline__ unsigned long long thread_weights(const Draw &w, int e, float out[kPerT]) {
  constexpr int es = (DT == SPECDEC_F32) ? 4 : 2;
  constexpr int nvec = kPerT * es / 16;
  uint32_t lw[kPerT], qw[kPerT];
  if (w.vec_ok && e + kPerT <= w.V) {
    uint4 lv[nvec], qv[nvec];
    const uint4 *lp = reinterpret_cast<const uint4 *>(w.lrow + (size_t)e * es);
#pragma unroll
    for (int k = 0; k < nvec; ++k) lv[k] = __ldg(lp + k);
    if (w.use_q) {
      const uint4 *qp = reinterpret_cast<const uint4 *>(w.qrow + (size_t)e * es);
#pragma unroll
      for (int k = 0; k < nvec; ++k) qv[k] = __ldg(qp + k);
    }
#pragma unroll
    for (int k = 0; k < nvec; ++k) {
      const uint32_t a[4] = {lv[k].x, lv[k].y, lv[k].z, lv[k].w};
      const uint32_t bq[4] = {w.use_q ? qv[k].x : 0u, w.use_q ? qv[k].y : 0u,
                              w.use_q ? qv[k].z : 0u, w.use_q ? qv[k].w : 0u};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        if (DT == SPECDEC_F32) {
          lw[4 * k + t] = a[t];
          qw[4 * k + t] = bq[t];
        } else {
          lw[8 * k + 2 * t] = a[t] & 0xFFFFu;
          lw[8 * k + 2 * t + 1] = a[t] >> 16;
          qw[8 * k + 2 * t] = bq[t] & 0xFFFFu;
          qw[8 * k + 2 * t + 1] = bq[t] >> 16;
        }
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < kPerT; ++k) {
      const int v = e + k;
      const bool in = v < w.V;
      if (DT == SPECDEC_F32) {
        lw[k] = in ? __float_as_uint(__ldg(reinterpret_cast<const float *>(w.lrow) + v)) : 0xFF800000u;
        qw[k] = (in && w.use_q) ? __float_as_uint(__ldg(reinterpret_cast<const float *>(w.qrow) + v)) : 0u;
      } else {
        lw[k] = in ? (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(w.lrow) + v) : 0xFF80u;
        qw[k] = (in && w.use_q) ? (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(w.qrow) + v) : 0u;
      }
    }
  }
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < kPerT; ++k) {
    const float ev = ex2_approx((bits_to_f<DT>(lw[k]) - w.M) * w.c);
    const float x = w.use_q ? fmaxf(fmaf(-w.K, bits_to_f<DT>(qw[k]), ev), 0.0f) : ev;
    out[k] = (e + k < w.V) ? x : 0.0f;
    s += out[k];
  }
  return to_fixed40(s);
}

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v,
                                                            unsigned long long *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v += shfl_xor_u64(v, d);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  unsigned long long s = 0;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) s += red[i];
  return s;
}

// Exclusive block scan of one u64 per thread; also returns the block total.
__device__ __forceinline__ unsigned long long block_exscan_u64(unsigned long long v,
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
  for (int i = 0; i < kWarps; ++i) {
    if (i < warp) pre += red[i];
    tot += red[i];
  }
  total = tot;
  return pre + inc - v;
}

template <int DT>
__global__ void __launch_bounds__(kThreads) linear_draw_sums_kernel(const LinearFinalizeParams p) {
  __shared__ unsigned long long red[kWarps];
  const long long b = (long long)p.B - 1 - blockIdx.x / p.nchunk;
  const int chunk = (int)(blockIdx.x % p.nchunk);
  const LinearDecision d = p.dec[b];
  if (d.status || d.greedy) return;
  const Draw w = make_draw<DT>(p, b, d);
  float out[kPerT];
  const unsigned long long f = thread_weights<DT>(w, chunk * kChunk + threadIdx.x * kPerT, out);
  const unsigned long long tot = block_sum_u64(f, red);
  if (threadIdx.x == 0) p.chunk_tot[b * p.nchunk + chunk] = tot;
}

template <int DT>
__global__ void __launch_bounds__(kThreads) linear_draw_search_kernel(const LinearFinalizeParams p) {
  __shared__ unsigned long long red[kWarps];
  __shared__ unsigned long long s_base;
  __shared__ int s_chunk;
  const long long b = blockIdx.x;
  const int tid = threadIdx.x;
  const LinearDecision d = p.dec[b];
  if (d.status || d.greedy) return;
  Draw w = make_draw<DT>(p, b, d);
  const int nch = p.nchunk;
  float out[kPerT];

  // chunk totals (recomputed with the target row's weights if the residual is empty)
  unsigned long long mine = (tid < nch) ? p.chunk_tot[b * nch + tid] : 0ull;
  unsigned long long Z;
  unsigned long long pre = block_exscan_u64(mine, red, Z);
  if (Z == 0 && w.use_q) {
    // residual mass 0 (only by rounding): draw from p itself
    w.use_q = false;
    __syncthreads();
    for (int ch = 0; ch < nch; ++ch) {
      const unsigned long long f = thread_weights<DT>(w, ch * kChunk + tid * kPerT, out);
      const unsigned long long t = block_sum_u64(f, red);
      if (tid == ch) mine = t;
      __syncthreads();
    }
    pre = block_exscan_u64(mine, red, Z);
  }
  const float U = __ldg(p.uniforms + b * (p.gamma + 1) + p.gamma);
  const unsigned long long target = uniform_target(U, Z);
  if (tid == 0) s_chunk = -1;
  __syncthreads();
  if (tid < nch && pre <= target && target - pre < mine) {
    s_chunk = tid;
    s_base = pre;
  }
  __syncthreads();
  const int ch = s_chunk;
  if (ch < 0) return;  // no weight at all: unreachable for a usable row
  const unsigned long long base = s_base;
  const int e = ch * kChunk + tid * kPerT;
  const unsigned long long f = thread_weights<DT>(w, e, out);
  __syncthreads();
  unsigned long long ctot;
  const unsigned long long excl = base + block_exscan_u64(f, red, ctot);
  if (excl <= target && target - excl < f) {
    float run = 0.0f;
    int v = e + kPerT - 1;
#pragma unroll
    for (int k = 0; k < kPerT; ++k) {
      run += out[k];
      if (excl + to_fixed40(run) > target) {
        v = e + k;
        break;
      }
    }
    p.final_token[b] = v;
    p.out_tokens[b * (p.gamma + 1) + d.k] = v;
  }
}

template <int DT>
cudaError_t launch_dt(const LinearFinalizeParams &p, cudaStream_t stream) {
  linear_decide_kernel<DT><<<(unsigned)p.B, kThreads, 0, stream>>>(p);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  linear_draw_sums_kernel<DT><<<(unsigned)((long long)p.B * p.nchunk), kThreads, 0, stream>>>(p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  linear_draw_search_kernel<DT><<<(unsigned)p.B, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_linear_finalize(const LinearFinalizeParams &p, cudaStream_t stream) {
  if (p.B <= 0) return cudaSuccess;
  return p.dtype == SPECDEC_F32 ? launch_dt<SPECDEC_F32>(p, stream)
                                : launch_dt<SPECDEC_BF16>(p, stream);
}

}  // namespace specdec
