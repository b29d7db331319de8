// Quantities the adaptive policies of "Chapter 15: Decoding acceleration"
// read off a verify step, from the stats pass's stage partials:
//   * the entropy -sum p ln p of every target row (the adaptive draft length
//     of the multi-token-prediction section keys on it);
//   * the log-probability of the emitted path, sum_i ln p(x_i | prefix_i)
//     (the path-probability passage of the tree section);
//   * the acceptance rate sum_v min(p_i(v), q_i(v)) of every drafted row
//     (Lemma 1 of section 15.1.2; the sliding-window draft length averages
//     it), a second pass over the drafted logits and q rows.
// Each stage partial holds (m, s = sum 2^((l - m) c), a = sum 2^((l - m) c)
// (l - m)) for non-greedy rows; merging to the row max M gives S and
// A = sum_v e_v (l_v - M) with e_v = exp((l_v - M) / T), and then
//     H = ln S - A / (T S),      ln p(x) = (l_x - M) / T - ln S.
// Every term of A is <= 0, so neither formula cancels.  One warp per row
// (entropy) or per request (path).
#include "common.cuh"

namespace specdec {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct RowMoments {
  float M, S, A;
  int arg, flags;
};

// Merge of a row's stage partials by one warp, keeping A (the partial's
// `arg` field holds a's float bits for non-greedy rows, the first arg-max
// for greedy ones).
__device__ __forceinline__ RowMoments warp_moments(const RowPartial *part, long long row, int spr,
                                                   float c, bool greedy, int lane) {
  const RowPartial *pr = part + row * (long long)spr;
  float m = -INFINITY, s = 0.0f, a = 0.0f;
  int arg = 0x7FFFFFFF, fl = 0;
  for (int j = lane; j < spr; j += 32) {
    const RowPartial x = pr[j];
    fl |= x.flags;
    const float a2 = greedy ? 0.0f : __int_as_float(x.arg);  // NaN without the entropy sums
    if (x.m == -INFINITY) continue;
    if (m == -INFINITY) {
      m = x.m;
      s = x.s;
      a = a2;
      arg = x.arg;
      continue;
    }
    const float M = fmax_nan(m, x.m);
    const float f1 = ex2_approx((m - M) * c), f2 = ex2_approx((x.m - M) * c);
    a = f1 * (a + (m - M) * s) + f2 * (a2 + (x.m - M) * x.s);
    s = s * f1 + x.s * f2;
    arg = (m > x.m) ? arg : (x.m > m) ? x.arg : min(arg, x.arg);
    m = M;
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, d);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, d);
    const float a2 = __shfl_xor_sync(0xffffffffu, a, d);
    const int g2 = __shfl_xor_sync(0xffffffffu, arg, d);
    fl |= __shfl_xor_sync(0xffffffffu, fl, d);
    if (m2 == -INFINITY) continue;
    if (m == -INFINITY) {
      m = m2;
      s = s2;
      a = a2;
      arg = g2;
      continue;
    }
    const float M = fmax_nan(m, m2);
    const float f1 = ex2_approx((m - M) * c), f2 = ex2_approx((m2 - M) * c);
    // symmetric in the two operands, so both lanes of a pair agree
    a = f1 * (a + (m - M) * s) + f2 * (a2 + (m2 - M) * s2);
    s = s * f1 + s2 * f2;
    arg = (m > m2) ? arg : (m2 > m) ? g2 : min(arg, g2);
    m = M;
  }
  RowMoments r;
  r.M = m;
  r.S = s;
  r.A = a;
  r.arg = arg;
  r.flags = fl;
  return r;
}

__device__ __forceinline__ bool usable(const RowMoments &r) {
  return r.flags == 0 && r.M > -INFINITY && r.M <= kMaxLogit && r.S > 0.0f && r.S < INFINITY;
}

__global__ void __launch_bounds__(kThreads) row_entropy_kernel(const RowPartial *part,
                                                               const float *temperature, int R,
                                                               long long rows, int spr,
                                                               float *entropy) {
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float T = __ldg(temperature + row / R);
  const bool greedy = (T == 0.0f);
  const RowMoments r = warp_moments(part, row, spr, temperature_scale(T), greedy, lane);
  if (lane != 0) return;
  float h;
  if (!temperature_valid(T) || !usable(r)) h = __int_as_float(0x7fc00000);
  else if (greedy) h = 0.0f;
  else h = logf(r.S) - r.A / (T * r.S);
  entropy[row] = h;
}

__global__ void __launch_bounds__(kThreads) path_logprob_kernel(const PathLogprobParams p) {
  const int lane = threadIdx.x & 31;
  const long long b = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (b >= p.B) return;
  const float T = __ldg(p.temperature + b);
  const bool greedy = (T == 0.0f);
  const float c = temperature_scale(T);
  const int k = __ldg(p.n_accepted + b);
  bool bad = (p.row_status && __ldg(p.row_status + b) != 0) || !temperature_valid(T) || k < 0 ||
             k >= p.path_len;
  float sum = 0.0f;
  for (int j = 0; !bad && j <= k; ++j) {
    const int row = p.path_nodes ? __ldg(p.path_nodes + b * p.path_len + j) : j;
    const int tok = __ldg(p.out_tokens + b * p.path_len + j);
    if (row < 0 || row >= p.R || tok < 0 || tok >= p.V) {
      bad = true;
      break;
    }
    const RowMoments r = warp_moments(p.part, b * p.R + row, p.spr, c, greedy, lane);
    if (!usable(r)) {
      bad = true;
      break;
    }
    if (greedy) {
      if (tok != r.arg) sum = -INFINITY;
    } else {
      const float lx = load_elem(p.logits, p.dtype, (b * p.R + row) * (long long)p.V + tok);
      sum += (lx - r.M) / T - logf(r.S);
    }
  }
  if (lane == 0) p.logprob[b] = bad ? __int_as_float(0x7fc00000) : sum;
}

// alpha of drafted row j = b * gamma + i: sum_v min(p(v), q(v)), p from the
// merged statistics of target row (b, i), q row (b, i) as stored.  One CTA
// per drafted row streams both rows once (16-byte loads, kAlphaU vectors of
// each in flight per thread), sums in float per thread and in double over
// the CTA.  Greedy rows: p is one-hot at the first arg-max, alpha = min(1,
// q(argmax)).  NaN for an invalid temperature or an unusable row.
constexpr int kAlphaU = 4;

template <int DT>
__device__ __forceinline__ float2 elem_pair(const uint4 &lv, const uint4 &qv, int k) {
  // element k of a 16-byte vector of logits and of q, as float32
  const uint32_t lw[4] = {lv.x, lv.y, lv.z, lv.w};
  const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
  if (DT == SPECDEC_F32) return make_float2(__uint_as_float(lw[k]), __uint_as_float(qw[k]));
  const uint32_t l = lw[k >> 1], q = qw[k >> 1];
  return (k & 1) ? make_float2(bf16_hi(l), bf16_hi(q)) : make_float2(bf16_lo(l), bf16_lo(q));
}

__device__ __forceinline__ float min_pq(float l, float q, float M, float c, float inv_s) {
  const float pv = ex2_approx((l - M) * c) * inv_s;
  return (pv < q) ? pv : q;  // NaN q propagates, as in a plain sum of min(p, q)
}

template <int DT>
__global__ void __launch_bounds__(kThreads) row_alpha_kernel(const void *logits, const void *q,
                                                             const RowPartial *part,
                                                             const float *temperature, int gamma,
                                                             int V, int spr, float *alpha) {
  __shared__ float sh[4];
  __shared__ double red[kWarps];
  constexpr int es = (DT == SPECDEC_F32) ? 4 : 2;
  constexpr int kN = 16 / es;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long j = blockIdx.x;
  const long long b = j / gamma;
  const int i = (int)(j - b * gamma);
  const long long row = b * (gamma + 1) + i;
  const float T = __ldg(temperature + b);
  const bool greedy = (T == 0.0f);
  const float c = temperature_scale(T);
  if (warp == 0) {
    const RowMoments r = warp_moments(part, row, spr, c, greedy, lane);
    if (lane == 0) {
      const bool ok = temperature_valid(T) && usable(r);
      sh[0] = r.M;
      sh[1] = 1.0f / r.S;
      sh[2] = ok ? 1.0f : 0.0f;
      sh[3] = __int_as_float(r.arg);
    }
  }
  __syncthreads();
  if (sh[2] == 0.0f) {
    if (tid == 0) alpha[j] = __int_as_float(0x7fc00000);
    return;
  }
  const uint8_t *lrow = reinterpret_cast<const uint8_t *>(logits) + (size_t)row * V * es;
  const uint8_t *qrow = reinterpret_cast<const uint8_t *>(q) + (size_t)j * V * es;
  if (greedy) {
    if (tid == 0) {
      const float qa = load_elem(qrow, DT, __float_as_int(sh[3]));
      alpha[j] = (1.0f < qa) ? 1.0f : qa;
    }
    return;
  }
  const float M = sh[0], inv_s = sh[1];
  float acc = 0.0f;
  int v_done = 0;  // elements covered by the vector loop
  if (((reinterpret_cast<uintptr_t>(lrow) | reinterpret_cast<uintptr_t>(qrow)) & 15) == 0) {
    const int nvec = V / kN;
    const uint4 *l4 = reinterpret_cast<const uint4 *>(lrow);
    const uint4 *q4 = reinterpret_cast<const uint4 *>(qrow);
    for (int base = 0; base < nvec; base += kThreads * kAlphaU) {
      uint4 lv[kAlphaU], qv[kAlphaU];
#pragma unroll
      for (int u = 0; u < kAlphaU; ++u) {
        const int vi = base + u * kThreads + tid;
        lv[u] = (vi < nvec) ? __ldg(l4 + vi) : make_uint4(0u, 0u, 0u, 0u);
        qv[u] = (vi < nvec) ? __ldg(q4 + vi) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kAlphaU; ++u) {
        if (base + u * kThreads + tid >= nvec) continue;
#pragma unroll
        for (int k = 0; k < kN; ++k) {
          const float2 x = elem_pair<DT>(lv[u], qv[u], k);
          acc += min_pq(x.x, x.y, M, c, inv_s);
        }
      }
    }
    v_done = nvec * kN;
  }
  for (int v = v_done + tid; v < V; v += kThreads)
    acc += min_pq(load_elem(lrow, DT, v), load_elem(qrow, DT, v), M, c, inv_s);
  double d = (double)acc;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
  if (lane == 0) red[warp] = d;
  __syncthreads();
  if (tid == 0) {
    double t = 0.0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t += red[w];
    alpha[j] = (float)t;
  }
}

}  // namespace

cudaError_t launch_row_alpha(const void *logits, const void *q, int dtype, const RowPartial *part,
                             const float *temperature, int B, int gamma, int V, int spr,
                             float *alpha, cudaStream_t stream) {
  const long long rows = (long long)B * gamma;
  if (rows <= 0) return cudaSuccess;
  if (dtype == SPECDEC_F32)
    row_alpha_kernel<SPECDEC_F32><<<(unsigned)rows, kThreads, 0, stream>>>(logits, q, part, temperature,
                                                                          gamma, V, spr, alpha);
  else
    row_alpha_kernel<SPECDEC_BF16><<<(unsigned)rows, kThreads, 0, stream>>>(logits, q, part, temperature,
                                                                           gamma, V, spr, alpha);
  return cudaGetLastError();
}

cudaError_t launch_row_entropy(const RowPartial *part, const float *temperature, int B, int R,
                               int spr, float *entropy, cudaStream_t stream) {
  const long long rows = (long long)B * R;
  if (rows <= 0) return cudaSuccess;
  const unsigned grid = (unsigned)((rows + kWarps - 1) / kWarps);
  row_entropy_kernel<<<grid, kThreads, 0, stream>>>(part, temperature, R, rows, spr, entropy);
  return cudaGetLastError();
}

cudaError_t launch_path_logprob(const PathLogprobParams &p, cudaStream_t stream) {
  if (p.B <= 0) return cudaSuccess;
  const unsigned grid = (unsigned)(((long long)p.B + kWarps - 1) / kWarps);
  path_logprob_kernel<<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace specdec
