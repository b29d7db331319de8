// Quantities the adaptive policies of "Chapter 15: Decoding acceleration"
// read off a verify step, from the stats pass's stage partials:
//   * the entropy -sum p ln p of every target row (the adaptive draft length
//     of the multi-token-prediction section keys on it);
//   * the log-probability of the emitted path, sum_i ln p(x_i | prefix_i)
//     (the path-probability passage of the tree section).
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

}  // namespace

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
