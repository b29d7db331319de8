// Linear verify with the top-k truncated residual, phase 2 (the approximate
// mode of specdec_verify_linear_topk): the implementation note of "Chapter
// 15: Decoding acceleration", section 15.1.2, precomputes the residual
// max(0, p - q) on the top-k candidates instead of the whole vocabulary.
// The accept test and the bonus draw are exact; a rejected position's token
// is drawn from the residual restricted to the k most probable tokens of p
// (ties to the lower index), in index order.
#include <cstring>
#include <cuda_bf16.h>

#include "linear_decision.cuh"

namespace specdec {

using lindec::request_decision;
using namespace drawc;

namespace {


// Candidate selection of the top-k residual: the K largest logits of the
// rejected row (ties to the lower index), in index order.
//
// Fast path, one pass over the row: a threshold estimated from a strided
// sample of at most kSample keys (the key with about 2K row elements above
// it), then every element at or above it kept in shared memory, each warp
// appending in index order to its own region for its contiguous segment of
// the row, and the exact K-th largest found among the kept ones.  A sample
// that keeps fewer than K, or overflows a region, is taken again at another
// rank; rows no rank serves (long runs of equal logits) take the full radix
// select over the row, with the same per-warp segments so that the digit
// counts give each warp its output offset.
// One CTA of 512 threads per request (16 warps; at most 64 registers, so two
// CTAs share an SM and a B=256 batch runs in one wave): the phases are
// latency-bound, and more warps per request hide more of it.  These names
// shadow the 256-thread ones of the other draw kernels.
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

// Block reductions of this kernel's 16 warps (two scratch buffers used in
// turn, as for the other kernels).
struct Red {
  unsigned long long *buf;  // [2][kWarps]
  int phase;
  __device__ __forceinline__ unsigned long long *next() {
    unsigned long long *r = buf + phase * kWarps;
    phase ^= 1;
    return r;
  }
};

__device__ __forceinline__ unsigned long long block_exscan_u64(unsigned long long v, Red &rr,
                                                               unsigned long long &total) {
  unsigned long long *red = rr.next();
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

constexpr int kU = 8;                   // 16-byte vectors in flight per lane
constexpr int kUF = 4;                  // the same in the one-pass filter (measured faster
                                        // than 2 or 8 with 512 threads)
constexpr int kUB = 8;                  // the same in the bonus draw
constexpr int kCap = 4096;              // elements the filter may keep
constexpr int kReg = kCap / kWarps;     // per warp
constexpr int kSample = 4096;           // keys of the threshold sample (at most)
constexpr int kTries = 3;               // sample ranks tried before the full select

struct Smem {
  lindec::DecisionSmem d;
  union {
    unsigned int hist[kWarps][256];     // full select: per-warp digit counts
    uint32_t key[kCap];                 // fast path: sampled keys, then kept keys by region
  } u;
  int cidx[kCap];                       // fast path: kept indices by region
  unsigned int h[256];                  // digit counts of the shared-memory selections
  unsigned int above[kWarps];           // per warp: keys above the threshold (so far)
  unsigned int ties[kWarps];            // per warp: keys equal to the threshold
  unsigned int out_off[kWarps];         // per warp: first output slot
  unsigned int tie_off[kWarps];         // per warp: rank of its first tie
  unsigned int nw[kWarps];              // per warp: elements kept (may pass kReg)
  unsigned long long tot[kWarps];       // bonus draw: per-warp weight sums
  unsigned int prefix;                  // key bits fixed so far
  int need;                             // keys still to place among those with that prefix
  int dgt;                              // digit fixed by the last pass
  int eq;                               // keys equal to the selected one
  int tok;
  int cand[SPECDEC_MAX_TOPK];
  unsigned long long w[SPECDEC_MAX_TOPK];
  unsigned long long red[2 * kWarps];
};
static_assert(kThreads >= 256, "one digit per thread in the selections");

// Order-preserving unsigned key of a logit's bits (bf16: 16 bits; float32:
// 32), -0 taking the key of +0 so that equal values have equal keys.
template <int DT>
__device__ __forceinline__ uint32_t order_key_bits(uint32_t b) {
  if (DT == SPECDEC_F32) {
    if ((b << 1) == 0u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  }
  if ((b & 0x7FFFu) == 0u) b = 0u;
  return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}

// The value whose key is k (inverse of order_key_bits).
template <int DT>
__device__ __forceinline__ float key_value(uint32_t k) {
  if (DT == SPECDEC_F32) return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
  const uint32_t b = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
  return __uint_as_float(b << 16);
}

template <int DT>
struct Vec {
  static constexpr int kN = (DT == SPECDEC_F32) ? 4 : 8;  // elements per 16 bytes
};

// The 16 bytes at row + 16 vi of a row whose start is not 16-byte aligned
// (vi * kN < V): the aligned vector holding the first byte, and the next one
// when it holds a byte of the row, then whole-word and half-word shifts.
// Every vector read holds a byte of the row (an aligned 16-byte vector never
// straddles a page), so no read leaves the caller's buffer.  Elements at or
// past V read as zero bits.
template <int DT>
__device__ __forceinline__ uint4 load_vec_shifted(const uint8_t *row, int vi, int V) {
  constexpr int kN = Vec<DT>::kN;
  constexpr int es = 16 / kN;
  const uintptr_t a = reinterpret_cast<uintptr_t>(row) + (uintptr_t)vi * 16u;
  const uintptr_t end = reinterpret_cast<uintptr_t>(row) + (uintptr_t)V * es;
  const unsigned mis = (unsigned)(a & 15u);
  const uint4 *c = reinterpret_cast<const uint4 *>(a - mis);
  const uint4 x0 = __ldg(c);
  const uint4 x1 = (a - mis + 16u < end) ? __ldg(c + 1) : make_uint4(0u, 0u, 0u, 0u);
  const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
  const unsigned ws = mis >> 2, hs = (mis & 2u) ? 16u : 0u;
  uint32_t d[5];
#pragma unroll
  for (int j = 0; j < 5; ++j) d[j] = ws == 0 ? w[j] : ws == 1 ? w[j + 1] : ws == 2 ? w[j + 2] : w[j + 3];
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) o[j] = __funnelshift_r(d[j], d[j + 1], hs);
  const int n = V - vi * kN;  // elements of the row in this vector (>= 1)
  if (n < kN) {
#pragma unroll
    for (int e = 0; e < kN; ++e) {
      if (e < n) continue;
      if (DT == SPECDEC_F32) o[e] = 0u;
      else o[e >> 1] &= (e & 1) ? 0x0000FFFFu : 0xFFFF0000u;
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// The 16 bytes of vector vi of a row (shifted aligned vectors on a row that
// is not 16-byte aligned; element loads for the ragged last vector of an
// aligned row; the missing elements read as zero bits and are masked by the
// caller).
template <int DT>
__device__ __forceinline__ uint4 load_vec(const uint8_t *row, bool aligned, int vi, int V, bool valid) {
  constexpr int kN = Vec<DT>::kN;
  const int v0 = vi * kN;
  if (valid && aligned && v0 + kN <= V) return __ldg(reinterpret_cast<const uint4 *>(row) + vi);
  if (valid && !aligned && v0 < V) return load_vec_shifted<DT>(row, vi, V);
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int e = 0; e < kN; ++e) {
    const int v = v0 + e;
    if (!valid || v >= V) continue;
    if (DT == SPECDEC_F32) w[e] = __ldg(reinterpret_cast<const uint32_t *>(row) + v);
    else w[e >> 1] |= (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(row) + v) << (16 * (e & 1));
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// NU vectors per lane, vector base + u * 32 + lane for u < NU: plain 16-byte
// loads, all in flight together, when the whole batch is aligned and inside
// [.., end) and the row; else vector by vector.
template <int DT, int NU>
__device__ __forceinline__ void load_batch(uint4 (&x)[NU], const uint8_t *row, bool aligned, int base,
                                           int end, int V, int lane) {
  constexpr int kN = Vec<DT>::kN;
  const int last = base + NU * 32;
  if (aligned && last <= end && last * kN <= V) {
    const uint4 *r4 = reinterpret_cast<const uint4 *>(row) + base + lane;
#pragma unroll
    for (int u = 0; u < NU; ++u) x[u] = __ldg(r4 + u * 32);
  } else {
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int vi = base + u * 32 + lane;
      x[u] = load_vec<DT>(row, aligned, vi, V, vi < end);
    }
  }
}

template <int DT>
__device__ __forceinline__ uint32_t elem_bits(const uint4 &x, int e) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  return (DT == SPECDEC_F32) ? w[e] : ((w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
}

template <int DT>
__device__ __forceinline__ uint32_t key_of(const uint4 &x, int e) {
  return order_key_bits<DT>(elem_bits<DT>(x, e));
}

// Number of valid elements of vector vi (0 at or past `end`).
template <int DT>
__device__ __forceinline__ int vec_valid(int vi, int end, int V) {
  constexpr int kN = Vec<DT>::kN;
  if (vi >= end) return 0;
  const int r = V - vi * kN;
  return r < kN ? r : kN;
}

// Bit e set for each element e of the vector with value >= t (packed bf16
// compares for bf16 rows).
template <int DT>
__device__ __forceinline__ unsigned ge_mask(const uint4 &x, float t) {
  if (DT == SPECDEC_F32) {
    return (__uint_as_float(x.x) >= t ? 1u : 0u) | (__uint_as_float(x.y) >= t ? 2u : 0u) |
           (__uint_as_float(x.z) >= t ? 4u : 0u) | (__uint_as_float(x.w) >= t ? 8u : 0u);
  }
  const __nv_bfloat162 tt = __float2bfloat162_rn(t);  // t is a bf16 value: exact
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  unsigned m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 v;
    memcpy(&v, &w[i], 4);
    const unsigned r = __hge2_mask(v, tt);
    m |= ((r & 1u) | ((r >> 15) & 2u)) << (2 * i);
  }
  return m;
}

__device__ __forceinline__ unsigned warp_exscan_u32(unsigned v, int lane, unsigned &total) {
  unsigned inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const unsigned y = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += y;
  }
  total = __shfl_sync(0xffffffffu, inc, 31);
  return inc - v;
}

// One digit count (a shared-memory add; lanes adding to one digit are
// serialised by the hardware, which measured cheaper here than aggregating
// them with a match).
__device__ __forceinline__ void count_digit(unsigned *hist, bool match, uint32_t digit) {
  if (match) atomicAdd(&hist[digit], 1u);
}

// After a pass's counts (sm.h for the block, or the sum of the per-warp
// counts): the digit holding the need-th largest key is fixed.  Thread t
// holds digit 255 - t, so an exclusive scan in thread order sums the larger
// digits.
__device__ __forceinline__ void fix_digit(unsigned cnt, uint32_t prefix, int shift, Smem &sm, Red &rr) {
  const int mine = 255 - (int)threadIdx.x;  // negative past 255: count 0, never selected
  unsigned long long total;
  const unsigned long long larger = block_exscan_u64(cnt, rr, total);
  const unsigned long long nd = (unsigned long long)sm.need;
  __syncthreads();
  if (larger < nd && larger + cnt >= nd) {
    sm.need = (int)(nd - larger);
    sm.eq = (int)cnt;
    sm.dgt = mine;
    sm.prefix = prefix | ((uint32_t)mine << shift);
  }
  __syncthreads();
}

// The K-th largest of keys[0, n) (1 <= K <= the number of nonzero keys; zero
// keys are never selected), by 8-bit digits from the top of kBits-bit keys.
// Returns it with `need` = how many keys equal to it complete the K largest;
// sm.eq = how many keys equal it.
template <int kBits>
__device__ __forceinline__ uint32_t smem_select(const uint32_t *keys, int n, int K, int &need,
                                                Smem &sm, Red &rr) {
  const int tid = threadIdx.x;
  __syncthreads();
  if (tid == 0) {
    sm.prefix = 0;
    sm.need = K;
  }
#pragma unroll 1
  for (int shift = kBits - 8; shift >= 0; shift -= 8) {
    __syncthreads();
    if (tid < 256) sm.h[tid] = 0u;
    __syncthreads();
    const uint32_t prefix = sm.prefix;
    const uint32_t hi_mask = (shift + 8 >= 32) ? 0u : (0xFFFFFFFFu << (shift + 8));
    for (int j = tid; j < n; j += kThreads) {
      const uint32_t key = keys[j];
      count_digit(sm.h, key != 0u && (key & hi_mask) == (prefix & hi_mask), (key >> shift) & 0xFFu);
    }
    __syncthreads();
    fix_digit(tid < 256 ? sm.h[255 - tid] : 0u, prefix, shift, sm, rr);
  }
  need = sm.need;
  return sm.prefix;
}

// Writes sm.cand[0, K) in index order from per-warp sequences of keys in
// index order (warp w: keys[w * stride + i] for i < count_w, with
// index[w * stride + i]): the keys above thr, and the first need_eq keys
// equal to it.  Ballot ranks within a warp, per-warp offsets from a first
// counting sweep.
__device__ __forceinline__ void ordered_pick(const uint32_t *keys, const int *index, int stride,
                                             int count_w, uint32_t thr, int need_eq, Smem &sm) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned lt = (1u << lane) - 1u;
  const uint32_t *kw = keys + warp * stride;
  const int *iw = index + warp * stride;
  unsigned na = 0, nt = 0;
  for (int r = 0; r < count_w; r += 32) {
    const uint32_t key = (r + lane < count_w) ? kw[r + lane] : 0u;
    na += __popc(__ballot_sync(0xffffffffu, key > thr));
    nt += __popc(__ballot_sync(0xffffffffu, key == thr));
  }
  if (lane == 0) {
    sm.above[warp] = na;
    sm.ties[warp] = nt;
  }
  __syncthreads();
  if (tid == 0) {
    unsigned ties = 0, out = 0;
    for (int w = 0; w < kWarps; ++w) {
      const unsigned t = sm.ties[w];
      const unsigned take = ((int)ties >= need_eq) ? 0u : min(t, (unsigned)need_eq - ties);
      sm.tie_off[w] = ties;
      sm.out_off[w] = out;
      ties += t;
      out += sm.above[w] + take;
    }
  }
  __syncthreads();
  unsigned out = sm.out_off[warp], trank = sm.tie_off[warp];
  for (int r = 0; r < count_w; r += 32) {
    const uint32_t key = (r + lane < count_w) ? kw[r + lane] : 0u;
    const unsigned tie = __ballot_sync(0xffffffffu, key == thr);
    const bool take = key > thr || (key == thr && trank + __popc(tie & lt) < (unsigned)need_eq);
    const unsigned sel = __ballot_sync(0xffffffffu, take);
    if (take) sm.cand[out + __popc(sel & lt)] = iw[r + lane];
    out += __popc(sel);
    trank += __popc(tie);
  }
}

// Fast path.  Returns false (CTA-uniform) when no sampled rank kept between
// K and kCap elements without overflowing a region; otherwise sm.cand[0, K)
// holds the K largest in index order.
template <int DT>
__device__ __forceinline__ bool topk_filter(const uint8_t *row, bool aligned, int V, int K,
                                            Smem &sm, Red &rr) {
  constexpr int kN = Vec<DT>::kN;
  constexpr int kBits = (DT == SPECDEC_F32) ? 32 : 16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nvec = (V + kN - 1) / kN;
  const int segw = (((nvec + kWarps - 1) / kWarps) + 31) & ~31;
  const int s0 = min(nvec, warp * segw), s1 = min(nvec, s0 + segw);
  constexpr int kSampleVec = kSample / kN;
  const int stride = (nvec + kSampleVec - 1) / kSampleVec;
  const int ns = (nvec + stride - 1) / stride;       // sampled vectors (every stride-th)
  const int ns_valid = (ns - 1) * kN + 1;            // at least this many sampled keys are valid
  // the sampled key ranked j has about tgt row elements above it
  const long long tgt = min(max(2 * K, 256), kCap / 2);
  int j = (int)max(1ll, min((long long)ns_valid, tgt * ns * kN / V));
#pragma unroll 1
  for (int attempt = 0; attempt < kTries; ++attempt) {
    __syncthreads();
    for (int s = tid; s < ns; s += kThreads) {
      const int vi = s * stride;
      const uint4 x = load_vec<DT>(row, aligned, vi, V, true);
      const int nv = vec_valid<DT>(vi, nvec, V);
#pragma unroll
      for (int e = 0; e < kN; ++e) sm.u.key[s * kN + e] = (e < nv) ? key_of<DT>(x, e) : 0u;
    }
    int unused;
    const uint32_t t_key = smem_select<kBits>(sm.u.key, ns * kN, j, unused, sm, rr);
    const float t_val = key_value<DT>(t_key);
    __syncthreads();
    // ---- one pass: each warp keeps, in index order, its elements >= t_val --
    unsigned kept = 0;
    uint32_t *kreg = sm.u.key + warp * kReg;
    int *ireg = sm.cidx + warp * kReg;
    for (int base = s0; base < s1; base += kUF * 32) {
      uint4 x[kUF];
      load_batch<DT>(x, row, aligned, base, s1, V, lane);
#pragma unroll
      for (int u = 0; u < kUF; ++u) {
        const int vi = base + u * 32 + lane;
        const int nv = vec_valid<DT>(vi, s1, V);
        const unsigned mask = ge_mask<DT>(x[u], t_val) & ((1u << nv) - 1u);
        if (!__any_sync(0xffffffffu, mask != 0u)) continue;
        unsigned tot;
        unsigned pos = kept + warp_exscan_u32((unsigned)__popc(mask), lane, tot);
        kept += tot;
#pragma unroll
        for (int e = 0; e < kN; ++e) {
          if ((mask >> e) & 1u) {
            if (pos < (unsigned)kReg) {
              kreg[pos] = key_of<DT>(x[u], e);
              ireg[pos] = vi * kN + e;
            }
            ++pos;
          }
        }
      }
    }
    for (int i = (int)kept + lane; i < kReg; i += 32) kreg[i] = 0u;
    if (lane == 0) sm.nw[warp] = kept;
    __syncthreads();
    unsigned total = 0, most = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      total += sm.nw[w];
      most = max(most, sm.nw[w]);
    }
    if (total >= (unsigned)K && most <= (unsigned)kReg) {
      // ---- the K largest kept, in index order --------------------------------
      int need_eq;
      const uint32_t thr = smem_select<kBits>(sm.u.key, kCap, K, need_eq, sm, rr);
      ordered_pick(sm.u.key, sm.cidx, kReg, (int)min(sm.nw[warp], (unsigned)kReg), thr, need_eq, sm);
      return true;
    }
    // another rank: lower when too few were kept, higher when a region overflowed
    const int j2 = (total < (unsigned)K) ? min(ns_valid, 4 * j) : max(1, j / 4);
    if (j2 == j) break;
    j = j2;
  }
  return false;
}

// One radix pass over this warp's segment [s0, s1) of vectors: counts of the
// digit (key >> shift) & 255 over the keys whose bits above the digit equal
// the prefix, then the digit of the need-th largest is fixed and each warp
// adds its keys with a larger digit to its `above` count.
template <int DT>
__device__ __forceinline__ void radix_pass(const uint8_t *row, bool aligned, int V, int s0, int s1,
                                           int shift, Smem &sm, Red &rr) {
  constexpr int kN = Vec<DT>::kN;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __syncthreads();  // every warp is done with the previous pass's counts
  for (int i = tid; i < kWarps * 256; i += kThreads) (&sm.u.hist[0][0])[i] = 0u;
  __syncthreads();
  const uint32_t prefix = sm.prefix;
  const uint32_t hi_mask = (shift + 8 >= 32) ? 0u : (0xFFFFFFFFu << (shift + 8));
  unsigned int *hist = sm.u.hist[warp];
  for (int base = s0; base < s1; base += kU * 32) {
    uint4 x[kU];
    load_batch<DT>(x, row, aligned, base, s1, V, lane);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int nv = vec_valid<DT>(base + u * 32 + lane, s1, V);
#pragma unroll
      for (int e = 0; e < kN; ++e) {
        const uint32_t key = key_of<DT>(x[u], e);
        count_digit(hist, e < nv && (key & hi_mask) == (prefix & hi_mask), (key >> shift) & 0xFFu);
      }
    }
  }
  __syncthreads();
  unsigned cnt = 0;
#pragma unroll
  for (int w = 0; w < kWarps && tid < 256; ++w) cnt += sm.u.hist[w][255 - tid];
  fix_digit(cnt, prefix, shift, sm, rr);
  const int dgt = sm.dgt;
  unsigned a = 0;
#pragma unroll
  for (int i = lane; i < 256; i += 32) a += (i > dgt) ? hist[i] : 0u;
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) a += __shfl_xor_sync(0xffffffffu, a, d);
  if (lane == 0) sm.above[warp] += a;
}

// Full radix select and stable compaction (rows the fast path declines).
template <int DT>
__device__ __forceinline__ void full_select(const uint8_t *lrow, bool aligned, int V, int K,
                                            Smem &sm, Red &rr) {
  constexpr int kBits = (DT == SPECDEC_F32) ? 32 : 16;
  constexpr int kN = Vec<DT>::kN;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nvec = (V + kN - 1) / kN;
  const int segw = (((nvec + kWarps - 1) / kWarps) + 31) & ~31;
  const int s0 = min(nvec, warp * segw), s1 = min(nvec, s0 + segw);
  __syncthreads();
  if (tid == 0) {
    sm.prefix = 0;
    sm.need = K;
  }
  if (tid < kWarps) sm.above[tid] = 0;
  for (int shift = kBits - 8; shift >= 0; shift -= 8) radix_pass<DT>(lrow, aligned, V, s0, s1, shift, sm, rr);
  __syncthreads();
  const uint32_t thr = sm.prefix;  // the K-th largest key
  const int need_eq = sm.need;     // keys equal to it that are candidates (the first by index)
  if (tid == 0) {
    // the last pass's count of the final digit is each warp's count of keys equal to thr
    unsigned ties = 0, out = 0;
    for (int w = 0; w < kWarps; ++w) {
      const unsigned t = sm.u.hist[w][sm.dgt];
      const unsigned take = ((int)ties >= need_eq) ? 0u : min(t, (unsigned)need_eq - ties);
      sm.tie_off[w] = ties;
      sm.out_off[w] = out;
      ties += t;
      out += sm.above[w] + take;
    }
  }
  __syncthreads();
  // ---- stable compaction: keys above thr, and the first need_eq ties --------
  const unsigned lt = (1u << lane) - 1u;
  unsigned out = sm.out_off[warp], trank = sm.tie_off[warp];
  for (int base = s0; base < s1; base += kU * 32) {
    uint4 x[kU];
    load_batch<DT>(x, lrow, aligned, base, s1, V, lane);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int vi = base + u * 32 + lane;
      const int nv = vec_valid<DT>(vi, s1, V);
      unsigned ab = 0, eq = 0;
#pragma unroll
      for (int e = 0; e < kN; ++e) {
        const uint32_t key = key_of<DT>(x[u], e);
        ab |= (e < nv && key > thr) ? (1u << e) : 0u;
        eq |= (e < nv && key == thr) ? (1u << e) : 0u;
      }
      if (!__any_sync(0xffffffffu, (ab | eq) != 0u)) continue;
      unsigned eq_tot;
      unsigned r = trank + warp_exscan_u32((unsigned)__popc(eq), lane, eq_tot);
      trank += eq_tot;
      unsigned sel = ab;
#pragma unroll
      for (int e = 0; e < kN; ++e) {
        if ((eq >> e) & 1u) {
          if (r < (unsigned)need_eq) sel |= 1u << e;
          ++r;
        }
      }
      unsigned sel_tot;
      unsigned pos = out + warp_exscan_u32((unsigned)__popc(sel), lane, sel_tot);
      out += sel_tot;
#pragma unroll
      for (int e = 0; e < kN; ++e)
        if ((sel >> e) & 1u) sm.cand[pos++] = vi * kN + e;
    }
  }
  (void)lt;
}

// The residual draw over the K candidates sm.cand[0, K) (index order):
// weights max(0, p - q) in 40-bit fixed point, p itself when they sum to 0.
template <int DT>
__device__ __forceinline__ void draw_candidates(const LinearFinalizeParams &p, long long b, int k,
                                                const LinearDecision &d, const uint8_t *lrow,
                                                const uint8_t *qrow, int K, Smem &sm, Red &rr) {
  const int tid = threadIdx.x;
  const int R = p.gamma + 1, gamma = p.gamma;
  constexpr int kPer = SPECDEC_MAX_TOPK / kThreads;  // candidates per thread
  static_assert(kPer * kThreads == SPECDEC_MAX_TOPK, "candidates split evenly");
  const int j0 = tid * kPer;
  unsigned long long zk = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = j0 + i;
    if (j >= K) break;
    const int v = sm.cand[j];
    const float lv = load_elem(lrow, DT, v), qv = load_elem(qrow, DT, v);
    const float ev = ex2_approx((lv - d.M) * d.c);
    const unsigned long long f = to_fixed40(fmaxf(fmaf(-d.S, qv, ev), 0.0f));
    sm.w[j] = f;
    zk += f;
  }
  unsigned long long Z;
  unsigned long long pre = block_exscan_u64(zk, rr, Z);
  if (Z == 0) {  // no residual mass on the candidates: p on them
    zk = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int j = j0 + i;
      if (j >= K) break;
      const float lv = load_elem(lrow, DT, sm.cand[j]);
      sm.w[j] = to_fixed40(ex2_approx((lv - d.M) * d.c));
      zk += sm.w[j];
    }
    pre = block_exscan_u64(zk, rr, Z);
  }
  const unsigned long long target = uniform_target(__ldg(p.uniforms + b * R + gamma), Z);
  if (tid == 0) p.ws.mass[b] = draw_mass(Z, d.S);  // the restricted residual's mass
  unsigned long long run = pre;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = j0 + i;
    if (j >= K) break;
    const unsigned long long nx = run + sm.w[j];
    if (run <= target && nx > target) sm.tok = sm.cand[j];
    run = nx;
  }
  __syncthreads();
  if (tid == 0) {
    const int tok = sm.tok >= 0 ? sm.tok : sm.cand[K - 1];
    p.final_token[b] = tok;
    p.out_tokens[b * R + k] = tok;
  }
}

// Elements of a vector at or past nv read as -inf (weight 0).
template <int DT>
__device__ __forceinline__ uint4 pad_neg_inf(uint4 x, int nv) {
  constexpr int kN = Vec<DT>::kN;
  if (nv >= kN) return x;
  uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int e = 0; e < kN; ++e) {
    if (e < nv) continue;
    if (DT == SPECDEC_F32) w[e] = 0xFF800000u;
    else w[e >> 1] = (e & 1) ? ((w[e >> 1] & 0xFFFFu) | 0xFF800000u) : ((w[e >> 1] & 0xFFFF0000u) | 0xFF80u);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Bonus draw, exact, from p over the whole final row: per-vector weight sums
// (the vector-ordered CDF of the bulk draw), summed per round of kUB * 32
// vectors of each warp's segment; the round holding U * Z is then walked
// again by its warp.
constexpr int kMaxRounds = sizeof(((Smem *)nullptr)->u) / sizeof(unsigned long long) / kWarps;

template <int DT>
__device__ __forceinline__ void bonus_draw(const LinearFinalizeParams &p, long long b,
                                           const LinearDecision &d, Smem &sm) {
  constexpr int kN = Vec<DT>::kN;
  constexpr int es = (DT == SPECDEC_F32) ? 4 : 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gamma = p.gamma, R = gamma + 1, V = p.V;
  const uint8_t *row = reinterpret_cast<const uint8_t *>(p.logits) + (size_t)(b * R + gamma) * V * es;
  const bool aligned = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
  const int nvec = (V + kN - 1) / kN;
  const int segw = (((nvec + kWarps - 1) / kWarps) + 31) & ~31;
  const int s0 = min(nvec, warp * segw), s1 = min(nvec, s0 + segw);
  const int nround = (s1 - s0 + kUB * 32 - 1) / (kUB * 32);
  constexpr int kMaxSeg = (((SPECDEC_MAX_V / 4 + kWarps - 1) / kWarps) + 31) & ~31;
  static_assert((kMaxSeg + kUB * 32 - 1) / (kUB * 32) <= kMaxRounds, "round sums fit in shared memory");
  unsigned long long *rs = reinterpret_cast<unsigned long long *>(&sm.u) + warp * kMaxRounds;
  const uint4 none = make_uint4(0u, 0u, 0u, 0u);
  unsigned long long wsum = 0;
  for (int r = 0; r < nround; ++r) {
    const int base = s0 + r * kUB * 32;
    uint4 x[kUB];
    load_batch<DT>(x, row, aligned, base, s1, V, lane);
    unsigned long long acc = 0;
#pragma unroll
    for (int u = 0; u < kUB; ++u) {
      const int vi = base + u * 32 + lane;
      if (vi < s1)
        acc += to_fixed40(drawc::vec_sum<DT>(pad_neg_inf<DT>(x[u], vec_valid<DT>(vi, s1, V)), none, d, false));
    }
    acc = drawc::warp_sum_u64(acc);
    if (lane == 0) rs[r] = acc;
    wsum += acc;
  }
  if (lane == 0) sm.tot[warp] = wsum;
  __syncthreads();
  unsigned long long Z = 0, before = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) before += sm.tot[w];
    Z += sm.tot[w];
  }
  const unsigned long long target = uniform_target(__ldg(p.uniforms + b * R + gamma), Z);
  if (threadIdx.x == 0) p.ws.mass[b] = draw_mass(Z, d.S);
  if (!(target >= before && target < before + sm.tot[warp])) return;
  // this warp's segment holds the target: its round, then the vector in u order
  int r = 0;
  unsigned long long run = before;
  while (r < nround - 1 && run + rs[r] <= target) run += rs[r++];
  const int base = s0 + r * kUB * 32;
  uint4 x[kUB];
  load_batch<DT>(x, row, aligned, base, s1, V, lane);
#pragma unroll
  for (int u = 0; u < kUB; ++u) {
    const int vi = base + u * 32 + lane;
    const uint4 xv = pad_neg_inf<DT>(x[u], vec_valid<DT>(vi, s1, V));
    const unsigned long long f = (vi < s1) ? to_fixed40(drawc::vec_sum<DT>(xv, none, d, false)) : 0ull;
    const unsigned long long incl = drawc::warp_incl_scan_u64(f, lane);
    const unsigned long long ut = __shfl_sync(0xffffffffu, incl, 31);
    if (run + ut > target) {
      const unsigned long long lo = run + incl - f;
      if (lo <= target && lo + f > target) {
        const int tok = vi * kN + drawc::vec_find<DT>(xv, none, d, false, lo, target);
        p.final_token[b] = tok;
        p.out_tokens[b * R + gamma] = tok;
      }
      return;
    }
    run += ut;
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 2) topk_draw_kernel(const LinearFinalizeParams p, int topk) {
  pdl_wait();
  __shared__ Smem sm;
  const int tid = threadIdx.x;
  const long long b = blockIdx.x;
  const int gamma = p.gamma, R = gamma + 1, V = p.V;
  const LinearDecision d = request_decision<DT, kThreads>(p, b, true, sm.d);
  if (d.status || d.greedy) return;
  const int k = d.k;
  Red rr{sm.red, 0};
  if (k == gamma) {
    bonus_draw<DT>(p, b, d, sm);
    return;
  }
  constexpr int es = (DT == SPECDEC_F32) ? 4 : 2;
  const uint8_t *lrow = reinterpret_cast<const uint8_t *>(p.logits) + (size_t)(b * R + k) * V * es;
  const uint8_t *qrow = reinterpret_cast<const uint8_t *>(p.q) + (size_t)(b * gamma + k) * V * es;
  const bool aligned = (reinterpret_cast<uintptr_t>(lrow) & 15) == 0;
  const int K = min(topk, V);
  if (tid == 0) sm.tok = -1;
  if (!topk_filter<DT>(lrow, aligned, V, K, sm, rr)) full_select<DT>(lrow, aligned, V, K, sm, rr);
  __syncthreads();
  draw_candidates<DT>(p, b, k, d, lrow, qrow, K, sm, rr);
}

}  // namespace

cudaError_t launch_linear_topk(const LinearFinalizeParams &p, int topk, cudaStream_t stream) {
  if (p.B <= 0) return cudaSuccess;
  if (p.dtype == SPECDEC_F32)
    return launch_pdl(topk_draw_kernel<SPECDEC_F32>, dim3((unsigned)p.B), dim3(kThreads), 0,
                      stream, p, topk);
  return launch_pdl(topk_draw_kernel<SPECDEC_BF16>, dim3((unsigned)p.B), dim3(kThreads), 0,
                    stream, p, topk);
}

}  // namespace specdec
