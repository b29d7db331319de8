// Linear verify, phase 2: the accept test and the final draw ("Chapter 15:
// Decoding acceleration", section 15.1.2 steps 3 and 4: accept x~_i while
// u_i <= min(1, p_i(x~_i) / q_i(x~_i)), stop at the first rejection and draw
// its replacement from max(0, p - q) / Z; the bonus draw from the last target
// row when every draft is accepted follows section 15.1.3's expected count
// (1 - a^(g+1)) / (1 - a) of emitted tokens per step).
//
// Two kernels.  Rows that are 16-byte aligned take the bulk-copy draw
// (namespace bulk, further down).  The others take the chunked draw, one CTA
// per (request, 8192-element chunk of its final row), described here:
//
// * every CTA merges its request's row partials (16 lanes per row) and runs
//   the accept test in one warp, lane i testing draft i with the logit and q
//   value the stats pass gathered; a ballot gives the first rejection k.  All
//   CTAs of a request compute the same decision bit for bit (same data, same
//   instruction sequence), which costs a few KB of L2 reads per CTA and needs
//   no cross-CTA handshake;
// * the CTA of chunk 0 writes the request's outputs but the final token
//   (accepted tokens and count, bonus flag, status, p_draft); greedy and
//   malformed requests are complete with it;
// * every CTA sums the draw weights of its chunk: with e_v = 2^((l_v - M) c),
//   the weights are max(0, e_v - S q_v) = S max(0, p - q) after a rejection and
//   e_v = S p for the bonus draw; each thread sums its 32 contiguous weights in
//   float32 and the CTA adds the thread sums in 40-bit fixed point;
// * the last CTA of a request to finish (an atomic ticket that the stats pass
//   zeroed) scans the chunk totals, finds the chunk holding U * Z, recomputes
//   that chunk's thread sums (the same arithmetic, the same order), scans
//   them, and the thread holding the crossing finds the token among its 32
//   weights.  Integer sums make the crossing exact for the weights computed.
//
// Requests are taken in reverse order so that the rows the stats pass read
// last, still in L2, come first.
#include <cfloat>
#include <cstring>
#include <cuda_bf16.h>

#include "linear_decision.cuh"

namespace specdec {
namespace {

using namespace drawc;
using lindec::request_decision;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPerT = 32;                  // contiguous elements per thread
constexpr int kChunk = kThreads * kPerT;   // elements per chunk (8192)
#ifndef SPECDEC_DRAW_MIN_BLOCKS
#define SPECDEC_DRAW_MIN_BLOCKS 4
#endif
constexpr int kMinBlocks = SPECDEC_DRAW_MIN_BLOCKS;  // resident CTAs per SM the registers allow
static_assert(kChunk == SPECDEC_DRAW_CHUNK, "chunk size shared with the workspace layout");

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

// Two 16-byte vectors of the bytes at p (2-byte aligned, not necessarily
// 16-byte aligned): the aligned 16-byte vectors that overlap those 32 bytes
// (three, or two when p is 16-byte aligned), then whole-word and half-word
// shifts.  Each vector read holds at least one of the 32 bytes, and an
// aligned 16-byte vector never straddles a page, so no read leaves the pages
// of the caller's buffer.
__device__ __forceinline__ void load32_shifted(const uint8_t *p, uint4 &o0, uint4 &o1) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const unsigned mis = (unsigned)(a & 15u);
  const uint4 *v = reinterpret_cast<const uint4 *>(a - mis);
  const uint4 x0 = __ldg(v), x1 = __ldg(v + 1);
  const uint4 x2 = mis ? __ldg(v + 2) : make_uint4(0u, 0u, 0u, 0u);
  const uint32_t w[12] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w, x2.x, x2.y, x2.z, x2.w};
  const unsigned ws = mis >> 2, hs = (mis & 2u) ? 16u : 0u;
  uint32_t d[9];
#pragma unroll
  for (int j = 0; j < 9; ++j)
    d[j] = ws == 0 ? w[j] : ws == 1 ? w[j + 1] : ws == 2 ? w[j + 2] : w[j + 3];
  o0 = make_uint4(__funnelshift_r(d[0], d[1], hs), __funnelshift_r(d[1], d[2], hs),
                  __funnelshift_r(d[2], d[3], hs), __funnelshift_r(d[3], d[4], hs));
  o1 = make_uint4(__funnelshift_r(d[4], d[5], hs), __funnelshift_r(d[5], d[6], hs),
                  __funnelshift_r(d[6], d[7], hs), __funnelshift_r(d[7], d[8], hs));
}

// Elements are read 32 bytes (two 16-byte vectors) per array at a time: 16
// bf16 or 8 float32 values.
template <int DT>
struct Sub {
  static constexpr int kEs = (DT == SPECDEC_F32) ? 4 : 2;
  static constexpr int kElems = 32 / kEs;
  uint4 l[2], q[2];

  // the raw bits of element i (a compile-time index after unrolling)
  __device__ __forceinline__ static uint32_t word(const uint4 (&v)[2], int j) {
    const uint4 x = v[j >> 2];
    return (j & 3) == 0 ? x.x : (j & 3) == 1 ? x.y : (j & 3) == 2 ? x.z : x.w;
  }
  __device__ __forceinline__ static float value(const uint4 (&v)[2], int i) {
    if (DT == SPECDEC_F32) return __uint_as_float(word(v, i));
    const uint32_t w = word(v, i >> 1);
    return (i & 1) ? bf16_hi(w) : bf16_lo(w);
  }

  // Elements [e, e + kElems): 16-byte loads inside the row (shifted into
  // place when the row is not 16-byte aligned); element loads in the row's
  // last partial group, with l = -inf, q = 0 beyond V (weight 0 there).
  __device__ __forceinline__ void load(const Draw &w, int e) {
    if (e + kElems <= w.V) {
      const uint8_t *lb = w.lrow + (size_t)e * kEs;
      const uint8_t *qb = w.qrow + (size_t)e * kEs;
      if (w.vec_ok) {
        const uint4 *lp = reinterpret_cast<const uint4 *>(lb);
        const uint4 *qp = reinterpret_cast<const uint4 *>(qb);
#pragma unroll
        for (int k = 0; k < 2; ++k) l[k] = __ldg(lp + k);
#pragma unroll
        for (int k = 0; k < 2; ++k) q[k] = w.use_q ? __ldg(qp + k) : make_uint4(0u, 0u, 0u, 0u);
        return;
      }
      load32_shifted(lb, l[0], l[1]);
      if (w.use_q) {
        load32_shifted(qb, q[0], q[1]);
      } else {
        q[0] = q[1] = make_uint4(0u, 0u, 0u, 0u);
      }
      return;
    }
    uint32_t lw[8], qw[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) lw[j] = qw[j] = 0u;
#pragma unroll
    for (int i = 0; i < kElems; ++i) {
      const int v = e + i;
      const bool in = v < w.V;
      if (DT == SPECDEC_F32) {
        lw[i] = in ? __float_as_uint(__ldg(reinterpret_cast<const float *>(w.lrow) + v)) : 0xFF800000u;
        qw[i] = (in && w.use_q) ? __float_as_uint(__ldg(reinterpret_cast<const float *>(w.qrow) + v)) : 0u;
      } else {
        const uint32_t lb = in ? (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(w.lrow) + v) : 0xFF80u;
        const uint32_t qb = (in && w.use_q) ? (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(w.qrow) + v) : 0u;
        lw[i >> 1] |= (i & 1) ? (lb << 16) : lb;
        qw[i >> 1] |= (i & 1) ? (qb << 16) : qb;
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      l[k] = make_uint4(lw[4 * k], lw[4 * k + 1], lw[4 * k + 2], lw[4 * k + 3]);
      q[k] = make_uint4(qw[4 * k], qw[4 * k + 1], qw[4 * k + 2], qw[4 * k + 3]);
    }
  }

  // weight of element i: e_v, or max(0, e_v - K q_v) after a rejection
  __device__ __forceinline__ float weight(const Draw &w, int i) const {
    const float ev = ex2_approx((value(l, i) - w.M) * w.c);
    return w.use_q ? fmaxf(fmaf(-w.K, value(q, i), ev), 0.0f) : ev;
  }
};

// The float32 sum, in index order, of the 32 weights of elements [e, e + 32)
// (zero at and beyond V), as 40-bit fixed point.
template <int DT>
__device__ __forceinline__ unsigned long long thread_sum(const Draw &w, int e) {
  constexpr int n = Sub<DT>::kElems;
  float s = 0.0f;
#pragma unroll
  for (int h = 0; h < kPerT / n; ++h) {
    Sub<DT> x;
    x.load(w, e + h * n);
#pragma unroll
    for (int i = 0; i < n; ++i) s += x.weight(w, i);
  }
  return to_fixed40(s);
}

// The element of [e, e + 32) at which base + (running float32 sum, as in
// thread_sum) first exceeds target.
template <int DT>
__device__ __forceinline__ int thread_find(const Draw &w, int e, unsigned long long base,
                                           unsigned long long target) {
  constexpr int n = Sub<DT>::kElems;
  float run = 0.0f;
#pragma unroll
  for (int h = 0; h < kPerT / n; ++h) {
    Sub<DT> x;
    x.load(w, e + h * n);
#pragma unroll
    for (int i = 0; i < n; ++i) {
      run += x.weight(w, i);
      if (base + to_fixed40(run) > target) return e + h * n + i;
    }
  }
  return e + kPerT - 1;
}

// Shared-memory scratch of the block reductions, two buffers used in turn:
// a buffer is written again only after a barrier that every reader of its
// previous contents has passed.
struct Red {
  unsigned long long *buf;  // [2][kWarps]
  int phase;
  __device__ __forceinline__ unsigned long long *next() {
    unsigned long long *r = buf + phase * kWarps;
    phase ^= 1;
    return r;
  }
};

__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, Red &rr) {
  unsigned long long *red = rr.next();
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

struct DrawSmem {
  unsigned long long red[2 * kWarps];
  unsigned long long base;
  int chunk, last;
  RowStat rs[SPECDEC_MAX_GAMMA + 1];
  LinearDecision dec;
};

// The token of request b from its chunk totals (all chunks summed): the
// chunk holding U * Z, then the thread of that chunk, then the element.
template <int DT>
__device__ __forceinline__ void request_search(const LinearFinalizeParams &p, long long b, int k,
                                               Draw w, Red &rr, DrawSmem &sm) {
  const int tid = threadIdx.x;
  const int gamma = p.gamma, R = gamma + 1;
  const int nch = p.nchunk;
  static_assert(SPECDEC_MAX_V / kChunk <= kThreads, "one chunk total per thread");
  unsigned long long mine = (tid < nch) ? __ldcg(p.ws.chunk_tot + b * p.ntot + tid) : 0ull;
  unsigned long long Z;
  unsigned long long pre = block_exscan_u64(mine, rr, Z);
  if (Z == 0 && w.use_q) {
    // residual mass 0 (only by rounding): draw from p itself
    w.use_q = false;
    for (int ch = 0; ch < nch; ++ch) {
      const unsigned long long t = block_sum_u64(thread_sum<DT>(w, ch * kChunk + tid * kPerT), rr);
      if (tid == ch) mine = t;
    }
    pre = block_exscan_u64(mine, rr, Z);
  }
  const float U = __ldg(p.uniforms + b * R + gamma);
  const unsigned long long target = uniform_target(U, Z);
  if (tid == 0) {
    sm.chunk = -1;
    p.ws.draw_cnt[b] = 0;  // phase 2 may run again on the same phase-1 result
    p.ws.mass[b] = draw_mass(Z, w.K);
  }
  __syncthreads();
  if (tid < nch && pre <= target && target - pre < mine) {
    sm.chunk = tid;
    sm.base = pre;
  }
  __syncthreads();
  const int ch = sm.chunk;
  const unsigned long long base = sm.base;
  if (ch < 0) return;  // no weight at all: unreachable for a usable row
  const int e = ch * kChunk + tid * kPerT;
  const unsigned long long fe = thread_sum<DT>(w, e);
  unsigned long long ctot;
  const unsigned long long excl = base + block_exscan_u64(fe, rr, ctot);
  if (excl <= target && target - excl < fe) {
    const int v = thread_find<DT>(w, e, excl, target);
    p.final_token[b] = v;
    p.out_tokens[b * R + k] = v;
  }
}

// Persistent: CTA i takes the items [n i / G, n (i + 1) / G) of the sequence
// of (request, chunk) pairs, requests in reverse order, so that it decides
// about one or two requests and sums several chunks of each.  A request's
// chunks are counted on its ticket once per CTA; the CTA that completes the
// count runs the search.
template <int DT>
__global__ void __launch_bounds__(kThreads, kMinBlocks) linear_draw_kernel(const LinearFinalizeParams p) {
  pdl_launch_dependents();  // a next call's stats pass waits for this grid's completion itself
  pdl_wait();
  __shared__ DrawSmem sm;
  const int tid = threadIdx.x;
  Red rr{sm.red, 0};
  const long long nch = p.nchunk;
  const long long n = (long long)p.B * nch;
  const long long lo = n * blockIdx.x / gridDim.x;
  const long long hi = n * (blockIdx.x + 1) / gridDim.x;
  for (long long t0 = lo; t0 < hi;) {
    const long long rb = t0 / nch;
    const long long t1 = min(hi, (rb + 1) * nch);
    const long long b = (long long)p.B - 1 - rb;
    const int c0 = (int)(t0 - rb * nch), c1 = (int)(t1 - rb * nch);
    t0 = t1;
    const LinearDecision d = request_decision<DT, kThreads>(p, b, c0 == 0, sm);
    if (d.status || d.greedy) continue;  // nothing to draw
    const Draw w = make_draw<DT>(p, b, d);
    for (int ch = c0; ch < c1; ++ch) {
      const unsigned long long tot = block_sum_u64(thread_sum<DT>(w, ch * kChunk + tid * kPerT), rr);
      if (tid == 0) p.ws.chunk_tot[b * p.ntot + ch] = tot;
    }
    if (tid == 0) {
      __threadfence();
      sm.last = atomicAdd(p.ws.draw_cnt + b, (unsigned)(c1 - c0)) + (unsigned)(c1 - c0) == (unsigned)nch;
    }
    __syncthreads();
    if (sm.last) {
      __threadfence();
      request_search<DT>(p, b, d.k, w, rr, sm);
    }
  }
}


// ---------------------------------------------------------------------------
// The draw over 16-byte aligned rows: bulk copies into shared memory and one
// warp per 4 KB stage of the final row, after the row-statistics kernel's
// pattern.  Persistent, one CTA per SM; CTA i takes a contiguous run of the
// sequence of (request, 16 KB unit) pairs, requests in reverse order.
//
// * Head: 16-lane segments merge the partials of every row of the run's
//   requests (at most kMaxReq), then warp j runs request j's accept test; the
//   CTA holding a request's first unit writes its outputs.
// * Pipeline: one producer thread copies each unit's logits (and, after a
//   rejection, its q values) into a ring of kSlots slots; stage t of a unit
//   goes to consumer warp (local stage index) mod kWarps.  A lane takes the
//   16-byte vectors lane, lane + 32, ... of the stage, sums each vector's
//   weights in float32 in index order and adds the sums as 40-bit fixed
//   point; the warp's total is the stage total.  Vectors in index order are
//   therefore the units of the inverse CDF above the float32 level.
// * Tail: after a barrier, thread 0 adds the run's stage count of each
//   request to the request's ticket; warp j searches request j if its count
//   completed the ticket: stage, then vector (in index order), then element.
// ---------------------------------------------------------------------------
namespace bulk {

using namespace drawc;

constexpr int kUnitStages = 4;
constexpr int kUnitBytes = kStage * kUnitStages;    // one bulk copy of logits (+ one of q)
constexpr int kSlots = 6;
constexpr int kWarps = 15;                          // consumer warps
constexpr int kThreads = (kWarps + 1) * 32;         // + the producer warp
constexpr int kMaxReq = 8;                          // requests in one CTA's run
static_assert(kWarps <= kSlots * kUnitStages, "no more consumer warps than ring stages");
constexpr unsigned kAbort = 1u << 24;               // ticket increment of a CTA whose wait ran out

struct Smem {
  alignas(128) uint8_t l[kSlots][kUnitBytes];
  alignas(128) uint8_t q[kSlots][kUnitBytes];
  alignas(8) uint64_t full[kSlots];
  alignas(8) uint64_t empty[kSlots];
  RowStat rs[kMaxReq][SPECDEC_MAX_GAMMA + 1];
  LinearDecision dec[kMaxReq];
  int search[kMaxReq];  // 0: not this CTA's; 1: search; 2: search, but a wait ran out somewhere
  volatile int abort_flag;
};

// kEarly: launched right after the stats pass of the same call (a plain
// launch, so everything before it is complete and visible), the call's own
// inputs may be read before waiting for the stats pass, which does not write
// them.  Launched after an arbitrary kernel, everything waits.
template <int DT, bool kEarly>
__global__ void __launch_bounds__(kThreads, 1) draw_bulk_kernel(const LinearFinalizeParams p) {
  pdl_launch_dependents();  // a next call's stats pass waits for this grid's completion itself
  if (!kEarly) pdl_wait();
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
  constexpr int es = (DT == SPECDEC_F32) ? 4 : 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gamma = p.gamma, R = gamma + 1;
  const int rowbytes = p.V * es;
  const int nst = (rowbytes + kStage - 1) / kStage;
  const int upr = (nst + kUnitStages - 1) / kUnitStages;  // units per row
  const long long units = (long long)p.B * upr;
  const long long lo = units * blockIdx.x / gridDim.x;
  const long long hi = units * (blockIdx.x + 1) / gridDim.x;
  const long long rb0 = lo / upr;
  const int nreq = (hi > lo) ? (int)((hi - 1) / upr - rb0 + 1) : 0;  // <= kMaxReq (host check)

  if (tid == 0) {
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], kUnitStages);  // one arrival per stage of the unit
    }
    sm.abort_flag = 0;
    fence_mbar_init();
  }

  // ---- head: row merges (16-lane segments over (request, row) pairs) ------
  // warp j, which runs request j's accept test, loads its inputs first so that
  // their round trip overlaps the merges (the call's own inputs before the
  // wait for the stats pass when kEarly; its gathered values after)
  DraftIn din;
  float Tj = 0.0f;
  if (warp < nreq) {
    const long long b = (long long)p.B - 1 - (rb0 + warp);
    Tj = __ldg(p.temperature + b);
    din = load_draft_inputs(p, b, lane);
  }
  if (kEarly) pdl_wait();
  if (warp < nreq) load_draft_gather(p, (long long)p.B - 1 - (rb0 + warp), lane, din);
  const int pairs = nreq * R;
  for (int base = 0; base < pairs; base += kThreads / kSeg) {
    if (base + warp * (32 / kSeg) >= pairs) continue;  // both segments of this warp idle
    const int pr = base + tid / kSeg;
    const bool active = pr < pairs;
    const int j = active ? pr / R : 0, r = active ? pr - j * R : 0;
    const long long b = (long long)p.B - 1 - (rb0 + j);
    const float c = temperature_scale(__ldg(p.temperature + b));
    const RowStat st = segment_merge_row(p.part, b * R + r, active, p.spr, c, tid % kSeg);
    if (active && tid % kSeg == 0) sm.rs[j][r] = st;
  }
  __syncthreads();
  // ---- head: accept tests, warp j for request j ----------------------------
  if (warp < nreq) {
    const long long rb = rb0 + warp;
    const long long b = (long long)p.B - 1 - rb;
    float pd;
    const LinearDecision d = decide(p, din, Tj, temperature_scale(Tj), sm.rs[warp], lane, pd);
    if (lane == 0) sm.dec[warp] = d;
    if (rb * upr >= lo) write_outputs_warp(p, b, d, pd, lane);  // this CTA holds unit 0
  }
  __syncthreads();

  long long n = 0;  // producer: units issued
  if (warp == kWarps) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      long long rb = rb0;
      int ju = (int)(lo - rb0 * upr);
      for (; lo + n < hi; ++n) {
        const uint32_t slot = (uint32_t)(n % kSlots), use = (uint32_t)(n / kSlots);
        if (use > 0 && !mbar_wait_bounded(&sm.empty[slot], (use - 1) & 1)) {
          sm.abort_flag = 1;
          break;
        }
        if (sm.abort_flag) break;
        const LinearDecision d = sm.dec[rb - rb0];
        if (d.status || d.greedy) {
          mbar_arrive(&sm.full[slot]);  // nothing to draw: an empty unit
        } else {
          const Req rq = make_req<DT>(p, rb, d.k);
          const bool use_q = d.k < gamma;
          const int bytes = min(kUnitBytes, rq.rowbytes - ju * kUnitBytes);
          mbar_arrive_expect_tx(&sm.full[slot], (uint32_t)(bytes * (use_q ? 2 : 1)));
          bulk_copy_g2s(sm.l[slot], rq.lrow + (size_t)ju * kUnitBytes, (uint32_t)bytes, &sm.full[slot]);
          if (use_q)
            bulk_copy_g2s(sm.q[slot], rq.qrow + (size_t)ju * kUnitBytes, (uint32_t)bytes, &sm.full[slot]);
        }
        if (++ju == upr) {
          ju = 0;
          ++rb;
        }
      }
    }
  } else {
    // ------------------------------ consumers -----------------------------
    const long long n_stages_local = (hi - lo) * kUnitStages;
    for (long long cst = warp; cst < n_stages_local; cst += kWarps) {
      const long long n = cst / kUnitStages;
      const int t = (int)(cst - n * kUnitStages);
      const long long i = lo + n;
      const long long rb = i / upr;
      const int ju = (int)(i - rb * upr);
      const uint32_t slot = (uint32_t)(n % kSlots), use = (uint32_t)(n / kSlots);
      const LinearDecision d = sm.dec[rb - rb0];
      const int s = ju * kUnitStages + t;  // stage within the row
      const bool real = !(d.status || d.greedy) && s < nst;
      const bool use_q = d.k < gamma;
      // the slot's previous use released first (see the stats pass: a parity
      // wait tells only two phases apart, and copies land in any order)
      const bool ok = __all_sync(0xffffffffu,  // one outcome for the whole warp
                                 !sm.abort_flag &&
                                     (use == 0 || mbar_wait_bounded(&sm.empty[slot], (use - 1) & 1,
                                                                    kConsumerWaitNs)) &&
                                     mbar_wait_bounded(&sm.full[slot], use & 1, kConsumerWaitNs));
      if (!ok) sm.abort_flag = 1;
      uint4 lv[kVec], qv[kVec];
      const int sbytes = (ok && real) ? min(kStage, rowbytes - s * kStage) : 0;
      load_stage<DT>(lv, qv, sm.l[slot] + t * kStage, sm.q[slot] + t * kStage, sbytes, use_q, lane,
                     false);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[slot]);  // this stage is in registers now
      if (!real || !ok) continue;
      unsigned long long acc = 0;
#pragma unroll
      for (int k = 0; k < kVec; ++k) acc += to_fixed40(vec_sum<DT>(lv[k], qv[k], d, use_q));
      acc = warp_sum_u64(acc);
      if (lane == 0) p.ws.chunk_tot[((long long)p.B - 1 - rb) * p.ntot + s] = acc;
    }
  }
  __syncthreads();
  // after any wait of the CTA gave up, consumers stopped waiting for copies:
  // the CTA stays until every copy the producer issued has landed
  if (sm.abort_flag && warp == kWarps && lane == 0) drain_ring(sm.full, kSlots, n);

  // ---- tail: tickets (thread j for request j), then the searches -------------
  if (tid < nreq) {
    __threadfence();
    const unsigned abort_add = sm.abort_flag ? kAbort : 0u;
    const int j = tid;
    const LinearDecision d = sm.dec[j];
    sm.search[j] = 0;
    if (!(d.status || d.greedy)) {
      const long long rb = rb0 + j;
      const long long u0 = max(lo, rb * upr), u1 = min(hi, (rb + 1) * upr);
      const int s0 = (int)(u0 - rb * upr) * kUnitStages;
      const int s1 = min(nst, (int)(u1 - rb * upr) * kUnitStages);
      const unsigned add = (unsigned)(s1 - s0) + abort_add;
      const long long b = (long long)p.B - 1 - rb;
      const unsigned now = atomicAdd(p.ws.draw_cnt + b, add) + add;
      if ((now & (kAbort - 1)) == (unsigned)nst) sm.search[j] = (now >= kAbort) ? 2 : 1;
    }
  }
  __syncthreads();
  if (warp < nreq && sm.search[warp]) {
    __threadfence();
    const LinearDecision d = sm.dec[warp];
    const Req rq = make_req<DT>(p, rb0 + warp, d.k);
    if (lane == 0) p.ws.draw_cnt[rq.b] = 0;  // phase 2 may run again on the same phase-1 result
    search_warp<DT>(p, rq, d, sm.search[warp] == 2, lane, GlobalTotals{p.ws.chunk_tot + rq.b * p.ntot});
  }
}

}  // namespace bulk

}  // namespace

namespace {

// The bulk-copy draw needs 16-byte aligned rows (base pointers and row
// length) and at most bulk::kMaxReq requests in any CTA's run.
bool bulk_draw_applies(const LinearFinalizeParams &p, int grid) {
  const int es = (p.dtype == SPECDEC_F32) ? 4 : 2;
  const long long rowbytes = (long long)p.V * es;
  if (rowbytes % 16 != 0) return false;
  if ((reinterpret_cast<uintptr_t>(p.logits) & 15) || (reinterpret_cast<uintptr_t>(p.q) & 15))
    return false;
  const long long nst = (rowbytes + bulk::kStage - 1) / bulk::kStage;
  const long long upr = (nst + bulk::kUnitStages - 1) / bulk::kUnitStages;
  const long long units = (long long)p.B * upr;
  const long long per_cta = (units + grid - 1) / grid;
  return (per_cta + upr - 1) / upr + 1 <= bulk::kMaxReq;
}

template <int DT, bool kEarly>
cudaError_t launch_bulk(const LinearFinalizeParams &p, unsigned grid, cudaStream_t stream) {
  static DeviceOnce once;
  const int smem = (int)sizeof(bulk::Smem);
  const cudaError_t err = smem_opt_in_once(once, bulk::draw_bulk_kernel<DT, kEarly>, smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(bulk::draw_bulk_kernel<DT, kEarly>, dim3(grid), dim3(bulk::kThreads),
                    (size_t)smem, stream, p);
}


}  // namespace

namespace {

cudaError_t launch_finalize(const LinearFinalizeParams &p, cudaStream_t stream, bool after_stats) {
  if (p.B <= 0) return cudaSuccess;
  {
    const int es = (p.dtype == SPECDEC_F32) ? 4 : 2;
    const long long nst = ((long long)p.V * es + bulk::kStage - 1) / bulk::kStage;
    const long long units = (long long)p.B * ((nst + bulk::kUnitStages - 1) / bulk::kUnitStages);
    const long long sms = device_sm_count();
    const int grid = (int)(units < sms ? units : sms);
    if (bulk_draw_applies(p, grid)) {
      const unsigned g = (unsigned)grid;
      if (after_stats)
        return (p.dtype == SPECDEC_F32) ? launch_bulk<SPECDEC_F32, true>(p, g, stream)
                                        : launch_bulk<SPECDEC_BF16, true>(p, g, stream);
      return (p.dtype == SPECDEC_F32) ? launch_bulk<SPECDEC_F32, false>(p, g, stream)
                                      : launch_bulk<SPECDEC_BF16, false>(p, g, stream);
    }
  }
  const long long items = (long long)p.B * p.nchunk;
  const long long slots = (long long)device_sm_count() * kMinBlocks;
  const unsigned grid = (unsigned)(items < slots ? items : slots);
  if (p.dtype == SPECDEC_F32)
    return launch_pdl(linear_draw_kernel<SPECDEC_F32>, dim3(grid), dim3(kThreads), 0, stream, p);
  return launch_pdl(linear_draw_kernel<SPECDEC_BF16>, dim3(grid), dim3(kThreads), 0, stream, p);
}

}  // namespace

cudaError_t launch_linear_finalize(const LinearFinalizeParams &p, cudaStream_t stream) {
  return launch_finalize(p, stream, false);
}

// Right after the stats pass of the same call (launched by this library as a
// plain launch): the draw may read the call's inputs before its dependency wait.
cudaError_t launch_linear_finalize_after_stats(const LinearFinalizeParams &p,
                                               cudaStream_t stream) {
  return launch_finalize(p, stream, true);
}

}  // namespace specdec
