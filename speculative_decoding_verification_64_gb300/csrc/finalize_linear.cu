// Linear verify, phase 2: accept test with early stop and the final draw
// ("Chapter 15: Decoding acceleration", section 15.1.2 steps 3 and 4; the
// bonus draw from the last target row follows section 15.1.3's expected
// count (1 - a^(g+1)) / (1 - a) of emitted tokens per step).
//
// One 8-CTA cluster per request.  In every CTA the warps merge the stage
// partials of the request's rows in parallel while warp 0 gathers q_i(x~_i)
// and l_i(x~_i); warp 0 then runs the accept test and finds the first
// rejection k with a ballot and find-first-set.  All CTAs of a cluster reach
// the same decision from the same data.  The final row (rejected row k, or
// the bonus row) is drawn by inverse CDF split across the cluster in one pass
// over its logits (and q): weights max(0, e_v - S q_v) = S max(0, p - q) for
// a rejection, e_v = S p for the bonus, with e_v = 2^((l_v - M) c); CTA
// totals meet through distributed shared memory and the CTA holding the
// crossing U * Z finds the token.  Greedy requests (T = 0) take the first
// arg-max and need no pass.  Clusters take the requests in reverse order so
// the rows the stats pass read last, still in L2, are drawn first.
#include "finalize_common.cuh"

namespace specdec {
namespace {

using namespace fin;

constexpr int kMaxRows = SPECDEC_MAX_GAMMA + 1;

struct LinSmem {
  DrawSmem ds;
  RowStat row[kMaxRows];
  int k, status, greedy;
};

template <int DT>
__global__ void __cluster_dims__(kG, 1, 1) __launch_bounds__(kThreads, 2)
    linear_finalize_kernel(const LinearFinalizeParams p) {
  __shared__ LinSmem sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const long long b = (long long)p.B - 1 - blockIdx.x / kG;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gamma = p.gamma, R = gamma + 1, V = p.V;
  constexpr int es = (DT == SPECDEC_F32) ? 4 : 2;

  const float T = __ldg(p.temperature + b);
  const bool greedy = (T == 0.0f);
  const float c = temperature_scale(T);

  // ---- gathers (warp 0) and row merges (all warps) -------------------------
  int x = -1;
  float lx = 0.0f, qx = 1.0f, u = 0.0f;
  if (warp == 0 && lane < gamma) {
    x = __ldg(p.tokens + b * gamma + lane);
    u = __ldg(p.uniforms + b * R + lane);
    if (x >= 0 && x < V) {
      lx = load_elem(p.logits, DT, (b * R + lane) * (long long)V + x);
      qx = load_elem(p.q, DT, (b * gamma + lane) * (long long)V + x);
    }
  }
  for (int i = warp; i < R; i += kWarps) {
    const RowStat r = warp_merge_row(p.part, b * R + i, p.spr, c, lane);
    if (lane == 0) sm.row[i] = r;
  }
  __syncthreads();

  // ---- accept test ---------------------------------------------------------
  if (warp == 0) {
    int status = temperature_valid(T) ? 0 : SPECDEC_ROW_BAD_TEMP;
    for (int i = lane; i < R; i += 32) {
      status |= sm.row[i].flags;
      if (!row_usable(sm.row[i])) status |= SPECDEC_ROW_NONFINITE;
    }
    bool acc = true;
    float pd = 0.0f;
    if (lane < gamma) {
      if (x < 0 || x >= V) {
        status |= SPECDEC_ROW_BAD_TOKEN;
      } else {
        if (!(qx > 0.0f) || qx == INFINITY) status |= SPECDEC_ROW_BAD_Q;
        if (greedy) {
          acc = (x == sm.row[lane].arg);
          pd = acc ? 1.0f : 0.0f;
        } else {
          pd = target_prob(lx, sm.row[lane], c);
          // u <= min(1, p/q)  <=>  u q <= p  for q > 0, u < 1 (exact products in float64)
          acc = ((double)u * (double)qx <= (double)pd);
        }
      }
    }
    status = __reduce_or_sync(0xffffffffu, status);
    const unsigned rej = __ballot_sync(0xffffffffu, lane < gamma && !acc);
    const int k = rej ? (__ffs(rej) - 1) : gamma;
    if (rank == 0) {
      if (status) {
        for (int j = lane; j < R; j += 32) p.out_tokens[b * R + j] = -1;
        if (p.p_draft && lane < gamma) p.p_draft[b * gamma + lane] = __int_as_float(0x7fc00000);
        if (lane == 0) {
          p.n_accepted[b] = 0;
          p.final_token[b] = -1;
          p.is_bonus[b] = 0;
          p.row_status[b] = status;
        }
      } else {
        for (int j = lane; j < R; j += 32) {
          if (j < k) p.out_tokens[b * R + j] = __ldg(p.tokens + b * gamma + j);
          else if (j > k) p.out_tokens[b * R + j] = -1;
        }
        if (p.p_draft && lane < gamma) p.p_draft[b * gamma + lane] = pd;
        if (lane == 0) {
          p.n_accepted[b] = k;
          p.is_bonus[b] = (uint8_t)(k == gamma);
          p.row_status[b] = 0;
          if (greedy) {
            p.final_token[b] = sm.row[k].arg;
            p.out_tokens[b * R + k] = sm.row[k].arg;
          }
        }
      }
    }
    if (lane == 0) {
      sm.k = k;
      sm.status = status;
      sm.greedy = greedy;
    }
  }
  __syncthreads();
  if (sm.status || sm.greedy) return;  // uniform across the cluster

  // ---- inverse-CDF draw of the final row -------------------------------------
  const int k = sm.k;
  DrawRow r;
  r.V = V;
  r.M = sm.row[k].M;
  r.c = c;
  r.lrow = reinterpret_cast<const uint8_t *>(p.logits) + (size_t)(b * R + k) * V * es;
  r.qrow = (k < gamma)
               ? reinterpret_cast<const uint8_t *>(p.q) + (size_t)(b * gamma + k) * V * es
               : r.lrow;
  r.use_q = (k < gamma);  // residual max(0, e - S q) = S max(0, p - q); bonus: e = S p
  r.K = sm.row[k].S;
  r.vec_ok = ((reinterpret_cast<uintptr_t>(r.lrow) & 15) == 0) &&
             ((reinterpret_cast<uintptr_t>(r.qrow) & 15) == 0);
  int t0, t1;
  cta_tiles(V, rank, t0, t1);
  draw_sums<DT>(sm.ds, r, t0, t1, 0);
  draw_exchange(sm.ds, cluster, 0);
  if (r.use_q && sm.ds.Z == 0) {
    // residual mass 0 (only by rounding): draw from p itself
    r.use_q = false;
    draw_sums<DT>(sm.ds, r, t0, t1, 1);
    draw_exchange(sm.ds, cluster, 1);
  }
  const float U = __ldg(p.uniforms + b * R + gamma);
  const unsigned long long target = uniform_target(U, sm.ds.Z);
  const int v = draw_search<DT>(sm.ds, r, t0, t1, target);
  if (tid == 0 && v >= 0) {
    p.final_token[b] = v;
    p.out_tokens[b * R + k] = v;
  }
  cluster.sync();  // keep this CTA's shared memory alive for the others' reads
}

}  // namespace

cudaError_t launch_linear_finalize(const LinearFinalizeParams &p, cudaStream_t stream) {
  if (p.B <= 0) return cudaSuccess;
  if (p.dtype == SPECDEC_F32)
    linear_finalize_kernel<SPECDEC_F32><<<(unsigned)(p.B * kG), kThreads, 0, stream>>>(p);
  else
    linear_finalize_kernel<SPECDEC_BF16><<<(unsigned)(p.B * kG), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace specdec
