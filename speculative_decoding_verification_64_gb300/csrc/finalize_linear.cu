// Linear verify, phase 2: accept test with early stop and the final draw
// ("Chapter 15: Decoding acceleration", section 15.1.2 steps 3 and 4; the
// bonus draw from the last target row follows section 15.1.3's expected
// count (1 - a^(g+1)) / (1 - a) of emitted tokens per step).
//
// One 8-CTA cluster per request.  Warp 0 of every CTA merges the row
// statistics of the request, gathers p_i(x~_i) and q_i(x~_i), and finds the
// first rejection with a warp ballot and find-first-set; all CTAs of the
// cluster reach the same decision.  The final row (the rejected row k, or the
// bonus row) is then drawn by inverse CDF: the cluster splits the vocabulary
// into tiles, sums the weights max(0, p - q) (or p) in 52-bit fixed point,
// exchanges the CTA totals through distributed shared memory and the CTA that
// holds the crossing U * Z locates the exact token.  Greedy requests (T = 0)
// take the first arg-max and need no pass over the vocabulary.
#include "finalize_common.cuh"

namespace specdec {
namespace {

using namespace fin;

constexpr int kMaxRows = SPECDEC_MAX_GAMMA + 1;

struct LinSmem {
  DrawSmem ds;
  float rowM[kMaxRows];
  float rowS[kMaxRows];
  int rowA[kMaxRows];   // exact arg-max (greedy requests)
  int k, status, greedy;
  float c;
};

__global__ void __cluster_dims__(kG, 1, 1) __launch_bounds__(kThreads)
    linear_finalize_kernel(const LinearFinalizeParams p) {
  __shared__ LinSmem sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const long long b = blockIdx.x / kG;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gamma = p.gamma, R = gamma + 1, V = p.V;

  if (warp == 0) {
    const float T = __ldg(p.temperature + b);
    const bool tvalid = temperature_valid(T);
    const bool greedy = (T == 0.0f);
    const float c = temperature_scale(T);
    int status = tvalid ? 0 : SPECDEC_ROW_BAD_TEMP;
    for (int i = lane; i < R; i += 32) {
      const long long row = b * R + i;
      const RowStat r = merge_row(p.part, row, p.P, c);
      status |= r.flags;
      if (!row_usable(r)) status |= SPECDEC_ROW_NONFINITE;
      sm.rowM[i] = r.M;
      sm.rowS[i] = r.S;
      sm.rowA[i] = (greedy && row_usable(r)) ? exact_argmax(p.logits, p.dtype, row * V, V, r) : 0;
    }
    __syncwarp();
    bool acc = true;
    float pd = 0.0f;
    int x = -1;
    if (lane < gamma) {
      x = __ldg(p.tokens + b * gamma + lane);
      if (x < 0 || x >= V) {
        status |= SPECDEC_ROW_BAD_TOKEN;
      } else {
        const long long row = b * R + lane;
        const float lx = load_elem(p.logits, p.dtype, row * V + x);
        const float qx = load_elem(p.q, p.dtype, (b * gamma + lane) * (long long)V + x);
        if (!(qx > 0.0f) || qx == INFINITY) status |= SPECDEC_ROW_BAD_Q;
        if (greedy) {
          acc = (x == sm.rowA[lane]);
          pd = acc ? 1.0f : 0.0f;
        } else {
          pd = exp2f((lx - sm.rowM[lane]) * c) / sm.rowS[lane];
          const float u = __ldg(p.uniforms + b * R + lane);
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
            p.final_token[b] = sm.rowA[k];
            p.out_tokens[b * R + k] = sm.rowA[k];
          }
        }
      }
    }
    if (lane == 0) {
      sm.k = k;
      sm.status = status;
      sm.greedy = greedy;
      sm.c = c;
    }
  }
  __syncthreads();
  if (sm.status || sm.greedy) return;  // uniform across the cluster

  // ---- inverse-CDF draw of the final row -----------------------------------
  const int k = sm.k;
  const int es = (p.dtype == SPECDEC_F32) ? 4 : 2;
  DrawRow r;
  r.dtype = p.dtype;
  r.V = V;
  r.M = sm.rowM[k];
  r.c = sm.c;
  r.invS = 1.0f / sm.rowS[k];
  r.lrow = reinterpret_cast<const uint8_t *>(p.logits) + (size_t)(b * R + k) * V * es;
  r.qrow = (k < gamma)
               ? reinterpret_cast<const uint8_t *>(p.q) + (size_t)(b * gamma + k) * V * es
               : nullptr;
  r.cq = (k < gamma) ? 1.0f : 0.0f;
  r.vec_ok = ((reinterpret_cast<uintptr_t>(r.lrow) & 15) == 0) &&
             (r.qrow == nullptr || (reinterpret_cast<uintptr_t>(r.qrow) & 15) == 0);
  const int nt = (V + kTile - 1) / kTile;
  const int tpc = (nt + kG - 1) / kG;
  const int t0 = min(nt, rank * tpc), t1 = min(nt, t0 + tpc);

  draw_sums(sm.ds, r, t0, t1, 0);
  draw_exchange(sm.ds, cluster, 0);
  if (sm.ds.Z == 0 && r.cq != 0.0f) {
    // residual mass 0 (only by rounding): draw from p itself
    r.cq = 0.0f;
    draw_sums(sm.ds, r, t0, t1, 1);
    draw_exchange(sm.ds, cluster, 1);
  }
  const float U = __ldg(p.uniforms + b * R + gamma);
  const unsigned long long target = uniform_target(U, sm.ds.Z);
  const int v = draw_search(sm.ds, r, t0, t1, target);
  if (tid == 0 && v >= 0) {
    p.final_token[b] = v;
    p.out_tokens[b * R + k] = v;
  }
  cluster.sync();  // keep this CTA's shared memory alive for the others' reads
}

}  // namespace

cudaError_t launch_linear_finalize(const LinearFinalizeParams &p, cudaStream_t stream) {
  if (p.B <= 0) return cudaSuccess;
  linear_finalize_kernel<<<(unsigned)(p.B * kG), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace specdec
