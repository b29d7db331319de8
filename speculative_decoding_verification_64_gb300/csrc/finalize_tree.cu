// Token-tree verify, phase 2: the sibling walk.
//
// The candidate tree of "Chapter 15: Decoding acceleration" (section 15.4.1,
// T = (V, E, P)) is verified with the speculative sampling test of section
// 15.1.2 applied to several i.i.d. drafts of the same position: the children
// of the current node are tried in ascending node index; the first accepted
// child becomes the current node; after a rejected child the current target
// distribution P is replaced by max(0, P - q) / sum (residual renormalised);
// when all children are rejected the final token is drawn from that residual,
// and at a leaf a bonus token is drawn from the leaf's own target row.
//
// The kernel never stores a residual row.  By induction, after j rejections
//     P_j = max(0, p - c_j q) / N_j,  c_0 = 0, N_0 = 1,
//     c_{j+1} = c_j + N_j,  N_{j+1} = sum_v max(0, p_v - c_{j+1} q_v),
// so each rejection costs one reduction over the (L2-resident) logits and q
// rows of the current node, and the test of the next sibling needs only its
// gathered p(t) and q(t).
//
// One 8-CTA cluster per request.  Every CTA validates the tree, merges the
// row statistics and gathers p_parent(t_n), q_parent(t_n) for all nodes; the
// walk itself is replicated in every CTA (the decisions depend only on those
// shared values and on exact fixed-point cluster sums, so all CTAs agree);
// reductions over the vocabulary are split across the cluster.
#include "finalize_common.cuh"

namespace specdec {
namespace {

using namespace fin;

constexpr int kMaxN = SPECDEC_MAX_TREE_NODES;

struct TreeSmem {
  DrawSmem ds;
  int par[kMaxN];
  int anc[kMaxN];
  int dep[kMaxN];
  int kids[kMaxN];
  float pg[kMaxN];    // p_parent(t_n) before renormalisation (greedy: 1 / 0)
  float qg[kMaxN];    // q_parent(t_n)
  float rowM[kMaxN];
  float rowS[kMaxN];
  int rowA[kMaxN];    // exact arg-max (greedy requests)
  int path[SPECDEC_MAX_TREE_DEPTH + 1];
  int status, nkids;
};

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__global__ void __cluster_dims__(kG, 1, 1) __launch_bounds__(kThreads)
    tree_finalize_kernel(const TreeFinalizeParams p) {
  __shared__ TreeSmem sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const long long b = blockIdx.x / kG;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = p.N, V = p.V, D1 = p.max_depth + 1;
  const long long nodebase = b * (long long)N;

  const float T = __ldg(p.temperature + b);
  const bool greedy = (T == 0.0f);
  const float c = temperature_scale(T);
  if (tid == 0) sm.status = temperature_valid(T) ? 0 : SPECDEC_ROW_BAD_TEMP;
  __syncthreads();

  // ---- structure, tokens, row statistics ---------------------------------
  int st = 0;
  for (int n = tid; n < N; n += kThreads) {
    const int a = __ldg(p.parent + nodebase + n);
    sm.par[n] = a;
    if (n == 0 ? (a != -1) : (a < 0 || a >= n)) st |= SPECDEC_ROW_BAD_TREE;
    sm.anc[n] = (n == 0) ? -1 : a;
    sm.dep[n] = (n == 0) ? 0 : 1;
    const RowStat r = merge_row(p.part, nodebase + n, p.P, c);
    st |= r.flags;
    const bool ok = row_usable(r);
    if (!ok) st |= SPECDEC_ROW_NONFINITE;
    sm.rowM[n] = r.M;
    sm.rowS[n] = r.S;
    sm.rowA[n] = (greedy && ok) ? exact_argmax(p.logits, p.dtype, (nodebase + n) * V, V, r) : 0;
  }
  if (st) atomicOr(&sm.status, st);
  __syncthreads();
  const bool tree_ok = !(sm.status & SPECDEC_ROW_BAD_TREE);
  if (tree_ok) {
    // depths by pointer jumping (parent[n] < n, so every chain ends at the root)
    for (int it = 0; it < 11; ++it) {
      int na[kMaxN / kThreads], nd[kMaxN / kThreads];
#pragma unroll
      for (int k = 0; k < kMaxN / kThreads; ++k) {
        const int n = tid + k * kThreads;
        if (n < N) {
          const int a = sm.anc[n];
          na[k] = (a > 0) ? sm.anc[a] : a;
          nd[k] = (a > 0) ? sm.dep[n] + sm.dep[a] : sm.dep[n];
        }
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kMaxN / kThreads; ++k) {
        const int n = tid + k * kThreads;
        if (n < N) {
          sm.anc[n] = na[k];
          sm.dep[n] = nd[k];
        }
      }
      __syncthreads();
    }
  }
  st = 0;
  for (int n = tid; n < N; n += kThreads) {
    if (tree_ok && sm.dep[n] > p.max_depth) st |= SPECDEC_ROW_BAD_TREE;
    if (n == 0) {
      sm.pg[0] = 0.0f;
      sm.qg[0] = 1.0f;
      continue;
    }
    const int t = __ldg(p.tokens + nodebase + n);
    const int a = sm.par[n];
    sm.pg[n] = 0.0f;
    sm.qg[n] = 1.0f;
    if (t < 0 || t >= V) {
      st |= SPECDEC_ROW_BAD_TOKEN;
      continue;
    }
    if (a < 0 || a >= n) continue;
    const long long prow = nodebase + a;
    const float qt = load_elem(p.q, p.dtype, prow * V + t);
    if (!(qt > 0.0f) || qt == INFINITY) st |= SPECDEC_ROW_BAD_Q;
    sm.qg[n] = qt;
    if (greedy) {
      sm.pg[n] = (t == sm.rowA[a]) ? 1.0f : 0.0f;
    } else {
      const float lt = load_elem(p.logits, p.dtype, prow * V + t);
      sm.pg[n] = exp2f((lt - sm.rowM[a]) * c) / sm.rowS[a];
    }
  }
  if (st) atomicOr(&sm.status, st);
  __syncthreads();
  const int status = sm.status;

  if (status) {
    if (rank == 0) {
      for (int j = tid; j < D1; j += kThreads) {
        p.path_nodes[b * D1 + j] = -1;
        p.out_tokens[b * D1 + j] = -1;
      }
      if (p.p_node)
        for (int n = tid; n < N; n += kThreads) p.p_node[nodebase + n] = __int_as_float(0x7fc00000);
      if (tid == 0) {
        p.n_accepted[b] = 0;
        p.final_token[b] = -1;
        p.is_bonus[b] = 0;
        p.row_status[b] = status;
      }
    }
    return;  // uniform across the cluster
  }
  if (rank == 0 && p.p_node)
    for (int n = tid; n < N; n += kThreads) p.p_node[nodebase + n] = sm.pg[n];

  // ---- the walk ------------------------------------------------------------
  const int es = (p.dtype == SPECDEC_F32) ? 4 : 2;
  const int nt = (V + kTile - 1) / kTile;
  const int tpc = (nt + kG - 1) / kG;
  const int t0 = min(nt, rank * tpc), t1 = min(nt, t0 + tpc);
  int cur = 0, nacc = 0, pass = 0;
  float cj = 0.0f;       // c_j of the current node
  double Nj = 1.0;       // N_j of the current node
  bool sums_match = false;  // the draw sums in smem are those of (cur, cj)
  bool bonus = false;
  if (tid == 0) sm.path[0] = 0;
  DrawRow r;
  r.dtype = p.dtype;
  r.V = V;
  r.c = c;
  for (;;) {
    __syncthreads();  // every thread is done with the previous node's child list
    // children of cur, ascending
    if (warp == 0) {
      int cnt = 0;
      for (int base = cur + 1; base < N; base += 32) {
        const int n = base + lane;
        const bool is = (n < N) && sm.par[n] == cur;
        const unsigned m = __ballot_sync(0xffffffffu, is);
        if (is) sm.kids[cnt + __popc(m & lanemask_lt())] = n;
        cnt += __popc(m);
      }
      if (lane == 0) sm.nkids = cnt;
    }
    __syncthreads();
    const int nk = sm.nkids;
    cj = 0.0f;
    Nj = 1.0;
    sums_match = false;
    if (nk == 0) {
      bonus = true;
      break;
    }
    r.lrow = reinterpret_cast<const uint8_t *>(p.logits) + (size_t)(nodebase + cur) * V * es;
    r.qrow = reinterpret_cast<const uint8_t *>(p.q) + (size_t)(nodebase + cur) * V * es;
    r.M = sm.rowM[cur];
    r.invS = 1.0f / sm.rowS[cur];
    r.vec_ok = ((reinterpret_cast<uintptr_t>(r.lrow) & 15) == 0) &&
               ((reinterpret_cast<uintptr_t>(r.qrow) & 15) == 0);
    int accepted = -1;
    for (int i = 0; i < nk; ++i) {
      const int child = sm.kids[i];
      const double pt = sm.pg[child], qt = sm.qg[child];
      bool acc;
      if (greedy) {
        acc = (pt == 1.0);
      } else {
        // u <= min(1, P_j(t) / q(t)),  P_j(t) = max(0, p(t) - c_j q(t)) / N_j
        const double u = __ldg(p.uniforms + nodebase + child);
        const double num = fmax(pt - (double)cj * qt, 0.0);
        acc = (u * qt * Nj <= num);
      }
      if (acc) {
        accepted = child;
        break;
      }
      if (greedy) continue;
      // rejected: N_{j+1} = sum max(0, p - c_{j+1} q) over the vocabulary
      const float cn = (float)((double)cj + Nj);
      r.cq = cn;
      draw_sums(sm.ds, r, t0, t1, pass);
      draw_exchange(sm.ds, cluster, pass);
      ++pass;
      const unsigned long long Zn = sm.ds.Z;
      if (Zn > 0) {
        cj = cn;
        Nj = (double)Zn * 0x1p-52;
        sums_match = true;
      } else {
        sums_match = false;  // keep P (rounding-only case)
      }
    }
    if (accepted < 0) break;
    ++nacc;
    cur = accepted;
    if (tid == 0) sm.path[nacc] = cur;
  }

  // ---- final draw -------------------------------------------------------------
  int fin_tok = -1;
  if (greedy) {
    fin_tok = sm.rowA[cur];
  } else {
    if (bonus) {
      r.lrow = reinterpret_cast<const uint8_t *>(p.logits) + (size_t)(nodebase + cur) * V * es;
      r.qrow = nullptr;
      r.M = sm.rowM[cur];
      r.invS = 1.0f / sm.rowS[cur];
      r.vec_ok = (reinterpret_cast<uintptr_t>(r.lrow) & 15) == 0;
    }
    r.cq = bonus ? 0.0f : cj;
    if (!sums_match) {
      draw_sums(sm.ds, r, t0, t1, pass);
      draw_exchange(sm.ds, cluster, pass);
      ++pass;
    }
    const float U = __ldg(p.uniforms + nodebase);
    const unsigned long long target = uniform_target(U, sm.ds.Z);
    const int v = draw_search(sm.ds, r, t0, t1, target);
    if (tid == 0 && v >= 0) {
      p.final_token[b] = v;
      p.out_tokens[b * D1 + nacc] = v;
    }
  }
  __syncthreads();
  if (rank == 0) {
    for (int j = tid; j < D1; j += kThreads) {
      p.path_nodes[b * D1 + j] = (j <= nacc) ? sm.path[j] : -1;
      if (j < nacc) p.out_tokens[b * D1 + j] = __ldg(p.tokens + nodebase + sm.path[j + 1]);
      else if (j > nacc) p.out_tokens[b * D1 + j] = -1;
    }
    if (tid == 0) {
      p.n_accepted[b] = nacc;
      p.is_bonus[b] = (uint8_t)bonus;
      p.row_status[b] = 0;
      if (greedy) {
        p.final_token[b] = fin_tok;
        p.out_tokens[b * D1 + nacc] = fin_tok;
      }
    }
  }
  if (!greedy) cluster.sync();  // the other CTAs may still read this CTA's smem
}

}  // namespace

cudaError_t launch_tree_finalize(const TreeFinalizeParams &p, cudaStream_t stream) {
  if (p.B <= 0) return cudaSuccess;
  tree_finalize_kernel<<<(unsigned)(p.B * kG), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace specdec
