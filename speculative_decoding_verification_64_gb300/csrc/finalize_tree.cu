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
//     c_{j+1} = c_j + N_j,  N_{j+1} = sum_v max(0, p_v - c_{j+1} q_v).
// In units of the row maximum (e_v = 2^((l_v - M) c), p = e / S) this reads
//     P_j = max(0, e - K_j q) / E_j,  K_0 = 0, E_0 = S,  K_{j+1} = K_j + E_j,
//     E_{j+1} = sum_v max(0, e_v - K_{j+1} q_v),
// so a rejection costs one reduction over the current node's logits and q
// rows (L2-resident after the first), and the next sibling's test needs only
// its gathered logit and q value.
//
// One 8-CTA cluster per request.  Every CTA validates the tree and gathers
// l_parent(t_n), q_parent(t_n) for all nodes; the row statistics are merged
// one eighth per CTA and pushed to the other CTAs' shared memory by
// asynchronous remote stores; then one warp finds the depths while the others
// form p_parent(t_n).  The walk is replicated in
// every CTA (the decisions depend only on those values and on exact
// fixed-point cluster sums, so all CTAs agree); reductions over the
// vocabulary are split across the cluster.
#include "finalize_common.cuh"

namespace specdec {
namespace {

using namespace fin;

constexpr int kMaxN = SPECDEC_MAX_TREE_NODES;

struct TreeSmem {
  DrawSmem ds;
  int par[kMaxN];
  int dep[kMaxN];
  int kids[kMaxN];
  float lg[kMaxN];    // l_parent(t_n)
  float pg[kMaxN];    // p_parent(t_n) before renormalisation (greedy: 1 / 0)
  float qg[kMaxN];    // q_parent(t_n)
  float rowM[kMaxN];
  float rowS[kMaxN];
  int rowA[kMaxN];    // first arg-max (greedy requests)
  int rowF[kMaxN];    // status bits of the row (partial flags, unusable statistics)
  int tok[kMaxN];     // t_n
  float uu[kMaxN];    // the request's uniforms (slot 0: final draw; slot n: test of node n)
  int path[SPECDEC_MAX_TREE_DEPTH + 1];
  int wst[kWarps];  // status bits found by each warp
  int nkids;
  alignas(8) uint64_t rbar;  // the other CTAs' merged rows have arrived
};

// warp_merge_row of a row of at most 32 stages whose partial x this lane
// holds (has: lane < the row's stage count): the same merges in the same
// order, so the result is bit-identical.
__device__ __forceinline__ RowStat warp_merge_one(const float4 x, bool has, float c) {
  float m = -INFINITY, s = 0.0f;
  int a = 0x7FFFFFFF, fl = 0;
  if (has) {
    fl |= __float_as_int(x.w);
    merge2(m, s, a, x.x, x.y, __float_as_int(x.z), c);
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

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

template <int DT>
__global__ void __cluster_dims__(kG, 1, 1) __launch_bounds__(kThreads, 2)
    tree_finalize_kernel(const TreeFinalizeParams p) {
  __shared__ TreeSmem sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const long long b = (long long)p.B - 1 - blockIdx.x / kG;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = p.N, V = p.V, D1 = p.max_depth + 1;
  const long long nodebase = b * (long long)N;
  constexpr int es = (DT == SPECDEC_F32) ? 4 : 2;

  const float T = __ldg(p.temperature + b);
  if (tid == 0) {
    exchange_init(sm.ds);
    mbar_init(&sm.rbar, 1);
    fence_mbar_init();
    // the request's status starts clean: a CTA whose exchange wait gives up
    // ORs SPECDEC_ROW_INTERNAL into it at the end (ordered after this store
    // by the cluster barrier)
    if (rank == 0) p.row_status[b] = 0;
  }
  // every CTA of the cluster is running, with its barriers initialised, before
  // any other CTA stores into its shared memory (arrive now, wait before the
  // first remote store)
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");

  // The stage partials of the first row this warp merges (rows of at most 32
  // stages: one partial a lane), loaded now so that their round trip overlaps
  // the structure loads below rather than following them.
  const int n_first = rank + kG * warp;
  const bool hoisted = p.spr <= 32;
  float4 x_first = make_float4(-INFINITY, 0.0f, __int_as_float(0x7FFFFFFF), 0.0f);
  if (hoisted && n_first < N && lane < p.spr)
    x_first = reinterpret_cast<const float4 *>(p.part + (nodebase + n_first) * (long long)p.spr)[lane];
  // ---- structure, the drafted tokens' logits and q values ---------------------
  int st = 0;
  for (int n = tid; n < N; n += kThreads) {
    const int a = __ldg(p.parent + nodebase + n);
    sm.par[n] = a;
    if (n == 0 ? (a != -1) : (a < 0 || a >= n)) st |= SPECDEC_ROW_BAD_TREE;
    sm.lg[n] = 0.0f;
    sm.qg[n] = 1.0f;
    sm.uu[n] = __ldg(p.uniforms + nodebase + n);  // the walk then needs no global load per test
    if (n == 0) continue;
    const int t = __ldg(p.tokens + nodebase + n);
    sm.tok[n] = t;
    if (t < 0 || t >= V) {
      st |= SPECDEC_ROW_BAD_TOKEN;
      continue;
    }
    if (a < 0 || a >= n) continue;
    const long long prow = nodebase + a;
    const float qt = load_elem(p.q, DT, prow * V + t);
    const float lt = load_elem(p.logits, DT, prow * V + t);
    if (!(qt > 0.0f) || qt == INFINITY) st |= SPECDEC_ROW_BAD_Q;
    sm.qg[n] = qt;
    sm.lg[n] = lt;
  }

  const bool greedy = (T == 0.0f);
  const float c = temperature_scale(T);
  if (!temperature_valid(T)) st |= SPECDEC_ROW_BAD_TEMP;
  // ---- row statistics: row n merged by warp (n / kG) % kWarps of CTA n % kG,
  // then pushed to the other CTAs by asynchronous remote stores that complete
  // on their barrier rbar (one round trip, no cluster-wide barrier)
  for (int n = rank + kG * warp; n < N; n += kG * kWarps) {
    const RowStat r = (hoisted && n == n_first) ? warp_merge_one(x_first, lane < p.spr, c)
                                                : warp_merge_row(p.part, nodebase + n, p.spr, c, lane);
    if (lane == 0) {
      sm.rowM[n] = r.M;
      sm.rowS[n] = r.S;
      sm.rowA[n] = r.arg;
      sm.rowF[n] = r.flags | (row_usable(r) ? 0 : SPECDEC_ROW_NONFINITE);
    }
  }
  const int own = (N - rank + kG - 1) / kG;  // rows n = rank + kG k of this CTA
  if (tid == 0)  // 4 words of every other CTA's row, from the kG - 1 others
    mbar_arrive_expect_tx(&sm.rbar, (uint32_t)((N - own) * 16));
  __syncthreads();  // this CTA's rows are in shared memory
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  for (int i = tid; i < own * (kG - 1) * 4; i += kThreads) {
    const int f = i & 3, rest = i >> 2;
    const int k = rest / (kG - 1), d = rest - k * (kG - 1);
    const uint32_t dst = (uint32_t)(d < rank ? d : d + 1);  // every rank but this one
    const int n = rank + kG * k;
    uint32_t *word = (f == 0) ? reinterpret_cast<uint32_t *>(&sm.rowM[n])
                     : (f == 1) ? reinterpret_cast<uint32_t *>(&sm.rowS[n])
                     : (f == 2) ? reinterpret_cast<uint32_t *>(&sm.rowA[n])
                                : reinterpret_cast<uint32_t *>(&sm.rowF[n]);
    st_async_u32(cluster_addr(smem_addr(word), dst), *word, cluster_addr(smem_addr(&sm.rbar), dst));
  }
  // the other CTAs' rows (one outcome for the CTA: a lost row would make
  // this CTA's walk differ from the others')
  if (!__syncthreads_and(mbar_wait_cluster_bounded(&sm.rbar, 0)) && tid == 0) sm.ds.lost = 1;
  for (int n = tid; n < N; n += kThreads) st |= sm.rowF[n];
  st = __reduce_or_sync(0xffffffffu, st);
  if (lane == 0) sm.wst[warp] = st;
  __syncthreads();

  // ---- depths (warp 0) and p_parent of every drafted token (the others) -------
  if (warp == 0) {
    // parent[n] < n: the depths of 32 nodes at a time, from the final depths
    // of earlier nodes and, for parents among the 32, by shuffles (a chain
    // within 32 nodes resolves one link a step)
    bool deep = false;
    for (int base = 0; base < N; base += 32) {
      const int n = base + lane;
      int a = -1, d = 0;
      bool done = true;
      if (n < N && n > 0) {
        a = sm.par[n];
        if (a >= 0 && a < n) {  // (a malformed parent is reported already)
          if (a < base) d = sm.dep[a] + 1;
          else done = false;
        }
      }
      for (int it = 0; it < 32; ++it) {
        if (!__ballot_sync(0xffffffffu, !done)) break;
        const int src = done ? lane : a - base;
        const int dp = __shfl_sync(0xffffffffu, d, src);
        const int pdone = __shfl_sync(0xffffffffu, (int)done, src);
        if (!done && pdone) {
          d = dp + 1;
          done = true;
        }
      }
      if (n < N) {
        sm.dep[n] = d;
        deep |= d > p.max_depth;
      }
      __syncwarp();
    }
    if (__any_sync(0xffffffffu, deep) && lane == 0) sm.wst[0] |= SPECDEC_ROW_BAD_TREE;
  } else {
    for (int n = tid - 32; n < N; n += kThreads - 32) {
      sm.pg[n] = 0.0f;
      if (n == 0) continue;
      const int t = sm.tok[n];
      const int a = sm.par[n];
      if (t < 0 || t >= V || a < 0 || a >= n) continue;
      if (greedy) {
        sm.pg[n] = (t == sm.rowA[a]) ? 1.0f : 0.0f;
      } else {
        RowStat r;
        r.M = sm.rowM[a];
        r.S = sm.rowS[a];
        sm.pg[n] = target_prob(sm.lg[n], r, c);
      }
    }
  }
  __syncthreads();
  int status_bits = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) status_bits |= sm.wst[w];
  const int status = status_bits;

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
        p.mass[b] = kNoMass;
      }
    }
    return;  // uniform across the cluster
  }
  if (rank == 0 && p.p_node)
    for (int n = tid; n < N; n += kThreads) p.p_node[nodebase + n] = sm.pg[n];

  // ---- the walk ------------------------------------------------------------
  // State of the current node in units of its row maximum: P_j = max(0, e - K q) / E,
  // starting from (K, E) = (0, S) with S the merged sum of the stats pass.
  int cur = 0, nacc = 0, pass = 0;
  float K = 0.0f, E = 0.0f;
  bool rejected_any = false;  // the node has a rejected child (state (K, E) in use)
  bool sums_match = false;    // the draw sums in smem are those of (cur, K)
  bool bonus = false;
  if (tid == 0) sm.path[0] = 0;
  DrawRow r;
  cta_slice(V, rank, r.v0, r.v1);
  r.c = c;
  r.use_q = false;
  r.K = 0.0f;
  for (;;) {
    __syncthreads();  // every thread is done with the previous node's child list
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
    K = 0.0f;
    E = sm.rowS[cur];
    rejected_any = false;
    sums_match = false;
    r.lrow = reinterpret_cast<const uint8_t *>(p.logits) + (size_t)(nodebase + cur) * V * es;
    r.qrow = reinterpret_cast<const uint8_t *>(p.q) + (size_t)(nodebase + cur) * V * es;
    r.M = sm.rowM[cur];
    r.vec_ok = ((reinterpret_cast<uintptr_t>(r.lrow) & 15) == 0) &&
               ((reinterpret_cast<uintptr_t>(r.qrow) & 15) == 0);
    if (nk == 0) {
      bonus = true;
      break;
    }
    int accepted = -1;
    for (int i = 0; i < nk; ++i) {
      const int child = sm.kids[i];
      const float qt = sm.qg[child];
      const float u = sm.uu[child];
      bool acc;
      if (greedy) {
        acc = (sm.pg[child] == 1.0f);
      } else if (!rejected_any) {
        // first sibling: the plain test u <= min(1, p(t) / q(t)), i.e. u q <= p
        acc = (u * qt <= sm.pg[child]);
      } else {
        // u <= min(1, P_j(t) / q(t)),  P_j(t) = max(0, e(t) - K q(t)) / E
        const float et = elem_e(r, sm.lg[child]);
        acc = (u * qt * E <= fmaxf(fmaf(-K, qt, et), 0.0f));
      }
      if (acc) {
        accepted = child;
        break;
      }
      if (greedy) continue;
      rejected_any = true;
      // rejected: K' = K + E, E' = sum max(0, e - K' q)
      const float Kn = K + E;
      r.K = Kn;
      r.use_q = true;
      draw_sums<DT>(sm.ds, r, pass);
      draw_exchange(sm.ds, cluster, pass);
      ++pass;
      if (sm.ds.Z > 0) {
        K = Kn;
        E = sm.ds.Zf;
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
    r.use_q = !bonus && K > 0.0f;
    r.K = K;
    if (!(sums_match && r.use_q)) {
      draw_sums<DT>(sm.ds, r, pass);
      draw_exchange(sm.ds, cluster, pass);
      ++pass;
    }
    const float U = sm.uu[0];
    const unsigned long long target = uniform_target(U, sm.ds.Z);
    if (rank == 0 && tid == 0) p.mass[b] = draw_mass(sm.ds.Z, sm.rowS[cur]);
    const int v = draw_search<DT>(sm.ds, r, target);
    if (tid == 0 && v >= 0) {
      p.final_token[b] = v;
      p.out_tokens[b * D1 + nacc] = v;
    }
  }
  __syncthreads();
  if (rank == 0) {
    for (int j = tid; j < D1; j += kThreads) {
      p.path_nodes[b * D1 + j] = (j <= nacc) ? sm.path[j] : -1;
      if (j < nacc) p.out_tokens[b * D1 + j] = sm.tok[sm.path[j + 1]];
      else if (j > nacc) p.out_tokens[b * D1 + j] = -1;
    }
    if (tid == 0) {
      p.n_accepted[b] = nacc;
      p.is_bonus[b] = (uint8_t)bonus;
      if (greedy) {
        p.final_token[b] = fin_tok;
        p.out_tokens[b * D1 + nacc] = fin_tok;
        p.mass[b] = kNoMass;
      }
    }
  }
  if (tid == 0 && sm.ds.lost) atomicOr(&p.row_status[b], SPECDEC_ROW_INTERNAL);
  // Every store into this CTA's shared memory has landed once its last
  // exchange wait completed (each exchange waits for all kG stores), and no
  // CTA stores after its last exchange, so CTAs leave freely.
}

}  // namespace

// A plain launch: with programmatic dependent launch the cluster grid's
// replays in a CUDA graph measured 11 us slower per step (B=32, N=64).
cudaError_t launch_tree_finalize(const TreeFinalizeParams &p, cudaStream_t stream) {
  if (p.B <= 0) return cudaSuccess;
  if (p.dtype == SPECDEC_F32)
    tree_finalize_kernel<SPECDEC_F32><<<(unsigned)(p.B * kG), kThreads, 0, stream>>>(p);
  else
    tree_finalize_kernel<SPECDEC_BF16><<<(unsigned)(p.B * kG), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace specdec
