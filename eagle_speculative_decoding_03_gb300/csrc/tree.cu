// Tree bookkeeping of the draft step: roots, per-depth expansion, final rerank.
//
// Node ids per request: 0 is the root; generated nodes are numbered in generation
// order (depth, then the frontier slot of the expanded row, then token id).  A node's
// path value V = V(parent) + log p(token) is the log of the product of draft
// confidences along its path ("EAGLE-2 - context-aware dynamic tree", zackli.ai
// "Speculative Decoding Deep Dive III"; "EAGLE-2: expand and rerank", aicassindra.com).
// Static trees (EAGLE-1, "Drafting a Tree, Not a Chain", stable-lab) expand every
// child; dynamic trees keep the top-k children of the depth by V as the next frontier
// and the top-m of all generated nodes at the end.  Every selection uses one total
// order: larger value first, ties to the smaller token id / node id.
#include "common.cuh"
#include "internal.h"

namespace eagle {

// ---------------------------------------------------------------- roots
__global__ void tree_init_kernel(const TreeArgs t, const RowMeta r0) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= t.B) return;
  int nb = __ldg(t.cu_seqlens + b + 1) - __ldg(t.cu_seqlens + b);
  if (nb < 0 || nb > t.max_prefix) {
    atomicOr(t.err, DEVERR_PREFIX);
    nb = nb < 0 ? 0 : t.max_prefix;
  }
  t.n_eff[b] = nb;
  int tok = __ldg(t.root_tok + b);
  if (tok < 0 || tok >= t.vocab) {       // never let a bad id reach an embedding-row address
    atomicOr(t.err, DEVERR_TOKEN);
    tok = 0;
  }
  const size_t nbase = static_cast<size_t>(b) * t.max_nodes;
  t.node_tok[nbase] = tok;
  t.node_parent[nbase] = -1;
  t.node_depth[nbase] = 0;
  t.node_row[nbase] = -1;
  t.node_logv[nbase] = 0.f;
  t.slot_mask[static_cast<size_t>(b) * t.tree_rows] = 1ull;
  r0.req[b] = b;
  r0.slot[b] = 0;
  r0.pos[b] = nb;
  r0.tok[b] = tok;
  r0.feat[b] = b;
  r0.node[b] = 0;
  r0.mask[b] = 1ull;
}

// ---------------------------------------------- merge of LM-head partials
// One warp merges the G per-CTA partial states of GEMM row n: log-sum-exp and the
// top-`kout` (value, id).  Lane r < kout returns the r-th best (descending).
// `cand` is the warp's shared-memory staging area (G * kp entries).
EAGLE_DEV void merge_lm_row(const LmPartials& lm, int N, int kp, int n, int kout, float2* cand,
                            float& lse, float& my_val, int& my_id, int lane) {
  const int G = lm.G, T = lm.T;
  float M = -INFINITY;
  for (int t = lane; t < T; t += 32) M = fmaxf(M, __ldcg(lm.max + static_cast<size_t>(t) * N + n));
  M = warp_max(M);
  float s = 0.f;
  for (int t = lane; t < T; t += 32) {
    const float mt = __ldcg(lm.max + static_cast<size_t>(t) * N + n);
    if (mt != -INFINITY) s += __ldcg(lm.sum + static_cast<size_t>(t) * N + n) * expf(mt - M);
  }
  s = warp_sum(s);
  lse = M + logf(s);

  const int tot = G * kp;
  for (int c = lane; c < tot; c += 32) {
    const int g = c / kp, j = c - g * kp;
    const size_t o = (static_cast<size_t>(g) * N + n) * kp + j;
    cand[c] = make_float2(__ldcg(lm.val + o), __int_as_float(__ldcg(lm.id + o)));
  }
  __syncwarp();
  float lastv = INFINITY;
  int lasti = -1;
  my_val = -INFINITY;
  my_id = -1;
  for (int r = 0; r < kout; ++r) {
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int c = lane; c < tot; c += 32) {
      const float2 e = cand[c];
      const int id = __float_as_int(e.y);
      if (id < 0) continue;
      if ((r == 0 || beats(lastv, lasti, e.x, id)) && beats(e.x, id, bv, bi)) { bv = e.x; bi = id; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (beats(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (bi == INT_MAX) break;
    if (lane == r) { my_val = bv; my_id = bi; }
    lastv = bv;
    lasti = bi;
  }
  __syncwarp();
}

// ------------------------------------------------------------ expansion
constexpr int EXP_WARPS = 8;

__global__ void __launch_bounds__(EXP_WARPS * 32)
expand_kernel(const TreeArgs t, const int s, const LmPartials lm, const RowMeta cur, const RowMeta nxt,
              const ExpandTrace tr, const int kp) {
  extern __shared__ float2 exp_smem[];
  __shared__ int sel_rank[256];
  __shared__ int sel_pos[256];
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = t.rows[s - 1], kids = t.kids[s - 1];
  const int N = t.B * R;
  const size_t nb0 = static_cast<size_t>(b) * t.max_nodes;
  const int base = t.node_base[s - 1];
  float2* cand = exp_smem + static_cast<size_t>(warp) * lm.G * kp;

  // children of every row of this request
  for (int i = warp; i < R; i += EXP_WARPS) {
    const int n = b * R + i;
    float lse, v;
    int id;
    merge_lm_row(lm, N, kp, n, kids, cand, lse, v, id, lane);
    // order the kids winners by token id
    int rank = 0;
    for (int j = 0; j < kids; ++j) {
      const int oj = __shfl_sync(0xffffffffu, id, j);
      rank += (lane < kids && oj < id) ? 1 : 0;
    }
    const int u = __ldcg(cur.node + n);
    const float vu = __ldcg(t.node_logv + nb0 + u);
    if (lane < kids) {
      const int c = base + i * kids + rank;
      const float lp = v - lse;
      t.node_tok[nb0 + c] = id;
      t.node_parent[nb0 + c] = u;
      t.node_depth[nb0 + c] = s;
      t.node_row[nb0 + c] = __ldcg(cur.slot + n);
      t.node_logv[nb0 + c] = vu + lp;
      if (tr.children) {
        tr.children[static_cast<size_t>(n) * tr.k_max + rank] = id;
        tr.child_logp[static_cast<size_t>(n) * tr.k_max + rank] = lp;
      }
    }
    if (tr.lse && lane == 0) tr.lse[n] = lse;
  }
  if (s >= t.depth) return;
  __syncthreads();

  // next frontier among the R * kids children of this depth
  const int nc = R * kids;
  const int F = t.rows[s];
  if (t.tree_kind == 1) {  // static: every child, in generation order
    for (int c = tid; c < nc; c += blockDim.x) sel_pos[c] = c;
  } else {
    for (int c = tid; c < nc; c += blockDim.x) {
      const float vc = __ldcg(t.node_logv + nb0 + base + c);
      int rk = 0;
      for (int c2 = 0; c2 < nc; ++c2) {
        const float v2 = __ldcg(t.node_logv + nb0 + base + c2);
        rk += beats(v2, c2, vc, c) ? 1 : 0;
      }
      sel_rank[c] = rk;
    }
    __syncthreads();
    for (int c = tid; c < nc; c += blockDim.x) {
      if (sel_rank[c] >= F) continue;
      int p = 0;
      for (int c2 = 0; c2 < c; ++c2) p += sel_rank[c2] < F ? 1 : 0;
      sel_pos[p] = c;
    }
  }
  __syncthreads();
  const int slot0 = t.row_base[s];
  for (int j = tid; j < F; j += blockDim.x) {
    const int u = base + sel_pos[j];
    const int n2 = b * F + j;
    const int slot = slot0 + j;
    const int srow = __ldcg(t.node_row + nb0 + u);
    const unsigned long long m = __ldcg(t.slot_mask + static_cast<size_t>(b) * t.tree_rows + srow) |
                                 (1ull << slot);
    t.slot_mask[static_cast<size_t>(b) * t.tree_rows + slot] = m;
    t.frontier[b * 64 + j] = u;
    nxt.req[n2] = b;
    nxt.slot[n2] = slot;
    nxt.pos[n2] = __ldcg(t.n_eff + b) + s;
    nxt.tok[n2] = __ldcg(t.node_tok + nb0 + u);
    nxt.feat[n2] = b * R + (srow - t.row_base[s - 1]);
    nxt.node[n2] = u;
    nxt.mask[n2] = m;
    if (tr.frontier) tr.frontier[b * tr.f_max + j] = u;
  }
}

// ---------------------------------------------------------------- rerank
constexpr int RR_THREADS = 1024;

__global__ void __launch_bounds__(RR_THREADS) rerank_kernel(const TreeArgs t, const OutArgs o) {
  __shared__ int keep[RR_THREADS];
  __shared__ int scan[RR_THREADS];
  __shared__ int slot_node[64];
  __shared__ int slot_par[64];
  __shared__ unsigned long long anc[64];
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, tid = threadIdx.x;
  const size_t nb0 = static_cast<size_t>(b) * t.max_nodes;
  const int G = t.node_base[t.depth] - 1;     // generated nodes: ids 1..G
  const int S = t.slots;
  // kept flags (node c = tid + 1)
  int kf = 0;
  if (tid < G) {
    const int c = tid + 1;
    if (t.tree_kind == 1) {
      kf = 1;
    } else {
      const float vc = __ldcg(t.node_logv + nb0 + c);
      int rk = 0;
      for (int c2 = 1; c2 <= G; ++c2) rk += beats(__ldcg(t.node_logv + nb0 + c2), c2, vc, c) ? 1 : 0;
      kf = rk < t.m;
    }
  }
  keep[tid] = kf;
  scan[tid] = kf;
  __syncthreads();
  for (int off = 1; off < RR_THREADS; off <<= 1) {
    const int add = tid >= off ? scan[tid - off] : 0;
    __syncthreads();
    scan[tid] += add;
    __syncthreads();
  }
  if (tid == 0) slot_node[0] = 0;
  if (tid < G && keep[tid]) slot_node[scan[tid]] = tid + 1;   // inclusive scan: slot = 1 + #kept before
  __syncthreads();
  // parents as slots: binary search of the parent node among kept slots (sorted ids)
  if (tid < S) {
    const int c = slot_node[tid];
    int ps = -1;
    if (tid > 0) {
      const int p = __ldcg(t.node_parent + nb0 + c);
      int lo = 0, hi = S - 1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (slot_node[mid] < p) lo = mid + 1; else hi = mid;
      }
      ps = slot_node[lo] == p ? lo : -1;
    }
    slot_par[tid] = ps;
    const size_t ob = static_cast<size_t>(b) * S + tid;
    o.tokens[ob] = __ldcg(t.node_tok + nb0 + c);
    o.parents[ob] = ps;
    o.positions[ob] = __ldcg(t.n_eff + b) + __ldcg(t.node_depth + nb0 + c);
    o.logv[ob] = __ldcg(t.node_logv + nb0 + c);
    if (o.final_nodes) o.final_nodes[ob] = c;
  }
  __syncthreads();
  if (tid == 0) {
    for (int i = 0; i < S; ++i) anc[i] = (i == 0 || slot_par[i] < 0 ? 0ull : anc[slot_par[i]]) | (1ull << i);
  }
  __syncthreads();
  for (int idx = tid; idx < S * S; idx += RR_THREADS) {
    const int i = idx / S, j = idx - i * S;
    o.mask[static_cast<size_t>(b) * S * S + idx] = static_cast<unsigned char>((anc[i] >> j) & 1ull);
  }
}

// ----------------------------------------------------- standalone merge
__global__ void __launch_bounds__(EXP_WARPS * 32)
lm_merge_kernel(const LmPartials lm, int N, int k, int* ids, float* logp, float* lse_out) {
  extern __shared__ float2 mg_smem[];
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * EXP_WARPS + warp;
  if (n >= N) return;
  float2* cand = mg_smem + static_cast<size_t>(warp) * lm.G * k;
  float lse, v;
  int id;
  merge_lm_row(lm, N, k, n, k, cand, lse, v, id, lane);
  if (lane < k) {
    ids[static_cast<size_t>(n) * k + lane] = id;
    logp[static_cast<size_t>(n) * k + lane] = v - lse;
  }
  if (lane == 0) lse_out[n] = lse;
}

// ================================================================== host side
static cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                                   cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.stream = st;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  return cfg;
}

cudaError_t tree_setup_attributes() {
  cudaError_t e = allow_max_smem(reinterpret_cast<const void*>(expand_kernel));
  if (e != cudaSuccess) return e;
  return allow_max_smem(reinterpret_cast<const void*>(lm_merge_kernel));
}

cudaError_t launch_tree_init(const TreeArgs& t, const RowMeta& rows0, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3((t.B + 63) / 64), dim3(64), 0, st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, tree_init_kernel, t, rows0);
}

static size_t merge_smem(int G, int kp) { return sizeof(float2) * EXP_WARPS * static_cast<size_t>(G) * kp; }

cudaError_t launch_expand(const TreeArgs& t, int s, const LmPartials& lm, const RowMeta& cur,
                          const RowMeta& next, const ExpandTrace& tr, cudaStream_t st, bool pdl) {
  const int kp = t.kids[s - 1];
  const size_t smem = merge_smem(lm.G, kp);
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(t.B), dim3(EXP_WARPS * 32), smem, st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, expand_kernel, t, s, lm, cur, next, tr, kp);
}

cudaError_t launch_rerank(const TreeArgs& t, const OutArgs& o, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(t.B), dim3(RR_THREADS), 0, st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, rerank_kernel, t, o);
}

cudaError_t launch_lm_merge(const LmPartials& lm, int N, int k, int* ids, float* logp, float* lse,
                            cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg =
      make_cfg(dim3((N + EXP_WARPS - 1) / EXP_WARPS), dim3(EXP_WARPS * 32), merge_smem(lm.G, k), st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, lm_merge_kernel, lm, N, k, ids, logp, lse);
}

}  // namespace eagle
