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
  r0.v[b] = 0.f;
}

// ------------------------------------------------------- fc operand copy
// One item = 8 consecutive columns of one row: a feature chunk (copied hi/lo, or split
// from fp32) or an embedding chunk (hi = the bf16 value, lo = 0).
__global__ void __launch_bounds__(256) fc_operand_kernel(const FcOperandArgs a) {
  // Trigger first: the fc GEMM that follows launches now and streams its weights while
  // this kernel still waits for the frontier; it reads this kernel's rows only after its
  // own wait.
  pdl_trigger();
  pdl_wait();
  const int chunks = a.d / 8;
  const long long total = static_cast<long long>(a.N) * 2 * chunks;
  const size_t ld = 2 * static_cast<size_t>(a.d);
  for (long long it = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; it < total;
       it += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(it / (2 * chunks)), c = static_cast<int>(it - static_cast<long long>(n) * 2 * chunks);
    uint4* hi = reinterpret_cast<uint4*>(a.out + 2 * static_cast<size_t>(n) * ld) + c;
    uint4* lo = reinterpret_cast<uint4*>(a.out + (2 * static_cast<size_t>(n) + 1) * ld) + c;
    if (c < chunks) {
      const int f = __ldcg(a.row_feat + n);
      if (a.feat_hl) {
        const uint4 h = __ldcg(reinterpret_cast<const uint4*>(a.feat_hl + 2 * static_cast<size_t>(f) * a.d) + c);
        const uint4 l = __ldcg(reinterpret_cast<const uint4*>(a.feat_hl + (2 * static_cast<size_t>(f) + 1) * a.d) + c);
        *hi = h;
        *lo = l;
      } else {
        const float4* src = reinterpret_cast<const float4*>(a.feat + static_cast<size_t>(f) * a.ldf) + 2 * c;
        const float4 x0 = __ldcg(src), x1 = __ldcg(src + 1);
        const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        uint16_t hv[8], lv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) split_hilo(xv[e], hv[e], lv[e]);
        *hi = make_uint4(hv[0] | (uint32_t(hv[1]) << 16), hv[2] | (uint32_t(hv[3]) << 16), hv[4] | (uint32_t(hv[5]) << 16),
                         hv[6] | (uint32_t(hv[7]) << 16));
        *lo = make_uint4(lv[0] | (uint32_t(lv[1]) << 16), lv[2] | (uint32_t(lv[3]) << 16), lv[4] | (uint32_t(lv[5]) << 16),
                         lv[6] | (uint32_t(lv[7]) << 16));
      }
    } else {
      int t = __ldcg(a.row_tok + n);
      t = (t < 0 || t >= a.vocab) ? 0 : t;   // never an address outside the table
      *hi = __ldg(reinterpret_cast<const uint4*>(a.emb + static_cast<size_t>(t) * a.d) + (c - chunks));
      *lo = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// Operand copy of bf16 rows (EAGLE-3's fused root features): row n of x [N][K] (stride ldx)
// -> rows 2n (the values) and 2n + 1 (zeros) of out [2N][K]; one item = 8 columns.
__global__ void __launch_bounds__(256) bf16_operand_kernel(const uint16_t* x, int N, int K, int ldx, uint16_t* out) {
  pdl_trigger();
  pdl_wait();
  const int chunks = K / 8;
  const long long total = static_cast<long long>(N) * chunks;
  for (long long it = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; it < total;
       it += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int n = static_cast<int>(it / chunks), c = static_cast<int>(it - static_cast<long long>(n) * chunks);
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(n) * ldx) + c);
    reinterpret_cast<uint4*>(out + 2 * static_cast<size_t>(n) * K)[c] = v;
    reinterpret_cast<uint4*>(out + (2 * static_cast<size_t>(n) + 1) * K)[c] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// ---------------------------------------------- merge of LM-head partials
constexpr int MERGE_MAX_G = 256;   // CTAs (lists) one warp can merge: 8 lists per lane

// The top-`kout` of G sorted (best first) lists of kp entries staged in shared memory,
// as a tournament: kout rounds of warp arg-max over the list heads, advancing the
// winner's list.  Lane r < kout returns the r-th best.
EAGLE_DEV void tournament(const float2* cand, int G, int kp, int kout, float& my_val, int& my_id, int lane) {
  int ptr[MERGE_MAX_G / 32];
#pragma unroll
  for (int i = 0; i < MERGE_MAX_G / 32; ++i) ptr[i] = 0;
  my_val = -INFINITY;
  my_id = -1;
  for (int r = 0; r < kout; ++r) {
    float bv = -INFINITY;
    int bi = INT_MAX, bl = -1;
#pragma unroll
    for (int i = 0; i < MERGE_MAX_G / 32; ++i) {
      const int c = lane + 32 * i;
      if (c < G && ptr[i] < kp) {
        const float2 e = cand[c * kp + ptr[i]];
        const int id = __float_as_int(e.y);
        if (id >= 0 && beats(e.x, id, bv, bi)) {
          bv = e.x;
          bi = id;
          bl = i;
        }
      }
    }
    float wv = bv;
    int wi = bi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, wv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, wi, o);
      if (beats(ov, oi, wv, wi)) { wv = ov; wi = oi; }
    }
    if (wi == INT_MAX) break;
    if (bi == wi) {   // token ids are unique: this lane holds the winning head
#pragma unroll
      for (int i = 0; i < MERGE_MAX_G / 32; ++i)
        if (i == bl) ++ptr[i];
    }
    if (lane == r) {
      my_val = wv;
      my_id = wi;
    }
  }
  __syncwarp();
}

// One warp merges the partial states of GEMM row n: the log-sum-exp over the per-tile
// (max, sum of exp) pairs, and the top-`kout` (value, id) of the G per-CTA top-kp lists
// (each sorted best first).  The lists are staged in shared memory (`cand`, G * kp) and
// merged as a tournament: kout rounds of warp arg-max over the list heads, advancing the
// winner's list.  Lane r < kout returns the r-th best.
EAGLE_DEV void merge_lm_row(const LmPartials& lm, int N, int kp, int n, int kout, float2* cand,
                            float& lse, float& my_val, int& my_id, int lane) {
  // log-sum-exp: loads issued in independent batches, combined online per lane in tile
  // order, then a symmetric butterfly (every lane ends with the same value)
  float m = -INFINITY, sm = 0.f;
  for (int t0 = 0; t0 < lm.T; t0 += 32 * 8) {
    float mb[8], sb[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int t = t0 + u * 32 + lane;
      mb[u] = t < lm.T ? __ldcg(lm.max + static_cast<size_t>(n) * lm.T + t) : -INFINITY;
      sb[u] = t < lm.T ? __ldcg(lm.sum + static_cast<size_t>(n) * lm.T + t) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (mb[u] == -INFINITY) continue;
      if (mb[u] > m) {
        sm = sm * expf(m - mb[u]) + sb[u];
        m = mb[u];
      } else {
        sm += sb[u] * expf(mb[u] - m);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o);
    const float os = __shfl_xor_sync(0xffffffffu, sm, o);
    const float M = fmaxf(m, om);
    sm = (m == -INFINITY ? 0.f : sm * expf(m - M)) + (om == -INFINITY ? 0.f : os * expf(om - M));
    m = M;
  }
  lse = m + logf(sm);

  // stage the lists (loads issued in independent batches of 8 per lane)
  const int G = lm.G, tot = G * kp;
  for (int c0 = 0; c0 < tot; c0 += 32 * 8) {
    float vb[8];
    int ib[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int c = c0 + u * 32 + lane;
      if (c < tot) {
        const size_t o = static_cast<size_t>(n) * tot + c;
        vb[u] = __ldcg(lm.val + o);
        ib[u] = __ldcg(lm.id + o);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int c = c0 + u * 32 + lane;
      if (c < tot) cand[c] = make_float2(vb[u], __int_as_float(ib[u]));
    }
  }
  __syncwarp();
  tournament(cand, G, kp, kout, my_val, my_id, lane);
}

// --------------------------------------------- LM-head selection from logits
// For launches with many rows the LM-head GEMM only stores the rows' logits; this kernel
// then takes, per (row, vocabulary part), the part's log-sum-exp state and its top-k keys,
// in the per-CTA-list / per-tile-state layout the expansion merges (lists = parts, tiles =
// parts).  Keys are the logits, or (sampled drafting) the logits plus the row's Gumbel
// noise.  Exact top-k on order-preserving 32-bit images of the keys, ties to the lower
// token id.  One warp per part of 1024 keys (32 in each lane's registers): every reduction
// is a shuffle and nothing waits on a block barrier.
constexpr int SEL_WARPS = 8;                       // parts per CTA
constexpr int SEL_PER = 32;                        // keys per lane: key i of a part in lane i % 32
constexpr int SEL_SPAN = 32 * SEL_PER;             // 1024 keys per part
constexpr int SEL_MAX_PARTS = 256;                 // lists the expansion merges per row
constexpr int SEL_CAP = 64;                        // candidates the threshold gather keeps per warp
static_assert(KMAX <= 32, "the threshold takes the k-th largest of the 32 lane maxima");

// order-preserving image of a float: larger float -> larger integer; NaN -> 0 (below all)
EAGLE_DEV uint32_t key_bits(float x) {
  if (x != x) return 0u;
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
EAGLE_DEV float key_float(uint32_t b) {
  return __uint_as_float((b & 0x80000000u) ? (b & 0x7FFFFFFFu) : ~b);
}
// Scratch of block_select_top: a 256-bin histogram, per-warp totals, the chosen digit.
struct SelectScratch {
  int hist[256];
  int wtot[32];
  int bin, above;
};

// The k best of up to NT keys, one per thread (0 = no key): larger key first, ties to the lower
// thread index.  A radix select on 8-bit digits from the top (histogram updates aggregated per
// warp over lanes with the same digit), then the keys equal to the k-th in thread order.  Every
// thread of the block calls it; returns whether this thread's key is among the k.
template <int NT>
EAGLE_DEV bool block_select_top(uint32_t kb, int k, SelectScratch& sc) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int present = __syncthreads_count(kb != 0u);
  int krem = min(k, present);
  if (krem <= 0) return false;
  uint32_t prefix = 0u, pmask = 0u;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += NT) sc.hist[i] = 0;
    __syncthreads();
    const bool in = kb != 0u && (kb & pmask) == prefix;
    const uint32_t dig = (kb >> shift) & 255u;
    const unsigned act = __ballot_sync(0xffffffffu, in);
    if (in) {
      const unsigned peers = __match_any_sync(act, dig);
      if (lane == __ffs(peers) - 1) atomicAdd(sc.hist + dig, __popc(peers));
    }
    __syncthreads();
    if (warp == 0) {   // the bin holding the krem-th largest, scanning down from bin 255
      int c[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = sc.hist[255 - (lane * 8 + j)];
        tot += c[j];
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - tot;
      if (excl < krem && incl >= krem) {
        int run = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (run < krem && run + c[j] >= krem) {
            sc.bin = 255 - (lane * 8 + j);
            sc.above = run;
          }
          run += c[j];
        }
      }
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(sc.bin) << shift;
    pmask |= 255u << shift;
    krem -= sc.above;
    __syncthreads();   // every thread has read bin / above before the next pass
  }
  const bool eq = kb != 0u && kb == prefix;
  const unsigned bal = __ballot_sync(0xffffffffu, eq);
  if (lane == 0) sc.wtot[warp] = __popc(bal);
  __syncthreads();
  int before = __popc(bal & ((1u << lane) - 1u));
  for (int w = 0; w < warp; ++w) before += sc.wtot[w];
  const bool keep = kb > prefix || (eq && before < krem);
  __syncthreads();   // the scratch may be reused by the caller
  return keep;
}

// Per-warp scratch: the gathered candidates, and the radix histogram of the fallback.
struct WarpSelect {
  uint32_t key[SEL_CAP];
  int id[SEL_CAP];
  int hist[256];
};

// Descending bitonic sort of one float per lane across the warp (NaN-free inputs).
EAGLE_DEV float warp_sort_desc(float x, int lane) {
#pragma unroll
  for (int k2 = 2; k2 <= 32; k2 <<= 1)
#pragma unroll
    for (int j2 = k2 >> 1; j2 > 0; j2 >>= 1) {
      const float y = __shfl_xor_sync(0xffffffffu, x, j2);
      x = (((lane & j2) == 0) == ((lane & k2) == 0)) ? fmaxf(x, y) : fminf(x, y);
    }
  return x;
}

// Selection values s (the logits, or with SAMPLED the logits plus the row's Gumbel noise) of
// one 1024-key part, key i = lane + 32 j in s[j] of each lane; past the part: -inf.  The
// fast path compares floats: theta, the ks-th largest of the 32 lane maxima, is at most the
// ks-th largest key (ks lanes hold a value >= theta), so the top ks are among the values
// >= theta (usually a few more than ks); those are ranked exactly on order-preserving keys.
// A part with NaN, theta = -inf or more than SEL_CAP such values takes the radix select.
template <bool SAMPLED>
__global__ void __launch_bounds__(SEL_WARPS * 32, SAMPLED ? 2 : 4)
lm_select_kernel(const float* __restrict__ logits, int V, int parts, int items, int k,
                 const unsigned long long* seeds, int sample_rows, int sample_depth, int row0,
                 float* out_max, float* out_sum, float* out_val, int* out_id) {
  __shared__ WarpSelect ws_all[SEL_WARPS];
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int item = blockIdx.x * SEL_WARPS + warp;
  if (item >= items) return;   // whole warps only: nothing below waits on the block
  WarpSelect& ws = ws_all[warp];
  const unsigned lt = (1u << lane) - 1u;
  const int n = item / parts, part = item - n * parts;   // n: row of this launch
  const int base = part * SEL_SPAN;
  const int len = max(0, min(SEL_SPAN, V - base));
  const float* x = logits + static_cast<size_t>(n) * V + base;
  float s[SEL_PER];
#pragma unroll
  for (int j = 0; j < SEL_PER; ++j) {
    const int i = lane + 32 * j;
    s[j] = i < len ? __ldcg(x + i) : -INFINITY;
  }
  // the part's log-sum-exp state: its maximum m, and the sum of exp(logit - m) (NaN when a
  // logit is NaN: the maximum skips NaN, the sum does not)
  float lmax = -INFINITY;
#pragma unroll
  for (int j = 0; j < SEL_PER; ++j) lmax = fmaxf(lmax, s[j]);
  float m = lmax;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float ms = m == -INFINITY ? 0.f : m;
  int ks = min(k, len);   // keys to select when no logit is NaN
  float sm = 0.f, theta;
  int cnt = 0;
  if (!SAMPLED) {
    theta = __shfl_sync(0xffffffffu, warp_sort_desc(lmax, lane), ks - 1);
#pragma unroll
    for (int j = 0; j < SEL_PER; ++j) {
      sm += __expf(s[j] - ms);
      cnt += s[j] >= theta;
    }
  } else {
#pragma unroll
    for (int j = 0; j < SEL_PER; ++j) sm += __expf(s[j] - ms);
    // Gumbel noise of token t = base + lane + 32 j: word j % 4 of the Philox block of
    // counter (32 (t / 128) + t % 32, row, depth, 0), shared by j = 4q .. 4q + 3
    const int gr = row0 + n, sb = gr / sample_rows;
    const unsigned long long sd = __ldg(seeds + sb);
    lmax = -INFINITY;
#pragma unroll
    for (int q = 0; q < SEL_PER / 4; ++q) {
      const uint4 w = philox4x32_10(make_uint4(32u * static_cast<uint32_t>((base >> 7) + q) + lane,
                                               static_cast<uint32_t>(gr - sb * sample_rows),
                                               static_cast<uint32_t>(sample_depth), 0u),
                                    static_cast<uint32_t>(sd), static_cast<uint32_t>(sd >> 32));
      const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 4 * q + e;
        if (lane + 32 * j < len) s[j] += gumbel_of_word(wd[e]);
        lmax = fmaxf(lmax, s[j]);
      }
    }
    theta = __shfl_sync(0xffffffffu, warp_sort_desc(lmax, lane), ks - 1);
#pragma unroll
    for (int j = 0; j < SEL_PER; ++j) cnt += s[j] >= theta;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
  int incl = cnt;   // inclusive prefix of the counts over lanes
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  int nc = __shfl_sync(0xffffffffu, incl, 31);
  if (lane == 0) {
    out_max[static_cast<size_t>(n) * parts + part] = m;
    out_sum[static_cast<size_t>(n) * parts + part] = sm;
  }
  if (sm == sm && theta > -INFINITY && nc <= SEL_CAP) {
    int pos = incl - cnt;
#pragma unroll
    for (int j = 0; j < SEL_PER; ++j)
      if (s[j] >= theta) {
        ws.key[pos] = key_bits(s[j]);
        ws.id[pos] = base + lane + 32 * j;
        ++pos;
      }
  } else {
    // radix select on 8-bit digits of the keys (0 = past the part or NaN) from the top, then
    // the keys equal to the k-th in id order; the keys replace the values in s (their bits)
    int nv = 0;
#pragma unroll
    for (int j = 0; j < SEL_PER; ++j) {
      const uint32_t kb = lane + 32 * j < len ? key_bits(s[j]) : 0u;
      nv += kb != 0u;
      s[j] = __uint_as_float(kb);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nv += __shfl_xor_sync(0xffffffffu, nv, o);
    ks = min(k, nv);
    uint32_t prefix = 0u, pmask = 0u;
    int krem = ks;
    for (int shift = 24; shift >= 0 && ks > 0; shift -= 8) {
      for (int b = lane; b < 256; b += 32) ws.hist[b] = 0;
      __syncwarp();
#pragma unroll
      for (int j = 0; j < SEL_PER; ++j) {
        const uint32_t kb = __float_as_uint(s[j]);
        if (kb != 0u && (kb & pmask) == prefix) atomicAdd(ws.hist + ((kb >> shift) & 255u), 1);
      }
      __syncwarp();
      int c[8], tot = 0;   // bins 255 - (8 lane + jj), scanned from the top
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        c[jj] = ws.hist[255 - (lane * 8 + jj)];
        tot += c[jj];
      }
      int hi = tot;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, hi, d);
        if (lane >= d) hi += y;
      }
      const int excl = hi - tot;
      int bin = 0, above = 0;
      if (excl < krem && hi >= krem) {
        int run = excl;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          if (run < krem && run + c[jj] >= krem) {
            bin = 255 - (lane * 8 + jj);
            above = run;
          }
          run += c[jj];
        }
      }
      const unsigned who = __ballot_sync(0xffffffffu, excl < krem && hi >= krem);
      const int src = __ffs(who) - 1;
      bin = __shfl_sync(0xffffffffu, bin, src);
      above = __shfl_sync(0xffffffffu, above, src);
      prefix |= static_cast<uint32_t>(bin) << shift;
      pmask |= 255u << shift;
      krem -= above;
      __syncwarp();   // every lane has read the histogram before the next pass clears it
    }
    // keys above the k-th: all; keys equal to it: the krem of lowest id (id order: j, then lane)
    int eq_seen = 0, taken = 0;
#pragma unroll
    for (int j = 0; j < SEL_PER; ++j) {
      const uint32_t kb = __float_as_uint(s[j]);
      const bool eq = ks > 0 && kb == prefix;
      const unsigned em = __ballot_sync(0xffffffffu, eq);
      const bool take = ks > 0 && (kb > prefix || (eq && eq_seen + __popc(em & lt) < krem));
      eq_seen += __popc(em);
      const unsigned tm = __ballot_sync(0xffffffffu, take);
      if (take) {
        const int pos = taken + __popc(tm & lt);
        ws.key[pos] = kb;
        ws.id[pos] = base + lane + 32 * j;
      }
      taken += __popc(tm);
    }
    nc = taken;   // == ks
  }
  __syncwarp();
  // the ks best candidates, best first (larger key, then lower id); empty places: -inf / -1
  const size_t o = (static_cast<size_t>(n) * parts + part) * k;
  for (int c = lane; c < nc; c += 32) {
    const uint32_t kk = ws.key[c];
    const int id = ws.id[c];
    int rank = 0;
    for (int c2 = 0; c2 < nc; ++c2) rank += ws.key[c2] > kk || (ws.key[c2] == kk && ws.id[c2] < id);
    if (rank < ks) {
      out_val[o + rank] = key_float(kk);
      out_id[o + rank] = id;
    }
  }
  if (lane >= ks && lane < k) {
    out_val[o + lane] = -INFINITY;
    out_id[o + lane] = -1;
  }
}

// ------------------------------------------------------------ expansion
// One CTA per row (frontier node) of the depth: log-sum-exp and top-k children of the
// row, written to the node table; the last CTA of a request to finish (arrival counter)
// selects the request's next frontier and writes the next depth's row metadata.
constexpr int EXR_THREADS = 256;
constexpr int EXR_WARPS = EXR_THREADS / 32;
constexpr int EXR_CAND = 4096;          // candidates a row can keep (G <= 256 lists of <= 16)

__global__ void __launch_bounds__(EXR_THREADS)
expand_kernel(const TreeArgs t, const int s, const LmPartials lm, const RowMeta cur, const RowMeta nxt,
              const ExpandTrace tr, const int kp, int* counters, float* scratch_v, int* scratch_tok) {
  extern __shared__ float2 cand[];                 // [EXR_CAND]
  __shared__ float red_m[EXR_WARPS], red_s[EXR_WARPS];
  __shared__ float wb_v[EXR_WARPS];
  __shared__ int wb_i[EXR_WARPS];
  __shared__ float2 sel[KMAX];
  __shared__ int ncand;
  __shared__ float s_lse;
  __shared__ int s_last;
  __shared__ float sv[256];
  __shared__ int spos[256];
  __shared__ int wcount[EXR_WARPS];
  __shared__ int s_u, s_slot, s_neff;
  __shared__ float s_vu;
  __shared__ unsigned long long s_pmask[64];
  __shared__ SelectScratch ex_sel;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = t.rows[s - 1], kids = t.kids[s - 1];
  const int n = blockIdx.x, b = n / R, i = n - b * R;
  const size_t nb0 = static_cast<size_t>(b) * t.max_nodes;
  const int base = t.node_base[s - 1];
  const int G = lm.G;

  // Metadata, loaded into registers together with the partials (one round trip): the
  // row's node, value and slot, the prefix length, and the masks of the request's rows
  // (parents of the next frontier, used by the request's last row to finish).
  int r_u = 0, r_slot = 0, r_neff = 0;
  float r_vu = 0.f;
  unsigned long long r_mask = 0ull;
  if (tid == 0) {
    r_u = __ldcg(cur.node + n);
    r_vu = __ldcg(cur.v + n);
    r_slot = __ldcg(cur.slot + n);
    r_neff = __ldcg(t.n_eff + b);
  }
  if (tid < R && s < t.depth) r_mask = __ldcg(cur.mask + b * R + tid);

  // ---- log-sum-exp over the row's per-tile pairs (loads batched ahead of the arithmetic)
  float m = -INFINITY, sm = 0.f;
  const float* pm = lm.max + static_cast<size_t>(n) * lm.T;
  const float* ps = lm.sum + static_cast<size_t>(n) * lm.T;
  for (int t0 = tid; t0 < lm.T; t0 += 4 * EXR_THREADS) {
    float mt[4], st[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int tt = t0 + j * EXR_THREADS;
      mt[j] = tt < lm.T ? __ldcg(pm + tt) : -INFINITY;
      st[j] = tt < lm.T ? __ldcg(ps + tt) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (mt[j] == -INFINITY) continue;
      if (mt[j] > m) {
        sm = sm * expf(m - mt[j]) + st[j];
        m = mt[j];
      } else {
        sm += st[j] * expf(mt[j] - m);
      }
    }
  }
  // this thread's CTA list, whole (sorted best first; empty entries have id -1)
  float lv[KMAX];
  int li[KMAX];
  const size_t lbase = static_cast<size_t>(n) * G * kp;
  if (tid < G) {
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < kp) {
        lv[j] = __ldcg(lm.val + lbase + static_cast<size_t>(tid) * kp + j);
        li[j] = __ldcg(lm.id + lbase + static_cast<size_t>(tid) * kp + j);
      }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o);
    const float os = __shfl_xor_sync(0xffffffffu, sm, o);
    const float M = fmaxf(m, om);
    sm = (m == -INFINITY ? 0.f : sm * expf(m - M)) + (om == -INFINITY ? 0.f : os * expf(om - M));
    m = M;
  }
  if (lane == 0) {
    red_m[warp] = m;
    red_s[warp] = sm;
  }
  // a row with fewer than kids valid candidates (non-finite logits) keeps distinct
  // out-of-range placeholders, caught below before they can index anything
  if (tid < KMAX) sel[tid] = make_float2(-INFINITY, __int_as_float(-1 - tid));
  if (tid == 0) {
    ncand = 0;
    s_u = r_u;
    s_vu = r_vu;
    s_slot = r_slot;
    s_neff = r_neff;
  }
  if (tid < R) s_pmask[tid] = r_mask;
  __syncthreads();
  // Pruning bound: in each warp, the kids-th best of its lanes' list heads; then the best
  // of those.  The kids best heads of any subset of the lists are distinct entries no
  // worse than the subset's kids-th head, so each of the row's top-kids entries is no
  // worse than the bound (value-then-id order): only entries the bound does not beat can
  // be kept.  Ranks within a warp come from shuffles, not shared-memory loops.
  {
    float hv = -INFINITY;
    int hid = INT_MAX;   // empty
    if (tid < G && li[0] >= 0) {
      hv = lv[0];
      hid = li[0];
    }
    int rk = 0;
#pragma unroll 8
    for (int o = 1; o < 32; ++o) {
      const int src = (lane + o) & 31;
      const float ov = __shfl_sync(0xffffffffu, hv, src);
      const int oi = __shfl_sync(0xffffffffu, hid, src);
      rk += (oi != INT_MAX) & ((ov > hv) | ((ov == hv) & (oi < hid)));
    }
    const int nv = __popc(__ballot_sync(0xffffffffu, hid != INT_MAX));
    if (lane == 0) {
      wb_v[warp] = -INFINITY;
      wb_i[warp] = INT_MAX;
    }
    __syncwarp();
    if (nv >= kids && hid != INT_MAX && rk == kids - 1) {
      wb_v[warp] = hv;
      wb_i[warp] = hid;
    }
  }
  if (tid == 32) {
    float M = -INFINITY, S = 0.f;
    for (int w = 0; w < EXR_WARPS; ++w) {
      const float mw = red_m[w], sw = red_s[w];
      const float MM = fmaxf(M, mw);
      S = (M == -INFINITY ? 0.f : S * expf(M - MM)) + (mw == -INFINITY ? 0.f : sw * expf(mw - MM));
      M = MM;
    }
    s_lse = M + logf(S);
  }
  __syncthreads();
  // ---- candidates: list entries that the bound does not beat
  if (tid < G) {
    float tv = -INFINITY;
    int ti = INT_MAX;
#pragma unroll
    for (int w = 0; w < EXR_WARPS; ++w)
      if (wb_i[w] != INT_MAX && beats(wb_v[w], wb_i[w], tv, ti)) {
        tv = wb_v[w];
        ti = wb_i[w];
      }
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < kp && li[j] >= 0 && !beats(tv, ti, lv[j], li[j]))
        cand[atomicAdd(&ncand, 1)] = make_float2(lv[j], __int_as_float(li[j]));
  }
  __syncthreads();
  const int nc = ncand;
  for (int c = tid; c < nc; c += EXR_THREADS) {
    const float2 e = cand[c];
    const int id = __float_as_int(e.y);
    int rank = 0;
#pragma unroll 8
    for (int c2 = 0; c2 < nc; ++c2) {
      const float2 f = cand[c2];
      const int fid = __float_as_int(f.y);
      rank += (f.x > e.x) | ((f.x == e.x) & (fid < id));
    }
    if (rank < kids) sel[rank] = e;
  }
  __syncthreads();
  // ---- children in token-id order (greedy) or draw order (sampled)
  const int u = s_u;
  if (tid < kids) {
    float v = sel[tid].x;
    int id = __float_as_int(sel[tid].y);
    int rank = 0;
    if (t.seeds) {
      // sampled drafting: sel holds logit + Gumbel noise in draw order; the children keep
      // that order and their log-probabilities drop the noise again
      rank = tid;
      if (id >= 0 && id < t.vocab) v -= token_gumbel(id, i, s, __ldg(t.seeds + b));
    } else {
      for (int j = 0; j < kids; ++j) rank += __float_as_int(sel[j].y) < id ? 1 : 0;
    }
    if (id < 0 || id >= t.vocab) {
      atomicOr(t.err, DEVERR_SELECT);
      id = 0;
    }
    const int c = i * kids + rank;
    const float lp = v - s_lse;
    const float vc = s_vu + lp;
    t.node_tok[nb0 + base + c] = id;
    t.node_parent[nb0 + base + c] = u;
    t.node_depth[nb0 + base + c] = s;
    t.node_row[nb0 + base + c] = s_slot;
    t.node_logv[nb0 + base + c] = vc;
    scratch_v[b * 256 + c] = vc;
    scratch_tok[b * 256 + c] = id;
    if (tr.children) {
      tr.children[static_cast<size_t>(n) * tr.k_max + rank] = id;
      tr.child_logp[static_cast<size_t>(n) * tr.k_max + rank] = lp;
    }
  }
  if (tr.lse && tid == 0) tr.lse[n] = s_lse;
  if (s >= t.depth) return;

  // ---- the last row of the request to finish selects the next frontier
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(counters + b, 1) == R - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid == 0) counters[b] = 0;
  const int nc2 = R * kids;
  const int F = t.rows[s];
  if (t.tree_kind == 1) {  // static: every child, in generation order
    for (int c = tid; c < nc2; c += EXR_THREADS) {
      spos[c] = c;
      sv[c] = rank_value(__ldcg(scratch_v + b * 256 + c));
    }
  } else {
    // the F best children (value, then generation index), kept in generation order: block
    // radix select over the depth's children (one per thread, nc2 <= 256)
    const float vc = tid < nc2 ? rank_value(__ldcg(scratch_v + b * 256 + tid)) : -INFINITY;
    if (tid < nc2) sv[tid] = vc;
    const bool keep = block_select_top<EXR_THREADS>(tid < nc2 ? key_bits(vc) : 0u, F, ex_sel);
    const int idc = tid;
    const unsigned kb = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) wcount[warp] = __popc(kb);
    __syncthreads();
    if (keep) {
      int p = __popc(kb & ((1u << lane) - 1u));
      for (int w = 0; w < warp; ++w) p += wcount[w];
      spos[p] = idc;
    }
  }
  __syncthreads();
  const int slot0 = t.row_base[s];
  const int neff = s_neff;
  for (int j = tid; j < F; j += EXR_THREADS) {
    const int c = spos[j];
    const int uu = base + c;
    const int pi = c / kids;                        // the row that generated the child
    const int n2 = b * F + j;
    const int slot = slot0 + j;
    const unsigned long long mk = s_pmask[pi] | (1ull << slot);
    t.slot_mask[static_cast<size_t>(b) * t.tree_rows + slot] = mk;
    t.frontier[b * 64 + j] = uu;
    nxt.req[n2] = b;
    nxt.slot[n2] = slot;
    nxt.pos[n2] = neff + s;
    nxt.tok[n2] = __ldcg(scratch_tok + b * 256 + c);
    nxt.feat[n2] = b * R + pi;
    nxt.node[n2] = uu;
    nxt.mask[n2] = mk;
    nxt.v[n2] = sv[c];
    if (tr.frontier) tr.frontier[b * tr.f_max + j] = uu;
  }
}

// ---------------------------------------------------------------- rerank
constexpr int RR_THREADS = 1024;

__global__ void __launch_bounds__(RR_THREADS) rerank_kernel(const TreeArgs t, const OutArgs o) {
  __shared__ int keep[RR_THREADS];
  __shared__ int scan[RR_THREADS];
  __shared__ float vals[RR_THREADS];        // node tid + 1: value as ranked
  __shared__ int npar[RR_THREADS];          // node tid + 1: parent node
  __shared__ int slot_of[RR_THREADS + 1];   // node -> kept slot (-1: not kept)
  __shared__ int ntok[RR_THREADS + 1], ndep[RR_THREADS + 1];
  __shared__ float nlogv[RR_THREADS + 1];
  __shared__ int slot_node[64];
  __shared__ int slot_par[64];
  __shared__ unsigned long long anc[64];
  __shared__ SelectScratch rr_sel;
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, tid = threadIdx.x;
  const size_t nb0 = static_cast<size_t>(b) * t.max_nodes;
  const int G = t.node_base[t.depth] - 1;     // generated nodes: ids 1..G (node 0: the root)
  const int S = t.slots;
  // one batch of loads: every node's value, parent, token and depth, and the prefix length
  for (int c = tid; c <= G; c += RR_THREADS) {   // G + 1 <= 1025 nodes
    const float lv = __ldcg(t.node_logv + nb0 + c);
    nlogv[c] = lv;
    ntok[c] = __ldcg(t.node_tok + nb0 + c);
    ndep[c] = __ldcg(t.node_depth + nb0 + c);
    slot_of[c] = -1;
    if (c >= 1) {
      vals[c - 1] = rank_value(lv);
      npar[c - 1] = __ldcg(t.node_parent + nb0 + c);
    }
  }
  const int neff = __ldcg(t.n_eff + b);
  __syncthreads();
  // kept flags (node c = tid + 1): static trees keep every node, dynamic ones the m best by V
  // (ties to the lower generation index = the lower thread), by block radix select
  int kf = 0;
  if (t.tree_kind == 1) {
    kf = tid < G;
  } else {
    kf = block_select_top<RR_THREADS>(tid < G ? key_bits(vals[tid]) : 0u, t.m, rr_sel);
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
  if (tid == 0) {
    slot_node[0] = 0;
    slot_of[0] = 0;
  }
  if (tid < G && keep[tid] && scan[tid] < S) {   // inclusive scan: slot = 1 + #kept before
    slot_node[scan[tid]] = tid + 1;
    slot_of[tid + 1] = scan[tid];
  }
  __syncthreads();
  // emitted slots in generation order; parents as slots (a kept node's parent is kept:
  // V never increases along a path and a parent precedes its children in the tie order)
  if (tid < S) {
    const int c = slot_node[tid];
    const int ps = tid > 0 ? slot_of[npar[c - 1]] : -1;
    slot_par[tid] = ps;
    const size_t ob = static_cast<size_t>(b) * S + tid;
    o.tokens[ob] = ntok[c];
    o.parents[ob] = ps;
    o.positions[ob] = neff + ndep[c];
    o.logv[ob] = nlogv[c];
    if (o.final_nodes) o.final_nodes[ob] = c;
  }
  __syncthreads();
  if (tid < S) {   // ancestor-or-self bits: walk the slot's parent chain
    unsigned long long a = 0ull;
    for (int j = tid, step = 0; j >= 0 && step < 64; j = slot_par[j], ++step) a |= 1ull << j;
    anc[tid] = a;
  }
  __syncthreads();
  for (int idx = tid; idx < S * S; idx += RR_THREADS) {
    const int i = idx / S, j = idx - i * S;
    o.mask[static_cast<size_t>(b) * S * S + idx] = static_cast<unsigned char>((anc[i] >> j) & 1ull);
  }
}

// ----------------------------------------------------- standalone merge
constexpr size_t MERGE_SMEM_BUDGET = 180 * 1024;
constexpr int MG_MAX_WARPS = 16;
static int merge_warps(int G, int kp) {
  const size_t per = sizeof(float2) * static_cast<size_t>(G) * kp;
  int w = static_cast<int>(MERGE_SMEM_BUDGET / per);
  return w < 1 ? 1 : (w > MG_MAX_WARPS ? MG_MAX_WARPS : w);
}

__global__ void __launch_bounds__(MG_MAX_WARPS * 32)
lm_merge_kernel(const LmPartials lm, int N, int k, int* ids, float* logp, float* lse_out) {
  extern __shared__ float2 mg_smem[];
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * (blockDim.x >> 5) + warp;
  if (n >= N) return;
  if (lm.poison_if && __ldcg(lm.poison_if) != 0u) {
    // the LM-head kernel gave up part-way: its partials are incomplete, so no row is merged
    if (lane < k) {
      ids[static_cast<size_t>(n) * k + lane] = -1;
      logp[static_cast<size_t>(n) * k + lane] = __int_as_float(0x7fc00000);
    }
    if (lane == 0) lse_out[n] = __int_as_float(0x7fc00000);
    return;
  }
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
  cudaError_t e = cudaFuncSetAttribute(expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sizeof(float2) * EXR_CAND));
  if (e != cudaSuccess) return e;
  return allow_max_smem(reinterpret_cast<const void*>(lm_merge_kernel));
}

cudaError_t launch_tree_init(const TreeArgs& t, const RowMeta& rows0, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3((t.B + 63) / 64), dim3(64), 0, st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, tree_init_kernel, t, rows0);
}

static size_t merge_smem(int G, int kp) {
  return sizeof(float2) * merge_warps(G, kp) * static_cast<size_t>(G) * kp;
}

cudaError_t launch_expand(const TreeArgs& t, int s, const LmPartials& lm, const RowMeta& cur,
                          const RowMeta& next, const ExpandTrace& tr, cudaStream_t st, bool pdl) {
  const int kp = t.kids[s - 1];
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(t.B * t.rows[s - 1]), dim3(EXR_THREADS), sizeof(float2) * EXR_CAND, st,
                                    pdl, attr);
  return cudaLaunchKernelEx(&cfg, expand_kernel, t, s, lm, cur, next, tr, kp, t.exp_counters, t.exp_v, t.exp_tok);
}

cudaError_t launch_rerank(const TreeArgs& t, const OutArgs& o, cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(t.B), dim3(RR_THREADS), 0, st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, rerank_kernel, t, o);
}

cudaError_t launch_bf16_operand(const uint16_t* x, int N, int K, int ldx, uint16_t* out, cudaStream_t st, bool pdl) {
  if (N < 1 || K % 8 != 0 || ldx % 8 != 0) return cudaErrorInvalidValue;
  const long long items = static_cast<long long>(N) * (K / 8);
  long long blocks = (items + 255) / 256;
  if (blocks > 1216) blocks = 1216;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, bf16_operand_kernel, x, N, K, ldx, out);
}

cudaError_t launch_fc_operand(const FcOperandArgs& a, cudaStream_t st, bool pdl) {
  const long long items = static_cast<long long>(a.N) * 2 * (a.d / 8);
  long long blocks = (items + 255) / 256;
  if (blocks > 1216) blocks = 1216;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, fc_operand_kernel, a);
}

cudaError_t launch_lm_merge(const LmPartials& lm, int N, int k, int* ids, float* logp, float* lse,
                            cudaStream_t st, bool pdl) {
  cudaLaunchAttribute attr[1];
  const int w = merge_warps(lm.G, k);
  cudaLaunchConfig_t cfg = make_cfg(dim3((N + w - 1) / w), dim3(w * 32), merge_smem(lm.G, k), st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, lm_merge_kernel, lm, N, k, ids, logp, lse);
}

}  // namespace eagle

namespace eagle {

// the vocabulary parts of 1024 keys, or 0 past 256 parts (no select kernel: the LM head then
// keeps its fused top-k epilogue)
int lm_select_parts(int vocab) {
  const int parts = (vocab + SEL_SPAN - 1) / SEL_SPAN;
  return vocab > 0 && parts <= SEL_MAX_PARTS ? parts : 0;
}

cudaError_t launch_lm_select(const float* logits, int N, int vocab, int k, const unsigned long long* seeds,
                             int sample_rows, int sample_depth, int row0, const LmPartials& lm, cudaStream_t st,
                             bool pdl) {
  const int parts = lm_select_parts(vocab);
  if (parts == 0 || N < 1 || k < 1 || k > KMAX || lm.G != parts || lm.T != parts) return cudaErrorInvalidValue;
  if (seeds && sample_rows < 1) return cudaErrorInvalidValue;
  const long long items = static_cast<long long>(N) * parts;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(static_cast<unsigned>((items + SEL_WARPS - 1) / SEL_WARPS)),
                                    dim3(SEL_WARPS * 32), 0, st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, seeds ? lm_select_kernel<true> : lm_select_kernel<false>, logits, vocab, parts,
                            static_cast<int>(items), k, seeds, sample_rows, sample_depth, row0,
                            lm.max + static_cast<size_t>(row0) * parts,
                            lm.sum + static_cast<size_t>(row0) * parts, lm.val + static_cast<size_t>(row0) * parts * k,
                            lm.id + static_cast<size_t>(row0) * parts * k);
}

}  // namespace eagle
