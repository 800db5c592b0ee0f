// Skinny-M GEMMs of the draft step: y[row][m] = sum_k W[m][k] * x[row][k].
//
// W (the weights, [M][K] row-major) is streamed from HBM once per launch; the rows
// (frontier nodes, at most a few hundred) are the N side.  Two mainloops share one
// operand loader and one set of fused epilogues:
//   * gemm_tc_kernel: bf16 weights.  Persistent CTAs split the (tile, k-block) space
//     evenly; a TMA warp streams 128x64 weight tiles into a shared-memory ring, loader
//     warps build the activation tile (gather / RMSNorm / SwiGLU applied on the fly,
//     fp32 split into bf16 hi + lo rows), one thread issues tcgen05.mma with the
//     accumulator in TMEM, and four epilogue warps drain TMEM.  Tiles split across CTAs
//     are finished by the last CTA to arrive (fixed summation order: deterministic).
//   * gemm_simt_kernel: f32 weights (small shapes), one CTA per 128-feature tile.
// Epilogues: EPI_STORE (residual add, per-tile sums of squares for the next RMSNorm),
// EPI_QKV (rotary embedding, queries and tree KV rows), EPI_LMHEAD (online log-sum-exp
// and per-row top-k over the vocabulary; no logits are written).
#include "common.cuh"
#include "internal.h"

#include <cooperative_groups.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

namespace eagle {

// ============================================================== operand loader
EAGLE_DEV void f4_to(float* v, float4 a, float4 b) {
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
EAGLE_DEV void bf8_to(float* v, uint4 u) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
EAGLE_DEV float silu_f(float x) { return x / (1.0f + expf(-x)); }

// Eight consecutive activation values x[row n][k .. k+7] of the GEMM operand.
EAGLE_DEV void load_b8(const BSrc& b, int n, int k, const float* rstd, float* v) {
  switch (b.mode) {
    case B_F32: {
      const float4* p = reinterpret_cast<const float4*>(b.x + static_cast<size_t>(n) * b.ldx + k);
      f4_to(v, __ldcg(p), __ldcg(p + 1));
      break;
    }
    case B_NORM: {
      const float4* p = reinterpret_cast<const float4*>(b.x + static_cast<size_t>(n) * b.ldx + k);
      const float4* gp = reinterpret_cast<const float4*>(b.gamma + k);
      float g[8];
      f4_to(v, __ldcg(p), __ldcg(p + 1));
      f4_to(g, __ldg(gp), __ldg(gp + 1));
      const float r = rstd[n];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = v[i] * r * g[i];
      break;
    }
    case B_FC: {
      if (k < b.split) {
        const int fr = __ldcg(b.row_feat + n);
        const float4* p = reinterpret_cast<const float4*>(b.x + static_cast<size_t>(fr) * b.ldx + k);
        f4_to(v, __ldcg(p), __ldcg(p + 1));
      } else {
        const int t = __ldcg(b.row_tok + n);
        const size_t off = static_cast<size_t>(t) * b.split + (k - b.split);
        if (b.emb_bf16) {
          bf8_to(v, __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(b.emb) + off)));
        } else {
          const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(b.emb) + off);
          f4_to(v, __ldg(p), __ldg(p + 1));
        }
      }
      break;
    }
    case B_SWIGLU: {
      const float* row = b.x + static_cast<size_t>(n) * b.ldx;
      const float4* gp = reinterpret_cast<const float4*>(row + k);
      const float4* up = reinterpret_cast<const float4*>(row + b.split + k);
      float gg[8], uu[8];
      f4_to(gg, __ldcg(gp), __ldcg(gp + 1));
      f4_to(uu, __ldcg(up), __ldcg(up + 1));
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = silu_f(gg[i]) * uu[i];
      break;
    }
    default: {  // B_BF16
      bf8_to(v, __ldcg(reinterpret_cast<const uint4*>(b.xb + static_cast<size_t>(n) * b.ldx + k)));
      break;
    }
  }
}

// 1 / sqrt(mean(x^2) + eps) of each row from the producer's per-tile sums of squares
// (summed in tile order).
EAGLE_DEV void compute_rstd(const BSrc& b, int N, float* rstd, int tid, int nthreads) {
  if (b.mode != B_NORM) return;
  for (int n = tid; n < N; n += nthreads) {
    float s = 0.f;
    for (int t = 0; t < b.ss_tiles; ++t) s += __ldcg(b.ss + static_cast<size_t>(t) * b.ss_ld + n);
    rstd[n] = 1.0f / sqrtf(s / static_cast<float>(b.dnorm) + b.eps);
  }
}

// ==================================================================== epilogues
// Shared-memory scratch of the 128 epilogue threads.
struct EpiScratch {
  float xch[16][BM];       // row-major exchange tile (rotary partners, LM-head transpose;
                           // STORE: the chunk's output rows before the vector stores)
  float red[4][16];        // per-warp partial sums of squares
  int meta[3][16];         // rows of the chunk: position, request, request-local slot
};
// Views of the epilogue's shared memory (the pointers themselves live in registers).
struct EpiSmem {
  EpiScratch* s;
  float* st_max;           // LM head, per row: running max, running sum of exp, list length
  float* st_sum;
  int* st_cnt;
  float* lv;               // [N][k] running top-k values (sorted)
  int* li;                 // [N][k] and their token ids
  float* rstd;             // [N] factored RMSNorm scale of each row (EPI_QKV / EPI_SWIGLU)
  uint16_t* shl;            // STORE / SWIGLU: [32][BM] operand-copy rows (hi, lo) before the vector stores
};

EAGLE_DEV EpiSmem epi_views(void* scratch, void* lm, int N, int topk) {
  EpiSmem es;
  es.s = reinterpret_cast<EpiScratch*>(scratch);
  es.shl = reinterpret_cast<uint16_t*>(lm);   // STORE / SWIGLU only (no LM-head lists then)
  float* f = reinterpret_cast<float*>(lm);
  es.st_max = f;
  es.st_sum = f + N;
  es.st_cnt = reinterpret_cast<int*>(f + 2 * N);
  es.lv = f + 3 * N;
  es.li = reinterpret_cast<int*>(f + 3 * N + N * topk);
  es.rstd = nullptr;
  return es;
}

// hi / lo rows of the operand copy the next GEMM loads with TMA
EAGLE_DEV void write_hl(const EpiArgs& e, int n, int m, float val, float gamma = 1.f) {
  val *= gamma;   // hl_gamma[m], loaded once by the caller
  uint16_t hi, lo;
  split_hilo(val, hi, lo);
  e.hl[static_cast<size_t>(2 * n) * e.hl_ld + m] = hi;
  e.hl[static_cast<size_t>(2 * n + 1) * e.hl_ld + m] = lo;
}

// 1 / sqrt(mean(x^2) + eps) per row from the producer's per-tile sums of squares.
EAGLE_DEV void epi_rstd(const EpiArgs& e, int N, float* rstd, int tl) {
  for (int n = tl; n < N; n += 128) {
    float s = 0.f;
    for (int t = 0; t < e.nss_tiles; ++t) s += __ldcg(e.nss + static_cast<size_t>(t) * e.nss_ld + n);
    rstd[n] = 1.0f / sqrtf(s / static_cast<float>(e.nss_d) + e.nss_eps);
  }
  named_bar(1, 128);
}

// AND of a predicate over the 128 epilogue threads (named barrier 1).
EAGLE_DEV bool epi_all(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\t"
      "setp.ne.u32 a, %1, 0;\n\t"
      "bar.red.and.pred b, 1, 128, a;\n\t"
      "selp.u32 %0, 1, 0, b;\n\t}"
      : "=r"(r)
      : "r"(p ? 1u : 0u)
      : "memory");
  return r != 0;
}

// Merge a warp's 128 new (value, id) candidates (4 per lane) into a row's sorted top-k
// list (length cnt <= k) held in shared memory: k rounds of warp arg-max.  Used to fill
// a list that is not full yet.
EAGLE_DEV void warp_topk_merge(float* lv, int* li, int* cnt_p, int k, const float* nv, const int* nid,
                               int lane) {
  const int cnt = *cnt_p;
  float cv[5];
  int ci[5];
#pragma unroll
  for (int j = 0; j < 4; ++j) { cv[j] = nv[j]; ci[j] = nid[j]; }
  cv[4] = lane < cnt ? lv[lane] : -INFINITY;
  ci[4] = lane < cnt ? li[lane] : INT_MAX;
  unsigned taken = 0;
  float outv = -INFINITY;
  int outi = INT_MAX;
  int rounds = 0;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = INT_MAX;
#pragma unroll
    for (int j = 0; j < 5; ++j)
      if (!(taken >> j & 1u) && ci[j] != INT_MAX && beats(cv[j], ci[j], bv, bi)) { bv = cv[j]; bi = ci[j]; }
    float wv = bv;
    int wi = bi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, wv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, wi, o);
      if (beats(ov, oi, wv, wi)) { wv = ov; wi = oi; }
    }
    if (wi == INT_MAX) break;
#pragma unroll
    for (int j = 0; j < 5; ++j)
      if (ci[j] == wi) taken |= 1u << j;
    if (lane == r) { outv = wv; outi = wi; }
    ++rounds;
  }
  __syncwarp();
  if (lane < rounds) { lv[lane] = outv; li[lane] = outi; }
  if (lane == 0) *cnt_p = rounds;
  __syncwarp();
}

// Insert the warp's candidates that beat the current k-th entry of a full list (best
// first, in shared memory).  The list lives one entry per lane while inserting; each
// candidate costs a ballot, a popcount and a shuffle-shift.  Only a few values per tile
// qualify once the list holds the best of earlier tiles.
EAGLE_DEV void warp_topk_insert(float* lv, int* li, int k, const float* nv, int* nid, int lane) {
  float myv = lane < k ? lv[lane] : -INFINITY;
  int myi = lane < k ? li[lane] : INT_MAX;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    for (;;) {
      const float kv = __shfl_sync(0xffffffffu, myv, k - 1);
      const int ki = __shfl_sync(0xffffffffu, myi, k - 1);
      const unsigned m = __ballot_sync(0xffffffffu, nid[j] != INT_MAX && beats(nv[j], nid[j], kv, ki));
      if (!m) break;
      const int src = __ffs(m) - 1;
      const float cv = __shfl_sync(0xffffffffu, nv[j], src);
      const int ci = __shfl_sync(0xffffffffu, nid[j], src);
      // entries better than the candidate stay; the rest move down one place
      const int pos = __popc(__ballot_sync(0xffffffffu, lane < k && beats(myv, myi, cv, ci)));
      const float upv = __shfl_up_sync(0xffffffffu, myv, 1);
      const int upi = __shfl_up_sync(0xffffffffu, myi, 1);
      if (lane > pos) {
        myv = upv;
        myi = upi;
      }
      if (lane == pos) {
        myv = cv;
        myi = ci;
      }
      if (lane == src) nid[j] = INT_MAX;   // consumed
    }
  }
  __syncwarp();
  if (lane < k) {
    lv[lane] = myv;
    li[lane] = myi;
  }
  __syncwarp();
}

// One 16-row chunk of accumulators: thread tl (0..127) holds feature m0 + tl of rows
// n0 .. n0+15 in v[].  All 128 epilogue threads call this together.
// The global inputs of one 16-row chunk's epilogue, loaded ahead (all loads of a batch in
// flight together): STORE: a[] = residuals; QKV: row metadata -> es.s->meta, a[] / b[] =
// rotary cos / sin of this thread's feature.  Called by all 128 epilogue threads.
EAGLE_DEV void epilogue_prefetch(const GemmArgs& g, EpiSmem& es, int mt, int n0, int tl, float* a, float* b) {
  const EpiArgs& e = g.e;
  const int m = mt * BM + tl;
  const bool mvalid = m < g.M;
  if (e.kind == EPI_STORE) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      a[i] = (e.resid && n0 + i < g.N && mvalid) ? __ldcg(e.resid + static_cast<size_t>(n0 + i) * e.ldr + m) : 0.f;
    b[0] = e.hl && e.hl_gamma && mvalid ? __ldg(e.hl_gamma + m) : 1.f;
  } else if (e.kind == EPI_QKV) {
    const int hd = e.hd, half = hd >> 1;
    const int head = m / hd, i = m - head * hd;
    const bool rotate = head < e.Hq + e.Hkv;
    if (tl < 16) {
      const int n = n0 + tl;
      es.s->meta[0][tl] = n < g.N ? __ldcg(e.row_pos + n) : 0;
      es.s->meta[1][tl] = n < g.N ? __ldcg(e.row_req + n) : 0;
      es.s->meta[2][tl] = n < g.N ? __ldcg(e.row_slot + n) : 0;
    }
    named_bar(1, 128);
    const int j = i < half ? i : i - half;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const bool ok = n0 + r < g.N && mvalid && rotate;
      const size_t o = static_cast<size_t>(es.s->meta[0][r]) * half + j;
      a[r] = ok ? __ldg(e.rope_cos + o) : 1.f;
      b[r] = ok ? __ldg(e.rope_sin + o) : 0.f;
    }
  }
}

// pre_a / pre_b (optional): this thread's inputs for the chunk, loaded earlier by
// epilogue_prefetch (STORE: residuals; QKV: rotary cos / sin, with the row metadata
// already in es.s->meta).
EAGLE_DEV void epilogue_chunk(const GemmArgs& g, EpiSmem& es, int mt, int n0, const float* v, int tl,
                              const float* pre_a = nullptr, const float* pre_b = nullptr) {
  const EpiArgs& e = g.e;
  const int m = mt * BM + tl;
  const bool mvalid = m < g.M;
  const int warp_q = tl >> 5, lane = tl & 31;
  if (e.kind == EPI_STORE) {
    // every residual load is issued before the first store (a store may alias a later
    // load, which would otherwise serialise the round trips)
    float rv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      rv[i] = pre_a ? pre_a[i]
                    : (e.resid && n0 + i < g.N && mvalid) ? __ldcg(e.resid + static_cast<size_t>(n0 + i) * e.ldr + m) : 0.f;
    const float gam = pre_b ? pre_b[0] : (e.hl && e.hl_gamma && mvalid ? __ldg(e.hl_gamma + m) : 1.f);
    float sq[16];
    // Rows are staged in shared memory and written with 16-byte vector stores of whole
    // rows (a tile row is contiguous in out and in the operand copy): 8 stores per thread
    // per chunk instead of 48 scalar ones.  Needs a full tile and 16-byte aligned rows.
    const bool vec = g.M % BM == 0 && e.ldo % 4 == 0 && reinterpret_cast<uintptr_t>(e.out) % 16 == 0 &&
                     (!e.hl || (e.hl_ld % 8 == 0 && reinterpret_cast<uintptr_t>(e.hl) % 16 == 0));
    if (vec) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float val = v[i] + rv[i];
        es.s->xch[i][tl] = val;
        sq[i] = n0 + i < g.N ? val * val : 0.f;
        if (e.hl) {
          uint16_t hi, lo;
          split_hilo(val * gam, hi, lo);
          es.shl[(2 * i) * BM + tl] = hi;
          es.shl[(2 * i + 1) * BM + tl] = lo;
        }
      }
      named_bar(1, 128);
      const int rows = min(16, g.N - n0), m0 = mt * BM;
      for (int idx = tl; idx < rows * (BM / 4); idx += 128) {   // out: 32 float4 per row
        const int r = idx / (BM / 4), q = idx - r * (BM / 4);
        *reinterpret_cast<float4*>(e.out + static_cast<size_t>(n0 + r) * e.ldo + m0 + 4 * q) =
            *reinterpret_cast<const float4*>(&es.s->xch[r][4 * q]);
      }
      if (e.hl) {
        for (int idx = tl; idx < 2 * rows * (BM / 8); idx += 128) {   // hi / lo rows: 16 uint4 per row
          const int r = idx / (BM / 8), q = idx - r * (BM / 8);
          const int n2 = 2 * n0 + r;   // row 2n = hi, 2n + 1 = lo
          *reinterpret_cast<uint4*>(e.hl + static_cast<size_t>(n2) * e.hl_ld + m0 + 8 * q) =
              *reinterpret_cast<const uint4*>(es.shl + r * BM + 8 * q);
        }
      }
      named_bar(1, 128);   // the staging rows are read before the next chunk writes them
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int n = n0 + i;
        float val = v[i] + rv[i];
        sq[i] = 0.f;
        if (n < g.N && mvalid) {
          e.out[static_cast<size_t>(n) * e.ldo + m] = val;
          if (e.hl) write_hl(e, n, m, val, gam);
          sq[i] = val * val;
        }
      }
    }
    if (e.ss) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float s = warp_sum(sq[i]);
        if (lane == 0) es.s->red[warp_q][i] = s;
      }
      named_bar(1, 128);
      if (tl < 16 && n0 + tl < g.N)
        e.ss[static_cast<size_t>(mt) * e.ss_ld + n0 + tl] =
            es.s->red[0][tl] + es.s->red[1][tl] + es.s->red[2][tl] + es.s->red[3][tl];
      named_bar(1, 128);
    }
  } else if (e.kind == EPI_QKV) {
    const int hd = e.hd, half = hd >> 1;
    const int head = m / hd, i = m - head * hd;
    const bool rotate = head < e.Hq + e.Hkv;
    float vn[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      vn[r] = (e.nss && n0 + r < g.N) ? v[r] * es.rstd[n0 + r] : v[r];
      es.s->xch[r][tl] = vn[r];
    }
    // row metadata (one load per row, shared), then the rotary table entries, all loaded
    // before the first store
    float rc[16], rsn[16];
    if (pre_a) {
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        rc[r] = pre_a[r];
        rsn[r] = pre_b[r];
      }
    } else {
      epilogue_prefetch(g, es, mt, n0, tl, rc, rsn);
    }
    named_bar(1, 128);
    const int partner = tl + (i < half ? half : -half);
    if (hd == BM && g.M % BM == 0) {
      // one head per tile: rotate, stage the rows, then 16-byte vector stores of whole
      // head rows (q, or the request's tree K / V row)
      float rv[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        rv[r] = vn[r];
        if (rotate) {
          const float p = es.s->xch[r][partner];
          rv[r] = i < half ? vn[r] * rc[r] - p * rsn[r] : vn[r] * rc[r] + p * rsn[r];
        }
      }
      named_bar(1, 128);
#pragma unroll
      for (int r = 0; r < 16; ++r) es.s->xch[r][tl] = rv[r];
      named_bar(1, 128);
      const int rows = min(16, g.N - n0);
      for (int idx = tl; idx < rows * (BM / 4); idx += 128) {
        const int r = idx / (BM / 4), q4 = idx - r * (BM / 4);
        float* dst;
        if (head < e.Hq) {
          dst = e.q + static_cast<size_t>(n0 + r) * e.Hq * hd + static_cast<size_t>(head) * hd;
        } else {
          const int b = es.s->meta[1][r], slot = es.s->meta[2][r];
          const bool isk = head < e.Hq + e.Hkv;
          const int kvh = isk ? head - e.Hq : head - e.Hq - e.Hkv;
          dst = (isk ? e.tk : e.tv) + ((static_cast<size_t>(b) * e.tree_rows + slot) * e.Hkv + kvh) * hd;
        }
        *reinterpret_cast<float4*>(dst + 4 * q4) = *reinterpret_cast<const float4*>(&es.s->xch[r][4 * q4]);
      }
      named_bar(1, 128);
      return;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int n = n0 + r;
      if (n >= g.N || !mvalid) continue;
      float val = vn[r];
      if (rotate) {
        const float c = rc[r], s = rsn[r];
        const float p = es.s->xch[r][partner];
        val = i < half ? val * c - p * s : val * c + p * s;
      }
      if (head < e.Hq) {
        e.q[static_cast<size_t>(n) * e.Hq * hd + m] = val;
      } else {
        const int b = es.s->meta[1][r], slot = es.s->meta[2][r];
        const bool isk = head < e.Hq + e.Hkv;
        const int kvh = isk ? head - e.Hq : head - e.Hq - e.Hkv;
        float* dst = isk ? e.tk : e.tv;
        dst[((static_cast<size_t>(b) * e.tree_rows + slot) * e.Hkv + kvh) * hd + i] = val;
      }
    }
    named_bar(1, 128);
  } else if (e.kind == EPI_SWIGLU) {
    // tile = 64 gate rows (threads 0-63) + the 64 matching up rows (threads 64-127)
#pragma unroll
    for (int r = 0; r < 16; ++r) es.s->xch[r][tl] = v[r];
    named_bar(1, 128);
    if (!e.out && e.hl && e.hl_ld % 8 == 0 && reinterpret_cast<uintptr_t>(e.hl) % 16 == 0) {
      // operand copy only: hi / lo rows staged, then 16-byte vector stores (64 columns)
      if (tl < 64) {
        const int j = mt * (BM / 2) + tl;
        const float gam = e.hl_gamma ? __ldg(e.hl_gamma + j) : 1.f;
#pragma unroll 4
        for (int r = 0; r < 16; ++r) {
          float gt = es.s->xch[r][tl], up = es.s->xch[r][tl + 64];
          if (e.nss && n0 + r < g.N) {
            gt *= es.rstd[n0 + r];
            up *= es.rstd[n0 + r];
          }
          uint16_t hi, lo;
          split_hilo(silu_f(gt) * up * gam, hi, lo);
          es.shl[(2 * r) * BM + tl] = hi;
          es.shl[(2 * r + 1) * BM + tl] = lo;
        }
      }
      named_bar(1, 128);
      const int rows = min(16, g.N - n0), j0 = mt * (BM / 2);
      for (int idx = tl; idx < 2 * rows * (BM / 16); idx += 128) {   // 8 uint4 per 64-column row
        const int r = idx / (BM / 16), q8 = idx - r * (BM / 16);
        *reinterpret_cast<uint4*>(e.hl + static_cast<size_t>(2 * n0 + r) * e.hl_ld + j0 + 8 * q8) =
            *reinterpret_cast<const uint4*>(es.shl + r * BM + 8 * q8);
      }
      named_bar(1, 128);
      return;
    }
    if (tl < 64) {
      const int j = mt * (BM / 2) + tl;
      const float gam = e.hl && e.hl_gamma ? __ldg(e.hl_gamma + j) : 1.f;
#pragma unroll 4
      for (int r = 0; r < 16; ++r) {
        const int n = n0 + r;
        if (n < g.N) {
          float gt = es.s->xch[r][tl], up = es.s->xch[r][tl + 64];
          if (e.nss) {
            gt *= es.rstd[n];
            up *= es.rstd[n];
          }
          const float sv = silu_f(gt) * up;
          if (e.out) e.out[static_cast<size_t>(n) * e.ldo + j] = sv;
          if (e.hl) write_hl(e, n, j, sv, gam);
        }
      }
    }
    named_bar(1, 128);
  } else if (e.kind == EPI_LOGITS) {
    // the rows' logits only (a separate kernel takes the log-sum-exp and the top-k): one
    // coalesced 512-byte row segment per row
    const int tok = mt * BM + tl;
    if (tok < g.M) {
#pragma unroll
      for (int r = 0; r < 16; ++r)
        if (n0 + r < g.N)
          e.logits[static_cast<size_t>(n0 + r) * g.M + tok] = e.nss ? v[r] * es.rstd[n0 + r] : v[r];
    }
  } else {  // EPI_LMHEAD
    // (with a factored RMSNorm of the operand, e.g. a final norm before the LM head, the
    // row scale is applied here)
#pragma unroll
    for (int r = 0; r < 16; ++r) es.s->xch[r][tl] = (e.nss && n0 + r < g.N) ? v[r] * es.rstd[n0 + r] : v[r];
    if (e.logits && mt * BM + tl < g.M) {   // (optional) the full logits as well
#pragma unroll
      for (int r = 0; r < 16; ++r)
        if (n0 + r < g.N) e.logits[static_cast<size_t>(n0 + r) * g.M + mt * BM + tl] = es.s->xch[r][tl];
    }
    named_bar(1, 128);
    const int k = e.topk;
    for (int r = warp_q; r < 16; r += 4) {
      const int n = n0 + r;
      if (n >= g.N) continue;                       // warp-uniform
      float val[4];
      int id[4];
      float lmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        id[j] = mt * BM + lane + 32 * j;
        val[j] = id[j] < g.M ? es.s->xch[r][lane + 32 * j] : -INFINITY;
        if (id[j] >= g.M) id[j] = INT_MAX;
        lmax = fmaxf(lmax, val[j]);
      }
      // this tile's log-sum-exp state (max, sum of exp) of the row, merged later in tile order
      const float tmax = warp_max(lmax);
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) s += id[j] != INT_MAX ? expf(val[j] - tmax) : 0.f;
      s = warp_sum(s);
      if (lane == 0) {
        e.lm_max[static_cast<size_t>(n) * g.MT + mt] = tmax;
        e.lm_sum[static_cast<size_t>(n) * g.MT + mt] = s;
      }
      // top-k (sampled drafting: of logit + Gumbel noise; one Philox call gives the lane's
      // four tokens, t = tile * 128 + lane + 32 j -> word j of counter 32 tile + lane)
      if (e.seeds) {
        const int gr = e.sample_row0 + n;
        const int b = gr / e.sample_rows, i = gr - b * e.sample_rows;
        const unsigned long long sd = __ldg(e.seeds + b);
        const uint4 w = philox4x32_10(make_uint4(32u * static_cast<uint32_t>(mt) + lane, static_cast<uint32_t>(i),
                                                 static_cast<uint32_t>(e.sample_depth), 0u),
                                      static_cast<uint32_t>(sd), static_cast<uint32_t>(sd >> 32));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (id[j] != INT_MAX) val[j] += gumbel_of_word(ws[j]);
      }
      const int cnt = es.st_cnt[n];
      float* lv = es.lv + static_cast<size_t>(n) * k;
      int* li = es.li + static_cast<size_t>(n) * k;
      const float tv = cnt < k ? -INFINITY : lv[k - 1];
      const int ti = cnt < k ? INT_MAX : li[k - 1];
      bool cand = false;
#pragma unroll
      for (int j = 0; j < 4; ++j) cand |= id[j] != INT_MAX && beats(val[j], id[j], tv, ti);
      __syncwarp();
      if (__any_sync(0xffffffffu, cand)) {
        if (cnt < k) warp_topk_merge(lv, li, es.st_cnt + n, k, val, id, lane);
        else warp_topk_insert(lv, li, k, val, id, lane);
      }
      __syncwarp();
    }
    named_bar(1, 128);
  }
}

// Per-CTA LM-head state: reset before the first tile, written out after the last.
EAGLE_DEV void lmhead_init(const GemmArgs& g, EpiSmem& es, int tl) {
  for (int n = tl; n < g.N; n += 128) es.st_cnt[n] = 0;
  named_bar(1, 128);
}
EAGLE_DEV void lmhead_flush(const GemmArgs& g, EpiSmem& es, int cta, int ncta, int tl) {
  const EpiArgs& e = g.e;
  const int k = e.topk;
  named_bar(1, 128);
  for (int n = tl; n < g.N; n += 128) {
    const size_t o = static_cast<size_t>(n) * ncta + cta;   // lists of one row are contiguous
    const int cnt = es.st_cnt[n];
    for (int j = 0; j < k; ++j) {
      e.lm_val[o * k + j] = j < cnt ? es.lv[static_cast<size_t>(n) * k + j] : -INFINITY;
      e.lm_id[o * k + j] = j < cnt ? es.li[static_cast<size_t>(n) * k + j] : -1;
    }
  }
}

// ============================================================ work decomposition
struct Sched {
  long long total;
  int grid;
  EAGLE_DEV long long begin(int c) const { return static_cast<long long>(c) * total / grid; }
  // CTA whose range holds unit index i
  EAGLE_DEV int owner(long long i) const {
    return static_cast<int>(((i + 1) * grid + total - 1) / total - 1);
  }
};

// Segment sg of a CTA's unit range [u0, u1) in processing order (false: no more).  With
// `reorder`, the tiles the CTA shares with a neighbour come first (its last tile, then its
// first) and its whole tiles last, so the cross-CTA fix-ups happen while the CTAs still
// have work rather than at the end of the kernel.
EAGLE_DEV bool range_segment(long long u0, long long u1, int KB, bool reorder, int sg, long long& b, long long& e) {
  if (u1 <= u0) return false;
  const long long ft = u0 / KB, lt = (u1 - 1) / KB;
  if (!reorder || ft == lt) {
    b = u0;
    e = u1;
    return sg == 0;
  }
  const bool hsplit = u0 % KB != 0, tsplit = u1 % KB != 0;
  const long long mb = hsplit ? (ft + 1) * KB : u0, me = tsplit ? lt * KB : u1;
  int k = 0;
  if (tsplit && k++ == sg) { b = lt * KB; e = u1; return true; }
  if (hsplit && k++ == sg) { b = u0; e = (ft + 1) * KB; return true; }
  if (me > mb && k++ == sg) { b = mb; e = me; return true; }
  return false;
}

// ============================================================ tcgen05 mainloop
struct TcLayout {
  uint32_t stage_bytes, b_off;
  uint32_t bar_off, misc_off, idx_off, epi_off, rstd_off, erstd_off, lm_off;
};

// Shared memory of gemm_tc_kernel: [stages x (A tile 16 KB | B tile npad*256 B)] |
// mbarriers | misc words | gathered row indices | epilogue scratch | rstd | LM-head lists.
// With kpair a stage holds two K blocks: [A(kb) | A(kb+1) | B(kb) | B(kb+1)].
__host__ __device__ inline TcLayout tc_layout(int npad, int stages, int kpair = 0) {
  TcLayout L;
  const uint32_t kp = kpair ? 2u : 1u;
  L.b_off = kp * A_STAGE_BYTES;
  L.stage_bytes = kp * (A_STAGE_BYTES + npad * 256);
  L.bar_off = L.stage_bytes * stages;
  L.misc_off = L.bar_off + (3 * stages + 4) * 8;
  L.idx_off = (L.misc_off + 64 + 15) & ~15u;
  L.epi_off = (L.idx_off + 2 * 256 * 4 + 127) & ~127u;
  L.rstd_off = L.epi_off + static_cast<uint32_t>((sizeof(EpiScratch) + 127) & ~size_t(127));
  L.erstd_off = L.rstd_off + sizeof(float) * 256;
  L.lm_off = L.erstd_off + sizeof(float) * 256;
  return L;
}
// The region at lm_off holds the LM head's per-row lists, or (STORE epilogue) the
// operand-copy staging rows.
__host__ __device__ inline uint32_t tc_smem_bytes(int npad, int stages, int lm_rows, int topk, bool store,
                                                  int kpair = 0) {
  TcLayout L = tc_layout(npad, stages, kpair);
  uint32_t tail = static_cast<uint32_t>(lm_rows) * (3 + 2 * topk) * 4;
  if (store && tail < 32 * BM * 2) tail = 32 * BM * 2;
  return L.lm_off + tail + 1024;  // +1024: base alignment
}

EAGLE_DEV void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

constexpr int TC_NCW = 4;                       // converter warps
constexpr int TC_THREADS = (7 + TC_NCW) * 32;   // A producer, MMA, 4 epilogue, B producer, converters
constexpr int TC_THREADS_TMA = 7 * 32;          // operand tile by TMA: no converter warps
constexpr uint32_t TC_SMEM_OCC2 = 113 * 1024;   // two CTAs per SM

// Warp roles: 0 = weight TMA producer, 1 = MMA issuer, 2-5 = epilogue (TMEM lanes by
// warp % 4), 6 = activation producer (bulk copies of the source rows into the B tile),
// 7.. = converters (in place: fp32 / bf16 row -> bf16 hi row + bf16 lo row, swizzled).
// B tile rows are interleaved: row 2r = hi of GEMM row r, row 2r+1 = its lo part, so the
// accumulator column 2r + 1 holds the low-order correction of column 2r.
// NT = TC_THREADS (converter warps present, one CTA per SM) or 7 warps (operand by TMA only;
// MINB = 1: the whole register file, MINB = 2: two CTAs per SM).
//
// PAIR: a cluster of two CTAs on the same (tile, K block) units, rank r on its own rows (its
// own argument block g_r and operand map tmB_r): rank 0 loads each weight stage once, by TMA
// multicast into both CTAs; each CTA's MMA commits release the stage in both, so a stage is
// refilled only when both have consumed it.
template <int NT, int MINB, bool SEG, bool PAIR = false>
__global__ void __launch_bounds__(NT, MINB)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tm0, const __grid_constant__ CUtensorMap tm1,
               const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ GemmArgs g0,
               const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ GemmArgs g1) {
  uint32_t crank = 0;
  if (PAIR) crank = cooperative_groups::this_cluster().block_rank();
  const GemmArgs& g = (PAIR && crank) ? g1 : g0;
  const CUtensorMap& tmB = (PAIR && crank) ? tmB1 : tmB0;
  const int cta = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);   // schedule index
  const int ncta = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const TcLayout L = tc_layout(g.npad, g.stages, g.kpair);
  const int KP = g.kpair ? 2 : 1;   // K blocks per stage
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + L.bar_off;
  const uint32_t bar_empty = bar_full + 8 * g.stages;
  const uint32_t bar_bfull = bar_empty + 8 * g.stages;
  const uint32_t bar_accf = bar_bfull + 8 * g.stages;
  const uint32_t bar_acce = bar_accf + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc_off);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc_off + 4);
  int* last_flag = reinterpret_cast<int*>(smem + L.misc_off + 8);
  int* s_feat = reinterpret_cast<int*>(smem + L.idx_off);
  int* s_tok = s_feat + 256;
  float* rstd = reinterpret_cast<float*>(smem + L.rstd_off);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = g.KB;
  const long long wlim = g.wait_limit > 0 ? g.wait_limit : WAIT_LIMIT_CYCLES;
  const int npad = g.npad, nrb = g.nrb, np2 = 2 * npad;
  const Sched sc{static_cast<long long>(g.MT) * KB, ncta};
  // units [u0, u1): stream-K range, or (csplit) K range r of tile blockIdx.x / S
  const int cs_t = g.csplit > 0 ? static_cast<int>(blockIdx.x) / g.csplit : 0;
  const int cs_r = g.csplit > 0 ? static_cast<int>(blockIdx.x) - cs_t * g.csplit : 0;
  const long long u0 = g.csplit > 0 ? static_cast<long long>(cs_t) * KB + static_cast<long long>(cs_r) * KB / g.csplit
                                    : sc.begin(cta);
  const long long u1 = g.csplit > 0
                           ? static_cast<long long>(cs_t) * KB + static_cast<long long>(cs_r + 1) * KB / g.csplit
                           : sc.begin(cta + 1);
  const bool reorder = SEG && g.csplit == 0;   // (compiled out of the other instances)

  if (threadIdx.x == 0) {
    for (int s = 0; s < g.stages; ++s) {
      mbar_init(bar_full + 8 * s, 2);            // weight bytes + activation (TMA bytes or converter)
      mbar_init(bar_empty + 8 * s, PAIR ? 2 : 1);   // tcgen05.commit (of both CTAs of a pair)
      mbar_init(bar_bfull + 8 * s, 1);           // bulk-copy bytes of the source rows
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_accf + 8 * b, 1);
      mbar_init(bar_acce + 8 * b, 4);            // one arrive per epilogue warp
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), g.tmem_cols);
    tmem_relinquish();
  }
  if (warp == 1 && lane == 0) {
    tma_prefetch_desc(&tm0);
    tma_prefetch_desc(&tm1);
    if (g.b_tma) tma_prefetch_desc(&tmB);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (PAIR) cooperative_groups::this_cluster().sync();   // both CTAs' barriers exist before any remote use
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer (weights)
    // Weights never depend on the previous kernel: streaming starts before its end.
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int sg = 0; ok; ++sg) {
        long long s0, s1;
        if (!range_segment(u0, u1, KB, reorder, sg, s0, s1)) break;
        for (long long i = s0; i < s1 && ok;) {
          const int mt = static_cast<int>(i / KB), kb0 = static_cast<int>(i % KB);
          const int kb1 = static_cast<int>(min(static_cast<long long>(KB), kb0 + (s1 - i)));
          const bool second = !g.a_pair && mt * BM >= g.m_split;
          const CUtensorMap* tm = second ? &tm1 : &tm0;
          const int mrow = g.a_pair ? mt * (BM / 2) : (second ? mt * BM - g.m_split : mt * BM);
          for (int kb = kb0; kb < kb1 && ok;) {
            const int nk = min(KP, kb1 - kb);   // K blocks of this stage
            for (int rb = 0; rb < nrb && ok; ++rb) {
              if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, g.err, abort_flag, wlim)) { ok = false; break; }
              const uint32_t dst = sbase + stage * L.stage_bytes;
              mbar_arrive_expect_tx(bar_full + 8 * stage, nk * A_STAGE_BYTES);
              for (int u = 0; u < nk && (!PAIR || crank == 0); ++u) {
                const uint32_t du = dst + u * A_STAGE_BYTES;
                if (PAIR) {      // one load, into both CTAs of the pair
                  if (g.a_pair) {
                    tma_load_2d_mc(du, &tm0, (kb + u) * BK, mrow, bar_full + 8 * stage, pol, 3);
                    tma_load_2d_mc(du + A_STAGE_BYTES / 2, &tm1, (kb + u) * BK, mrow, bar_full + 8 * stage, pol, 3);
                  } else {
                    tma_load_2d_mc(du, tm, (kb + u) * BK, mrow, bar_full + 8 * stage, pol, 3);
                  }
                } else if (g.a_pair) {  // rows 0-63 from map 0 (gate), rows 64-127 from map 1 (up)
                  tma_load_2d(du, &tm0, (kb + u) * BK, mrow, bar_full + 8 * stage, pol);
                  tma_load_2d(du + A_STAGE_BYTES / 2, &tm1, (kb + u) * BK, mrow, bar_full + 8 * stage, pol);
                } else {
                  tma_load_2d(du, tm, (kb + u) * BK, mrow, bar_full + 8 * stage, pol);
                }
              }
              if (++stage == g.stages) { stage = 0; phase ^= 1; }
            }
            kb += nk;
          }
          i += kb1 - kb0;
        }
      }
      if (!ok) {
        // let copies already issued land before the CTA releases its shared memory
        const long long t0 = clock64();
        while (clock64() - t0 < 4000000) {
        }
      } else if (PAIR) {
        // every stage released once more: all of both CTAs' commits (remote arrivals on this
        // CTA's barriers) have landed before the pair's closing cluster barrier
        for (int s = 0; s < g.stages && ok; ++s) {
          ok = mbar_wait(bar_empty + 8 * stage, phase ^ 1, g.err, abort_flag, wlim);
          if (++stage == g.stages) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, np2);
      // Stage 0's operand descriptors; a stage or a 16-wide K step only moves the start
      // address field (bits 0-13, in 16-byte units, far from carrying), so the loop adds.
      const uint64_t adesc0 = smem_desc_sw128(sbase), bdesc0 = smem_desc_sw128(sbase + L.b_off);
      const uint64_t dstep = L.stage_bytes >> 4;
      const uint64_t astep2 = A_STAGE_BYTES >> 4, bstep2 = (static_cast<uint32_t>(npad) * 256u) >> 4;
      int stage = 0;
      uint32_t phase = 0;
      long long uc = 0;
      bool ok = true;
      for (int sg = 0; ok; ++sg) {
        long long s0, s1;
        if (!range_segment(u0, u1, KB, reorder, sg, s0, s1)) break;
        for (long long i = s0; i < s1 && ok; ++uc) {
          const int kb0 = static_cast<int>(i % KB);
          const int kb1 = static_cast<int>(min(static_cast<long long>(KB), kb0 + (s1 - i)));
          const int ab = static_cast<int>(uc % g.nbuf);
          const uint32_t ap = static_cast<uint32_t>((uc / g.nbuf) & 1);
          if (!mbar_wait(bar_acce + 8 * ab, ap ^ 1, g.err, abort_flag, wlim)) { ok = false; break; }
          tc_fence_after();
          // (the one-block loop is kept apart: this thread's per-stage work bounds the rate)
          if (KP == 1) {
            for (int kb = kb0; kb < kb1 && ok; ++kb) {
              for (int rb = 0; rb < nrb; ++rb) {
                if (!mbar_wait(bar_full + 8 * stage, phase, g.err, abort_flag, wlim)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>((ab * nrb + rb) * np2);
                const uint64_t ad = adesc0 + stage * dstep, bd = bdesc0 + stage * dstep;
  #pragma unroll
                for (int j = 0; j < BK / 16; ++j)   // 16 bf16 of K = 32 bytes = 2 descriptor units
                  tc_mma_bf16(d, ad + 2 * j, bd + 2 * j, idesc, (kb > kb0 || j > 0) ? 1u : 0u);
                if (PAIR) tc_commit_mc(bar_empty + 8 * stage, 3);
                else tc_commit(bar_empty + 8 * stage);
                if (++stage == g.stages) { stage = 0; phase ^= 1; }
              }
            }
          } else {   // one 16-row block (nrb == 1), two K blocks per stage
            const uint32_t d = tmem + static_cast<uint32_t>(ab * np2);
            for (int kb = kb0; kb < kb1 && ok;) {
              if (!mbar_wait(bar_full + 8 * stage, phase, g.err, abort_flag, wlim)) { ok = false; break; }
              tc_fence_after();
              const uint64_t ad = adesc0 + stage * dstep, bd = bdesc0 + stage * dstep;
  #pragma unroll
              for (int j = 0; j < BK / 16; ++j)
                tc_mma_bf16(d, ad + 2 * j, bd + 2 * j, idesc, (kb > kb0 || j > 0) ? 1u : 0u);
              if (kb + 1 < kb1) {   // the stage's second K block
  #pragma unroll
                for (int j = 0; j < BK / 16; ++j)
                  tc_mma_bf16(d, ad + astep2 + 2 * j, bd + bstep2 + 2 * j, idesc, 1u);
              }
              if (PAIR) tc_commit_mc(bar_empty + 8 * stage, 3);
              else tc_commit(bar_empty + 8 * stage);
              if (++stage == g.stages) { stage = 0; phase ^= 1; }
              kb += 2;
            }
          }
          if (ok) tc_commit(bar_accf + 8 * ab);
          i += kb1 - kb0;
        }
      }
      if (!ok) {
        // let MMAs already issued finish before TMEM is released
        const long long t0 = clock64();
        while (clock64() - t0 < 4000000) {
        }
      }
    }
  } else if (warp == 6 && g.b_tma) {
    // ------------------------- activation producer: TMA of the operand copy's tile
    // (written by the previous kernel: wait for it; the weight stream does not)
    if (lane == 0) {
      pdl_wait();
      uint64_t pol_b;
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_b));
      const uint32_t b_bytes = static_cast<uint32_t>(npad) * 256u;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int sg = 0; ok; ++sg) {
        long long s0, s1;
        if (!range_segment(u0, u1, KB, reorder, sg, s0, s1)) break;
        for (long long i = s0; i < s1 && ok;) {
          const int kb0 = static_cast<int>(i % KB);
          const int kb1 = static_cast<int>(min(static_cast<long long>(KB), kb0 + (s1 - i)));
          for (int kb = kb0; kb < kb1 && ok;) {
            const int nk = min(KP, kb1 - kb);
            for (int rb = 0; rb < nrb && ok; ++rb) {
              if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1, g.err, abort_flag, wlim)) { ok = false; break; }
              mbar_arrive_expect_tx(bar_full + 8 * stage, nk * b_bytes);
              for (int u = 0; u < nk; ++u)
                tma_load_2d(sbase + stage * L.stage_bytes + L.b_off + u * b_bytes, &tmB, (kb + u) * BK, rb * np2,
                            bar_full + 8 * stage, pol_b);
              if (++stage == g.stages) { stage = 0; phase ^= 1; }
            }
            kb += nk;
          }
          i += kb1 - kb0;
        }
      }
      if (!ok) {
        const long long t0 = clock64();
        while (clock64() - t0 < 4000000) {
        }
      }
    }
  } else if (warp == 6) {
    // ------------------------------- activation producer: bulk copies of source rows
    pdl_wait();
    if (g.b.mode == B_FC) {
      for (int n = lane; n < g.N; n += 32) {
        s_feat[n] = __ldcg(g.b.row_feat + n);
        s_tok[n] = __ldcg(g.b.row_tok + n);
      }
    }
    __syncwarp();
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int sg = 0; ok; ++sg) {
      long long s0, s1;
      if (!range_segment(u0, u1, KB, reorder, sg, s0, s1)) break;
      for (long long i = s0; i < s1 && ok;) {
        const int kb0 = static_cast<int>(i % KB);
        const int kb1 = static_cast<int>(min(static_cast<long long>(KB), kb0 + (s1 - i)));
        for (int kb = kb0; kb < kb1 && ok; ++kb) {
          const int k0 = kb * BK;
          const bool bf = g.b.mode == B_BF16 || (g.b.mode == B_FC && k0 >= g.b.split);
          const uint32_t rowbytes = bf ? 128u : 256u;
          for (int rb = 0; rb < nrb; ++rb) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar_empty + 8 * stage, phase ^ 1, g.err, abort_flag, wlim));
            if (!ok) break;
            const int r0 = rb * npad;
            const int rows = min(npad, g.N - r0);
            const uint32_t bdst = sbase + stage * L.stage_bytes + L.b_off;
            if (lane == 0) mbar_arrive_expect_tx(bar_bfull + 8 * stage, static_cast<uint32_t>(rows) * rowbytes);
            __syncwarp();
            for (int r = lane; r < rows; r += 32) {
              const int n = r0 + r;
              const void* src;
              if (g.b.mode == B_FC) {
                src = k0 < g.b.split
                          ? static_cast<const void*>(g.b.x + static_cast<size_t>(s_feat[n]) * g.b.ldx + k0)
                          : static_cast<const void*>(static_cast<const uint16_t*>(g.b.emb) +
                                                     static_cast<size_t>(s_tok[n]) * g.b.split + (k0 - g.b.split));
              } else if (g.b.mode == B_BF16) {
                src = g.b.xb + static_cast<size_t>(n) * g.b.ldx + k0;
              } else {
                src = g.b.x + static_cast<size_t>(n) * g.b.ldx + k0;
              }
              bulk_copy_g2s(bdst + 256u * r, src, rowbytes, bar_bfull + 8 * stage);
            }
            if (++stage == g.stages) { stage = 0; phase ^= 1; }
          }
        }
        i += kb1 - kb0;
      }
    }
    if (!ok) {
      const long long t0 = clock64();
      while (clock64() - t0 < 4000000) {
      }
    }
  } else if (warp >= 7 && !g.b_tma) {
    // ------------------------------------ converters: source row -> bf16 hi / lo rows
    // Stage-iteration it is converted by warp it % TC_NCW (all of its rows).
    const int cw = warp - 7;
    pdl_wait();
    compute_rstd(g.b, g.N, rstd, cw * 32 + lane, TC_NCW * 32);
    named_bar(2, TC_NCW * 32);
    int stage = 0;
    uint32_t phase = 0;
    long long it = 0;
    bool ok = true;
    const uint32_t cbyte = (4u * lane) & 15u;
    const int chunk = lane >> 2;
    for (int sg = 0; ok; ++sg) {
      long long s0, s1;
      if (!range_segment(u0, u1, KB, reorder, sg, s0, s1)) break;
      for (long long i = s0; i < s1 && ok;) {
        const int kb0 = static_cast<int>(i % KB);
        const int kb1 = static_cast<int>(min(static_cast<long long>(KB), kb0 + (s1 - i)));
        for (int kb = kb0; kb < kb1 && ok; ++kb) {
          const int k0 = kb * BK;
          const bool bf = g.b.mode == B_BF16 || (g.b.mode == B_FC && k0 >= g.b.split);
          for (int rb = 0; rb < nrb; ++rb, ++it) {
            if (it % TC_NCW == cw) {
              ok = __all_sync(0xffffffffu, mbar_wait(bar_bfull + 8 * stage, phase, g.err, abort_flag, wlim));
              if (!ok) break;
              float gm0 = 1.f, gm1 = 1.f;
              if (g.b.mode == B_NORM) {
                const float2 gg = __ldg(reinterpret_cast<const float2*>(g.b.gamma + k0) + lane);
                gm0 = gg.x;
                gm1 = gg.y;
              }
              const int r0 = rb * npad;
              const int rows = min(npad, g.N - r0);
              uint8_t* bs = smem + stage * L.stage_bytes + L.b_off;
              for (int r = 0; r < rows; ++r) {
                float x0, x1;
                if (bf) {
                  const uint32_t w = *reinterpret_cast<const uint32_t*>(bs + 256 * r + 4 * lane);
                  x0 = __uint_as_float(w << 16);
                  x1 = __uint_as_float(w & 0xFFFF0000u);
                } else {
                  const float2 f = *reinterpret_cast<const float2*>(bs + 256 * r + 8 * lane);
                  x0 = f.x;
                  x1 = f.y;
                }
                if (g.b.mode == B_NORM) {
                  const float rs = rstd[r0 + r];
                  x0 = x0 * rs * gm0;
                  x1 = x1 * rs * gm1;
                }
                uint16_t h0, l0, h1, l1;
                split_hilo(x0, h0, l0);
                split_hilo(x1, h1, l1);
                __syncwarp();   // every lane has read row r before it is overwritten
                *reinterpret_cast<uint32_t*>(bs + sw128_offset(2 * r, chunk) + cbyte) =
                    static_cast<uint32_t>(h0) | (static_cast<uint32_t>(h1) << 16);
                *reinterpret_cast<uint32_t*>(bs + sw128_offset(2 * r + 1, chunk) + cbyte) =
                    static_cast<uint32_t>(l0) | (static_cast<uint32_t>(l1) << 16);
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar_full + 8 * stage);
            }
            if (++stage == g.stages) { stage = 0; phase ^= 1; }
          }
        }
        i += kb1 - kb0;
      }
    }
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------ epilogue (warps 2-5)
    const int q = warp & 3;                 // TMEM lane quadrant of this warp
    const int tl = q * 32 + lane;           // feature row of the tile = TMEM lane
    EpiSmem es = epi_views(smem + L.epi_off, smem + L.lm_off, g.N, g.e.topk);
    es.rstd = reinterpret_cast<float*>(smem + L.erstd_off);
    pdl_wait();
    if (g.e.kind == EPI_LMHEAD) lmhead_init(g, es, tl);
    if (g.e.nss) epi_rstd(g.e, g.N, es.rstd, tl);
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int rows_total = nrb * npad;
    const size_t pbytes = static_cast<size_t>(rows_total) * BM * sizeof(float);   // one partial tile
    long long uc = 0, done = 0;
    bool ok = true;
    for (int sg = 0; ok; ++sg) {
      long long s0, s1;
      if (!range_segment(u0, u1, KB, reorder, sg, s0, s1)) break;
      for (long long i = s0; i < s1 && ok; ++uc) {
        const int mt = static_cast<int>(i / KB), kb0 = static_cast<int>(i % KB);
        const int kb1 = static_cast<int>(min(static_cast<long long>(KB), kb0 + (s1 - i)));
        const int ab = static_cast<int>(uc % g.nbuf);
        const uint32_t ap = static_cast<uint32_t>((uc / g.nbuf) & 1);
        ok = epi_all(mbar_wait(bar_accf + 8 * ab, ap, g.err, abort_flag, wlim));
        if (!ok) break;
        tc_fence_after();
        const bool complete = kb0 == 0 && kb1 == KB;
        const bool final_unit = (done += kb1 - kb0) == u1 - u0;   // this CTA's MMAs end with it
        const int slot = (mt == u0 / KB) ? 0 : 1;   // the CTA's first tile or its last
        float* mypart = g.part + (static_cast<size_t>(cta) * 2 + slot) * rows_total * BM;
        for (int rb = 0; rb < nrb; ++rb) {
          for (int c0 = 0; c0 < npad; c0 += 16) {
            const int n0 = rb * npad + c0;
            if (n0 >= g.N) break;
            const uint32_t col = static_cast<uint32_t>((ab * nrb + rb) * np2 + 2 * c0);
            float c[32], v[16];
            __syncwarp();
            tmem_ld16(tmem + lane_base + col, c);
            tmem_ld16(tmem + lane_base + col + 16, c + 16);
            tmem_wait_ld();
  #pragma unroll
            for (int r = 0; r < 16; ++r) v[r] = c[2 * r] + c[2 * r + 1];
            if (complete) {
              epilogue_chunk(g, es, mt, n0, v, tl);
            } else if (g.csplit > 1) {   // this rank's partial, in its (now idle) stage ring
              float* cpart = reinterpret_cast<float*>(smem);
  #pragma unroll
              for (int r = 0; r < 16; ++r) cpart[static_cast<size_t>(n0 + r) * BM + tl] = v[r];
            } else {
  #pragma unroll
              for (int r = 0; r < 16; ++r) mypart[static_cast<size_t>(n0 + r) * BM + tl] = v[r];
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_acce + 8 * ab);
        if (!complete && g.csplit == 0) {
          __threadfence();
          named_bar(1, 128);
          const int cf = sc.owner(static_cast<long long>(mt) * KB);
          const int cl = sc.owner(static_cast<long long>(mt + 1) * KB - 1);
          if (tl == 0) {
            const int old = atomicAdd(g.counters + mt, 1);
            *last_flag = (old == cl - cf);
          }
          named_bar(1, 128);
          const int P = cl - cf + 1;
          // After the CTA's last unit its stage ring is idle (every MMA has completed and no
          // load is left): with more than one 16-row chunk the tile's partials come in by
          // bulk copy, one transfer in place of a round trip per chunk (operand-by-TMA
          // launches, whose source-row barriers are otherwise unused).  (With one chunk the
          // direct loads are the shorter path.)
          const bool staged = *last_flag && final_unit && g.b_tma && rows_total > 16 &&
                              static_cast<size_t>(P) * pbytes <= static_cast<size_t>(g.stages) * L.stage_bytes;
          if (staged) {
            __threadfence();
            if (tl == 0) {
              g.counters[mt] = 0;
              asm volatile("fence.proxy.async.global;" ::: "memory");   // the partials: generic writes
              mbar_arrive_expect_tx(bar_bfull, static_cast<uint32_t>(P * pbytes));
              for (int c = cf; c <= cl; ++c) {
                const int sl = (sc.begin(c) / KB == mt) ? 0 : 1;
                bulk_copy_g2s(sbase + static_cast<uint32_t>((c - cf) * pbytes),
                              g.part + (static_cast<size_t>(c) * 2 + sl) * rows_total * BM,
                              static_cast<uint32_t>(pbytes), bar_bfull);
              }
            }
            ok = epi_all(mbar_wait(bar_bfull, 0, g.err, abort_flag, wlim));
            if (!ok) {   // let the copies land before the CTA releases its shared memory
              const long long t0 = clock64();
              while (clock64() - t0 < 4000000) {
              }
            }
            const float* sp = reinterpret_cast<const float*>(smem);
            for (int rb = 0; rb < nrb && ok; ++rb) {
              for (int c0 = 0; c0 < npad; c0 += 16) {
                const int n0 = rb * npad + c0;
                if (n0 >= g.N) break;
                float v[16];
  #pragma unroll
                for (int r = 0; r < 16; ++r) v[r] = 0.f;
                for (int pp = 0; pp < P; ++pp) {   // partials summed in CTA order
                  const float* q0 = sp + (static_cast<size_t>(pp) * rows_total + n0) * BM + tl;
  #pragma unroll
                  for (int r = 0; r < 16; ++r) v[r] += q0[static_cast<size_t>(r) * BM];
                }
                epilogue_chunk(g, es, mt, n0, v, tl);
              }
            }
          } else if (*last_flag) {
            __threadfence();
            if (tl == 0) g.counters[mt] = 0;
            for (int rb = 0; rb < nrb; ++rb) {
              for (int c0 = 0; c0 < npad; c0 += 16) {
                const int n0 = rb * npad + c0;
                if (n0 >= g.N) break;
                // partials summed in CTA order; loads of up to 4 segments issued together
                float v[16];
  #pragma unroll
                for (int r = 0; r < 16; ++r) v[r] = 0.f;
                for (int c0 = cf; c0 <= cl; c0 += 4) {
                  float pv[4][16];
  #pragma unroll
                  for (int u = 0; u < 4; ++u) {
                    const int c = c0 + u;
                    if (c <= cl) {
                      const int sl = (sc.begin(c) / KB == mt) ? 0 : 1;
                      const float* p = g.part + (static_cast<size_t>(c) * 2 + sl) * rows_total * BM;
  #pragma unroll
                      for (int r = 0; r < 16; ++r) pv[u][r] = __ldcg(p + static_cast<size_t>(n0 + r) * BM + tl);
                    }
                  }
  #pragma unroll
                  for (int u = 0; u < 4; ++u)
                    if (c0 + u <= cl) {
  #pragma unroll
                      for (int r = 0; r < 16; ++r) v[r] += pv[u][r];
                    }
                }
                epilogue_chunk(g, es, mt, n0, v, tl);
              }
            }
          }
          named_bar(1, 128);
        }
        i += kb1 - kb0;
      }
    }
    if (g.e.kind == EPI_LMHEAD) lmhead_flush(g, es, cta, ncta, tl);
  }

  if (g.csplit > 1) {
    // Every thread of every rank passes both cluster barriers (whatever its role did), so
    // no rank can wait on one that left.  The 16-row chunks are dealt round-robin to the
    // ranks; the rank of a chunk sums all ranks' partials of it in rank order.
    cooperative_groups::cluster_group cluster = cooperative_groups::this_cluster();
    const bool red = warp >= 2 && warp < 6;
    const bool pre_ok = red && cs_r == 0 && g.N <= 16;   // one chunk of rows: inputs load during the barrier
    const int tl = (warp & 3) * 32 + lane;
    EpiSmem es = epi_views(smem + L.epi_off, smem + L.lm_off, g.N, g.e.topk);
    es.rstd = reinterpret_cast<float*>(smem + L.erstd_off);
    float pre_a[16], pre_b[16];
    if (pre_ok) epilogue_prefetch(g, es, cs_t, 0, tl, pre_a, pre_b);
    cluster.sync();
    if (red) {
      int ci = 0;   // chunk counter, for the round-robin deal
      for (int rb = 0; rb < nrb; ++rb) {
        for (int c0 = 0; c0 < npad; c0 += 16, ++ci) {
          const int n0 = rb * npad + c0;
          if (n0 >= g.N) break;
          if (ci % g.csplit != cs_r) continue;
          float v[16];
#pragma unroll
          for (int r = 0; r < 16; ++r) v[r] = 0.f;
          for (int q0 = 0; q0 < g.csplit; q0 += 2) {   // loads of two ranks in flight together
            float pv[2][16];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              if (q0 + u < g.csplit) {
                const float* pq = cluster.map_shared_rank(reinterpret_cast<float*>(smem), q0 + u);
#pragma unroll
                for (int r = 0; r < 16; ++r) pv[u][r] = pq[static_cast<size_t>(n0 + r) * BM + tl];
              }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u)
              if (q0 + u < g.csplit) {
#pragma unroll
                for (int r = 0; r < 16; ++r) v[r] += pv[u][r];
              }
          }
          if (pre_ok) epilogue_chunk(g, es, cs_t, n0, v, tl, pre_a, pre_b);
          else epilogue_chunk(g, es, cs_t, n0, v, tl);
        }
      }
    }
    cluster.sync();   // the partials stay in place until every rank has read them
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, g.tmem_cols);
  }
  if (PAIR) cooperative_groups::this_cluster().sync();   // neither CTA leaves while the other may signal it
}

// ============================================================ SIMT mainloop (f32)
// One CTA (256 threads) per (128-feature tile, 16-row block); full K per CTA.
constexpr int SIMT_ROWS = 16;

__global__ void __launch_bounds__(256)
gemm_simt_kernel(const float* __restrict__ W0, const float* __restrict__ W1, const GemmArgs g) {
  extern __shared__ float sm[];
  float* xs = sm;                                   // [16][K] activation rows
  float* acc = xs + SIMT_ROWS * g.K;                // [16][128]
  float* rstd = acc + SIMT_ROWS * BM;               // [N]
  EpiScratch* scr = reinterpret_cast<EpiScratch*>(rstd + ((g.N + 31) & ~31));
  float* lm = reinterpret_cast<float*>(scr + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = blockIdx.x, n0 = blockIdx.y * SIMT_ROWS;
  pdl_wait();
  pdl_trigger();
  compute_rstd(g.b, g.N, rstd, tid, 256);
  __syncthreads();
  for (int idx = tid; idx < SIMT_ROWS * (g.K / 8); idx += 256) {
    const int r = idx / (g.K / 8), k = (idx % (g.K / 8)) * 8;
    float v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (n0 + r < g.N) load_b8(g.b, n0 + r, k, rstd, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) xs[r * g.K + k + i] = v[i];
  }
  __syncthreads();
  for (int f = warp; f < BM; f += 8) {
    const int m = mt * BM + f;
    float a[SIMT_ROWS];
#pragma unroll
    for (int r = 0; r < SIMT_ROWS; ++r) a[r] = 0.f;
    if (m < g.M) {
      const float* w = (m < g.m_split) ? W0 + static_cast<size_t>(m) * g.K
                                       : W1 + static_cast<size_t>(m - g.m_split) * g.K;
      for (int k = lane; k < g.K; k += 32) {
        const float wk = __ldg(w + k);
#pragma unroll
        for (int r = 0; r < SIMT_ROWS; ++r) a[r] += wk * xs[r * g.K + k];
      }
    }
#pragma unroll
    for (int r = 0; r < SIMT_ROWS; ++r) {
      const float s = warp_sum(a[r]);
      if (lane == 0) acc[r * BM + f] = s;
    }
  }
  __syncthreads();
  if (tid < 128) {
    EpiSmem es = epi_views(scr, lm, g.N, g.e.topk);
    if (g.e.kind == EPI_LMHEAD) lmhead_init(g, es, tid);
    float v[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) v[r] = acc[r * BM + tid];
    epilogue_chunk(g, es, mt, n0, v, tid);
    if (g.e.kind == EPI_LMHEAD) {
      // this CTA owns rows [n0, n0+16) of tile mt: partial slot = tile
      named_bar(1, 128);
      const int k = g.e.topk;
      for (int r = tid; r < SIMT_ROWS; r += 128) {
        const int n = n0 + r;
        if (n >= g.N) continue;
        const size_t o = static_cast<size_t>(n) * gridDim.x + mt;
        const int cnt = es.st_cnt[n];
        for (int j = 0; j < k; ++j) {
          g.e.lm_val[o * k + j] = j < cnt ? es.lv[static_cast<size_t>(n) * k + j] : -INFINITY;
          g.e.lm_id[o * k + j] = j < cnt ? es.li[static_cast<size_t>(n) * k + j] : -1;
        }
      }
    }
  }
}

// ================================================================== host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool make_weight_map(CUtensorMap* tm, const void* w, int M, int K, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {BK, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_kv_map(CUtensorMap* tm, const void* cache, long long tokens, int Hkv) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !cache || tokens < 1 || Hkv < 1) return false;
  const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(tokens)};
  const cuuint64_t strides[2] = {256, static_cast<cuuint64_t>(Hkv) * 256};
  const cuuint32_t box[3] = {64, 1, 64};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(cache), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_act_map(CUtensorMap* tm, const void* hl, int rows, int K, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {BK, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(hl), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// SM count of the current device, cached per device ordinal (GPUs of one host may differ).
constexpr int MAX_DEVICES = 64;
static int g_num_sms[MAX_DEVICES] = {};
int num_sms() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= MAX_DEVICES) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n;
  }
  if (!g_num_sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}

constexpr int TC_MAX_SMEM = 232448;
static size_t g_tc_smem_cap = 0, g_simt_smem_cap = 0;

size_t max_dyn_smem(const void* func) {
  int dev = 0, optin = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, func) != cudaSuccess) return 0;
  return optin > static_cast<int>(fa.sharedSizeBytes) ? optin - fa.sharedSizeBytes : 0;
}

cudaError_t allow_max_smem(const void* func, size_t* granted) {
  const size_t m = max_dyn_smem(func);
  if (granted) *granted = m;
  if (m == 0) return cudaErrorInvalidValue;
  return cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(m));
}

// Clusters of S CTAs of the one-CTA-per-SM kernel (full shared memory) the device holds
// at once; cached per device and size.
int gemm_active_clusters(int S) {
  static std::mutex mu;
  static int cache[MAX_DEVICES][9];
  static bool init = false;
  std::lock_guard<std::mutex> lk(mu);
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= MAX_DEVICES || S < 1 || S > 8) return 0;
  if (!init) {
    for (auto& row : cache)
      for (int& c : row) c = -1;
    init = true;
  }
  if (cache[dev][S] >= 0) return cache[dev][S];
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(S, 1, 1);
  cfg.blockDim = dim3(TC_THREADS, 1, 1);
  cfg.dynamicSmemBytes = g_tc_smem_cap ? g_tc_smem_cap : 200 * 1024;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<TC_THREADS, 1, false>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[dev][S] = n;
  return n;
}

GemmPlan gemm_plan(bool tc, const CUtensorMap& tm0, const CUtensorMap* tm1, const void* w0, const void* w1,
                   int M, int K, int m_split, float* part, int* counters, unsigned* err) {
  GemmPlan p;
  p.tc = tc;
  if (tc) {
    p.tm0 = tm0;
    p.tm1 = tm1 ? *tm1 : tm0;
  } else {
    p.w0f = static_cast<const float*>(w0);
    p.w1f = static_cast<const float*>(w1 ? w1 : w0);
  }
  GemmArgs& g = p.args;
  memset(&g, 0, sizeof(g));
  g.M = M;
  g.K = K;
  g.m_split = m_split;
  g.part = part;
  g.counters = counters;
  g.err = err;
  return p;
}

EpiArgs epi_store(float* out, int ldo, const float* resid, int ldr, float* ss, int ss_ld) {
  EpiArgs e;
  memset(&e, 0, sizeof(e));
  e.kind = EPI_STORE;
  e.out = out;
  e.ldo = ldo;
  e.resid = resid;
  e.ldr = ldr;
  e.ss = ss;
  e.ss_ld = ss_ld;
  return e;
}

// Fill the launch geometry of a GEMM over N rows.
bool plan_gemm(GemmPlan& p, int N) {
  GemmArgs& g = p.args;
  g.N = N;
  g.KB = (g.K + BK - 1) / BK;
  g.MT = (g.M + BM - 1) / BM;
  if (!p.tc) {
    p.grid = g.MT;
    p.grid_y = (N + SIMT_ROWS - 1) / SIMT_ROWS;
    p.smem = sizeof(float) * (SIMT_ROWS * g.K + SIMT_ROWS * BM + ((N + 31) & ~31)) + sizeof(EpiScratch) +
             static_cast<size_t>(N) * (3 + 2 * std::max(1, g.e.topk)) * 4 + 64;
    return p.smem <= (g_simt_smem_cap ? g_simt_smem_cap : static_cast<size_t>(TC_MAX_SMEM));
  }
  g.nrb = (N + MAX_ROWS_PER_BLOCK - 1) / MAX_ROWS_PER_BLOCK;
  const int per = (N + g.nrb - 1) / g.nrb;
  g.npad = std::max(16, (per + 15) / 16 * 16);
  const int accum_cols = g.nrb * 2 * g.npad;
  g.nbuf = (2 * accum_cols <= 512) ? 2 : 1;
  int cols = 32;
  while (cols < g.nbuf * accum_cols) cols <<= 1;
  g.tmem_cols = cols;
  const long long total = static_cast<long long>(g.MT) * g.KB;
  const int sms = num_sms();
  p.grid = p.pair ? 2 * static_cast<int>(std::min<long long>(sms / 2, total)) : static_cast<int>(std::min<long long>(sms, total));
  p.grid_y = 1;
  const int topk = std::max(1, g.e.topk);
  const int lm_rows = g.e.kind == EPI_LMHEAD ? N : 0;
  // Work split.  Few tiles (the small-N projections): S CTAs per tile in a cluster, each
  // on 1/S of K, reduced on chip, when the clusters cover >= 80% of the SMs; enough tiles
  // to fill the SMs: one tile per CTA; otherwise (the LM head, very wide layers, tile
  // counts the clusters would leave SMs idle for) the stream-K schedule.
  g.csplit = 0;
  const size_t part_bytes = static_cast<size_t>(g.nrb) * g.npad * BM * sizeof(float);
  if (g.e.kind != EPI_LMHEAD && g.e.kind != EPI_LOGITS && !p.stream_k) {
    int S = std::min(std::min(8, g.KB), sms / g.MT);
    while (S >= 2 && gemm_active_clusters(S) < g.MT) --S;
    // Long K (fc's 2d, the FFN's d_ff) takes the clusters too when the launch has one 16-row
    // chunk: the on-chip reduction's shorter tail outweighs the clusters' later start (each
    // waits for S free SMs where stream-K CTAs start SM by SM as the previous kernel
    // retires); with more rows the long-K stream-K launches measured faster.  With two or
    // more row blocks the stream-K partial tiles double and the accumulator loses its second
    // buffer, so the clusters win there.  (With more than one 16-row chunk the reduction
    // tail, spread over the ranks, matters more than covering every SM with the weight
    // stream.)
    if (S >= 2 && (g.K < 8192 || g.nrb > 1 || N <= 16) &&
        (5 * g.MT * S >= 4 * sms || (N > 16 && 2 * g.MT * S >= sms))) {
      g.csplit = S;
      p.occ = 1;
    } else if (S < 2 && 4 * g.MT >= 3 * sms && g.MT <= sms * (g.b_tma ? 2 : 1)) {
      g.csplit = 1;
      p.occ = g.MT > sms ? 2 : 1;
    }
    if (g.csplit > 0) p.grid = g.MT * g.csplit;
  }
  if (p.occ == 2 && (!g.b_tma || g.tmem_cols > 256)) {
    p.occ = 1;
    if (g.csplit == 1 && g.MT > sms) {   // one tile per CTA needs two CTAs per SM here
      g.csplit = 0;
      p.grid = static_cast<int>(std::min<long long>(sms, total));
    }
  }
  uint32_t cap = static_cast<uint32_t>(g_tc_smem_cap ? g_tc_smem_cap : TC_MAX_SMEM);
  if (p.occ == 2) cap = std::min(cap, TC_SMEM_OCC2);
  // Few rows (one 16-row block): the MMA issuer's per-stage work (barrier wait, commit,
  // loop) rather than the tensor core bounds its rate, so a stage carries two K blocks.
  g.kpair = g.b_tma && g.npad <= 16 ? 1 : 0;
  int stages = 12;
  const bool staged = g.e.kind == EPI_STORE || g.e.kind == EPI_SWIGLU;
  while (stages >= 2 && tc_smem_bytes(g.npad, stages, lm_rows, topk, staged, g.kpair) > cap) --stages;
  if (stages < 2) return false;
  if (g.csplit > 1 &&
      part_bytes > static_cast<size_t>(stages) * tc_layout(g.npad, stages, g.kpair).stage_bytes) {
    // the partial tile does not fit the stage ring it is parked in: stream-K instead
    g.csplit = 0;
    p.grid = static_cast<int>(std::min<long long>(sms, total));
  }
  if (p.pair && (g.csplit != 0 || p.occ != 1 || g.kpair)) return false;
  g.stages = stages;
  p.smem = tc_smem_bytes(g.npad, stages, lm_rows, topk, staged, g.kpair);
  if (g.b_tma) {
    // the operand copy holds 2 N rows (hi, lo); rows past them read as zero
    if (!p.b_hl || !make_act_map(&p.tmB, p.b_hl, 2 * N, g.K, 2 * g.npad)) return false;
  } else {
    p.tmB = p.tm0;
  }
  return true;
}

bool plan_gemm_pair(GemmPlan& p, int N, size_t part_half) {
  const int per = (N + 1) / 2, n1 = N - per;
  if (!p.tc || !p.args.b_tma || n1 < 1 || per > MAX_ROWS_PER_BLOCK) return false;
  const EpiKind ek = static_cast<EpiKind>(p.args.e.kind);
  if (ek != EPI_STORE && ek != EPI_QKV && ek != EPI_SWIGLU && ek != EPI_LOGITS) return false;
  p.pair = true;
  p.stream_k = true;
  p.occ = 1;
  const uint16_t* b_hl = p.b_hl;
  if (!plan_gemm(p, per)) return false;
  if (p.args.MT > 8192 || p.args.nrb != 1) return false;
  // rank 1: the same plan on rows [per, N)
  GemmArgs& g1 = p.args1;
  g1 = p.args;
  g1.N = n1;
  EpiArgs& e = g1.e;
  if (e.out) e.out += static_cast<size_t>(per) * e.ldo;
  if (e.resid) e.resid += static_cast<size_t>(per) * e.ldr;
  if (e.ss) e.ss += per;
  if (e.hl) e.hl += 2 * static_cast<size_t>(per) * e.hl_ld;
  if (e.nss) e.nss += per;
  if (e.q) e.q += static_cast<size_t>(per) * e.Hq * e.hd;
  if (e.row_req) e.row_req += per;
  if (e.row_slot) e.row_slot += per;
  if (e.row_pos) e.row_pos += per;
  if (e.logits) e.logits += static_cast<size_t>(per) * g1.M;
  if (e.seeds) e.sample_row0 += per;
  g1.counters = p.args.counters + 8192;
  g1.part = p.args.part + part_half;
  return make_act_map(&p.tmB1, b_hl + 2 * static_cast<size_t>(per) * g1.K, 2 * n1, g1.K, 2 * g1.npad);
}

cudaError_t gemm_setup_attributes() {
  cudaError_t e = allow_max_smem(reinterpret_cast<const void*>(gemm_tc_kernel<TC_THREADS, 1, false>), &g_tc_smem_cap);
  if (e != cudaSuccess) return e;
  e = allow_max_smem(reinterpret_cast<const void*>(gemm_tc_kernel<TC_THREADS_TMA, 1, false, true>));
  if (e != cudaSuccess) return e;
  e = allow_max_smem(reinterpret_cast<const void*>(gemm_tc_kernel<TC_THREADS_TMA, 2, false>));
  if (e != cudaSuccess) return e;
  e = allow_max_smem(reinterpret_cast<const void*>(gemm_tc_kernel<TC_THREADS_TMA, 1, false>));
  if (e != cudaSuccess) return e;
  e = allow_max_smem(reinterpret_cast<const void*>(gemm_tc_kernel<TC_THREADS_TMA, 1, true>));
  if (e != cudaSuccess) return e;
  return allow_max_smem(reinterpret_cast<const void*>(gemm_simt_kernel), &g_simt_smem_cap);
}

cudaError_t launch_gemm(const GemmPlan& p, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = p.tc && p.args.csplit > 1 ? p.args.csplit : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.tc && (p.args.csplit > 1 || p.pair) ? 2 : 1;
  cfg.stream = st;
  cfg.dynamicSmemBytes = p.smem;
  if (p.tc) {
    cfg.gridDim = dim3(p.grid, 1, 1);
    if (p.pair) {   // clusters of two CTAs sharing the weight stream
      attr[1].val.clusterDim.x = 2;
      cfg.blockDim = dim3(TC_THREADS_TMA, 1, 1);
      return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<TC_THREADS_TMA, 1, false, true>, p.tm0, p.tm1, p.tmB, p.args,
                                p.tmB1, p.args1);
    }
    if (p.occ == 2) {
      cfg.blockDim = dim3(TC_THREADS_TMA, 1, 1);
      return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<TC_THREADS_TMA, 2, false>, p.tm0, p.tm1, p.tmB, p.args, p.tmB,
                                p.args);
    }
    if (p.args.b_tma) {   // no converter warps: the full register file for 7 warps
      cfg.blockDim = dim3(TC_THREADS_TMA, 1, 1);
      if (p.args.e.kind == EPI_LMHEAD && p.args.N <= 16)   // stream-K with the split tiles first
        return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<TC_THREADS_TMA, 1, true>, p.tm0, p.tm1, p.tmB, p.args, p.tmB,
                                  p.args);
      return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<TC_THREADS_TMA, 1, false>, p.tm0, p.tm1, p.tmB, p.args, p.tmB,
                                p.args);
    }
    cfg.blockDim = dim3(TC_THREADS, 1, 1);
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<TC_THREADS, 1, false>, p.tm0, p.tm1, p.tmB, p.args, p.tmB, p.args);
  }
  cfg.gridDim = dim3(p.grid, p.grid_y, 1);
  cfg.blockDim = dim3(256, 1, 1);
  return cudaLaunchKernelEx(&cfg, gemm_simt_kernel, p.w0f, p.w1f, p.args);
}

}  // namespace eagle
