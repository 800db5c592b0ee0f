// Tree-masked grouped-query decode attention of one draft depth.
//
// Every row of the depth (a frontier node) attends to its request's whole verified
// prefix (post-RoPE KV cache, read once per KV head) and to the tree rows that are its
// ancestors or itself (ancestor bit mask; "Tree attention in one verification pass",
// aicassindra.com tm_eagle_deep).  All query heads of a KV group and all rows of the
// request share one pass over the prefix keys.
//
// Grid (cluster rank, kv head, request), one thread-block cluster per (request, kv head).
// The keys are cut into 64-key chunks (the prefix chunks, then one chunk holding the
// tree rows); CTA r of a cluster of cs takes chunks r, r + cs, ... and keeps an online
// softmax state per query vector; the cluster then merges the states through
// distributed shared memory, in a fixed order (deterministic).  Two kernels share this
// plan: an fp32 SIMT one (f32 caches, any head size) and a tensor-core one (bf16 cache,
// head size 128).
#include "common.cuh"
#include "internal.h"

#include <cooperative_groups.h>
#include <algorithm>
#include <cstdlib>
#include <mutex>
namespace cg = cooperative_groups;

namespace eagle {

constexpr int ATT_THREADS = 256;
constexpr int KT_LD = ATT_CHUNK;        // Kt row stride (floats)
constexpr int VS_LD = 132;              // Vs row stride: 128 + 4 keeps float4 rows on distinct banks
constexpr int ATT_MAX_CLUSTER = 16;
constexpr int ATT_MAX_BLOCKS = 4;       // 4x4 (query, dim) output blocks per thread: qv <= 128

struct AttSmem {
  float* qt;     // [hd][qvp]      queries, transposed, pre-scaled
  float* kt;     // [hd][KT_LD]    keys, transposed (reused for the final state [qv][hd])
  float* vs;     // [CH][VS_LD]
  float* pt;     // [CH][qvp]      scores, then probabilities
  float* mrow;   // [qvp]          running max
  float* lrow;   // [qvp]          running sum of exp
  float* alpha;  // [qvp]          rescale of this chunk
};

size_t attn_smem_bytes(int qv, int hd) {
  const int qvp = (qv + 3) & ~3;
  return sizeof(float) * (static_cast<size_t>(hd) * qvp + static_cast<size_t>(hd) * KT_LD +
                          static_cast<size_t>(ATT_CHUNK) * VS_LD + static_cast<size_t>(ATT_CHUNK) * qvp +
                          3 * qvp) + 16;
}

size_t attn_merge_capacity(int qv, int hd) {   // the final state [qv][hd] lives in kt + vs
  (void)qv;
  return static_cast<size_t>(hd) * KT_LD + static_cast<size_t>(ATT_CHUNK) * VS_LD;
}

EAGLE_DEV void bf8_to_f(const uint4 u, float* v) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// One cluster (gridDim.x CTAs) per (KV head, request).  CTA r of the cluster takes the
// 64-key chunks r, r + cs, ... of [prefix chunks..., tree chunk] and keeps an online
// softmax state per query vector; the cluster then merges the states through
// distributed shared memory (CTA order, deterministic).
__global__ void __launch_bounds__(ATT_THREADS)
tree_attention_kernel(const AttnArgs a) {
  extern __shared__ float4 att_smem4[];
  float* sm = reinterpret_cast<float*>(att_smem4);
  cg::cluster_group cluster = cg::this_cluster();
  const int cs = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hd = a.hd, gq = a.Hq / a.Hkv;
  const int qv = a.rows_per_req * gq, qvp = (qv + 3) & ~3;
  AttSmem S;
  S.qt = sm;
  S.kt = S.qt + hd * qvp;
  S.vs = S.kt + hd * KT_LD;
  S.pt = S.vs + ATT_CHUNK * VS_LD;
  S.mrow = S.pt + ATT_CHUNK * qvp;
  S.lrow = S.mrow + qvp;
  S.alpha = S.lrow + qvp;

  pdl_wait();
  pdl_trigger();
  const int nb = __ldcg(a.n_eff + b);
  const int npre = (nb + ATT_CHUNK - 1) / ATT_CHUNK;
  const int nchunks = npre + 1;                 // the last chunk holds the tree rows
  const int row0 = b * a.rows_per_req;
  const float scale = 1.0f / sqrtf(static_cast<float>(hd));
  const int dg_n = hd / 8;
  const int nvb = qvp / 4;
  const int nblk = nvb * (hd / 4);             // output blocks of 4 query vectors x 4 dims

  // queries (consecutive threads take consecutive query vectors: conflict-free transpose)
  for (int idx = tid; idx < qvp * (hd / 4); idx += ATT_THREADS) {
    const int v = idx % qvp, d4 = idx / qvp;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (v < qv) {
      const int i = v / gq, gh = v - i * gq;
      x = __ldcg(reinterpret_cast<const float4*>(a.q + (static_cast<size_t>(row0 + i) * a.Hq + kvh * gq + gh) * hd) + d4);
    }
    S.qt[(4 * d4 + 0) * qvp + v] = x.x * scale;
    S.qt[(4 * d4 + 1) * qvp + v] = x.y * scale;
    S.qt[(4 * d4 + 2) * qvp + v] = x.z * scale;
    S.qt[(4 * d4 + 3) * qvp + v] = x.w * scale;
  }
  for (int v = tid; v < qvp; v += ATT_THREADS) {
    S.mrow[v] = -INFINITY;
    S.lrow[v] = 0.f;
  }
  float acc[ATT_MAX_BLOCKS][4][4];
#pragma unroll
  for (int u = 0; u < ATT_MAX_BLOCKS; ++u)
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) acc[u][x][y] = 0.f;

  for (int c = rank; c < nchunks; c += cs) {
    const bool tree = c == npre;
    const int nkeys = tree ? a.tree_upto : min(ATT_CHUNK, nb - c * ATT_CHUNK);
    __syncthreads();   // the previous chunk's keys, values and probabilities are consumed
    // keys (transposed) and values: consecutive threads take consecutive keys
    for (int idx = tid; idx < ATT_CHUNK * dg_n; idx += ATT_THREADS) {
      const int j = idx % ATT_CHUNK, dg = idx / ATT_CHUNK;
      float kx[8], vx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) kx[e] = vx[e] = 0.f;
      if (j < nkeys) {
        if (tree) {
          const size_t o = ((static_cast<size_t>(b) * a.tree_rows + j) * a.Hkv + kvh) * hd + 8 * dg;
          const float4* kp = reinterpret_cast<const float4*>(a.tk + o);
          const float4* vp = reinterpret_cast<const float4*>(a.tv + o);
          const float4 k0 = __ldcg(kp), k1 = __ldcg(kp + 1), v0 = __ldcg(vp), v1 = __ldcg(vp + 1);
          kx[0] = k0.x; kx[1] = k0.y; kx[2] = k0.z; kx[3] = k0.w; kx[4] = k1.x; kx[5] = k1.y; kx[6] = k1.z; kx[7] = k1.w;
          vx[0] = v0.x; vx[1] = v0.y; vx[2] = v0.z; vx[3] = v0.w; vx[4] = v1.x; vx[5] = v1.y; vx[6] = v1.z; vx[7] = v1.w;
        } else {
          const size_t o =
              ((static_cast<size_t>(__ldg(a.cu_seqlens + b)) + c * ATT_CHUNK + j) * a.Hkv + kvh) * hd + 8 * dg;
          if (a.cache_bf16) {
            bf8_to_f(__ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.k_cache) + o)), kx);
            bf8_to_f(__ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.v_cache) + o)), vx);
          } else {
            const float4* kp = reinterpret_cast<const float4*>(static_cast<const float*>(a.k_cache) + o);
            const float4* vp = reinterpret_cast<const float4*>(static_cast<const float*>(a.v_cache) + o);
            const float4 k0 = __ldg(kp), k1 = __ldg(kp + 1), v0 = __ldg(vp), v1 = __ldg(vp + 1);
            kx[0] = k0.x; kx[1] = k0.y; kx[2] = k0.z; kx[3] = k0.w; kx[4] = k1.x; kx[5] = k1.y; kx[6] = k1.z; kx[7] = k1.w;
            vx[0] = v0.x; vx[1] = v0.y; vx[2] = v0.z; vx[3] = v0.w; vx[4] = v1.x; vx[5] = v1.y; vx[6] = v1.z; vx[7] = v1.w;
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) S.kt[(8 * dg + e) * KT_LD + j] = kx[e];
      float4* vdst = reinterpret_cast<float4*>(S.vs + j * VS_LD + 8 * dg);
      vdst[0] = make_float4(vx[0], vx[1], vx[2], vx[3]);
      vdst[1] = make_float4(vx[4], vx[5], vx[6], vx[7]);
    }
    __syncthreads();

    // scores: 4 query vectors x 4 keys per thread block
    for (int blk = tid; blk < nvb * (ATT_CHUNK / 4); blk += ATT_THREADS) {
      const int vb = blk / (ATT_CHUNK / 4), jb = blk - vb * (ATT_CHUNK / 4);
      float sc[4][4] = {};
#pragma unroll 4
      for (int d = 0; d < hd; ++d) {
        const float4 qq = *reinterpret_cast<const float4*>(S.qt + d * qvp + 4 * vb);
        const float4 kk = *reinterpret_cast<const float4*>(S.kt + d * KT_LD + 4 * jb);
        const float qa[4] = {qq.x, qq.y, qq.z, qq.w}, ka[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
          for (int y = 0; y < 4; ++y) sc[x][y] += qa[x] * ka[y];
      }
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        const int j = 4 * jb + y;
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int v = 4 * vb + x;
          bool vis = j < nkeys && v < qv;
          if (vis && tree) {
            const unsigned long long msk = __ldcg(a.row_mask + row0 + v / gq);
            vis = (msk >> j) & 1ull;
          }
          S.pt[j * qvp + v] = vis ? sc[x][y] : -INFINITY;
        }
      }
    }
    __syncthreads();

    // online softmax update per query vector
    for (int v = warp; v < qvp; v += ATT_THREADS / 32) {
      const float s0 = S.pt[lane * qvp + v], s1 = S.pt[(lane + 32) * qvp + v];
      const float mold = S.mrow[v];
      const float mnew = fmaxf(mold, warp_max(fmaxf(s0, s1)));
      float p0 = 0.f, p1 = 0.f;
      if (mnew != -INFINITY) {
        p0 = expf(s0 - mnew);
        p1 = expf(s1 - mnew);
      }
      S.pt[lane * qvp + v] = p0;
      S.pt[(lane + 32) * qvp + v] = p1;
      const float l = warp_sum(p0 + p1);
      if (lane == 0) {
        const float al = mold == -INFINITY ? 0.f : expf(mold - mnew);
        S.alpha[v] = al;
        S.lrow[v] = S.lrow[v] * al + l;
        S.mrow[v] = mnew;
      }
    }
    __syncthreads();

    // acc = acc * alpha + P V
#pragma unroll
    for (int u = 0; u < ATT_MAX_BLOCKS; ++u) {
      const int blk = tid + u * ATT_THREADS;
      if (blk >= nblk) break;
      const int vb = blk / (hd / 4), db = blk - vb * (hd / 4);
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float al = S.alpha[4 * vb + x];
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[u][x][y] *= al;
      }
      for (int j = 0; j < nkeys; ++j) {
        const float4 pp = *reinterpret_cast<const float4*>(S.pt + j * qvp + 4 * vb);
        const float4 vv = *reinterpret_cast<const float4*>(S.vs + j * VS_LD + 4 * db);
        const float pa[4] = {pp.x, pp.y, pp.z, pp.w}, va[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
          for (int y = 0; y < 4; ++y) acc[u][x][y] += pa[x] * va[y];
      }
    }
  }

  // publish this CTA's state [qv][hd] (in the key/value buffers) and merge across the cluster
  __syncthreads();
  float* st = S.kt;
#pragma unroll
  for (int u = 0; u < ATT_MAX_BLOCKS; ++u) {
    const int blk = tid + u * ATT_THREADS;
    if (blk >= nblk) break;
    const int vb = blk / (hd / 4), db = blk - vb * (hd / 4);
#pragma unroll
    for (int x = 0; x < 4; ++x)
      *reinterpret_cast<float4*>(st + (4 * vb + x) * hd + 4 * db) =
          make_float4(acc[u][x][0], acc[u][x][1], acc[u][x][2], acc[u][x][3]);
  }
  cluster.sync();
  const size_t ld = static_cast<size_t>(a.Hq) * hd;
  for (int idx = rank * ATT_THREADS + tid; idx < qv * (hd / 4); idx += cs * ATT_THREADS) {
    const int v = idx / (hd / 4), d4 = idx - v * (hd / 4);
    float M = -INFINITY;
    for (int r = 0; r < cs; ++r) M = fmaxf(M, cluster.map_shared_rank(S.mrow, r)[v]);
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r = 0; r < cs; ++r) {
      const float mr = cluster.map_shared_rank(S.mrow, r)[v];
      const float w = mr == -INFINITY ? 0.f : expf(mr - M);
      L += w * cluster.map_shared_rank(S.lrow, r)[v];
      const float4 x = *reinterpret_cast<const float4*>(cluster.map_shared_rank(st, r) + v * hd + 4 * d4);
      o.x += w * x.x;
      o.y += w * x.y;
      o.z += w * x.z;
      o.w += w * x.w;
    }
    const float inv = 1.0f / L;
    o.x *= inv;
    o.y *= inv;
    o.z *= inv;
    o.w *= inv;
    const int i = v / gq, gh = v - i * gq;
    const size_t col = static_cast<size_t>(kvh * gq + gh) * hd + 4 * d4;
    *reinterpret_cast<float4*>(a.out + static_cast<size_t>(row0 + i) * ld + col) = o;
    if (a.out_hl) {   // bf16 hi / lo rows: the O projection's operand copy
      const float ov[4] = {o.x, o.y, o.z, o.w};
      uint16_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) split_hilo(ov[e], hi[e], lo[e]);
      uint2* h2 = reinterpret_cast<uint2*>(a.out_hl + 2 * static_cast<size_t>(row0 + i) * ld + col);
      uint2* l2 = reinterpret_cast<uint2*>(a.out_hl + (2 * static_cast<size_t>(row0 + i) + 1) * ld + col);
      *h2 = make_uint2(hi[0] | (static_cast<uint32_t>(hi[1]) << 16), hi[2] | (static_cast<uint32_t>(hi[3]) << 16));
      *l2 = make_uint2(lo[0] | (static_cast<uint32_t>(lo[1]) << 16), lo[2] | (static_cast<uint32_t>(lo[3]) << 16));
    }
  }
  cluster.sync();   // the other CTAs' shared memory stays alive until every read is done
}

// ============================================================ tensor-core path
// bf16 prefix cache, head_dim 128.  Same cluster decomposition and merge as above; the
// inner products run on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate)
// with the fp32 operands (queries, probabilities, tree-row keys and values) split into
// bf16 hi + lo parts, so each product keeps ~16 significant bits: S = Qhi K + Qlo K,
// O += Phi V + Plo V (the bf16 cache is exact in bf16).  Warp (m, s) owns query vectors
// [16 m, 16 m + 16) and the 16-key groups s, s + KS, ... of every chunk; its online
// softmax state (row max, row sum, output tile) stays in registers.  Keys and values of
// the CTA's prefix chunks stream through a 4-stage cp.async ring.
constexpr int TA_HD = 128;
constexpr int TA_ROWB = TA_HD * 2 + 16;                 // smem row stride: conflict-free ldmatrix
constexpr int TA_TILE = ATT_CHUNK * TA_ROWB;             // one 64-key tile (bytes)
constexpr int TA_NST = 4;
constexpr size_t TA_RING = static_cast<size_t>(TA_NST) * 2 * TA_TILE;
constexpr size_t TA_TREE = static_cast<size_t>(4) * TA_TILE;   // tree keys / values, hi and lo
constexpr int TA_MAX_QV = 128;
constexpr size_t TA_SMEM = TA_RING + TA_TREE + 4 * sizeof(float) * 4 * TA_MAX_QV;
static_assert(sizeof(float) * TA_MAX_QV * TA_HD <= TA_RING, "merge state must fit the ring");

EAGLE_DEV void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;   // 0: fill with zeros, read nothing
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
EAGLE_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
EAGLE_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

EAGLE_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
EAGLE_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
EAGLE_DEV void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};"
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// bf16 hi / lo parts of two floats, packed (first float in the low half)
EAGLE_DEV void split2(float x, float y, uint32_t& hi, uint32_t& lo) {
  uint16_t hx, lx, hy, ly;
  split_hilo(x, hx, lx);
  split_hilo(y, hy, ly);
  hi = hx | (static_cast<uint32_t>(hy) << 16);
  lo = lx | (static_cast<uint32_t>(ly) << 16);
}

// key groups (of 16) per warp for WM query tiles of 16 vectors on 8 warps
__host__ __device__ inline int ta_key_splits(int wm) { return wm <= 2 ? 4 : (wm <= 4 ? 2 : 1); }

struct TaWarp {
  uint32_t qh[8][4], ql[8][4];     // query fragments (A), 8 k-steps of 16 dims
  float o[16][4];                  // output tile 16 x 128
  float m0, m1, l0, l1;            // rows g and g + 8: running max (log2 units), partial sums
  unsigned long long mk0, mk1;     // ancestor masks of the rows (tree chunk)
};

// one chunk (64 keys) for warp (its query tile, key groups ks, ks + KS, ...)
template <bool TREE>
EAGLE_DEV void ta_chunk(TaWarp& w, uint32_t khi, uint32_t klo, uint32_t vhi, uint32_t vlo, int nkeys, int ks,
                        int KS, int lane) {
  const int t4 = lane & 3;
  float s[4][2][4];
#pragma unroll
  for (int gi = 0; gi < 4; ++gi) {
    if (gi * KS + ks >= 4) break;
    const int kg = ks + gi * KS;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) s[gi][nt][e] = 0.f;
      const int key0 = kg * 16 + nt * 8;
      const uint32_t roff = (key0 + (lane & 7)) * TA_ROWB + (lane >> 3) * 16;
#pragma unroll
      for (int k2 = 0; k2 < 4; ++k2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(khi + roff + k2 * 64, b0, b1, b2, b3);
        mma_bf16(s[gi][nt], w.qh[2 * k2], b0, b1);
        mma_bf16(s[gi][nt], w.ql[2 * k2], b0, b1);
        mma_bf16(s[gi][nt], w.qh[2 * k2 + 1], b2, b3);
        mma_bf16(s[gi][nt], w.ql[2 * k2 + 1], b2, b3);
        if (TREE) {
          ldsm_x4(klo + roff + k2 * 64, b0, b1, b2, b3);
          mma_bf16(s[gi][nt], w.qh[2 * k2], b0, b1);
          mma_bf16(s[gi][nt], w.qh[2 * k2 + 1], b2, b3);
        }
      }
      // visibility: key inside the chunk, and (tree rows) an ancestor of the query's row
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = key0 + 2 * t4 + (e & 1);
        bool vis = key < nkeys;
        if (TREE) vis = vis && (((e < 2 ? w.mk0 : w.mk1) >> key) & 1ull);
        if (!vis) s[gi][nt][e] = -INFINITY;
      }
    }
  }
  // online softmax (log2 units; the queries carry log2(e) / sqrt(d))
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int gi = 0; gi < 4; ++gi) {
    if (gi * KS + ks >= 4) break;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      mx0 = fmaxf(mx0, fmaxf(s[gi][nt][0], s[gi][nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[gi][nt][2], s[gi][nt][3]));
    }
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
  }
  const float mn0 = fmaxf(w.m0, mx0), mn1 = fmaxf(w.m1, mx1);
  const float al0 = w.m0 == -INFINITY ? 0.f : exp2f(w.m0 - mn0);
  const float al1 = w.m1 == -INFINITY ? 0.f : exp2f(w.m1 - mn1);
  w.m0 = mn0;
  w.m1 = mn1;
  float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
  for (int gi = 0; gi < 4; ++gi) {
    if (gi * KS + ks >= 4) break;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float mn = e < 2 ? mn0 : mn1;
        const float pv = mn == -INFINITY ? 0.f : exp2f(s[gi][nt][e] - mn);
        s[gi][nt][e] = pv;
        if (e < 2) ps0 += pv; else ps1 += pv;
      }
    }
  }
  w.l0 = w.l0 * al0 + ps0;
  w.l1 = w.l1 * al1 + ps1;
#pragma unroll
  for (int dn = 0; dn < 16; ++dn) {
    w.o[dn][0] *= al0;
    w.o[dn][1] *= al0;
    w.o[dn][2] *= al1;
    w.o[dn][3] *= al1;
  }
  // O += P V over this warp's key groups
#pragma unroll
  for (int gi = 0; gi < 4; ++gi) {
    if (gi * KS + ks >= 4) break;
    const int kg = ks + gi * KS;
    uint32_t ph[4], pl[4];
    split2(s[gi][0][0], s[gi][0][1], ph[0], pl[0]);
    split2(s[gi][0][2], s[gi][0][3], ph[1], pl[1]);
    split2(s[gi][1][0], s[gi][1][1], ph[2], pl[2]);
    split2(s[gi][1][2], s[gi][1][3], ph[3], pl[3]);
    const int mi = lane >> 3;
    const uint32_t roff = (kg * 16 + (mi & 1) * 8 + (lane & 7)) * TA_ROWB + (mi >> 1) * 16;
#pragma unroll
    for (int d2 = 0; d2 < 8; ++d2) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vhi + roff + d2 * 32, b0, b1, b2, b3);
      mma_bf16(w.o[2 * d2], ph, b0, b1);
      mma_bf16(w.o[2 * d2], pl, b0, b1);
      mma_bf16(w.o[2 * d2 + 1], ph, b2, b3);
      mma_bf16(w.o[2 * d2 + 1], pl, b2, b3);
      if (TREE) {
        ldsm_x4_t(vlo + roff + d2 * 32, b0, b1, b2, b3);
        mma_bf16(w.o[2 * d2], ph, b0, b1);
        mma_bf16(w.o[2 * d2 + 1], ph, b2, b3);
      }
    }
  }
}

__global__ void __launch_bounds__(ATT_THREADS, 1)
tree_attention_tc_kernel(const AttnArgs a) {
  extern __shared__ __align__(128) uint8_t ta_smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const int cs = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  // blockIdx.z = request * row groups + group: a request's rows may be split into groups
  // of rows_per_group (each its own cluster, each reading the whole prefix) so that no CTA
  // holds more than TA_MAX_QV query vectors
  const int G = a.row_groups > 1 ? a.row_groups : 1;
  const int kvh = blockIdx.y, b = blockIdx.z / G, grp = blockIdx.z - (blockIdx.z / G) * G;
  const int rpg = G > 1 ? a.rows_per_group : a.rows_per_req;
  const int rfirst = grp * rpg;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
  const int gq = a.Hq / a.Hkv;
  const int qv = max(0, min(rpg, a.rows_per_req - rfirst)) * gq;
  const int WM = (qv + 15) >> 4, SROW = WM * 16;
  const int KS = ta_key_splits(WM);
  const int mt = warp / KS, ks = warp - mt * KS;
  const bool active = mt < WM;
  uint8_t* ring = ta_smem;
  uint8_t* trees = ta_smem + TA_RING;
  float* mst = reinterpret_cast<float*>(trees + TA_TREE);   // [KS][SROW]
  float* lst = mst + 4 * TA_MAX_QV;
  const uint32_t ring_u = smem_u32(ring), tree_u = smem_u32(trees);

  // The prefix keys and values are inputs of the draft step that none of its kernels
  // write, so the ring's first stages are issued before the wait on the previous kernel;
  // the prefix length is clamped here the way the roots kernel clamps (and reports) it.
  const int nb = min(max(__ldg(a.cu_seqlens + b + 1) - __ldg(a.cu_seqlens + b), 0), a.max_prefix);
  const int npre = (nb + ATT_CHUNK - 1) / ATT_CHUNK;
  const int row0 = b * a.rows_per_req + rfirst;
  const size_t kv_ld = static_cast<size_t>(a.Hkv) * TA_HD;
  const size_t base = (static_cast<size_t>(__ldg(a.cu_seqlens + b)) * a.Hkv + kvh) * TA_HD;
  const uint16_t* kc = static_cast<const uint16_t*>(a.k_cache) + base;
  const uint16_t* vc = static_cast<const uint16_t*>(a.v_cache) + base;
  const int np = rank < npre ? (npre - 1 - rank) / cs + 1 : 0;   // prefix chunks rank, rank + cs, ...
  const bool has_tree = npre % cs == rank;

  auto issue = [&](int i) {
    if (i < np) {
      const int c = rank + i * cs;
      const int nk = min(ATT_CHUNK, nb - c * ATT_CHUNK);
      const uint32_t kt = ring_u + (i % TA_NST) * 2 * TA_TILE, vt = kt + TA_TILE;
      for (int idx = tid; idx < ATT_CHUNK * 16; idx += ATT_THREADS) {
        const int j = idx >> 4, p = idx & 15;
        const bool ok = j < nk;
        const size_t off = static_cast<size_t>(c * ATT_CHUNK + j) * kv_ld + p * 8;
        cp_async16(kt + j * TA_ROWB + p * 16, ok ? kc + off : kc, ok);
        cp_async16(vt + j * TA_ROWB + p * 16, ok ? vc + off : vc, ok);
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int i = 0; i < TA_NST; ++i) issue(i);
  pdl_wait();
  pdl_trigger();
  // one batch of loads in flight together: tree rows (if this CTA has the tree chunk),
  // this warp's queries and its rows' ancestor masks (all written by the previous kernels)
  constexpr int PER = ATT_CHUNK * (TA_HD / 4) / ATT_THREADS;   // float4 of tree keys (and values) per thread
  float4 k4[PER], v4[PER];
  if (has_tree) {
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int idx = tid + u * ATT_THREADS;
      const int j = idx / (TA_HD / 4), d4 = idx - j * (TA_HD / 4);
      k4[u] = v4[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < a.tree_upto) {
        const size_t o = ((static_cast<size_t>(b) * a.tree_rows + j) * a.Hkv + kvh) * TA_HD + 4 * d4;
        k4[u] = __ldcg(reinterpret_cast<const float4*>(a.tk + o));
        v4[u] = __ldcg(reinterpret_cast<const float4*>(a.tv + o));
      }
    }
  }
  float2 qx[8][4];
  TaWarp w;
  w.mk0 = w.mk1 = 0ull;
  if (active) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
#pragma unroll
      for (int f = 0; f < 4; ++f) {
        const int v = mt * 16 + g + (f & 1) * 8;
        const int col = kk * 16 + 2 * t4 + (f >> 1) * 8;
        qx[kk][f] = make_float2(0.f, 0.f);
        if (v < qv) {
          const int i = v / gq, gh = v - i * gq;
          qx[kk][f] = __ldcg(reinterpret_cast<const float2*>(a.q + (static_cast<size_t>(row0 + i) * a.Hq + kvh * gq + gh) * TA_HD + col));
        }
      }
    const int v0 = mt * 16 + g, v1 = v0 + 8;
    if (v0 < qv) w.mk0 = __ldcg(a.row_mask + row0 + v0 / gq);
    if (v1 < qv) w.mk1 = __ldcg(a.row_mask + row0 + v1 / gq);
  }
  if (has_tree) {   // fp32 tree keys / values -> bf16 hi and lo tiles
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int idx = tid + u * ATT_THREADS;
      const int j = idx / (TA_HD / 4), d4 = idx - j * (TA_HD / 4);
      uint32_t h0, l0, h1, l1;
      const size_t so = static_cast<size_t>(j) * TA_ROWB + d4 * 8;
      split2(k4[u].x, k4[u].y, h0, l0);
      split2(k4[u].z, k4[u].w, h1, l1);
      *reinterpret_cast<uint2*>(trees + so) = make_uint2(h0, h1);
      *reinterpret_cast<uint2*>(trees + TA_TILE + so) = make_uint2(l0, l1);
      split2(v4[u].x, v4[u].y, h0, l0);
      split2(v4[u].z, v4[u].w, h1, l1);
      *reinterpret_cast<uint2*>(trees + 2 * TA_TILE + so) = make_uint2(h0, h1);
      *reinterpret_cast<uint2*>(trees + 3 * TA_TILE + so) = make_uint2(l0, l1);
    }
  }
  w.m0 = w.m1 = -INFINITY;
  w.l0 = w.l1 = 0.f;
#pragma unroll
  for (int dn = 0; dn < 16; ++dn)
#pragma unroll
    for (int e = 0; e < 4; ++e) w.o[dn][e] = 0.f;
  {
    const float qs = 1.4426950408889634f / sqrtf(static_cast<float>(TA_HD));
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
#pragma unroll
      for (int f = 0; f < 4; ++f) split2(qx[kk][f].x * qs, qx[kk][f].y * qs, w.qh[kk][f], w.ql[kk][f]);
  }
  for (int i = 0; i < np; ++i) {
    cp_async_wait<TA_NST - 1>();
    __syncthreads();
    if (active) {
      const int c = rank + i * cs;
      const uint32_t kt = ring_u + (i % TA_NST) * 2 * TA_TILE;
      ta_chunk<false>(w, kt, 0, kt + TA_TILE, 0, min(ATT_CHUNK, nb - c * ATT_CHUNK), ks, KS, lane);
    }
    __syncthreads();
    issue(i + TA_NST);
  }
  cp_async_wait<0>();
  __syncthreads();
  if (has_tree && active)
    ta_chunk<true>(w, tree_u, tree_u + TA_TILE, tree_u + 2 * TA_TILE, tree_u + 3 * TA_TILE, a.tree_upto, ks, KS, lane);
  __syncthreads();   // every warp is done with the ring: it now holds the states

  // publish the warp states: output [KS][SROW][hd], row max and row sum [KS][SROW]
  float* st = reinterpret_cast<float*>(ring);
  float* mcta = lst + 4 * TA_MAX_QV;   // [SROW] the CTA's merged state
  float* lcta = mcta + TA_MAX_QV;
  if (active) {
    float l0 = w.l0, l1 = w.l1;
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    const int v0 = mt * 16 + g;
    float* r0p = st + (static_cast<size_t>(ks) * SROW + v0) * TA_HD;
    float* r1p = r0p + 8 * TA_HD;
#pragma unroll
    for (int dn = 0; dn < 16; ++dn) {
      *reinterpret_cast<float2*>(r0p + dn * 8 + 2 * t4) = make_float2(w.o[dn][0], w.o[dn][1]);
      *reinterpret_cast<float2*>(r1p + dn * 8 + 2 * t4) = make_float2(w.o[dn][2], w.o[dn][3]);
    }
    if (t4 == 0) {
      mst[ks * SROW + v0] = w.m0;
      mst[ks * SROW + v0 + 8] = w.m1;
      lst[ks * SROW + v0] = l0;
      lst[ks * SROW + v0 + 8] = l1;
    }
  }
  __syncthreads();
  // merge the KS warp states of each query vector inside the CTA (into split 0)
  if (KS > 1) {
    for (int idx = tid; idx < SROW * (TA_HD / 4); idx += ATT_THREADS) {
      const int v = idx / (TA_HD / 4), d4 = idx - v * (TA_HD / 4);
      float M = -INFINITY;
      for (int k = 0; k < KS; ++k) M = fmaxf(M, mst[k * SROW + v]);
      float L = 0.f;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int k = 0; k < KS; ++k) {
        const float mk = mst[k * SROW + v];
        const float wk = mk == -INFINITY ? 0.f : exp2f(mk - M);
        L += wk * lst[k * SROW + v];
        const float4 x = *reinterpret_cast<const float4*>(st + (static_cast<size_t>(k) * SROW + v) * TA_HD + 4 * d4);
        o.x += wk * x.x;
        o.y += wk * x.y;
        o.z += wk * x.z;
        o.w += wk * x.w;
      }
      *reinterpret_cast<float4*>(st + static_cast<size_t>(v) * TA_HD + 4 * d4) = o;   // read by this thread only
      if (d4 == 0) {
        mcta[v] = M;
        lcta[v] = L;
      }
    }
  } else {
    for (int v = tid; v < SROW; v += ATT_THREADS) {
      mcta[v] = mst[v];
      lcta[v] = lst[v];
    }
  }
  cluster.sync();
  // merge the cluster's CTA states (rank order) and normalise
  const size_t ld = static_cast<size_t>(a.Hq) * TA_HD;
  for (int idx = rank * ATT_THREADS + tid; idx < qv * (TA_HD / 4); idx += cs * ATT_THREADS) {
    const int v = idx / (TA_HD / 4), d4 = idx - v * (TA_HD / 4);
    float mr[ATT_MAX_CLUSTER], lr[ATT_MAX_CLUSTER];
    float4 xr[ATT_MAX_CLUSTER];
#pragma unroll
    for (int r = 0; r < ATT_MAX_CLUSTER; ++r) {   // every remote load issued before any use
      mr[r] = -INFINITY;
      lr[r] = 0.f;
      xr[r] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < cs) {
        mr[r] = cluster.map_shared_rank(mcta, r)[v];
        lr[r] = cluster.map_shared_rank(lcta, r)[v];
        xr[r] = *reinterpret_cast<const float4*>(cluster.map_shared_rank(st, r) + static_cast<size_t>(v) * TA_HD + 4 * d4);
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < ATT_MAX_CLUSTER; ++r) M = fmaxf(M, mr[r]);
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < ATT_MAX_CLUSTER; ++r) {
      const float wr = mr[r] == -INFINITY ? 0.f : exp2f(mr[r] - M);
      L += wr * lr[r];
      o.x += wr * xr[r].x;
      o.y += wr * xr[r].y;
      o.z += wr * xr[r].z;
      o.w += wr * xr[r].w;
    }
    const float inv = 1.0f / L;
    o.x *= inv;
    o.y *= inv;
    o.z *= inv;
    o.w *= inv;
    const int i = v / gq, gh = v - i * gq;
    const size_t col = static_cast<size_t>(kvh * gq + gh) * TA_HD + 4 * d4;
    *reinterpret_cast<float4*>(a.out + static_cast<size_t>(row0 + i) * ld + col) = o;
    if (a.out_hl) {
      uint32_t h0, l0, h1, l1;
      split2(o.x, o.y, h0, l0);
      split2(o.z, o.w, h1, l1);
      *reinterpret_cast<uint2*>(a.out_hl + 2 * static_cast<size_t>(row0 + i) * ld + col) = make_uint2(h0, h1);
      *reinterpret_cast<uint2*>(a.out_hl + (2 * static_cast<size_t>(row0 + i) + 1) * ld + col) = make_uint2(l0, l1);
    }
  }
  cluster.sync();
}

static int rows_per_cta(const AttnArgs& a) {
  return a.row_groups > 1 ? std::min(a.rows_per_group, a.rows_per_req) : a.rows_per_req;
}

static bool use_tc(const AttnArgs& a) {
  return a.cache_bf16 && a.hd == TA_HD && rows_per_cta(a) * (a.Hq / a.Hkv) <= TA_MAX_QV;
}

int attn_rows_per_group(int Hq, int Hkv) { return TA_MAX_QV / (Hq / Hkv); }

static int g_att_cluster = 0;

cudaError_t attn_setup_attributes() {
  cudaError_t e = allow_max_smem(reinterpret_cast<const void*>(tree_attention_kernel));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(tree_attention_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(TA_SMEM));
  if (e != cudaSuccess) return e;
  if (!g_att_cluster) {
    // 16-CTA clusters when the device schedules them, else the portable 8
    g_att_cluster = 8;
    if (cudaFuncSetAttribute(tree_attention_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess &&
        cudaFuncSetAttribute(tree_attention_tc_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess)
      g_att_cluster = ATT_MAX_CLUSTER;
    cudaGetLastError();
  }
  return cudaSuccess;
}

// clusters of `cs` CTAs the device holds at once (cached per kernel, size and smem)
static int active_clusters(bool tc, int cs, size_t smem) {
  struct Entry { int dev, tc, cs; size_t smem; int n; };
  static Entry cache[128];
  static int used = 0;
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  int dev = 0;
  cudaGetDevice(&dev);
  for (int i = 0; i < used; ++i)
    if (cache[i].dev == dev && cache[i].tc == tc && cache[i].cs == cs && cache[i].smem == smem) return cache[i].n;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(ATT_THREADS, 1, 1);
  cfg.gridDim = dim3(cs, 1, 1);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  const cudaError_t e = tc ? cudaOccupancyMaxActiveClusters(&n, tree_attention_tc_kernel, &cfg)
                           : cudaOccupancyMaxActiveClusters(&n, tree_attention_kernel, &cfg);
  if (e != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  if (used < 128) cache[used++] = Entry{dev, tc ? 1 : 0, cs, smem, n};
  return n;
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t st, bool pdl) {
  const bool tc = use_tc(a);
  const int G = a.row_groups > 1 ? a.row_groups : 1;
  if (G > 1 && (!tc || static_cast<long long>(G) * a.rows_per_group < a.rows_per_req ||
                static_cast<long long>(G - 1) * a.rows_per_group >= a.rows_per_req))
    return cudaErrorInvalidValue;   // groups only on the tensor-core path, each with >= 1 row
  const int qv = rows_per_cta(a) * (a.Hq / a.Hkv);
  const size_t smem = tc ? TA_SMEM : attn_smem_bytes(qv, a.hd);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  cudaLaunchConfig_t cfg = {};
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cfg.stream = st;
  cfg.blockDim = dim3(ATT_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  // Cluster size: each CTA of a cluster of cs takes ceil(chunks / cs) chunks, and the
  // (request, kv head) clusters run in waves of as many as the device holds at once.
  // Estimated time ~ waves x (chunks per CTA + fixed cost of a CTA, ~4 chunks).
  const int total = a.Hkv * a.B * G;
  const int cmax = g_att_cluster ? g_att_cluster : 8;
  int best_cs = 0;
  long long best_cost = 0;
  for (int cs = 1; cs <= cmax; ++cs) {
    if (cs > a.max_splits) break;
    const int nca = active_clusters(tc, cs, smem);
    if (nca <= 0) continue;
    const long long waves = (total + nca - 1) / nca;
    const long long cost = waves * ((a.max_splits + cs - 1) / cs + 4);
    if (!best_cs || cost < best_cost || (cost == best_cost && cs > best_cs)) {
      best_cs = cs;
      best_cost = cost;
    }
  }
  // tuning override: EAGLE_ATTN_CLUSTER = a cluster size to use when the device holds such
  // clusters (sweeps of the launch shape); unset or 0 keeps the cost model's choice
  if (const char* ov = getenv("EAGLE_ATTN_CLUSTER")) {
    const int cs = atoi(ov);
    if (cs >= 1 && cs <= cmax && cs <= a.max_splits && active_clusters(tc, cs, smem) > 0) best_cs = cs;
  }
  if (!best_cs) return cudaErrorInvalidConfiguration;
  attr[1].val.clusterDim.x = best_cs;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3(best_cs, a.Hkv, a.B * G);
  if (tc) return cudaLaunchKernelEx(&cfg, tree_attention_tc_kernel, a);
  return cudaLaunchKernelEx(&cfg, tree_attention_kernel, a);
}

}  // namespace eagle
