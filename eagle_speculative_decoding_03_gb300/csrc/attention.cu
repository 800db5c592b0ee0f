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
#include <cstdio>
#include <cstdlib>
#include <cstring>
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

// ----------------------------------------------------------- shared helpers
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

// ============================================================ tensor-core path
// bf16 prefix cache, head size 128, at most 128 query vectors (rows x query heads of the KV
// group) per CTA.  The cluster decomposition and merge of the SIMT kernel over 128-key
// tiles (the tree rows: one tile, zero-padded past 64 rows); per tile
// the two products run on the 5th-generation tensor cores (tcgen05.mma) with every operand
// that the CTA produces itself held in tensor memory:
//   S [query x key]  = Q K^T   A = queries (TMEM, bf16 hi and lo parts), B = key tile (smem)
//   O [query x dim] += P V     A = probabilities (TMEM, hi and lo, written over S), B = value
//                              tile (smem, MN-major)
// so each product keeps ~16 significant bits of the fp32 operands (the bf16 cache is exact;
// tree-row keys and values, fp32, are split into hi and lo as well: three products).  Shared
// memory holds only the key / value ring, filled by TMA through a 3-D map over
// [token][kv head][dim] (a request's partial last tile is loaded shifted back to end on its
// last key, so no copy reads past the request; rows before its first new key are masked).
// S / P has two TMEM buffers, so one tile's QK^T overlaps the previous tile's softmax.
// (128 keys per tile: one QK^T instruction covers 128 keys, so a tile costs half the
// instructions per key of a 64-key tile and half the barrier round trips.)
// Warp roles: 0 TMA producer; 1 TMEM owner; 4 + q softmax for TMEM lane quadrant q (thread
// = query vector = TMEM lane), for the quadrants that hold query vectors; the MMA issuer on
// warp 3 (warp 1 when all four quadrants are in use); the other two of warps 1-3 convert
// the tree tile.  The running max is raised only when a
// tile exceeds it by more than 2^8 (the thread then rescales its row of O in TMEM), so
// probabilities stay below 2^8.
constexpr int UA_THREADS = 256;
constexpr int UA_HD = 128;
constexpr uint32_t UA_MISC = 1280;       // barriers, flags, merge m / l
constexpr float UA_RESCALE = 8.0f;       // log2 units
constexpr int UA_ST_LD = UA_HD + 4;      // row stride (floats) of the CTA's final state in shared memory
constexpr uint32_t UA_TMEM_COLS = 512;
// Per tile size CH (64 or 128 keys): a 64-dim half of a key or value tile is CH rows of
// 128 bytes (128-byte swizzle); a ring slot holds K (dims 0-63, 64-127) | V (same).
// TMEM columns: S / P buffers [0, CH), [CH, 2 CH); O [2 CH, 2 CH + 128); Q hi, Q lo: 64
// columns each after O (CH = 128 fills all 512).
__host__ __device__ constexpr uint32_t ua_kblk(int ch) { return static_cast<uint32_t>(ch) * 128u; }
__host__ __device__ constexpr uint32_t ua_slot(int ch) { return 4u * ua_kblk(ch); }
__host__ __device__ constexpr int ua_max_stages(int ch) { return ch == 64 ? 6 : 3; }
__host__ __device__ inline size_t ua_smem_bytes(int ch, int stages) {
  return static_cast<size_t>(stages) * ua_slot(ch) + UA_MISC + 1024;
}

// byte offset of 16-byte chunk c (0-7) of row r in a 128-byte-swizzled block of 128-byte rows
EAGLE_DEV uint32_t ua_sw(int r, int c) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// 8 floats -> 8 bf16 hi parts and 8 bf16 lo parts, packed
EAGLE_DEV void ua_split8(const float* x, uint4& hi, uint4& lo) {
  split2_packed(x[0], x[1], hi.x, lo.x);
  split2_packed(x[2], x[3], hi.y, lo.y);
  split2_packed(x[4], x[5], hi.z, lo.z);
  split2_packed(x[6], x[7], hi.w, lo.w);
}
EAGLE_DEV void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

template <int CH>
__global__ void __launch_bounds__(UA_THREADS, 1)
tree_attention_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                         const AttnArgs a, const int NS) {
  constexpr uint32_t UA_KBLK = ua_kblk(CH), UA_SLOT = ua_slot(CH);
  constexpr uint32_t UA_T_O = 2 * CH, UA_T_QHI = UA_T_O + 128, UA_T_QLO = UA_T_O + 192;
  constexpr int UA_PREFETCH = 256 / CH;   // tiles requested into L2 beyond the ring
  extern __shared__ uint8_t ua_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ua_raw) + 1023) & ~uintptr_t(1023));
  cg::cluster_group cluster = cg::this_cluster();
  const int cs = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  // blockIdx.z = (request order) * row groups + group (see the SIMT kernel)
  const int G = a.row_groups > 1 ? a.row_groups : 1;
  const int kvh = blockIdx.y, grp = blockIdx.z - (blockIdx.z / G) * G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t ring_u = smem_u32(sm);
  uint8_t* misc = sm + static_cast<uint32_t>(NS) * UA_SLOT;
  // With several requests the CTAs take them longest prefix first (then by index), so that
  // when the grid runs in waves the long requests start in the first and the short ones fill
  // the gaps: the o-th request in that order, ranked from the (input) prefix lengths.
  int b = blockIdx.z / G;
  if (a.B > 1) {
    int* s_req = reinterpret_cast<int*>(misc + 224);
    const int o = b;
    auto len = [&](int r) { return min(max(__ldg(a.cu_seqlens + r + 1) - __ldg(a.cu_seqlens + r), 0), a.max_prefix); };
    for (int r = tid; r < a.B; r += UA_THREADS) {
      const int lr = len(r);
      int rk = 0;
      for (int q = 0; q < a.B; ++q) {
        const int lq = len(q);
        rk += (lq > lr || (lq == lr && q < r)) ? 1 : 0;
      }
      if (rk == o) *s_req = r;
    }
    __syncthreads();
    b = *s_req;
  }
  const int rpg = G > 1 ? a.rows_per_group : a.rows_per_req;
  const int rfirst = grp * rpg;
  const int gq = a.Hq / a.Hkv;
  const int qv = max(0, min(rpg, a.rows_per_req - rfirst)) * gq;
  const int row0 = b * a.rows_per_req + rfirst;

  const uint32_t misc_u = smem_u32(misc);
  const uint32_t bar_kvf = misc_u, bar_kve = misc_u + 64, bar_sf = misc_u + 128, bar_pf = misc_u + 144,
                 bar_pe = misc_u + 160, bar_od = misc_u + 176, bar_tg = misc_u + 184, bar_tf = misc_u + 192,
                 bar_fin = misc_u + 200;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc + 208);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 212);
  int* tree_slot = reinterpret_cast<int*>(misc + 216);
  float* mcta = reinterpret_cast<float*>(misc + 256);   // [128] the CTA's final state per vector
  float* lcta = mcta + 128;
  float* st = reinterpret_cast<float*>(sm);             // [qv][UA_ST_LD] un-normalised output (ring, at the end)

  // this CTA's keys: prefix tiles rank, rank + cs, ... and (one CTA) the tree tile
  const int tok0 = __ldg(a.cu_seqlens + b);
  const int nb = min(max(__ldg(a.cu_seqlens + b + 1) - tok0, 0), a.max_prefix);
  const int npre = (nb + CH - 1) / CH;
  const int np = rank < npre ? (npre - 1 - rank) / cs + 1 : 0;
  const bool has_tree = npre % cs == rank;
  const int T = np + (has_tree ? 1 : 0);
  const long long wlim = a.wait_limit > 0 ? a.wait_limit : WAIT_LIMIT_CYCLES;
  // Softmax warps: one per TMEM lane quadrant that holds query vectors (warp 4 + q reads
  // quadrant q).  With three or fewer, the MMA issuer takes warp 3, whose SM sub-partition
  // then runs no softmax warp: the issue loop keeps its sub-partition's instruction cache
  // and issue slots to itself.
  const int nq = min(4, max(1, (qv + 31) / 32));
  const int mma_warp = nq <= 3 ? 3 : 1;

  if (tid == 0) {
    for (int s = 0; s < 8; ++s) {
      mbar_init(bar_kvf + 8 * s, 1);
      mbar_init(bar_kve + 8 * s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_sf + 8 * i, 1);
      mbar_init(bar_pf + 8 * i, nq);
      mbar_init(bar_pe + 8 * i, 1);
    }
    mbar_init(bar_od, 1);
    mbar_init(bar_tg, 1);
    mbar_init(bar_tf, 2);
    mbar_init(bar_fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), UA_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // first token of tile t (a partial tile is shifted back to end on the request's last key)
  auto tile_t0 = [&](int t) {
    const int c = rank + t * cs;
    return tok0 + c * CH - (CH - min(CH, nb - c * CH));
  };
  // tiles beyond the ring are also requested into L2, so a slot's refill comes from L2
  // (the maps' boxes are 64 tokens: two per 64-dim half)
  auto prefetch = [&](int t) {
    if (t >= np) return;
    const int t0 = tile_t0(t);
#pragma unroll
    for (int h = 0; h < CH; h += 64) {
      tma_prefetch_l2_3d(&tmk, 0, kvh, t0 + h);
      tma_prefetch_l2_3d(&tmk, 64, kvh, t0 + h);
      tma_prefetch_l2_3d(&tmv, 0, kvh, t0 + h);
      tma_prefetch_l2_3d(&tmv, 64, kvh, t0 + h);
    }
  };
  const uint64_t pol = a.kv_keep ? policy_evict_last() : policy_evict_first();
  auto issue = [&](int t) {
    const int slot = t % NS;
    const int t0 = tile_t0(t);
    const uint32_t dst = ring_u + slot * UA_SLOT, bar = bar_kvf + 8 * slot;
    mbar_arrive_expect_tx(bar, UA_SLOT);
    // 64 tokens of 128-byte rows per box: the second box continues the first's 8-row
    // swizzle groups, so each 64-dim half is one 128-row K-major block
#pragma unroll
    for (int h = 0; h < CH; h += 64) {
      const uint32_t o = static_cast<uint32_t>(h) * 128u;
      tma_load_3d(dst + o, &tmk, 0, kvh, t0 + h, bar, pol);
      tma_load_3d(dst + UA_KBLK + o, &tmk, 64, kvh, t0 + h, bar, pol);
      tma_load_3d(dst + 2 * UA_KBLK + o, &tmv, 0, kvh, t0 + h, bar, pol);
      tma_load_3d(dst + 3 * UA_KBLK + o, &tmv, 64, kvh, t0 + h, bar, pol);
    }
  };
  // The prefix cache is an input of the draft step that none of its kernels write: the
  // first ring slots are filled before the wait on the previous kernel.
  const int first = min(NS, np);
  if (warp == 0 && lane == 0 && np > 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
    for (int t = 0; t < first; ++t) issue(t);
    for (int t = first; t < first + UA_PREFETCH; ++t) prefetch(t);
  }
  pdl_wait();
  pdl_trigger();

  // queries (scaled by log2(e) / sqrt(hd)) -> bf16 hi / lo parts in TMEM, one lane per
  // query vector (lanes past qv hold zeros)
  if (warp >= 4 && warp - 4 < nq) {
    const int v = tid - 128;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const float qs = 1.4426950408889634f / sqrtf(static_cast<float>(UA_HD));
    const float* src = nullptr;
    if (v < qv) {
      const int i = v / gq, gh = v - i * gq;
      src = a.q + (static_cast<size_t>(row0 + i) * a.Hq + kvh * gq + gh) * UA_HD;
    }
#pragma unroll 1
    for (int c0 = 0; c0 < UA_HD; c0 += 64) {   // 64 dims = 32 packed columns per part
      uint32_t hi[32], lo[32];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (src) x = __ldcg(reinterpret_cast<const float4*>(src + c0 + 4 * e));
        split2_packed(x.x * qs, x.y * qs, hi[2 * e], lo[2 * e]);
        split2_packed(x.z * qs, x.w * qs, hi[2 * e + 1], lo[2 * e + 1]);
      }
      tmem_st32(tmem + lane_base + UA_T_QHI + c0 / 2, hi);
      tmem_st32(tmem + lane_base + UA_T_QLO + c0 / 2, lo);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  bool ok = true;
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      for (int t = first; t < np + (has_tree ? 2 : 0) && ok; ++t) {   // ring positions
        const int slot = t % NS;
        if (t >= NS) ok = mbar_wait_sleepy(bar_kve + 8 * slot, ((t / NS) & 1) ^ 1, a.err, abort_flag, wlim);
        if (!ok) break;
        if (t < np) {
          issue(t);
          prefetch(t + UA_PREFETCH);
        } else {
          tree_slot[t - np] = slot;   // the tree tile takes two free slots (keys | values)
        }
      }
      if (has_tree && ok) mbar_arrive(bar_tg);
      if (!ok) {   // let copies already issued land before the CTA releases its shared memory
        const long long t0 = clock64();
        while (clock64() - t0 < 4000000) {
        }
      }
    }
  } else if (warp == mma_warp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id1 = idesc_bf16_f32(128, CH);
      const uint32_t id2 = idesc_bf16_f32(128, UA_HD) | (1u << 16);   // B (values) MN-major
      const uint32_t tO = tmem + UA_T_O;
      // Step t issues QK^T of tile t (into S buffer t & 1) and P V of tile t - 1; the tree
      // tile (last) takes P V first, since its slots may wait for that product's release.
      // (One copy of each issue sequence: the issue loop stays small.)
      for (int t = 0; t <= T && ok; ++t) {
        const bool tree_step = t == np && t < T;
#pragma unroll 1
        for (int ph = 0; ph < 2 && ok; ++ph) {
          if ((ph == 0) != tree_step) {
            if (t == T) continue;
            // ---- S = Q K^T for tile t, once P V of tile t - 2 (same TMEM buffer) is done
            ok = tree_step ? mbar_wait(bar_tf, 0, a.err, abort_flag, wlim)
                           : mbar_wait(bar_kvf + 8 * (t % NS), (t / NS) & 1, a.err, abort_flag, wlim);
            ok = ok && mbar_wait(bar_pe + 8 * (t & 1), ((t >> 1) & 1) ^ 1, a.err, abort_flag, wlim);
            if (!ok) break;
            // (the tree tile's slots are known once the converters signalled)
            const uint32_t kb = tree_step ? ring_u + tree_slot[0] * UA_SLOT : ring_u + (t % NS) * UA_SLOT;
            tc_fence_after();
            const uint32_t d = tmem + (t & 1) * CH;
            // descriptors move only in their start-address field (16-byte units, no carry)
            const uint64_t dk = smem_desc_sw128(kb), dkl = dk + ((2 * UA_KBLK) >> 4);
#pragma unroll
            for (int j = 0; j < UA_HD / 16; ++j) {   // 16 dims: 8 packed Q columns, 32 bytes of K
              const uint32_t ko = ((j >> 2) * UA_KBLK + (j & 3) * 32) >> 4;
              tc_mma_bf16_ta(d, tmem + UA_T_QHI + 8 * j, dk + ko, id1, j > 0 ? 1u : 0u);
              tc_mma_bf16_ta(d, tmem + UA_T_QLO + 8 * j, dk + ko, id1, 1u);
              if (tree_step) tc_mma_bf16_ta(d, tmem + UA_T_QHI + 8 * j, dkl + ko, id1, 1u);
            }
            tc_commit(bar_sf + 8 * (t & 1));
          } else {
            if (t == 0) continue;
            // ---- O += P V for tile u = t - 1 (P hi / lo in S buffer u & 1)
            const int u = t - 1;
            const bool tree = u == np;
            ok = mbar_wait(bar_pf + 8 * (u & 1), (u >> 1) & 1, a.err, abort_flag, wlim);
            if (!ok) break;
            tc_fence_after();
            const uint32_t vb = tree ? ring_u + tree_slot[1] * UA_SLOT : ring_u + (u % NS) * UA_SLOT + 2 * UA_KBLK;
            const uint64_t dv = smem_desc_sw128_mn(vb, UA_KBLK, 1024), dvl = dv + ((2 * UA_KBLK) >> 4);
            const uint32_t tp = tmem + (u & 1) * CH;
#pragma unroll
            for (int j = 0; j < CH / 16; ++j) {   // 16 keys: 8 packed P columns, two 8-key V groups
              // P of keys [32 c, 32 c + 32) sits at columns 32 c (hi, 16) and 32 c + 16 (lo, 16)
              const uint32_t pa = tp + 32 * (j >> 1) + 8 * (j & 1);
              tc_mma_bf16_ta(tO, pa, dv + j * 128, id2, (u > 0 || j > 0) ? 1u : 0u);
              tc_mma_bf16_ta(tO, pa + 16, dv + j * 128, id2, 1u);
              if (tree) tc_mma_bf16_ta(tO, pa, dvl + j * 128, id2, 1u);
            }
            tc_commit(bar_pe + 8 * (u & 1));
            if (!tree) tc_commit(bar_kve + 8 * (u % NS));
            tc_commit(bar_od);
          }
        }
      }
      if (!ok) {   // let MMAs already issued finish before TMEM is released
        const long long t0 = clock64();
        while (clock64() - t0 < 4000000) {
        }
      }
      tc_commit(bar_fin);
    }
  } else if (warp < 4) {
    // ------------------------------ tree tile: fp32 keys / values -> bf16 hi / lo tiles
    // (the two of warps 1-3 that do not issue MMAs)
    if (has_tree) {
      const int ct = (warp - 1 - (warp > mma_warp ? 1 : 0)) * 32 + lane;
      if (mbar_wait_sleepy(bar_tg, 0, a.err, abort_flag, wlim)) {
        const uint32_t ks = ring_u + tree_slot[0] * UA_SLOT, vs = ring_u + tree_slot[1] * UA_SLOT;
        for (int it = ct; it < CH * 16; it += 64) {   // rows past the tree rows: zeros
          const int j = it >> 4, c16 = it & 15;
          float k8[8], v8[8];
          if (j < a.tree_upto) {
            const size_t o = ((static_cast<size_t>(b) * a.tree_rows + j) * a.Hkv + kvh) * UA_HD + c16 * 8;
            const float4 k0 = __ldcg(reinterpret_cast<const float4*>(a.tk + o));
            const float4 k1 = __ldcg(reinterpret_cast<const float4*>(a.tk + o + 4));
            const float4 v0 = __ldcg(reinterpret_cast<const float4*>(a.tv + o));
            const float4 v1 = __ldcg(reinterpret_cast<const float4*>(a.tv + o + 4));
            k8[0] = k0.x; k8[1] = k0.y; k8[2] = k0.z; k8[3] = k0.w; k8[4] = k1.x; k8[5] = k1.y; k8[6] = k1.z; k8[7] = k1.w;
            v8[0] = v0.x; v8[1] = v0.y; v8[2] = v0.z; v8[3] = v0.w; v8[4] = v1.x; v8[5] = v1.y; v8[6] = v1.z; v8[7] = v1.w;
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) k8[e] = v8[e] = 0.f;
          }
          uint4 kh, kl, vh, vl;
          ua_split8(k8, kh, kl);
          ua_split8(v8, vh, vl);
          const uint32_t off = (c16 >> 3) * UA_KBLK + ua_sw(j, c16 & 7);
          st_shared_v4(ks + off, kh);
          st_shared_v4(ks + 2 * UA_KBLK + off, kl);
          st_shared_v4(vs + off, vh);
          st_shared_v4(vs + 2 * UA_KBLK + off, vl);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tf);
    }
  } else if (warp - 4 < nq) {
    // ------------------------------------------------------------ softmax
    const int v = tid - 128;                       // query vector = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const bool live = v < qv;
    const unsigned long long mrow = (live && has_tree) ? __ldcg(a.row_mask + row0 + v / gq) : 0ull;
    // tree keys a vector sees: rows that exist so far and are ancestors of (or are) its row
    const unsigned long long vis_tree =
        mrow & (a.tree_upto >= 64 ? ~0ull : ((1ull << max(a.tree_upto, 0)) - 1ull));
    float m_run = -INFINITY, l_run = 0.f;
    const uint32_t tO = tmem + lane_base + UA_T_O;
    for (int t = 0; t < T; ++t) {
      const bool tree = t == np;
      ok = ok && mbar_wait_sleepy(bar_sf + 8 * (t & 1), (t >> 1) & 1, a.err, abort_flag, wlim);
      tc_fence_after();
      const uint32_t ts = tmem + lane_base + (t & 1) * CH;
      float s[CH];
#pragma unroll
      for (int c = 0; c < CH; c += 32) tmem_ld32(ts + c, s + c);
      tmem_wait_ld();
      // visible keys of the tile as 64-bit masks (two for 128 keys): prefix rows [lead, CH)
      // (a shifted partial tile starts late); the tree tile: rows that exist and are
      // ancestors of (or are) the vector's row, all in the first 64
      unsigned long long vis0 = vis_tree, vis1 = CH > 64 ? 0ull : ~0ull;
      if (!tree) {
        const int lead = CH - min(CH, nb - (rank + t * cs) * CH);
        vis0 = lead >= 64 ? 0ull : (~0ull << lead);
        vis1 = (CH == 64 || lead <= 64) ? ~0ull : (~0ull << (lead - 64));
      }
      const bool work = live && ok;
      if (work && (vis0 & vis1) != ~0ull) {
#pragma unroll
        for (int r = 0; r < 64; ++r) s[r] = ((vis0 >> r) & 1ull) ? s[r] : -INFINITY;
        if constexpr (CH > 64) {
#pragma unroll
          for (int r = 0; r < 64; ++r) s[64 + r] = ((vis1 >> r) & 1ull) ? s[64 + r] : -INFINITY;
        }
      }
      float mt = -INFINITY;
      if (work) {
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = s[e];
#pragma unroll
        for (int r = 8; r < CH; ++r) m8[r & 7] = fmaxf(m8[r & 7], s[r]);
        mt = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      }
      float f = 1.f;
      bool resc = false;
      if (mt != -INFINITY) {
        if (m_run == -INFINITY) {
          m_run = mt;
        } else if (mt > m_run + UA_RESCALE) {
          f = fast_exp2(m_run - mt);
          m_run = mt;
          resc = true;
        }
      }
      if (__any_sync(0xffffffffu, resc)) {
        // this warp's rows whose max rose: scale them in O once every earlier P V is done
        ok = ok && mbar_wait_sleepy(bar_od, (t - 1) & 1, a.err, abort_flag, wlim);
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < UA_HD; c0 += 32) {
          float x[32];
          tmem_ld32(tO + c0, x);
          tmem_wait_ld();
          uint32_t y[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) y[e] = __float_as_uint(x[e] * f);
          tmem_st32(tO + c0, y);
        }
        tmem_wait_st();
      }
      l_run *= f;
      // probabilities 2^(s - m) (a masked key gives 2^-inf = 0); rows without a key so far
      // (and padding rows) give zeros.  P (hi, lo) is written over this tile's S: keys
      // [32 c, 32 c + 32) as 16 packed hi columns at 32 c and 16 lo columns at 32 c + 16
      // (each group's S is in registers before its columns are overwritten).
      const bool pw = work && m_run != -INFINITY;
      float p8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) p8[e] = 0.f;
#pragma unroll
      for (int c = 0; c < CH; c += 32) {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float x0 = 0.f, x1 = 0.f;
          if (pw) {
            x0 = fast_exp2(s[c + 2 * e] - m_run);
            x1 = fast_exp2(s[c + 2 * e + 1] - m_run);
            p8[(2 * e) & 7] += x0;
            p8[(2 * e + 1) & 7] += x1;
          }
          split2_packed(x0, x1, pk[e], pk[16 + e]);
        }
        tmem_st32(ts + c, pk);
      }
      l_run += ((p8[0] + p8[1]) + (p8[2] + p8[3])) + ((p8[4] + p8[5]) + (p8[6] + p8[7]));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pf + 8 * (t & 1));
    }
    // the CTA's state: row v of O -> st[v][.], its m and l
    ok = mbar_wait_sleepy(bar_fin, 0, a.err, abort_flag, wlim) && ok;
    tc_fence_after();
    if (T > 0) {
#pragma unroll 1
      for (int c0 = 0; c0 < UA_HD; c0 += 32) {
        float x[32];
        tmem_ld32(tO + c0, x);
        tmem_wait_ld();
        if (live) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(st + static_cast<size_t>(v) * UA_ST_LD + c0 + e) =
                make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
        }
      }
    }
    mcta[v] = (live && T > 0 && ok) ? m_run : -INFINITY;
    lcta[v] = l_run;
  }
  tc_fence_before();
  __syncthreads();
  cluster.sync();
  // merge the cluster's CTA states (rank order) and normalise
  const size_t ld = static_cast<size_t>(a.Hq) * UA_HD;
  for (int idx = rank * UA_THREADS + tid; idx < qv * (UA_HD / 4); idx += cs * UA_THREADS) {
    const int v = idx / (UA_HD / 4), d4 = idx - v * (UA_HD / 4);
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
        xr[r] = *reinterpret_cast<const float4*>(cluster.map_shared_rank(st, r) + static_cast<size_t>(v) * UA_ST_LD + 4 * d4);
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < ATT_MAX_CLUSTER; ++r) M = fmaxf(M, mr[r]);
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < ATT_MAX_CLUSTER; ++r) {
      if (mr[r] == -INFINITY) continue;   // a CTA that saw no key of this vector
      const float wr = exp2f(mr[r] - M);
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
    const size_t col = static_cast<size_t>(kvh * gq + gh) * UA_HD + 4 * d4;
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
  if (warp == 1) tmem_dealloc(tmem, UA_TMEM_COLS);
}

static int rows_per_cta(const AttnArgs& a) {
  return a.row_groups > 1 ? std::min(a.rows_per_group, a.rows_per_req) : a.rows_per_req;
}

constexpr int UA_MAX_QV = 128;
static bool use_tc(const AttnArgs& a) {
  return a.cache_bf16 && a.hd == UA_HD && rows_per_cta(a) * (a.Hq / a.Hkv) <= UA_MAX_QV;
}

int attn_rows_per_group(int Hq, int Hkv) { return UA_MAX_QV / (Hq / Hkv); }

static int g_att_cluster = 0;
static size_t g_ua_smem_cap = 0;

cudaError_t attn_setup_attributes() {
  cudaError_t e = allow_max_smem(reinterpret_cast<const void*>(tree_attention_kernel));
  if (e != cudaSuccess) return e;
  e = allow_max_smem(reinterpret_cast<const void*>(tree_attention_tc_kernel<64>), &g_ua_smem_cap);
  if (e != cudaSuccess) return e;
  e = allow_max_smem(reinterpret_cast<const void*>(tree_attention_tc_kernel<128>));
  if (e != cudaSuccess) return e;
  if (!g_att_cluster) {
    // 16-CTA clusters when the device schedules them, else the portable 8
    g_att_cluster = 8;
    if (cudaFuncSetAttribute(tree_attention_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess &&
        cudaFuncSetAttribute(tree_attention_tc_kernel<64>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess &&
        cudaFuncSetAttribute(tree_attention_tc_kernel<128>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess)
      g_att_cluster = ATT_MAX_CLUSTER;
    cudaGetLastError();
  }
  return cudaSuccess;
}

// clusters of `cs` CTAs the device holds at once (cached per kernel, size and smem);
// tc = 0: the SIMT kernel, else the tensor-core kernel of tc-key tiles
static int active_clusters(int tc, int cs, size_t smem) {
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
  const cudaError_t e = tc == 128  ? cudaOccupancyMaxActiveClusters(&n, tree_attention_tc_kernel<128>, &cfg)
                       : tc == 64 ? cudaOccupancyMaxActiveClusters(&n, tree_attention_tc_kernel<64>, &cfg)
                                  : cudaOccupancyMaxActiveClusters(&n, tree_attention_kernel, &cfg);
  if (e != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  if (used < 128) cache[used++] = Entry{dev, tc, cs, smem, n};
  return n;
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t st, bool pdl) {
  const bool tc = use_tc(a);
  const int G = a.row_groups > 1 ? a.row_groups : 1;
  if (G > 1 && (!tc || static_cast<long long>(G) * a.rows_per_group < a.rows_per_req ||
                static_cast<long long>(G - 1) * a.rows_per_group >= a.rows_per_req))
    return cudaErrorInvalidValue;   // groups only on the tensor-core path, each with >= 1 row
  const int qv = rows_per_cta(a) * (a.Hq / a.Hkv);
  // Cluster size: each CTA of a cluster of cs takes ceil(tiles / cs) tiles, and the
  // (request, kv head) clusters run in waves of as many as the device holds at once.
  // Estimated time ~ waves x (tiles per CTA + fixed cost of a CTA, ~4 tiles).  max_splits
  // counts 64-key tiles, the tree tile included.
  auto plan = [&](int kind, int tiles, size_t smem, long long& cost) {
    const int total = a.Hkv * a.B * G;
    const int cmax = g_att_cluster ? g_att_cluster : 8;
    int best = 0;
    for (int cs = 1; cs <= cmax && cs <= tiles; ++cs) {
      const int nca = active_clusters(kind, cs, smem);
      if (nca <= 0) continue;
      const long long waves = (total + nca - 1) / nca;
      const long long c = waves * ((tiles + cs - 1) / cs + 4);
      if (!best || c < cost || (c == cost && cs > best)) {
        best = cs;
        cost = c;
      }
    }
    // tuning override: EAGLE_ATTN_CLUSTER = a cluster size to use when the device holds such
    // clusters (sweeps of the launch shape); unset or 0 keeps the cost model's choice
    if (const char* ov = getenv("EAGLE_ATTN_CLUSTER")) {
      const int cs = atoi(ov);
      if (cs >= 1 && cs <= cmax && cs <= tiles && active_clusters(kind, cs, smem) > 0) best = cs;
    }
    return best;
  };
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  cudaLaunchConfig_t cfg = {};
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cfg.stream = st;
  cfg.blockDim = dim3(ATT_THREADS, 1, 1);
  int best_cs = 0, ch = 0, stages = 0;
  long long cost = 0;
  if (tc) {
    // Tensor-core kernel over 64-key tiles, as many ring slots as fit but no more than a
    // CTA's tiles need (at least four: the final per-vector state, qv x 132 floats, is
    // parked in the ring); with 8 or more tiles per CTA, 128-key tiles instead (half the
    // instructions and barrier round trips per key; three 64 KB slots).
    int st64 = ua_max_stages(64);
    while (st64 > 4 && ua_smem_bytes(64, st64) > g_ua_smem_cap) --st64;
    if (ua_smem_bytes(64, st64) > g_ua_smem_cap) return cudaErrorInvalidConfiguration;
    best_cs = plan(64, a.max_splits, ua_smem_bytes(64, st64), cost);
    if (!best_cs) return cudaErrorInvalidConfiguration;
    const int per_cta = (a.max_splits + best_cs - 1) / best_cs;   // tiles, the tree tile's two slots included
    ch = 64;
    stages = std::max(4, std::min(st64, per_cta + 1));
    const int st128 = ua_max_stages(128);
    // tuning / test override: EAGLE_ATTN_TILE = 64 or 128 keys per tile; unset keeps the rule
    int want = per_cta >= 8 ? 128 : 64;
    if (const char* ov = getenv("EAGLE_ATTN_TILE")) {
      const int v = atoi(ov);
      if (v == 64 || v == 128) want = v;
    }
    if (want == 128 && ua_smem_bytes(128, st128) <= g_ua_smem_cap) {
      long long c128 = 0;
      const int cs128 = plan(128, a.max_splits / 2 + 1, ua_smem_bytes(128, st128), c128);
      if (cs128) {
        best_cs = cs128;
        ch = 128;
        stages = st128;
      }
    }
    cfg.dynamicSmemBytes = ua_smem_bytes(ch, stages);
  } else {
    const size_t smem = attn_smem_bytes(qv, a.hd);
    best_cs = plan(0, a.max_splits, smem, cost);
    if (!best_cs) return cudaErrorInvalidConfiguration;
    cfg.dynamicSmemBytes = smem;
  }
  attr[1].val.clusterDim.x = best_cs;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3(best_cs, a.Hkv, a.B * G);
  if (tc) {
    // key / value maps over every token the requests may hold (lengths are clamped to
    // max_prefix, and no tile reads past its request's last key)
    CUtensorMap tmk, tmv;
    memset(&tmk, 0, sizeof(tmk));
    memset(&tmv, 0, sizeof(tmv));
    const long long tokens = static_cast<long long>(a.B) * a.max_prefix;
    if (tokens > 0 && (!make_kv_map(&tmk, a.k_cache, tokens, a.Hkv) || !make_kv_map(&tmv, a.v_cache, tokens, a.Hkv)))
      return cudaErrorInvalidValue;
    if (ch == 128) return cudaLaunchKernelEx(&cfg, tree_attention_tc_kernel<128>, tmk, tmv, a, stages);
    return cudaLaunchKernelEx(&cfg, tree_attention_tc_kernel<64>, tmk, tmv, a, stages);
  }
  return cudaLaunchKernelEx(&cfg, tree_attention_kernel, a);
}

}  // namespace eagle
