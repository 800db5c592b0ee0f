// Tree-masked grouped-query decode attention of one draft depth.
//
// Every row of the depth (a frontier node) attends to its request's whole verified
// prefix (post-RoPE KV cache, read once per KV head) and to the tree rows that are its
// ancestors or itself (ancestor bit mask; "Tree attention in one verification pass",
// aicassindra.com tm_eagle_deep).  All query heads of a KV group and all rows of the
// request share one pass over the prefix keys.
//
// Grid (split, kv head, request): split s < ceil(n_b / 64) covers prefix keys
// [64 s, 64 s + 64); split ceil(n_b / 64) covers the tree rows; larger splits exit.  Each
// CTA writes its local softmax state (max, sum, unnormalised output) per query vector;
// the last CTA of a (request, kv head) merges them in split order.
#include "common.cuh"
#include "internal.h"

#include <cooperative_groups.h>
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

static int g_att_cluster = 0;

cudaError_t attn_setup_attributes() {
  cudaError_t e = allow_max_smem(reinterpret_cast<const void*>(tree_attention_kernel));
  if (e != cudaSuccess) return e;
  if (!g_att_cluster) {
    // 16-CTA clusters when the device schedules them, else the portable 8
    g_att_cluster = 8;
    if (cudaFuncSetAttribute(tree_attention_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
        cudaSuccess)
      g_att_cluster = ATT_MAX_CLUSTER;
    cudaGetLastError();
  }
  return cudaSuccess;
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t st, bool pdl) {
  const int qv = a.rows_per_req * (a.Hq / a.Hkv);
  const size_t smem = attn_smem_bytes(qv, a.hd);
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
  // the largest cluster size (<= the chunks of the longest request) that can be scheduled
  int cs = g_att_cluster ? g_att_cluster : 8;
  const int max_chunks = a.max_splits;
  while (cs > 1 && cs / 2 >= max_chunks) cs /= 2;
  for (; cs >= 1; cs /= 2) {
    attr[1].val.clusterDim.x = cs;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.gridDim = dim3(cs, a.Hkv, a.B);
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, tree_attention_kernel, &cfg) == cudaSuccess && nclusters > 0) break;
    cudaGetLastError();
  }
  if (cs < 1) return cudaErrorInvalidConfiguration;
  return cudaLaunchKernelEx(&cfg, tree_attention_kernel, a);
}

}  // namespace eagle
