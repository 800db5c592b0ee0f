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

namespace eagle {

constexpr int ATT_THREADS = 256;

struct AttSmem {
  float* qt;     // [hd][qvp]  queries, transposed
  float* kt;     // [hd][CH]   keys, transposed
  float* vs;     // [CH][hd]
  float* pt;     // [CH][qvp]  scores, then probabilities
  float* mrow;   // [qvp]
  float* lrow;   // [qvp]
};

size_t attn_smem_bytes(int qv, int hd) {
  const int qvp = (qv + 3) & ~3;
  return sizeof(float) * (static_cast<size_t>(hd) * qvp + 2 * static_cast<size_t>(hd) * ATT_CHUNK +
                          static_cast<size_t>(ATT_CHUNK) * qvp + 2 * qvp) + 16;
}

__global__ void __launch_bounds__(ATT_THREADS)
tree_attention_kernel(const AttnArgs a) {
  extern __shared__ float4 att_smem4[];
  float* sm = reinterpret_cast<float*>(att_smem4);
  const int sp = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hd = a.hd, gq = a.Hq / a.Hkv;
  const int qv = a.rows_per_req * gq, qvp = (qv + 3) & ~3;
  AttSmem S;
  S.qt = sm;
  S.kt = S.qt + hd * qvp;
  S.vs = S.kt + hd * ATT_CHUNK;
  S.pt = S.vs + ATT_CHUNK * hd;
  S.mrow = S.pt + ATT_CHUNK * qvp;
  S.lrow = S.mrow + qvp;

  pdl_wait();
  pdl_trigger();
  const int nb = __ldcg(a.n_eff + b);
  const int npre = (nb + ATT_CHUNK - 1) / ATT_CHUNK;
  const int nsplit = npre + 1;
  if (sp >= nsplit) return;
  const bool tree = sp == npre;
  const int nkeys = tree ? a.tree_upto : min(ATT_CHUNK, nb - sp * ATT_CHUNK);
  const int row0 = b * a.rows_per_req;
  const float scale = 1.0f / sqrtf(static_cast<float>(hd));

  // ---- stage queries (transposed, pre-scaled), keys (transposed) and values
  for (int idx = tid; idx < qvp * hd; idx += ATT_THREADS) {
    const int v = idx / hd, d = idx - v * hd;
    float x = 0.f;
    if (v < qv) {
      const int i = v / gq, gh = v - i * gq;
      x = __ldcg(a.q + (static_cast<size_t>(row0 + i) * a.Hq + kvh * gq + gh) * hd + d) * scale;
    }
    S.qt[d * qvp + v] = x;
  }
  for (int idx = tid; idx < ATT_CHUNK * hd; idx += ATT_THREADS) {
    const int j = idx / hd, d = idx - j * hd;
    float kx = 0.f, vx = 0.f;
    if (j < nkeys) {
      if (tree) {
        const size_t o = ((static_cast<size_t>(b) * a.tree_rows + j) * a.Hkv + kvh) * hd + d;
        kx = __ldcg(a.tk + o);
        vx = __ldcg(a.tv + o);
      } else {
        const size_t o = ((static_cast<size_t>(__ldg(a.cu_seqlens + b)) + sp * ATT_CHUNK + j) * a.Hkv + kvh) * hd + d;
        if (a.cache_bf16) {
          kx = bf16_to_f32(__ldg(static_cast<const uint16_t*>(a.k_cache) + o));
          vx = bf16_to_f32(__ldg(static_cast<const uint16_t*>(a.v_cache) + o));
        } else {
          kx = __ldg(static_cast<const float*>(a.k_cache) + o);
          vx = __ldg(static_cast<const float*>(a.v_cache) + o);
        }
      }
    }
    S.kt[d * ATT_CHUNK + j] = kx;
    S.vs[j * hd + d] = vx;
  }
  __syncthreads();

  // ---- scores: 4 query vectors x 4 keys per thread block
  const int nvb = qvp / 4;
  for (int blk = tid; blk < nvb * (ATT_CHUNK / 4); blk += ATT_THREADS) {
    const int vb = blk / (ATT_CHUNK / 4), jb = blk - vb * (ATT_CHUNK / 4);
    float acc[4][4] = {};
    for (int d = 0; d < hd; ++d) {
      const float4 qq = *reinterpret_cast<const float4*>(S.qt + d * qvp + 4 * vb);
      const float4 kk = *reinterpret_cast<const float4*>(S.kt + d * ATT_CHUNK + 4 * jb);
      const float qa[4] = {qq.x, qq.y, qq.z, qq.w}, ka[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] += qa[x] * ka[y];
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
        S.pt[j * qvp + v] = vis ? acc[x][y] : -INFINITY;
      }
    }
  }
  __syncthreads();

  // ---- local softmax state per query vector
  for (int v = warp; v < qv; v += ATT_THREADS / 32) {
    const float s0 = S.pt[lane * qvp + v], s1 = S.pt[(lane + 32) * qvp + v];
    const float mx = warp_max(fmaxf(s0, s1));
    float p0 = 0.f, p1 = 0.f;
    if (mx != -INFINITY) {
      p0 = expf(s0 - mx);
      p1 = expf(s1 - mx);
    }
    S.pt[lane * qvp + v] = p0;
    S.pt[(lane + 32) * qvp + v] = p1;
    const float l = warp_sum(p0 + p1);
    if (lane == 0) {
      S.mrow[v] = mx;
      S.lrow[v] = l;
    }
  }
  __syncthreads();

  // ---- unnormalised output: 4 query vectors x 4 dims per thread block
  const size_t pstride = static_cast<size_t>(hd) + 2;
  const size_t qv_cap = static_cast<size_t>(qv);
  float* part = a.part + ((static_cast<size_t>(b) * a.Hkv + kvh) * a.max_splits + sp) * qv_cap * pstride;
  for (int blk = tid; blk < nvb * (hd / 4); blk += ATT_THREADS) {
    const int vb = blk / (hd / 4), db = blk - vb * (hd / 4);
    float acc[4][4] = {};
    for (int j = 0; j < nkeys; ++j) {
      const float4 pp = *reinterpret_cast<const float4*>(S.pt + j * qvp + 4 * vb);
      const float4 vv = *reinterpret_cast<const float4*>(S.vs + j * hd + 4 * db);
      const float pa[4] = {pp.x, pp.y, pp.z, pp.w}, va[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] += pa[x] * va[y];
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int v = 4 * vb + x;
      if (v >= qv) continue;
#pragma unroll
      for (int y = 0; y < 4; ++y) part[v * pstride + 2 + 4 * db + y] = acc[x][y];
    }
  }
  for (int v = tid; v < qv; v += ATT_THREADS) {
    part[v * pstride] = S.mrow[v];
    part[v * pstride + 1] = S.lrow[v];
  }

  // ---- the last CTA of (request, kv head) merges the splits in order
  __threadfence();
  __syncthreads();
  __shared__ int last;
  if (tid == 0) {
    const int old = atomicAdd(a.counters + b * a.Hkv + kvh, 1);
    last = old == nsplit - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (tid == 0) a.counters[b * a.Hkv + kvh] = 0;
  const float* base = a.part + (static_cast<size_t>(b) * a.Hkv + kvh) * a.max_splits * qv_cap * pstride;
  for (int idx = tid; idx < qv * hd; idx += ATT_THREADS) {
    const int v = idx / hd, d = idx - v * hd;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, __ldcg(base + (s * qv_cap + v) * pstride));
    float L = 0.f, O = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float* ps = base + (s * qv_cap + v) * pstride;
      const float ms = __ldcg(ps);
      const float w = ms == -INFINITY ? 0.f : expf(ms - M);
      L += w * __ldcg(ps + 1);
      O += w * __ldcg(ps + 2 + d);
    }
    const int i = v / gq, gh = v - i * gq;
    const float val = O / L;
    a.out[(static_cast<size_t>(row0 + i) * a.Hq + kvh * gq + gh) * hd + d] = val;
    if (a.out_hl) {   // bf16 hi / lo rows: the O projection's operand copy
      uint16_t hi, lo;
      split_hilo(val, hi, lo);
      const size_t ld = static_cast<size_t>(a.Hq) * hd, col = static_cast<size_t>(kvh * gq + gh) * hd + d;
      a.out_hl[2 * static_cast<size_t>(row0 + i) * ld + col] = hi;
      a.out_hl[(2 * static_cast<size_t>(row0 + i) + 1) * ld + col] = lo;
    }
  }
}

cudaError_t attn_setup_attributes() {
  return allow_max_smem(reinterpret_cast<const void*>(tree_attention_kernel));
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t st, bool pdl) {
  const int qv = a.rows_per_req * (a.Hq / a.Hkv);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.stream = st;
  cfg.gridDim = dim3(a.max_splits, a.Hkv, a.B);
  cfg.blockDim = dim3(ATT_THREADS, 1, 1);
  cfg.dynamicSmemBytes = attn_smem_bytes(qv, a.hd);
  return cudaLaunchKernelEx(&cfg, tree_attention_kernel, a);
}

}  // namespace eagle
