// Multi-round speculative sampling over an emitted tree: which drafted tokens the target
// accepts, and the token it draws after the accepted path.  See include/eagle_draft.h.
//
// "Speculative Decoding Deep Dive III" (zackli.ai), EAGLE-1: verification is tree attention
// plus multi-round speculative sampling; "How speculative decoding works" (kaushalya.io):
// a drafted token is accepted with probability min(1, p/q), otherwise a token is drawn
// from the renormalised residual max(0, p - q).  Over a tree (the reading taken here):
// from the root, the children of the current slot are tried in slot order; child x is
// accepted when U * q(x) < p(x); on rejection the target becomes norm(max(0, p - q)) and x
// leaves the proposal (q restricted to the untried tokens, renormalised).  The walk moves
// to an accepted child; where no child is accepted (or at a leaf) one token is drawn from
// the current target by Gumbel-max and the walk ends.
//
// One CTA per request.  The residual after r rejections is elementwise in the row's p and
// q given r normalisers Z_i, the rejected tokens and their proposal mass, so every pass
// recomputes it per element from the two logit rows: no scratch memory.  All reductions
// run in a fixed order (deterministic).  Random numbers: Philox4x32-10 under the request's
// seed: the uniform that tries child slot c is word 0 of counter (c, 0, 0, 2); the noise of
// token t drawn at slot u after r rejections is word (t mod 128) / 32 of counter
// (32 (t / 128) + t mod 32, u, r, 1).
#include "../../include/eagle_draft.h"
#include "common.cuh"
#include "internal.h"

#include <cstdarg>
#include <cstdio>

using namespace eagle;

namespace {

constexpr int AC_THREADS = 1024;
constexpr int AC_WARPS = AC_THREADS / 32;
constexpr int AC_MAX_TRIES = 64;   // rejections at one slot (its children, <= 63)

struct SpecArgs {
  int B, S, V;
  const int* tokens;
  const int* parents;
  const float* logit_p;          // [B][S][V] target
  const float* logit_q;          // [B][S][V] draft
  const unsigned long long* seeds;
  int* accept_len;
  int* accept_slots;
  int* correction;
  unsigned* err;
};

struct AcShared {
  float red_a[AC_WARPS];
  float red_b[AC_WARPS];
  int red_i[AC_WARPS];
  float Z[AC_MAX_TRIES];         // normaliser of each rejection at the current slot
  float rem[AC_MAX_TRIES + 1];   // proposal mass removed before try i (rem[0] = 0)
  int xs[AC_MAX_TRIES];          // rejected tokens
  int tok[64], par[64];
  float bcast[4];
};

// block-wide max / sum, lanes then warps in index order: every thread gets the result
EAGLE_DEV float block_max(float v, AcShared& sh) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh.red_a[w] = v;
  __syncthreads();
  float m = sh.red_a[0];
  for (int i = 1; i < AC_WARPS; ++i) m = fmaxf(m, sh.red_a[i]);
  return m;
}
EAGLE_DEV float block_sum(float v, AcShared& sh) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sh.red_b[w] = v;
  __syncthreads();
  float s = 0.f;
  for (int i = 0; i < AC_WARPS; ++i) s += sh.red_b[i];
  return s;
}

// log-sum-exp of a row (max pass, then sum of exp)
EAGLE_DEV float row_lse(const float* x, int V, AcShared& sh) {
  float m = -INFINITY;
  for (int t = threadIdx.x; t < V; t += AC_THREADS) m = fmaxf(m, __ldg(x + t));
  m = block_max(m, sh);
  float s = 0.f;
  for (int t = threadIdx.x; t < V; t += AC_THREADS) s += expf(__ldg(x + t) - m);
  s = block_sum(s, sh);
  return m + logf(s);
}

// The current target after r rejections at this slot, at token t: the residual chain
// p_{i+1} = max(0, p_i - q_i) / Z_i with q_i = q restricted to the untried tokens,
// renormalised by 1 - rem[i].
EAGLE_DEV float residual_at(float p, float q, int t, int r, const AcShared& sh) {
  int tried = r;
  for (int j = 0; j < r; ++j)
    if (sh.xs[j] == t) { tried = j; break; }
  for (int i = 0; i < r; ++i) {
    const float qi = i <= tried ? q / (1.f - sh.rem[i]) : 0.f;   // t leaves the proposal after its own try
    if (sh.Z[i] > 0.f) p = fmaxf(p - qi, 0.f) / sh.Z[i];         // (Z = 0: p == q, the target stays)
  }
  return p;
}

__global__ void __launch_bounds__(AC_THREADS) spec_accept_kernel(const SpecArgs a) {
  __shared__ AcShared sh;
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, tid = threadIdx.x;
  const unsigned long long seed = __ldg(a.seeds + b);
  const uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
  if (tid < a.S) {
    const size_t o = static_cast<size_t>(b) * a.S + tid;
    int t = __ldg(a.tokens + o);
    if (t < 0 || t >= a.V) {
      atomicOr(a.err, DEVERR_TOKEN);
      t = 0;
    }
    int p = __ldg(a.parents + o);
    if (tid == 0) p = -1;
    else if (p < 0 || p >= tid) {
      atomicOr(a.err, DEVERR_TOKEN);
      p = -2;
    }
    sh.tok[tid] = t;
    sh.par[tid] = p;
    a.accept_slots[o] = -1;
  }
  __syncthreads();
  int u = 0, len = 0;
  for (;;) {
    const float* lp = a.logit_p + (static_cast<size_t>(b) * a.S + u) * a.V;
    const float* lq = a.logit_q + (static_cast<size_t>(b) * a.S + u) * a.V;
    const float lse_p = row_lse(lp, a.V, sh);
    const float lse_q = row_lse(lq, a.V, sh);
    int r = 0, nxt = -1;
    if (tid == 0) sh.rem[0] = 0.f;
    __syncthreads();
    for (int c = u + 1; c < a.S && nxt < 0; ++c) {
      if (sh.par[c] != u) continue;
      const int x = sh.tok[c];
      // this child's try: p_r(x) against q_r(x) (thread 0; broadcast)
      if (tid == 0) {
        const float px = residual_at(expf(__ldg(lp + x) - lse_p), expf(__ldg(lq + x) - lse_q), x, r, sh);
        bool again = false;   // (a repeated sibling token has left the proposal already)
        for (int j = 0; j < r; ++j) again |= sh.xs[j] == x;
        const float qx = again ? 0.f : expf(__ldg(lq + x) - lse_q) / (1.f - sh.rem[r]);
        const uint4 w = philox4x32_10(make_uint4(static_cast<uint32_t>(c), 0u, 0u, 2u), k0, k1);
        const float U = (static_cast<float>(w.x) + 0.5f) * 2.3283064365386963e-10f;
        sh.bcast[0] = (U * qx < px) ? 1.f : 0.f;
      }
      __syncthreads();
      if (sh.bcast[0] != 0.f) {
        nxt = c;
        break;
      }
      if (r >= AC_MAX_TRIES) {   // cannot happen with <= 64 slots; keeps the tables in bounds
        if (tid == 0) atomicOr(a.err, DEVERR_SELECT);
        break;
      }
      // rejected: normaliser of the next residual, sum over t of max(0, p_r(t) - q_r(t))
      float z = 0.f;
      for (int t = tid; t < a.V; t += AC_THREADS) {
        const float q = expf(__ldg(lq + t) - lse_q);
        const float pr = residual_at(expf(__ldg(lp + t) - lse_p), q, t, r, sh);
        int tried = r;
        for (int j = 0; j < r; ++j)
          if (sh.xs[j] == t) { tried = j; break; }
        const float qr = tried < r ? 0.f : q / (1.f - sh.rem[r]);
        z += fmaxf(pr - qr, 0.f);
      }
      z = block_sum(z, sh);
      if (tid == 0) {
        bool again = false;
        for (int j = 0; j < r; ++j) again |= sh.xs[j] == x;
        sh.Z[r] = z;
        sh.xs[r] = x;
        sh.rem[r + 1] = sh.rem[r] + (again ? 0.f : expf(__ldg(lq + x) - lse_q));
      }
      __syncthreads();
      ++r;
    }
    if (nxt >= 0) {
      if (tid == 0) a.accept_slots[static_cast<size_t>(b) * a.S + len] = nxt;
      ++len;
      u = nxt;
      continue;
    }
    // the token drawn at slot u: argmax over t of log p_r(t) + Gumbel noise (ties: lower id)
    float best = -INFINITY;
    int bid = INT_MAX;
    for (int t = tid; t < a.V; t += AC_THREADS) {
      const float pr = residual_at(expf(__ldg(lp + t) - lse_p), expf(__ldg(lq + t) - lse_q), t, r, sh);
      if (!(pr > 0.f)) continue;
      const uint4 w = philox4x32_10(make_uint4(32u * static_cast<uint32_t>(t >> 7) + (t & 31), static_cast<uint32_t>(u),
                                               static_cast<uint32_t>(r), 1u), k0, k1);
      const int j = (t & 127) >> 5;
      const float sc = logf(pr) + gumbel_of_word(j == 0 ? w.x : j == 1 ? w.y : j == 2 ? w.z : w.w);
      if (beats(sc, t, best, bid)) { best = sc; bid = t; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bid, o);
      if (beats(ov, oi, best, bid)) { best = ov; bid = oi; }
    }
    __syncthreads();
    if ((tid & 31) == 0) {
      sh.red_a[tid >> 5] = best;
      sh.red_i[tid >> 5] = bid;
    }
    __syncthreads();
    if (tid == 0) {
      float bv = sh.red_a[0];
      int bi = sh.red_i[0];
      for (int w = 1; w < AC_WARPS; ++w)
        if (beats(sh.red_a[w], sh.red_i[w], bv, bi)) { bv = sh.red_a[w]; bi = sh.red_i[w]; }
      if (bi == INT_MAX) {   // no token with positive probability (non-finite logits)
        atomicOr(a.err, DEVERR_SELECT);
        bi = 0;
      }
      a.accept_len[b] = len;
      a.correction[b] = bi;
    }
    return;
  }
}

}  // namespace

extern "C" eagle_status_t eagle_speculative_accept(int32_t B, int32_t S, int32_t vocab, const int32_t* tokens,
                                                   const int32_t* parents, const float* logits_target,
                                                   const float* logits_draft, const uint64_t* seeds,
                                                   int32_t* accept_len, int32_t* accept_slots, int32_t* correction,
                                                   uint32_t* err_word, void* stream) {
  if (!tokens || !parents || !logits_target || !logits_draft || !seeds || !accept_len || !accept_slots ||
      !correction || !err_word) {
    set_last_error("speculative_accept: null pointer argument");
    return EAGLE_ERR_INVALID_ARG;
  }
  if (B < 1 || S < 1 || S > 64 || vocab < 1) {
    set_last_error("speculative_accept: need B >= 1, 1 <= S <= 64, vocab >= 1");
    return EAGLE_ERR_INVALID_ARG;
  }
  SpecArgs a;
  a.B = B;
  a.S = S;
  a.V = vocab;
  a.tokens = tokens;
  a.parents = parents;
  a.logit_p = logits_target;
  a.logit_q = logits_draft;
  a.seeds = reinterpret_cast<const unsigned long long*>(seeds);
  a.accept_len = accept_len;
  a.accept_slots = accept_slots;
  a.correction = correction;
  a.err = err_word;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.gridDim = dim3(B);
  cfg.blockDim = dim3(AC_THREADS);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, spec_accept_kernel, a);
  if (e != cudaSuccess) {
    char buf[256];
    snprintf(buf, sizeof(buf), "speculative_accept: launch failed: %s", cudaGetErrorString(e));
    set_last_error(buf);
    return EAGLE_ERR_CUDA;
  }
  return EAGLE_OK;
}
