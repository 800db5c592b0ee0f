// C ABI of the verification side: the target's one pass over an emitted draft tree, and
// greedy acceptance of the deepest path it confirms.  See include/eagle_draft.h.
//
// "Tree attention in one verification pass" (aicassindra.com tm_eagle_deep): the tree's
// slots are laid out after the verified prefix and run through the target at once; each
// slot attends to the prefix and to its ancestors and itself only (the emitted mask), at
// position id prefix length + depth.  One pass gives, for every slot, the target's
// next-token distribution after exactly that slot's path.  Greedy acceptance ("How
// speculative decoding works", kaushalya.io; "Acceptance length under a tree",
// aicassindra.com): at temperature 0 a drafted token passes when it is the target's most
// likely token after its parent's path; the deepest passing path is kept and the target's
// most likely token after it is the correction token.
//
// The target here is one Llama-style decoder layer (the draft head's shapes, its own
// weights) between the frozen embedding and the frozen LM head, with a final RMSNorm:
//   embed rows    x = E[tok]; operand copy of RMSNorm-gained x; per-tile sums of squares;
//                 row metadata and the mask rows as ancestor bits
//   QKV GEMM      RMSNorm(x) -> q, the slots' K/V (rotary in the epilogue)
//   attention     prefix KV + the slots the mask row marks (query groups past 128 vectors)
//   O GEMM        y = x + W_o o
//   gate / up     RMSNorm(y) -> silu(g) * u
//   down GEMM     hidden = y + W_d s; operand copy of the final-norm-gained hidden
//   LM head       W_lm RMSNorm(hidden): per-tile log-sum-exp and the most likely token
//   merge         per slot: token, its log-probability, log-sum-exp
//   accept        one CTA per request walks the tree from the root (greedy)
#include "../../include/eagle_draft.h"
#include "common.cuh"
#include "internal.h"

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

using namespace eagle;

namespace {

eagle_status_t vfail(eagle_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  set_last_error(buf);
  return st;
}

#define VCU(call)                                                                          \
  do {                                                                                     \
    cudaError_t e_ = (call);                                                               \
    if (e_ != cudaSuccess)                                                                 \
      return vfail(EAGLE_ERR_CUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), \
                   __FILE__, __LINE__);                                                    \
  } while (0)

int cdiv(int a, int b) { return (a + b - 1) / b; }

constexpr int VMAX_ROWS = 256;   // slots of one call over all requests (split-K scratch, rstd)

// ------------------------------------------------------------- device kernels
struct EmbedArgs {
  int B, S, d, vocab, max_pos, max_prefix;
  const int* tokens;          // [B][S]
  const int* positions;       // [B][S]
  const unsigned char* mask;  // [B][S][S]
  const int* cu_seqlens;      // [B+1]
  const uint16_t* emb;        // [V][d] bf16
  const float* gamma;         // attention RMSNorm gain [d]
  float* x;                   // [N][d] residual stream
  uint16_t* x_hl;             // [2N][d] hi / lo of x * gamma
  float* ss;                  // [d/128][ss_ld] per-tile sums of squares of x
  int ss_ld;
  int* row_req;
  int* row_slot;
  int* row_pos;
  unsigned long long* row_mask;
  int* n_eff;
  unsigned* err;
};

// One CTA (128 threads) per slot row: the embedding row, its gained hi / lo copy, the
// per-128-column sums of squares (the factored RMSNorm the QKV GEMM applies), and the
// row's metadata: request, slot, position id (clamped to the rotary table) and the mask row
// as ancestor bits.
__global__ void __launch_bounds__(128) verify_embed_kernel(const EmbedArgs a) {
  __shared__ float red[4];
  pdl_wait();
  pdl_trigger();
  const int n = blockIdx.x, b = n / a.S, i = n - b * a.S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int tok = __ldg(a.tokens + n);
  if (tok < 0 || tok >= a.vocab) {
    if (tid == 0) atomicOr(a.err, DEVERR_TOKEN);
    tok = 0;
  }
  if (tid == 0) {
    int pos = __ldg(a.positions + n);
    if (pos < 0 || pos >= a.max_pos) {
      atomicOr(a.err, DEVERR_PREFIX);
      pos = pos < 0 ? 0 : a.max_pos - 1;
    }
    a.row_req[n] = b;
    a.row_slot[n] = i;
    a.row_pos[n] = pos;
    if (i == 0) {
      int nb = __ldg(a.cu_seqlens + b + 1) - __ldg(a.cu_seqlens + b);
      if (nb < 0 || nb > a.max_prefix) {
        atomicOr(a.err, DEVERR_PREFIX);
        nb = nb < 0 ? 0 : a.max_prefix;
      }
      a.n_eff[b] = nb;
    }
  }
  if (warp == 0) {   // mask row -> ancestor bits over the request's slots
    const unsigned char* mr = a.mask + (static_cast<size_t>(b) * a.S + i) * a.S;
    unsigned long long bits = 0ull;
    for (int j = lane; j < a.S; j += 32)
      if (__ldg(mr + j)) bits |= 1ull << j;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bits |= __shfl_xor_sync(0xffffffffu, bits, o);
    if (lane == 0) a.row_mask[n] = bits;
  }
  const uint16_t* er = a.emb + static_cast<size_t>(tok) * a.d;
  for (int t = 0; t < a.d / BM; ++t) {
    const int c = t * BM + tid;
    const float v = bf16_to_f32(__ldg(er + c));
    a.x[static_cast<size_t>(n) * a.d + c] = v;
    uint16_t hi, lo;
    split_hilo(v * __ldg(a.gamma + c), hi, lo);
    a.x_hl[static_cast<size_t>(2 * n) * a.d + c] = hi;
    a.x_hl[static_cast<size_t>(2 * n + 1) * a.d + c] = lo;
    const float sq = warp_sum(v * v);
    if (lane == 0) red[warp] = sq;
    __syncthreads();
    if (tid == 0) a.ss[static_cast<size_t>(t) * a.ss_ld + n] = red[0] + red[1] + red[2] + red[3];
    __syncthreads();
  }
}

struct AcceptArgs {
  int B, S;
  const int* top_id;          // [B][S] the target's most likely next token after each slot
  const int* tokens;          // [B][S]
  const int* parents;         // [B][S]
  int* accept_len;            // [B]
  int* accept_slots;          // [B][S] accepted slots in path order (root excluded), -1 after
  int* correction;            // [B]
  unsigned* err;
};

// One CTA per request.  From the root, the child whose token is the target's most likely
// next token is accepted (the first such slot: siblings carry distinct tokens) and the
// walk continues from it; it stops at a slot with no such child.
__global__ void __launch_bounds__(64) greedy_accept_kernel(const AcceptArgs a) {
  __shared__ int top[64], tok[64], par[64];
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, i = threadIdx.x;
  if (i < a.S) {
    const size_t o = static_cast<size_t>(b) * a.S + i;
    top[i] = __ldcg(a.top_id + o);
    tok[i] = __ldg(a.tokens + o);
    int p = __ldg(a.parents + o);
    if (i == 0) p = -1;
    else if (p < 0 || p >= i) {   // a parent precedes its child; anything else is cut off
      atomicOr(a.err, DEVERR_TOKEN);
      p = -2;
    }
    par[i] = p;
    a.accept_slots[o] = -1;
  }
  __syncthreads();
  if (i == 0) {
    int u = 0, len = 0;
    for (;;) {
      const int want = top[u];
      int nxt = -1;
      for (int j = u + 1; j < a.S; ++j)
        if (par[j] == u && tok[j] == want) { nxt = j; break; }
      if (nxt < 0) break;
      a.accept_slots[static_cast<size_t>(b) * a.S + len] = nxt;
      ++len;
      u = nxt;
    }
    a.accept_len[b] = len;
    a.correction[b] = top[u];
  }
}

cudaLaunchConfig_t small_cfg(dim3 grid, dim3 block, cudaStream_t st, bool pdl, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.stream = st;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  return cfg;
}

}  // namespace

// --------------------------------------------------------------------- handle
struct eagle_verify {
  eagle_verify_config_t cfg;
  eagle_verify_weights_t w;
  bool use_pdl = true;
  int n_max = 0, max_pos = 0, lm_G = 0;
  CUtensorMap tm_qkv, tm_o, tm_gate, tm_up, tm_down, tm_lm;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  float *x = nullptr, *y = nullptr, *hid = nullptr, *q = nullptr, *o = nullptr;
  float *ss_x = nullptr, *ss_y = nullptr, *ss_h = nullptr, *tk = nullptr, *tv = nullptr;
  float *rope_cos = nullptr, *rope_sin = nullptr, *part = nullptr;
  float *lm_max = nullptr, *lm_sum = nullptr, *lm_val = nullptr, *top_lp = nullptr, *top_lse = nullptr;
  uint16_t *x_hl = nullptr, *o_hl = nullptr, *xm_hl = nullptr, *s_hl = nullptr, *hf_hl = nullptr;
  int *lm_id = nullptr, *counters = nullptr, *top_id = nullptr;
  int *row_req = nullptr, *row_slot = nullptr, *row_pos = nullptr, *n_eff = nullptr;
  unsigned long long* row_mask = nullptr;
  unsigned* err = nullptr;
};

namespace {

struct VCarver {
  char* base;
  size_t off = 0;
  template <class T>
  T* take(size_t n) {
    off = (off + 255) & ~size_t(255);
    T* p = reinterpret_cast<T*>(base ? base + off : nullptr);
    off += n * sizeof(T);
    return p;
  }
};

void vcarve(eagle_verify* h, char* base, size_t* total) {
  const eagle_verify_config_t& c = h->cfg;
  const size_t n = h->n_max, d = c.d, hq = static_cast<size_t>(c.n_heads) * c.head_dim, ff = c.d_ff;
  const size_t dt = cdiv(c.d, BM), T = cdiv(c.vocab, BM);
  VCarver cv{base};
  h->x = cv.take<float>(n * d);
  h->y = cv.take<float>(n * d);
  h->hid = cv.take<float>(n * d);
  h->q = cv.take<float>(n * hq);
  h->o = cv.take<float>(n * hq);
  h->x_hl = cv.take<uint16_t>(2 * n * d);
  h->o_hl = cv.take<uint16_t>(2 * n * hq);
  h->xm_hl = cv.take<uint16_t>(2 * n * d);
  h->s_hl = cv.take<uint16_t>(2 * n * ff);
  h->hf_hl = cv.take<uint16_t>(2 * n * d);
  h->ss_x = cv.take<float>(dt * n);
  h->ss_y = cv.take<float>(dt * n);
  h->ss_h = cv.take<float>(dt * n);
  const size_t tkv = static_cast<size_t>(c.max_batch) * c.max_slots * c.n_kv_heads * c.head_dim;
  h->tk = cv.take<float>(tkv);
  h->tv = cv.take<float>(tkv);
  h->rope_cos = cv.take<float>(static_cast<size_t>(h->max_pos) * c.head_dim / 2);
  h->rope_sin = cv.take<float>(static_cast<size_t>(h->max_pos) * c.head_dim / 2);
  h->part = cv.take<float>(static_cast<size_t>(num_sms()) * 2 * VMAX_ROWS * BM);
  h->lm_max = cv.take<float>(T * n);
  h->lm_sum = cv.take<float>(T * n);
  h->lm_val = cv.take<float>(static_cast<size_t>(h->lm_G) * n);
  h->lm_id = cv.take<int>(static_cast<size_t>(h->lm_G) * n);
  h->counters = cv.take<int>(16384);
  h->top_id = cv.take<int>(n);
  h->top_lp = cv.take<float>(n);
  h->top_lse = cv.take<float>(n);
  h->row_req = cv.take<int>(n);
  h->row_slot = cv.take<int>(n);
  h->row_pos = cv.take<int>(n);
  h->row_mask = cv.take<unsigned long long>(n);
  h->n_eff = cv.take<int>(c.max_batch);
  h->err = cv.take<unsigned>(64);
  *total = cv.off + 256;
}

eagle_status_t vgemm(eagle_verify* h, GemmPlan& p, int N, cudaStream_t st) {
  if (!plan_gemm(p, N)) return vfail(EAGLE_ERR_UNSUPPORTED, "verify GEMM M=%d K=%d N=%d does not fit", p.args.M, p.args.K, N);
  VCU(launch_gemm(p, st, h->use_pdl));
  return EAGLE_OK;
}

GemmPlan vplan(eagle_verify* h, const CUtensorMap& tm0, const CUtensorMap* tm1, int M, int K) {
  return gemm_plan(true, tm0, tm1, nullptr, nullptr, M, K, M, h->part, h->counters, h->err);
}

eagle_status_t enqueue_verify(eagle_verify* h, const eagle_verify_inputs_t* in, const eagle_verify_outputs_t* out,
                              cudaStream_t st) {
  const eagle_verify_config_t& c = h->cfg;
  const int B = in->B, S = in->S, N = B * S, d = c.d, ff = c.d_ff, hq = c.n_heads * c.head_dim;
  const int dt = cdiv(d, BM), nmax = h->n_max;
  const bool pdl = h->use_pdl;
  cudaLaunchAttribute attr[1];
  {
    EmbedArgs a;
    a.B = B;
    a.S = S;
    a.d = d;
    a.vocab = c.vocab;
    a.max_pos = h->max_pos;
    a.max_prefix = c.max_prefix;
    a.tokens = in->tokens;
    a.positions = in->positions;
    a.mask = in->mask;
    a.cu_seqlens = in->cu_seqlens;
    a.emb = static_cast<const uint16_t*>(h->w.embed);
    a.gamma = h->w.attn_norm;
    a.x = h->x;
    a.x_hl = h->x_hl;
    a.ss = h->ss_x;
    a.ss_ld = nmax;
    a.row_req = h->row_req;
    a.row_slot = h->row_slot;
    a.row_pos = h->row_pos;
    a.row_mask = h->row_mask;
    a.n_eff = h->n_eff;
    a.err = h->err;
    cudaLaunchConfig_t cfg = small_cfg(dim3(N), dim3(128), st, pdl, attr);
    VCU(cudaLaunchKernelEx(&cfg, verify_embed_kernel, a));
  }
  eagle_status_t r;
  // RMSNorm + QKV + rotary: queries, and every slot's K / V as a tree row of its request
  {
    const int qkv = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
    GemmPlan p = vplan(h, h->tm_qkv, nullptr, qkv, d);
    tma_operand(p, h->x_hl);
    EpiArgs& e = p.args.e;
    memset(&e, 0, sizeof(e));
    e.kind = EPI_QKV;
    e.q = h->q;
    e.tk = h->tk;
    e.tv = h->tv;
    e.row_req = h->row_req;
    e.row_slot = h->row_slot;
    e.row_pos = h->row_pos;
    e.rope_cos = h->rope_cos;
    e.rope_sin = h->rope_sin;
    e.max_pos = h->max_pos;
    e.Hq = c.n_heads;
    e.Hkv = c.n_kv_heads;
    e.hd = c.head_dim;
    e.tree_rows = S;
    factored_norm(e, h->ss_x, dt, nmax, d, c.rms_eps);
    if ((r = vgemm(h, p, N, st)) != EAGLE_OK) return r;
  }
  // attention over the prefix and the slots of the row's mask
  {
    AttnArgs a;
    memset(&a, 0, sizeof(a));
    a.q = h->q;
    a.k_cache = in->k_cache;
    a.v_cache = in->v_cache;
    a.cache_bf16 = 1;
    a.cu_seqlens = in->cu_seqlens;
    a.n_eff = h->n_eff;
    a.max_prefix = c.max_prefix;
    a.tk = h->tk;
    a.tv = h->tv;
    a.row_mask = h->row_mask;
    a.rows_per_req = S;
    a.tree_rows = S;
    a.tree_upto = S;
    a.B = B;
    a.Hq = c.n_heads;
    a.Hkv = c.n_kv_heads;
    a.hd = c.head_dim;
    a.max_splits = cdiv(c.max_prefix, ATT_CHUNK) + 1;
    const int rpg = attn_rows_per_group(c.n_heads, c.n_kv_heads);
    if (S > rpg) {
      a.row_groups = cdiv(S, rpg);
      a.rows_per_group = cdiv(S, a.row_groups);   // balanced groups
    }
    a.out = h->o;
    a.out_hl = h->o_hl;
    VCU(launch_attention(a, st, pdl));
  }
  // O projection + residual (and the MLP's gained operand copy)
  {
    GemmPlan p = vplan(h, h->tm_o, nullptr, d, hq);
    tma_operand(p, h->o_hl);
    p.args.e = epi_store(h->y, d, h->x, d, h->ss_y, nmax);
    write_operand(p.args.e, h->xm_hl, d, h->w.mlp_norm);
    if ((r = vgemm(h, p, N, st)) != EAGLE_OK) return r;
  }
  // RMSNorm + gate | up -> silu(g) * u
  {
    GemmPlan p = vplan(h, h->tm_gate, &h->tm_up, 2 * ff, d);
    p.args.a_pair = 1;
    p.args.e = epi_store(nullptr, ff, nullptr, 0, nullptr, 0);
    p.args.e.kind = EPI_SWIGLU;
    tma_operand(p, h->xm_hl);
    factored_norm(p.args.e, h->ss_y, dt, nmax, d, c.rms_eps);
    write_operand(p.args.e, h->s_hl, ff, nullptr);
    if ((r = vgemm(h, p, N, st)) != EAGLE_OK) return r;
  }
  // down projection + residual -> the layer output; the LM head's operand carries the
  // final RMSNorm gain, its row scale comes from these sums of squares
  {
    GemmPlan p = vplan(h, h->tm_down, nullptr, d, ff);
    tma_operand(p, h->s_hl);
    p.args.e = epi_store(h->hid, d, h->y, d, h->ss_h, nmax);
    write_operand(p.args.e, h->hf_hl, d, h->w.final_norm);
    if ((r = vgemm(h, p, N, st)) != EAGLE_OK) return r;
  }
  // frozen LM head over RMSNorm(hidden): per-tile log-sum-exp and the most likely token
  const long long T = cdiv(c.vocab, BM);
  int G = 0;
  {
    const int parts = cdiv(N, MAX_ROWS_PER_BLOCK), per = cdiv(N, parts);
    for (int r0 = 0; r0 < N; r0 += per) {
      const int n = std::min(per, N - r0);
      GemmPlan p = vplan(h, h->tm_lm, nullptr, c.vocab, d);
      tma_operand(p, h->hf_hl + 2 * static_cast<size_t>(r0) * d);
      EpiArgs& e = p.args.e;
      e.kind = EPI_LMHEAD;
      e.topk = 1;
      factored_norm(e, h->ss_h + r0, dt, nmax, d, c.rms_eps);
      if (out->logits) e.logits = out->logits + static_cast<size_t>(r0) * c.vocab;
      if (!plan_gemm(p, n)) return vfail(EAGLE_ERR_UNSUPPORTED, "verify LM head does not fit");
      G = p.grid;
      e.lm_max = h->lm_max + r0 * T;
      e.lm_sum = h->lm_sum + r0 * T;
      e.lm_val = h->lm_val + static_cast<size_t>(r0) * G;
      e.lm_id = h->lm_id + static_cast<size_t>(r0) * G;
      VCU(launch_gemm(p, st, pdl));
    }
  }
  {
    LmPartials lm;
    lm.max = h->lm_max;
    lm.sum = h->lm_sum;
    lm.val = h->lm_val;
    lm.id = h->lm_id;
    lm.G = G;
    lm.T = static_cast<int>(T);
    lm.poison_if = nullptr;
    int* ids = out->top_id ? out->top_id : h->top_id;
    float* lp = out->top_logp ? out->top_logp : h->top_lp;
    float* ls = out->lse ? out->lse : h->top_lse;
    VCU(launch_lm_merge(lm, N, 1, ids, lp, ls, st, pdl));
    if (out->accept_len) {
      AcceptArgs a;
      a.B = B;
      a.S = S;
      a.top_id = ids;
      a.tokens = in->tokens;
      a.parents = in->parents;
      a.accept_len = out->accept_len;
      a.accept_slots = out->accept_slots;
      a.correction = out->correction;
      a.err = h->err;
      cudaLaunchConfig_t cfg = small_cfg(dim3(B), dim3(64), st, pdl, attr);
      VCU(cudaLaunchKernelEx(&cfg, greedy_accept_kernel, a));
    }
  }
  if (out->hidden)
    VCU(cudaMemcpyAsync(out->hidden, h->hid, sizeof(float) * static_cast<size_t>(N) * d, cudaMemcpyDeviceToDevice, st));
  return EAGLE_OK;
}

}  // namespace

extern "C" eagle_status_t eagle_verify_create(const eagle_verify_config_t* cfg, const eagle_verify_weights_t* w,
                                              eagle_verify_t** out) {
  if (!cfg || !w || !out) return vfail(EAGLE_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  const eagle_verify_config_t& c = *cfg;
  if (c.d <= 0 || c.n_heads <= 0 || c.n_kv_heads <= 0 || c.d_ff <= 0 || c.vocab <= 0 || c.n_heads % c.n_kv_heads)
    return vfail(EAGLE_ERR_INVALID_ARG, "verify: sizes must be positive and n_heads %% n_kv_heads == 0");
  if (c.max_batch < 1 || c.max_slots < 1 || c.max_prefix < 0)
    return vfail(EAGLE_ERR_INVALID_ARG, "verify: max_batch, max_slots >= 1, max_prefix >= 0");
  if (!(c.rms_eps >= 0.f) || !(c.rope_theta > 0.f)) return vfail(EAGLE_ERR_INVALID_ARG, "verify: rms_eps / rope_theta");
  if (c.dtype != EAGLE_DTYPE_BF16 || c.head_dim != 128)
    return vfail(EAGLE_ERR_UNSUPPORTED, "verify: bf16 weights with head_dim 128 only");
  const int qkv = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
  if (c.d % 128 || c.d_ff % 128 || c.vocab % 128 || qkv % 128)
    return vfail(EAGLE_ERR_UNSUPPORTED, "verify: d, d_ff, vocab, (Hq+2Hkv)hd must be multiples of 128");
  if (c.max_slots > 64) return vfail(EAGLE_ERR_UNSUPPORTED, "verify: more than 64 slots per request");
  if (static_cast<long long>(c.max_batch) * c.max_slots > VMAX_ROWS)
    return vfail(EAGLE_ERR_UNSUPPORTED, "verify: more than %d slots per call (max_batch * max_slots)", VMAX_ROWS);
  if (!w->embed || !w->attn_norm || !w->w_qkv || !w->w_o || !w->mlp_norm || !w->w_gate || !w->w_up || !w->w_down ||
      !w->final_norm || !w->w_lm)
    return vfail(EAGLE_ERR_INVALID_ARG, "verify: null weight pointer");
  eagle_verify* h = new eagle_verify();
  h->cfg = c;
  h->w = *w;
  h->use_pdl = !(c.flags & EAGLE_FLAG_NO_PDL);
  h->n_max = c.max_batch * c.max_slots;
  h->max_pos = c.max_prefix + c.max_slots + 1;
  h->lm_G = std::min<long long>(num_sms(), static_cast<long long>(cdiv(c.vocab, BM)) * cdiv(c.d, BK));
  cudaError_t e;
  if ((e = gemm_setup_attributes()) != cudaSuccess || (e = attn_setup_attributes()) != cudaSuccess ||
      (e = tree_setup_attributes()) != cudaSuccess) {
    delete h;
    return vfail(EAGLE_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  }
  const int d = c.d, ff = c.d_ff, hq = c.n_heads * c.head_dim;
  if (!(make_weight_map(&h->tm_qkv, w->w_qkv, qkv, d) && make_weight_map(&h->tm_o, w->w_o, d, hq) &&
        make_weight_map(&h->tm_gate, w->w_gate, ff, d, BM / 2) && make_weight_map(&h->tm_up, w->w_up, ff, d, BM / 2) &&
        make_weight_map(&h->tm_down, w->w_down, d, ff) && make_weight_map(&h->tm_lm, w->w_lm, c.vocab, d))) {
    delete h;
    return vfail(EAGLE_ERR_CUDA, "verify: cuTensorMapEncodeTiled failed (weights must be 16-byte aligned)");
  }
  size_t total = 0;
  vcarve(h, nullptr, &total);
  if (cudaMalloc(&h->ws, total) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return vfail(EAGLE_ERR_OOM, "verify: workspace of %zu bytes", total);
  }
  h->ws_bytes = total;
  vcarve(h, static_cast<char*>(h->ws), &total);
  if ((e = cudaMemset(h->ws, 0, h->ws_bytes)) != cudaSuccess) {
    cudaFree(h->ws);
    delete h;
    return vfail(EAGLE_ERR_CUDA, "cudaMemset: %s", cudaGetErrorString(e));
  }
  {   // rotary tables: angle = pos * theta^(-2j/hd), evaluated in double
    const int half = c.head_dim / 2;
    std::vector<float> cs(static_cast<size_t>(h->max_pos) * half), sn(cs.size());
    for (int p = 0; p < h->max_pos; ++p)
      for (int j = 0; j < half; ++j) {
        const double ang = p * std::pow(static_cast<double>(c.rope_theta), -2.0 * j / c.head_dim);
        cs[static_cast<size_t>(p) * half + j] = static_cast<float>(std::cos(ang));
        sn[static_cast<size_t>(p) * half + j] = static_cast<float>(std::sin(ang));
      }
    if (cudaMemcpy(h->rope_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(h->rope_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaFree(h->ws);
      delete h;
      return vfail(EAGLE_ERR_CUDA, "verify: rope table upload");
    }
  }
  *out = h;
  return EAGLE_OK;
}

extern "C" eagle_status_t eagle_verify_tree(eagle_verify_t* h, const eagle_verify_inputs_t* in,
                                            const eagle_verify_outputs_t* out, void* stream) {
  if (!h || !in || !out) return vfail(EAGLE_ERR_INVALID_ARG, "null argument");
  const eagle_verify_config_t& c = h->cfg;
  if (in->B < 1 || in->B > c.max_batch) return vfail(EAGLE_ERR_INVALID_ARG, "verify: B=%d outside 1..%d", in->B, c.max_batch);
  if (in->S < 1 || in->S > c.max_slots) return vfail(EAGLE_ERR_INVALID_ARG, "verify: S=%d outside 1..%d", in->S, c.max_slots);
  if (!in->tokens || !in->positions || !in->mask || !in->cu_seqlens ||
      (c.max_prefix > 0 && (!in->k_cache || !in->v_cache)))
    return vfail(EAGLE_ERR_INVALID_ARG, "verify: null input pointer");
  if (out->accept_len && (!out->accept_slots || !out->correction || !in->parents))
    return vfail(EAGLE_ERR_INVALID_ARG, "verify: acceptance needs parents, accept_slots and correction");
  return enqueue_verify(h, in, out, static_cast<cudaStream_t>(stream));
}

extern "C" eagle_status_t eagle_verify_check(eagle_verify_t* h, uint32_t* word) {
  if (!h) return vfail(EAGLE_ERR_INVALID_ARG, "null handle");
  VCU(cudaDeviceSynchronize());
  unsigned wv = 0;
  VCU(cudaMemcpy(&wv, h->err, sizeof(unsigned), cudaMemcpyDeviceToHost));
  if (word) *word = wv;
  if (wv) {
    VCU(cudaMemset(h->err, 0, sizeof(unsigned)));
    return vfail(EAGLE_ERR_DEVICE, "device error word 0x%x", wv);
  }
  return EAGLE_OK;
}

extern "C" void eagle_verify_destroy(eagle_verify_t* h) {
  if (!h) return;
  if (h->ws) cudaFree(h->ws);
  delete h;
}
