// Multi-layer decoder stacks over tree / block rows, behind two C entry points (see
// include/eagle_draft.h):
//
// * the target's one verification pass over an emitted draft tree, and greedy acceptance
//   of the deepest path it confirms.  "Tree attention in one verification pass"
//   (aicassindra.com tm_eagle_deep): the tree's slots are laid out after the verified
//   prefix and run through the target at once; each slot attends to the prefix and to its
//   ancestors and itself only (the emitted mask), at position id prefix length + depth, so
//   one pass gives every slot the target's next-token distribution after exactly that
//   slot's path.  Greedy acceptance ("How speculative decoding works", kaushalya.io;
//   "Acceptance length under a tree", aicassindra.com): at temperature 0 a drafted token
//   passes when it is the target's most likely token after its parent's path; the deepest
//   passing path is kept and the target's most likely token after it is the correction.
// * the DFlash block-parallel draft ("DFlash-1: parallel block + KV injection", zackli.ai
//   "Speculative Decoding Deep Dive III"; "DFlash", kaushalya.io): the block [anchor, MASK,
//   ..., MASK] runs through L draft layers in one pass, every row attending to the target's
//   fused context injected as per-layer keys / values and to all rows of its block
//   (bidirectional), then the shared frozen LM head gives the top-k tokens of each mask slot.
//
// One engine serves both: Llama-style layers (RMSNorm, QKV, rotary, grouped-query
// attention, O, RMSNorm, SwiGLU) between the frozen embedding and the frozen LM head, with a
// final RMSNorm:
//   embed rows    x = E[tok]; operand copy of the first layer's RMSNorm-gained x; per-tile
//                 sums of squares; row metadata and the visibility rows as ancestor bits
//   per layer     QKV GEMM (factored RMSNorm, rotary in the epilogue, the rows' K/V as tree
//                 rows) -> attention over the layer's prefix cache + the visible rows (query
//                 groups past 128 vectors) -> O GEMM (+ residual) -> gate / up (factored
//                 RMSNorm, SwiGLU) -> down GEMM (+ residual), whose epilogue writes the next
//                 layer's gained operand copy (after the last layer: the final norm's)
//   LM head       W_lm RMSNorm(x): per-tile log-sum-exp and the top-k tokens
//   merge         per row: tokens, log-probabilities, log-sum-exp
//   accept        (verification) one CTA per request walks the tree from the root
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
  const int* tokens;          // [B][S]   (tree rows), or
  const int* positions;       // [B][S]
  const unsigned char* mask;  // [B][S][S]
  const int* anchor;          // [B]      (block rows: anchor, then mask_token; positions n_b + j;
  int mask_token;             //           every row sees the whole block)
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
  int nb = __ldg(a.cu_seqlens + b + 1) - __ldg(a.cu_seqlens + b);
  const bool nb_bad = nb < 0 || nb > a.max_prefix;
  nb = nb < 0 ? 0 : (nb > a.max_prefix ? a.max_prefix : nb);
  int tok = a.anchor ? (i == 0 ? __ldg(a.anchor + b) : a.mask_token) : __ldg(a.tokens + n);
  if (tok < 0 || tok >= a.vocab) {
    if (tid == 0) atomicOr(a.err, DEVERR_TOKEN);
    tok = 0;
  }
  if (tid == 0) {
    int pos = a.anchor ? nb + i : __ldg(a.positions + n);
    if (pos < 0 || pos >= a.max_pos) {
      atomicOr(a.err, DEVERR_PREFIX);
      pos = pos < 0 ? 0 : a.max_pos - 1;
    }
    a.row_req[n] = b;
    a.row_slot[n] = i;
    a.row_pos[n] = pos;
    if (i == 0) {
      if (nb_bad) atomicOr(a.err, DEVERR_PREFIX);
      a.n_eff[b] = nb;
    }
  }
  if (a.anchor) {
    if (tid == 0) a.row_mask[n] = a.S == 64 ? ~0ull : ((1ull << a.S) - 1ull);   // the whole block
  } else if (warp == 0) {   // mask row -> ancestor bits over the request's slots
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


// ----------------------------------------------------------------------- engine
namespace {

constexpr int STACK_MAX_LAYERS = 16;

struct StackShapes {
  int d, Hq, Hkv, hd, ff, vocab;
  float eps, theta;
  int layers, max_batch, max_slots, max_prefix;
  bool pdl;
};

struct StackLayer {
  CUtensorMap tm_qkv, tm_o, tm_gate, tm_up, tm_down;
  const float* attn_norm;
  const float* mlp_norm;
};

struct Stack {
  StackShapes c;
  StackLayer layer[STACK_MAX_LAYERS];
  const void* embed = nullptr;
  const float* final_norm = nullptr;
  CUtensorMap tm_lm;
  int n_max = 0, max_pos = 0, lm_G = 0, topk_max = 1;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  float *x[2] = {nullptr, nullptr}, *y = nullptr, *q = nullptr, *o = nullptr;
  float *ss_x = nullptr, *ss_y = nullptr, *tk = nullptr, *tv = nullptr;
  float *rope_cos = nullptr, *rope_sin = nullptr, *part = nullptr;
  float *lm_max = nullptr, *lm_sum = nullptr, *lm_val = nullptr, *top_lp = nullptr, *top_lse = nullptr;
  uint16_t *x_hl = nullptr, *o_hl = nullptr, *xm_hl = nullptr, *s_hl = nullptr;
  int *lm_id = nullptr, *counters = nullptr, *top_id = nullptr;
  int *row_req = nullptr, *row_slot = nullptr, *row_pos = nullptr, *n_eff = nullptr;
  unsigned long long* row_mask = nullptr;
  unsigned* err = nullptr;
};

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

void stack_carve(Stack* h, char* base, size_t* total) {
  const StackShapes& c = h->c;
  const size_t n = h->n_max, d = c.d, hq = static_cast<size_t>(c.Hq) * c.hd, ff = c.ff;
  const size_t dt = cdiv(c.d, BM), T = cdiv(c.vocab, BM);
  VCarver cv{base};
  h->x[0] = cv.take<float>(n * d);
  h->x[1] = cv.take<float>(n * d);
  h->y = cv.take<float>(n * d);
  h->q = cv.take<float>(n * hq);
  h->o = cv.take<float>(n * hq);
  h->x_hl = cv.take<uint16_t>(2 * n * d);
  h->o_hl = cv.take<uint16_t>(2 * n * hq);
  h->xm_hl = cv.take<uint16_t>(2 * n * d);
  h->s_hl = cv.take<uint16_t>(2 * n * ff);
  h->ss_x = cv.take<float>(dt * n);
  h->ss_y = cv.take<float>(dt * n);
  const size_t tkv = static_cast<size_t>(c.max_batch) * c.max_slots * c.Hkv * c.hd;
  h->tk = cv.take<float>(tkv);
  h->tv = cv.take<float>(tkv);
  h->rope_cos = cv.take<float>(static_cast<size_t>(h->max_pos) * c.hd / 2);
  h->rope_sin = cv.take<float>(static_cast<size_t>(h->max_pos) * c.hd / 2);
  h->part = cv.take<float>(static_cast<size_t>(num_sms()) * 2 * VMAX_ROWS * BM);
  h->lm_max = cv.take<float>(T * n);
  h->lm_sum = cv.take<float>(T * n);
  h->lm_val = cv.take<float>(static_cast<size_t>(h->lm_G) * n * h->topk_max);
  h->lm_id = cv.take<int>(static_cast<size_t>(h->lm_G) * n * h->topk_max);
  h->counters = cv.take<int>(16384);
  h->top_id = cv.take<int>(n * h->topk_max);
  h->top_lp = cv.take<float>(n * h->topk_max);
  h->top_lse = cv.take<float>(n);
  h->row_req = cv.take<int>(n);
  h->row_slot = cv.take<int>(n);
  h->row_pos = cv.take<int>(n);
  h->row_mask = cv.take<unsigned long long>(n);
  h->n_eff = cv.take<int>(c.max_batch);
  h->err = cv.take<unsigned>(64);
  *total = cv.off + 256;
}

// The weights of layer l (device pointers) -> its TMA descriptors.
struct LayerPtrs {
  const float *attn_norm, *mlp_norm;
  const void *w_qkv, *w_o, *w_gate, *w_up, *w_down;
};

// Validates the shapes, builds the descriptors, allocates and fills the workspace.
eagle_status_t stack_init(Stack* h, const StackShapes& c, const LayerPtrs* lp, const void* embed, const float* final_norm,
                          const void* w_lm, int topk_max) {
  if (c.d <= 0 || c.Hq <= 0 || c.Hkv <= 0 || c.ff <= 0 || c.vocab <= 0 || c.Hq % c.Hkv)
    return vfail(EAGLE_ERR_INVALID_ARG, "sizes must be positive and n_heads %% n_kv_heads == 0");
  if (c.max_batch < 1 || c.max_slots < 1 || c.max_prefix < 0)
    return vfail(EAGLE_ERR_INVALID_ARG, "max_batch, slots >= 1, max_prefix >= 0");
  if (!(c.eps >= 0.f) || !(c.theta > 0.f)) return vfail(EAGLE_ERR_INVALID_ARG, "rms_eps / rope_theta");
  if (c.hd != 128) return vfail(EAGLE_ERR_UNSUPPORTED, "bf16 weights with head_dim 128 only");
  if (c.layers < 1 || c.layers > STACK_MAX_LAYERS) return vfail(EAGLE_ERR_INVALID_ARG, "layers must be 1..%d", STACK_MAX_LAYERS);
  const int qkv = (c.Hq + 2 * c.Hkv) * c.hd;
  if (c.d % 128 || c.ff % 128 || c.vocab % 128 || qkv % 128)
    return vfail(EAGLE_ERR_UNSUPPORTED, "d, d_ff, vocab, (Hq+2Hkv)hd must be multiples of 128");
  if (c.max_slots > 64) return vfail(EAGLE_ERR_UNSUPPORTED, "more than 64 rows per request");
  if (static_cast<long long>(c.max_batch) * c.max_slots > VMAX_ROWS)
    return vfail(EAGLE_ERR_UNSUPPORTED, "more than %d rows per call", VMAX_ROWS);
  if (topk_max < 1 || topk_max > KMAX) return vfail(EAGLE_ERR_INVALID_ARG, "k must be 1..%d", KMAX);
  if (!embed || !final_norm || !w_lm) return vfail(EAGLE_ERR_INVALID_ARG, "null weight pointer");
  for (int l = 0; l < c.layers; ++l)
    if (!lp[l].attn_norm || !lp[l].mlp_norm || !lp[l].w_qkv || !lp[l].w_o || !lp[l].w_gate || !lp[l].w_up ||
        !lp[l].w_down)
      return vfail(EAGLE_ERR_INVALID_ARG, "null weight pointer (layer %d)", l);
  h->c = c;
  h->embed = embed;
  h->final_norm = final_norm;
  h->topk_max = topk_max;
  h->n_max = c.max_batch * c.max_slots;
  h->max_pos = c.max_prefix + c.max_slots + 1;
  h->lm_G = std::min<long long>(num_sms(), static_cast<long long>(cdiv(c.vocab, BM)) * cdiv(c.d, BK));
  cudaError_t e;
  if ((e = gemm_setup_attributes()) != cudaSuccess || (e = attn_setup_attributes()) != cudaSuccess ||
      (e = tree_setup_attributes()) != cudaSuccess)
    return vfail(EAGLE_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  const int d = c.d, ff = c.ff, hq = c.Hq * c.hd;
  for (int l = 0; l < c.layers; ++l) {
    StackLayer& L = h->layer[l];
    L.attn_norm = lp[l].attn_norm;
    L.mlp_norm = lp[l].mlp_norm;
    if (!(make_weight_map(&L.tm_qkv, lp[l].w_qkv, qkv, d) && make_weight_map(&L.tm_o, lp[l].w_o, d, hq) &&
          make_weight_map(&L.tm_gate, lp[l].w_gate, ff, d, BM / 2) && make_weight_map(&L.tm_up, lp[l].w_up, ff, d, BM / 2) &&
          make_weight_map(&L.tm_down, lp[l].w_down, d, ff)))
      return vfail(EAGLE_ERR_CUDA, "cuTensorMapEncodeTiled failed (weights must be 16-byte aligned)");
  }
  if (!make_weight_map(&h->tm_lm, w_lm, c.vocab, d))
    return vfail(EAGLE_ERR_CUDA, "cuTensorMapEncodeTiled failed (LM head must be 16-byte aligned)");
  size_t total = 0;
  stack_carve(h, nullptr, &total);
  if (cudaMalloc(&h->ws, total) != cudaSuccess) {
    cudaGetLastError();
    h->ws = nullptr;
    return vfail(EAGLE_ERR_OOM, "workspace of %zu bytes", total);
  }
  h->ws_bytes = total;
  stack_carve(h, static_cast<char*>(h->ws), &total);
  if ((e = cudaMemset(h->ws, 0, h->ws_bytes)) != cudaSuccess)
    return vfail(EAGLE_ERR_CUDA, "cudaMemset: %s", cudaGetErrorString(e));
  // rotary tables: angle = pos * theta^(-2j/hd), evaluated in double
  const int half = c.hd / 2;
  std::vector<float> cs(static_cast<size_t>(h->max_pos) * half), sn(cs.size());
  for (int p = 0; p < h->max_pos; ++p)
    for (int j = 0; j < half; ++j) {
      const double ang = p * std::pow(static_cast<double>(c.theta), -2.0 * j / c.hd);
      cs[static_cast<size_t>(p) * half + j] = static_cast<float>(std::cos(ang));
      sn[static_cast<size_t>(p) * half + j] = static_cast<float>(std::sin(ang));
    }
  if (cudaMemcpy(h->rope_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(h->rope_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess)
    return vfail(EAGLE_ERR_CUDA, "rope table upload");
  return EAGLE_OK;
}

void stack_free(Stack* h) {
  if (h->ws) cudaFree(h->ws);
  h->ws = nullptr;
}

eagle_status_t vgemm(Stack* h, GemmPlan& p, int N, cudaStream_t st) {
  if (!plan_gemm(p, N)) return vfail(EAGLE_ERR_UNSUPPORTED, "GEMM M=%d K=%d N=%d does not fit", p.args.M, p.args.K, N);
  VCU(launch_gemm(p, st, h->c.pdl));
  return EAGLE_OK;
}

GemmPlan vplan(Stack* h, const CUtensorMap& tm0, const CUtensorMap* tm1, int M, int K) {
  return gemm_plan(true, tm0, tm1, nullptr, nullptr, M, K, M, h->part, h->counters, h->err);
}

// The rows of one call: B requests of S rows (tree slots or a block), their embedding.
struct StackRows {
  int B, S;
  const int* tokens;
  const int* positions;
  const unsigned char* mask;
  const int* anchor;
  int mask_token;
  const int* cu_seqlens;
  const void* const* k_cache;   // [layers] host array of device caches
  const void* const* v_cache;
};

// Every kernel of one pass up to the merge; the rows' top-k tokens, log-probabilities and
// log-sum-exp end in ids / lps [N][k] and lses [N].  hidden / logits (nullable) receive the
// last layer's output and the full logits.
eagle_status_t stack_enqueue(Stack* h, const StackRows& in, int k, int* ids, float* lps, float* lses, float* hidden,
                             float* logits, cudaStream_t st) {
  const StackShapes& c = h->c;
  const int B = in.B, S = in.S, N = B * S, d = c.d, ff = c.ff, hq = c.Hq * c.hd;
  const int dt = cdiv(d, BM), nmax = h->n_max;
  const bool pdl = c.pdl;
  cudaLaunchAttribute attr[1];
  {
    EmbedArgs a;
    a.B = B;
    a.S = S;
    a.d = d;
    a.vocab = c.vocab;
    a.max_pos = h->max_pos;
    a.max_prefix = c.max_prefix;
    a.tokens = in.tokens;
    a.positions = in.positions;
    a.mask = in.mask;
    a.anchor = in.anchor;
    a.mask_token = in.mask_token;
    a.cu_seqlens = in.cu_seqlens;
    a.emb = static_cast<const uint16_t*>(h->embed);
    a.gamma = h->layer[0].attn_norm;
    a.x = h->x[0];
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
  for (int l = 0; l < c.layers; ++l) {
    const StackLayer& L = h->layer[l];
    float* x_cur = h->x[l & 1];
    float* x_next = h->x[(l + 1) & 1];
    // RMSNorm + QKV + rotary: queries, and every row's K / V as a tree row of its request
    {
      const int qkv = (c.Hq + 2 * c.Hkv) * c.hd;
      GemmPlan p = vplan(h, L.tm_qkv, nullptr, qkv, d);
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
      e.Hq = c.Hq;
      e.Hkv = c.Hkv;
      e.hd = c.hd;
      e.tree_rows = S;
      factored_norm(e, h->ss_x, dt, nmax, d, c.eps);
      if ((r = vgemm(h, p, N, st)) != EAGLE_OK) return r;
    }
    // attention over the layer's prefix cache and the rows each row's bits mark
    {
      AttnArgs a;
      memset(&a, 0, sizeof(a));
      a.q = h->q;
      a.k_cache = in.k_cache[l];
      a.v_cache = in.v_cache[l];
      a.cache_bf16 = 1;
      a.cu_seqlens = in.cu_seqlens;
      a.n_eff = h->n_eff;
      a.max_prefix = c.max_prefix;
      a.tk = h->tk;
      a.tv = h->tv;
      a.row_mask = h->row_mask;
      a.rows_per_req = S;
      a.tree_rows = S;
      a.tree_upto = S;
      a.B = B;
      a.Hq = c.Hq;
      a.Hkv = c.Hkv;
      a.hd = c.hd;
      a.max_splits = cdiv(c.max_prefix, ATT_CHUNK) + 1;
      const int rpg = attn_rows_per_group(c.Hq, c.Hkv);
      if (S > rpg) {
        a.row_groups = cdiv(S, rpg);
        a.rows_per_group = cdiv(S, a.row_groups);   // balanced groups
      }
      a.out = h->o;
      a.out_hl = h->o_hl;
      a.err = h->err;
      VCU(launch_attention(a, st, pdl));
    }
    // O projection + residual (and the MLP's gained operand copy)
    {
      GemmPlan p = vplan(h, L.tm_o, nullptr, d, hq);
      tma_operand(p, h->o_hl);
      p.args.e = epi_store(h->y, d, x_cur, d, h->ss_y, nmax);
      write_operand(p.args.e, h->xm_hl, d, L.mlp_norm);
      if ((r = vgemm(h, p, N, st)) != EAGLE_OK) return r;
    }
    // RMSNorm + gate | up -> silu(g) * u
    {
      GemmPlan p = vplan(h, L.tm_gate, &L.tm_up, 2 * ff, d);
      p.args.a_pair = 1;
      p.args.e = epi_store(nullptr, ff, nullptr, 0, nullptr, 0);
      p.args.e.kind = EPI_SWIGLU;
      tma_operand(p, h->xm_hl);
      factored_norm(p.args.e, h->ss_y, dt, nmax, d, c.eps);
      write_operand(p.args.e, h->s_hl, ff, nullptr);
      if ((r = vgemm(h, p, N, st)) != EAGLE_OK) return r;
    }
    // down projection + residual -> the layer output; its epilogue writes the next layer's
    // gained operand copy (after the last layer: the final norm's, for the LM head) and the
    // sums of squares of the row scale
    {
      GemmPlan p = vplan(h, L.tm_down, nullptr, d, ff);
      tma_operand(p, h->s_hl);
      p.args.e = epi_store(x_next, d, h->y, d, h->ss_x, nmax);
      write_operand(p.args.e, h->x_hl, d, l + 1 < c.layers ? h->layer[l + 1].attn_norm : h->final_norm);
      if ((r = vgemm(h, p, N, st)) != EAGLE_OK) return r;
    }
  }
  float* x_out = h->x[c.layers & 1];
  // frozen LM head over RMSNorm(x): per-tile log-sum-exp and the top-k tokens
  const long long T = cdiv(c.vocab, BM);
  int G = 0;
  {
    const int parts = cdiv(N, MAX_ROWS_PER_BLOCK), per = cdiv(N, parts);
    for (int r0 = 0; r0 < N; r0 += per) {
      const int n = std::min(per, N - r0);
      GemmPlan p = vplan(h, h->tm_lm, nullptr, c.vocab, d);
      tma_operand(p, h->x_hl + 2 * static_cast<size_t>(r0) * d);
      EpiArgs& e = p.args.e;
      e.kind = EPI_LMHEAD;
      e.topk = k;
      factored_norm(e, h->ss_x + r0, dt, nmax, d, c.eps);
      if (logits) e.logits = logits + static_cast<size_t>(r0) * c.vocab;
      if (!plan_gemm(p, n)) return vfail(EAGLE_ERR_UNSUPPORTED, "LM head does not fit");
      G = p.grid;
      e.lm_max = h->lm_max + r0 * T;
      e.lm_sum = h->lm_sum + r0 * T;
      e.lm_val = h->lm_val + static_cast<size_t>(r0) * G * k;
      e.lm_id = h->lm_id + static_cast<size_t>(r0) * G * k;
      VCU(launch_gemm(p, st, pdl));
    }
  }
  LmPartials lm;
  lm.max = h->lm_max;
  lm.sum = h->lm_sum;
  lm.val = h->lm_val;
  lm.id = h->lm_id;
  lm.G = G;
  lm.T = static_cast<int>(T);
  lm.poison_if = nullptr;
  VCU(launch_lm_merge(lm, N, k, ids, lps, lses, st, pdl));
  if (hidden) VCU(cudaMemcpyAsync(hidden, x_out, sizeof(float) * static_cast<size_t>(N) * d, cudaMemcpyDeviceToDevice, st));
  return EAGLE_OK;
}

eagle_status_t stack_check(Stack* h, uint32_t* word) {
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

}  // namespace

// -------------------------------------------------------------- verification
struct eagle_verify {
  Stack s;
  eagle_verify_config_t cfg;
};

extern "C" eagle_status_t eagle_verify_create(const eagle_verify_config_t* cfg, const eagle_verify_weights_t* w,
                                              eagle_verify_t** out) {
  if (!cfg || !w || !out) return vfail(EAGLE_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  const eagle_verify_config_t& c = *cfg;
  if (c.dtype != EAGLE_DTYPE_BF16) return vfail(EAGLE_ERR_UNSUPPORTED, "verify: bf16 weights only");
  StackShapes sh{c.d, c.n_heads, c.n_kv_heads, c.head_dim, c.d_ff, c.vocab, c.rms_eps, c.rope_theta, 1,
                 c.max_batch, c.max_slots, c.max_prefix, !(c.flags & EAGLE_FLAG_NO_PDL)};
  LayerPtrs lp{w->attn_norm, w->mlp_norm, w->w_qkv, w->w_o, w->w_gate, w->w_up, w->w_down};
  eagle_verify* h = new eagle_verify();
  h->cfg = c;
  const eagle_status_t st = stack_init(&h->s, sh, &lp, w->embed, w->final_norm, w->w_lm, 1);
  if (st != EAGLE_OK) {
    stack_free(&h->s);
    delete h;
    return st;
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
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Stack* s = &h->s;
  StackRows rows{in->B, in->S, in->tokens, in->positions, in->mask, nullptr, 0, in->cu_seqlens, &in->k_cache,
                 &in->v_cache};
  int* ids = out->top_id ? out->top_id : s->top_id;
  eagle_status_t r = stack_enqueue(s, rows, 1, ids, out->top_logp ? out->top_logp : s->top_lp,
                                   out->lse ? out->lse : s->top_lse, out->hidden, out->logits, st);
  if (r != EAGLE_OK) return r;
  if (out->accept_len) {
    AcceptArgs a;
    a.B = in->B;
    a.S = in->S;
    a.top_id = ids;
    a.tokens = in->tokens;
    a.parents = in->parents;
    a.accept_len = out->accept_len;
    a.accept_slots = out->accept_slots;
    a.correction = out->correction;
    a.err = s->err;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = small_cfg(dim3(in->B), dim3(64), st, s->c.pdl, attr);
    VCU(cudaLaunchKernelEx(&cfg, greedy_accept_kernel, a));
  }
  return EAGLE_OK;
}

extern "C" eagle_status_t eagle_verify_check(eagle_verify_t* h, uint32_t* word) {
  if (!h) return vfail(EAGLE_ERR_INVALID_ARG, "null handle");
  return stack_check(&h->s, word);
}

extern "C" void eagle_verify_destroy(eagle_verify_t* h) {
  if (!h) return;
  stack_free(&h->s);
  delete h;
}

// ---------------------------------------------------------------- DFlash draft
struct eagle_dflash {
  Stack s;
  eagle_dflash_config_t cfg;
};

extern "C" eagle_status_t eagle_dflash_create(const eagle_dflash_config_t* cfg, const eagle_dflash_weights_t* w,
                                              eagle_dflash_t** out) {
  if (!cfg || !w || !out) return vfail(EAGLE_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  const eagle_dflash_config_t& c = *cfg;
  if (c.dtype != EAGLE_DTYPE_BF16) return vfail(EAGLE_ERR_UNSUPPORTED, "dflash: bf16 weights only");
  if (c.n_layers < 1 || c.n_layers > STACK_MAX_LAYERS)
    return vfail(EAGLE_ERR_INVALID_ARG, "dflash: n_layers must be 1..%d", STACK_MAX_LAYERS);
  if (c.gamma < 1 || c.gamma > 63) return vfail(EAGLE_ERR_INVALID_ARG, "dflash: gamma must be 1..63");
  if (c.mask_token < 0 || c.mask_token >= c.vocab) return vfail(EAGLE_ERR_INVALID_ARG, "dflash: mask_token outside the table");
  if (!w->attn_norm || !w->mlp_norm || !w->w_qkv || !w->w_o || !w->w_gate || !w->w_up || !w->w_down)
    return vfail(EAGLE_ERR_INVALID_ARG, "dflash: null per-layer weight array");
  StackShapes sh{c.d, c.n_heads, c.n_kv_heads, c.head_dim, c.d_ff, c.vocab, c.rms_eps, c.rope_theta, c.n_layers,
                 c.max_batch, c.gamma + 1, c.max_prefix, !(c.flags & EAGLE_FLAG_NO_PDL)};
  LayerPtrs lp[STACK_MAX_LAYERS];
  for (int l = 0; l < c.n_layers; ++l)
    lp[l] = LayerPtrs{w->attn_norm[l], w->mlp_norm[l], w->w_qkv[l], w->w_o[l], w->w_gate[l], w->w_up[l], w->w_down[l]};
  eagle_dflash* h = new eagle_dflash();
  h->cfg = c;
  const eagle_status_t st = stack_init(&h->s, sh, lp, w->embed, w->final_norm, w->w_lm, c.k);
  if (st != EAGLE_OK) {
    stack_free(&h->s);
    delete h;
    return st;
  }
  *out = h;
  return EAGLE_OK;
}

extern "C" eagle_status_t eagle_dflash_draft(eagle_dflash_t* h, const eagle_dflash_inputs_t* in,
                                             const eagle_dflash_outputs_t* out, void* stream) {
  if (!h || !in || !out) return vfail(EAGLE_ERR_INVALID_ARG, "null argument");
  const eagle_dflash_config_t& c = h->cfg;
  if (in->B < 1 || in->B > c.max_batch) return vfail(EAGLE_ERR_INVALID_ARG, "dflash: B=%d outside 1..%d", in->B, c.max_batch);
  if (!in->anchor || !in->cu_seqlens || !in->ctx_k || !in->ctx_v) return vfail(EAGLE_ERR_INVALID_ARG, "dflash: null input");
  for (int l = 0; l < c.n_layers; ++l)
    if (c.max_prefix > 0 && (!in->ctx_k[l] || !in->ctx_v[l]))
      return vfail(EAGLE_ERR_INVALID_ARG, "dflash: null context cache of layer %d", l);
  if (!out->tokens || !out->logp || !out->lse) return vfail(EAGLE_ERR_INVALID_ARG, "dflash: null output pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Stack* s = &h->s;
  const int S = c.gamma + 1, k = c.k;
  StackRows rows{in->B, S, nullptr, nullptr, nullptr, in->anchor, c.mask_token, in->cu_seqlens, in->ctx_k, in->ctx_v};
  eagle_status_t r = stack_enqueue(s, rows, k, s->top_id, s->top_lp, s->top_lse, out->hidden, nullptr, st);
  if (r != EAGLE_OK) return r;
  // the mask rows (1..gamma of every request's block) into the outputs
  const size_t w = static_cast<size_t>(c.gamma) * k;
  VCU(cudaMemcpy2DAsync(out->tokens, w * 4, s->top_id + k, static_cast<size_t>(S) * k * 4, w * 4, in->B,
                        cudaMemcpyDeviceToDevice, st));
  VCU(cudaMemcpy2DAsync(out->logp, w * 4, s->top_lp + k, static_cast<size_t>(S) * k * 4, w * 4, in->B,
                        cudaMemcpyDeviceToDevice, st));
  VCU(cudaMemcpy2DAsync(out->lse, static_cast<size_t>(c.gamma) * 4, s->top_lse + 1, static_cast<size_t>(S) * 4,
                        static_cast<size_t>(c.gamma) * 4, in->B, cudaMemcpyDeviceToDevice, st));
  return EAGLE_OK;
}

extern "C" eagle_status_t eagle_dflash_check(eagle_dflash_t* h, uint32_t* word) {
  if (!h) return vfail(EAGLE_ERR_INVALID_ARG, "null handle");
  return stack_check(&h->s, word);
}

extern "C" void eagle_dflash_destroy(eagle_dflash_t* h) {
  if (!h) return;
  stack_free(&h->s);
  delete h;
}
