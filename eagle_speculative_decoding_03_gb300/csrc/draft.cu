// C ABI of the draft-tree step: handle creation, workspace, the per-depth launch
// sequence, CUDA-graph replay.  See include/eagle_draft.h for the contract.
//
// Per depth s (rows = frontier nodes of every request):
//   fc GEMM    [feat ; emb(tok)] -> h                         (gather fused into the operand loader)
//   QKV GEMM   RMSNorm(h) -> q, tree K/V (rotary in the epilogue)
//   attention  prefix KV + ancestor rows -> o
//   O GEMM     h + W_o o -> y
//   gate/up    RMSNorm(y) -> [g | u]
//   down GEMM  y + W_d (silu(g) * u) -> a                      (SwiGLU fused into the operand loader)
//   LM head    W_lm a -> per-CTA log-sum-exp and top-k partials (no logits in memory)
//   expand     merge partials, create children, pick the next frontier
// then one rerank / emit kernel.
#include "../../include/eagle_draft.h"
#include "common.cuh"
#include "internal.h"

#include <cmath>
#include <cstdarg>
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

using namespace eagle;

static thread_local std::string g_last_error = "no error";

static eagle_status_t fail(eagle_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

#define CU(call)                                                                          \
  do {                                                                                    \
    cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess)                                                                \
      return fail(EAGLE_ERR_CUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), \
                  __FILE__, __LINE__);                                                    \
  } while (0)

// LM-head launches of at least this many rows store the logits and select in a second
// kernel; fewer rows (one 16-row chunk) keep the log-sum-exp and top-k in the GEMM's
// epilogue.  (The fused epilogue's per-row work grows with the rows of a tile; from the
// second chunk on, its tail after the last weight tile costs more than writing and
// re-reading the logits.)
constexpr int LM_LOGITS_MIN_ROWS = 17;

struct eagle_draft {
  eagle_draft_config_t cfg;
  eagle_draft_weights_t w;
  bool tc = false;
  bool use_graph = true, use_pdl = true, gemm_occ2 = false;
  long long wait_limit = 0;   // bounded waits of the GEMMs, clock cycles (0: the default)
  int kv_keep = 0;            // the whole prefix cache stays in L2 between depths (evict-last hint)
  int lm_logits_min_rows = LM_LOGITS_MIN_ROWS;
  int D = 0, R = 0, gen = 0, S = 0, n_max = 0, k_max = 0, f_max = 0, max_nodes = 0;
  int rows[EAGLE_MAX_DEPTH], kids[EAGLE_MAX_DEPTH];
  int row_base[EAGLE_MAX_DEPTH + 1], node_base[EAGLE_MAX_DEPTH + 1];
  int max_pos = 0, max_splits = 0, qv_max = 0, lm_G = 0;
  CUtensorMap tm_fc, tm_fc3, tm_qkv, tm_o, tm_gate, tm_up, tm_down, tm_lm;
  // workspace
  void* ws = nullptr;
  size_t ws_bytes = 0;
  float *h = nullptr, *y = nullptr, *a[2] = {nullptr, nullptr}, *q = nullptr, *o = nullptr, *gu = nullptr;
  float *ss_h = nullptr, *ss_y = nullptr, *g_root = nullptr, *tk = nullptr, *tv = nullptr;
  float *rope_cos = nullptr, *rope_sin = nullptr, *part = nullptr;
  float *lm_max = nullptr, *lm_sum = nullptr, *lm_val = nullptr;
  float* logits = nullptr;   // [N_max][vocab] LM heads over many rows: logits, then a select kernel
  // bf16 hi/lo operand copies [2 N_max][K] written by the producing epilogue (tensor-core path)
  uint16_t *xa_hl = nullptr, *o_hl = nullptr, *xm_hl = nullptr, *s_hl = nullptr, *a_hl = nullptr, *fc_hl = nullptr;
  int *lm_id = nullptr, *counters = nullptr;
  int *node_tok = nullptr, *node_parent = nullptr, *node_depth = nullptr, *node_row = nullptr;
  float* node_logv = nullptr;
  int *n_eff = nullptr, *frontier = nullptr, *exp_counters = nullptr, *exp_tok = nullptr;
  float* exp_v = nullptr;
  unsigned long long* slot_mask = nullptr;
  RowMeta meta[2];
  unsigned* err = nullptr;
  // graph cache
  cudaStream_t cap_stream = nullptr;
  cudaGraphExec_t graph = nullptr;
  std::vector<const void*> graph_key;
  int launches = 0;
  // profiling: (kind, start, stop) per launch
  bool profiling = false;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_used = 0;
  std::vector<int> ev_kind;
};

static const char* kKernelNames[EAGLE_K_COUNT] = {"init", "fc3", "fc", "qkv_rope", "attention", "o_proj",
                                                  "gate_up", "down", "lm_head", "expand", "rerank", "lm_merge", "fc_operand",
                                                  "lm_select"};

// Event pair around one launch (profiling mode only).
struct ProfScope {
  eagle_draft* h;
  cudaStream_t st;
  int kind;
  cudaEvent_t stop = nullptr;
  ProfScope(eagle_draft* h_, int kind_, cudaStream_t st_) : h(h_), st(st_), kind(kind_) {
    if (!h->profiling) return;
    while (h->ev_pool.size() < h->ev_used + 2) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return;
      h->ev_pool.push_back(e);
    }
    // External: inside a stream capture this becomes an event-record node of the graph
    cudaEventRecordWithFlags(h->ev_pool[h->ev_used], st, cudaEventRecordExternal);
    stop = h->ev_pool[h->ev_used + 1];
    h->ev_used += 2;
    h->ev_kind.push_back(kind);
  }
  ~ProfScope() {
    if (stop) cudaEventRecordWithFlags(stop, st, cudaEventRecordExternal);
  }
};

static int ceil_div(int a, int b) { return (a + b - 1) / b; }

// EAGLE_FAULT in the environment makes a step fail on the host, for tests of the error paths:
// "alloc" = the workspace allocation of eagle_draft_create, "launch" = a launch in the middle of
// eagle_draft_tree (depth 2's attention, or the last depth's if there is one).
static bool fault_injected(const char* what) {
  const char* f = getenv("EAGLE_FAULT");
  return f && strcmp(f, what) == 0;
}


// --------------------------------------------------------------- validation
static eagle_status_t validate(const eagle_draft_config_t& c, const eagle_draft_weights_t* w) {
  if (c.d <= 0 || c.n_heads <= 0 || c.n_kv_heads <= 0 || c.head_dim <= 0 || c.d_ff <= 0 || c.vocab <= 0)
    return fail(EAGLE_ERR_INVALID_ARG, "sizes must be positive");
  if (c.n_heads % c.n_kv_heads) return fail(EAGLE_ERR_INVALID_ARG, "n_heads %% n_kv_heads != 0");
  if (c.dtype != EAGLE_DTYPE_F32 && c.dtype != EAGLE_DTYPE_BF16) return fail(EAGLE_ERR_INVALID_ARG, "dtype");
  if (c.tree_kind != EAGLE_TREE_STATIC && c.tree_kind != EAGLE_TREE_DYNAMIC)
    return fail(EAGLE_ERR_INVALID_ARG, "tree_kind");
  if (c.feat_kind != EAGLE_FEAT_F && c.feat_kind != EAGLE_FEAT_FUSED) return fail(EAGLE_ERR_INVALID_ARG, "feat_kind");
  if (c.depth < 1 || c.depth > EAGLE_MAX_DEPTH) return fail(EAGLE_ERR_INVALID_ARG, "depth must be 1..%d", EAGLE_MAX_DEPTH);
  if (c.max_batch < 1 || c.max_prefix < 0) return fail(EAGLE_ERR_INVALID_ARG, "max_batch / max_prefix");
  if (!(c.rms_eps >= 0.f) || !(c.rope_theta > 0.f)) return fail(EAGLE_ERR_INVALID_ARG, "rms_eps / rope_theta");
  if (c.head_dim != 64 && c.head_dim != 128) return fail(EAGLE_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
  if (c.tree_kind == EAGLE_TREE_DYNAMIC) {
    if (c.k < 1 || c.k > KMAX) return fail(EAGLE_ERR_INVALID_ARG, "k must be 1..%d", KMAX);
  } else {
    for (int s = 0; s < c.depth; ++s)
      if (c.branching[s] < 1 || c.branching[s] > KMAX) return fail(EAGLE_ERR_INVALID_ARG, "branching must be 1..%d", KMAX);
  }
  if (!w || !w->embed || !w->w_fc || !w->attn_norm || !w->w_qkv || !w->w_o || !w->mlp_norm || !w->w_gate ||
      !w->w_up || !w->w_down || !w->w_lm || (c.feat_kind == EAGLE_FEAT_FUSED && !w->w_fc3))
    return fail(EAGLE_ERR_INVALID_ARG, "null weight pointer");
  const int qkv = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
  if (c.dtype == EAGLE_DTYPE_BF16) {
    if (c.d % 128 || c.d_ff % 128 || c.vocab % 128 || qkv % 128 || (c.n_heads * c.head_dim) % 64)
      return fail(EAGLE_ERR_UNSUPPORTED, "bf16 weights need d, d_ff, vocab, (Hq+2Hkv)hd multiples of 128");
  } else {
    if (c.d % 8 || c.d_ff % 8 || (c.n_heads * c.head_dim) % 8) return fail(EAGLE_ERR_UNSUPPORTED, "f32: d, d_ff multiples of 8");
  }
  return EAGLE_OK;
}

// ---------------------------------------------------------------- workspace
struct Carver {
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

static void carve(eagle_draft* h, char* base, size_t* total) {
  const eagle_draft_config_t& c = h->cfg;
  const int d = c.d, B = c.max_batch, hq = c.n_heads * c.head_dim, n = h->n_max;
  const int dt = ceil_div(d, BM);
  Carver cv{base};
  h->h = cv.take<float>(static_cast<size_t>(n) * d);
  h->y = cv.take<float>(static_cast<size_t>(n) * d);
  h->a[0] = cv.take<float>(static_cast<size_t>(n) * d);
  h->a[1] = cv.take<float>(static_cast<size_t>(n) * d);
  h->q = cv.take<float>(static_cast<size_t>(n) * hq);
  h->o = cv.take<float>(static_cast<size_t>(n) * hq);
  h->gu = cv.take<float>(static_cast<size_t>(n) * 2 * c.d_ff);
  h->xa_hl = cv.take<uint16_t>(static_cast<size_t>(2 * n) * d);
  h->o_hl = cv.take<uint16_t>(static_cast<size_t>(2 * n) * hq);
  h->xm_hl = cv.take<uint16_t>(static_cast<size_t>(2 * n) * d);
  h->s_hl = cv.take<uint16_t>(static_cast<size_t>(2 * n) * c.d_ff);
  h->a_hl = cv.take<uint16_t>(static_cast<size_t>(2 * n) * d);
  h->fc_hl = cv.take<uint16_t>(static_cast<size_t>(2 * n) * 2 * d);
  h->ss_h = cv.take<float>(static_cast<size_t>(dt) * n);
  h->ss_y = cv.take<float>(static_cast<size_t>(dt) * n);
  h->g_root = cv.take<float>(static_cast<size_t>(B) * d);
  const size_t tkv = static_cast<size_t>(B) * h->R * c.n_kv_heads * c.head_dim;
  h->tk = cv.take<float>(tkv);
  h->tv = cv.take<float>(tkv);
  h->rope_cos = cv.take<float>(static_cast<size_t>(h->max_pos) * c.head_dim / 2);
  h->rope_sin = cv.take<float>(static_cast<size_t>(h->max_pos) * c.head_dim / 2);
  h->part = cv.take<float>(static_cast<size_t>(num_sms()) * 2 * 256 * BM);
  const size_t lmn = static_cast<size_t>(h->lm_G) * n;
  const size_t lmt = static_cast<size_t>(ceil_div(c.vocab, BM)) * n;
  h->lm_max = cv.take<float>(lmt);
  h->lm_sum = cv.take<float>(lmt);
  h->lm_val = cv.take<float>(lmn * KMAX);
  h->lm_id = cv.take<int>(lmn * KMAX);
  h->counters = cv.take<int>(16384);
  h->logits = (h->tc && n >= h->lm_logits_min_rows && lm_select_parts(c.vocab) > 0)
                  ? cv.take<float>(static_cast<size_t>(n) * c.vocab)
                  : nullptr;
  const size_t nn = static_cast<size_t>(B) * h->max_nodes;
  h->node_tok = cv.take<int>(nn);
  h->node_parent = cv.take<int>(nn);
  h->node_depth = cv.take<int>(nn);
  h->node_row = cv.take<int>(nn);
  h->node_logv = cv.take<float>(nn);
  h->n_eff = cv.take<int>(B);
  h->exp_counters = cv.take<int>(B);
  h->exp_v = cv.take<float>(static_cast<size_t>(B) * 256);
  h->exp_tok = cv.take<int>(static_cast<size_t>(B) * 256);
  h->frontier = cv.take<int>(static_cast<size_t>(B) * 64);
  h->slot_mask = cv.take<unsigned long long>(static_cast<size_t>(B) * h->R);
  for (int i = 0; i < 2; ++i) {
    RowMeta& m = h->meta[i];
    m.req = cv.take<int>(n);
    m.slot = cv.take<int>(n);
    m.pos = cv.take<int>(n);
    m.tok = cv.take<int>(n);
    m.feat = cv.take<int>(n);
    m.node = cv.take<int>(n);
    m.mask = cv.take<unsigned long long>(n);
    m.v = cv.take<float>(n);
  }
  h->err = cv.take<unsigned>(64);
  *total = cv.off + 256;
}

// EAGLE-3's fused-feature GEMM takes its operand by TMA when fc's operand buffer
// ([2 n_max][2d]) holds the B rows' copy ([2B][3d]).
static bool fc3_by_tma(const eagle_draft* h, int B) {
  return 2 * static_cast<long long>(h->n_max) * 2 * h->cfg.d >= 2 * static_cast<long long>(B) * 3 * h->cfg.d &&
         h->cfg.d % 8 == 0;
}

// ------------------------------------------------------------------- create
extern "C" eagle_status_t eagle_draft_create(const eagle_draft_config_t* cfg, const eagle_draft_weights_t* weights,
                                             eagle_draft_t** out) {
  if (!cfg || !out) return fail(EAGLE_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  eagle_status_t st = validate(*cfg, weights);
  if (st != EAGLE_OK) return st;
  eagle_draft* h = new eagle_draft();
  h->cfg = *cfg;
  h->w = *weights;
  const eagle_draft_config_t& c = h->cfg;
  h->tc = c.dtype == EAGLE_DTYPE_BF16;
  h->use_graph = !(c.flags & EAGLE_FLAG_NO_GRAPH);
  h->use_pdl = !(c.flags & EAGLE_FLAG_NO_PDL);
  h->gemm_occ2 = (c.flags & EAGLE_FLAG_GEMM_TWO_CTA) != 0;
  // every depth reads the whole prefix cache again: when all of it fits in a third of L2
  // (the LM head streams past it with the evict-first hint) it is kept there
  // tuning override: EAGLE_LM_LOGITS_MIN_ROWS = the row count from which the LM head stores
  // logits for the select kernel (sweeps of the crossover); unset keeps the default
  if (const char* ov = getenv("EAGLE_LM_LOGITS_MIN_ROWS")) h->lm_logits_min_rows = std::max(1, atoi(ov));
  h->kv_keep = static_cast<double>(c.max_batch) * c.max_prefix * c.n_kv_heads * c.head_dim * 4.0 <= 40e6 ? 1 : 0;
  h->D = c.depth;
  // tree geometry
  int rb = 0, nb = 1, kmax = 0, fmax = 0, nmax_rows = 0;
  for (int s = 0; s < c.depth; ++s) {
    const int kids = c.tree_kind == EAGLE_TREE_STATIC ? c.branching[s] : c.k;
    int rows = 1;
    if (s > 0) rows = c.tree_kind == EAGLE_TREE_STATIC ? h->rows[s - 1] * h->kids[s - 1] : c.k;
    h->rows[s] = rows;
    h->kids[s] = kids;
    h->row_base[s] = rb;
    h->node_base[s] = nb;
    rb += rows;
    nb += rows * kids;
    kmax = std::max(kmax, kids);
    fmax = std::max(fmax, rows);
    nmax_rows = std::max(nmax_rows, rows);
    if (rows * kids > 256) {
      delete h;
      return fail(EAGLE_ERR_UNSUPPORTED, "more than 256 children per request at one depth");
    }
  }
  h->row_base[c.depth] = rb;
  h->node_base[c.depth] = nb;
  h->R = rb;
  h->gen = nb - 1;
  h->max_nodes = nb;
  h->S = (c.tree_kind == EAGLE_TREE_STATIC ? h->gen : c.m) + 1;
  h->k_max = kmax;
  h->f_max = fmax;
  h->n_max = c.max_batch * nmax_rows;
  if (h->R > 64) { delete h; return fail(EAGLE_ERR_UNSUPPORTED, "more than 64 rows per request"); }
  if (h->gen > 1024) { delete h; return fail(EAGLE_ERR_UNSUPPORTED, "more than 1024 generated nodes per request"); }
  if (fmax > 64) { delete h; return fail(EAGLE_ERR_UNSUPPORTED, "more than 64 rows at one depth"); }
  if (c.tree_kind == EAGLE_TREE_DYNAMIC && (c.m < 1 || c.m > h->gen))
    { delete h; return fail(EAGLE_ERR_INVALID_ARG, "m must be 1..%d (generated nodes)", h->gen); }
  if (h->S > 64) { delete h; return fail(EAGLE_ERR_UNSUPPORTED, "more than 63 kept nodes"); }
  h->max_pos = c.max_prefix + c.depth + 1;
  h->max_splits = ceil_div(c.max_prefix, ATT_CHUNK) + 1;
  h->qv_max = nmax_rows * (c.n_heads / c.n_kv_heads);
  if (static_cast<size_t>((h->qv_max + 3) & ~3) * c.head_dim > attn_merge_capacity(h->qv_max, c.head_dim)) {
    delete h;
    return fail(EAGLE_ERR_UNSUPPORTED, "too many query vectors per KV group (%d)", h->qv_max);
  }
  if (attn_smem_bytes(h->qv_max, c.head_dim) > 227 * 1024 - 64) {
    delete h;
    return fail(EAGLE_ERR_UNSUPPORTED, "too many query vectors per KV group (%d)", h->qv_max);
  }
  if (h->tc && h->n_max > 256) { delete h; return fail(EAGLE_ERR_UNSUPPORTED, "more than 256 rows per depth"); }
  // partial lists per row: the fused epilogue's one per CTA, or the select kernel's one per
  // vocabulary part
  h->lm_G = h->tc ? std::max(num_sms(), lm_select_parts(c.vocab)) : ceil_div(c.vocab, BM);
  if (h->lm_G > 256) { delete h; return fail(EAGLE_ERR_UNSUPPORTED, "more than 256 LM-head partial lists (SMs or vocabulary tiles)"); }

  cudaError_t e = cudaSuccess;
  if ((e = gemm_setup_attributes()) != cudaSuccess || (e = attn_setup_attributes()) != cudaSuccess ||
      (e = tree_setup_attributes()) != cudaSuccess) {
    delete h;
    return fail(EAGLE_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  }
  if (h->tc) {
    const int d = c.d, ff = c.d_ff, hq = c.n_heads * c.head_dim;
    const int qkv = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
    bool ok = make_weight_map(&h->tm_fc, h->w.w_fc, d, 2 * d) && make_weight_map(&h->tm_qkv, h->w.w_qkv, qkv, d) &&
              make_weight_map(&h->tm_o, h->w.w_o, d, hq) && make_weight_map(&h->tm_gate, h->w.w_gate, ff, d, BM / 2) &&
              make_weight_map(&h->tm_up, h->w.w_up, ff, d, BM / 2) && make_weight_map(&h->tm_down, h->w.w_down, d, ff) &&
              make_weight_map(&h->tm_lm, h->w.w_lm, c.vocab, d);
    if (ok && c.feat_kind == EAGLE_FEAT_FUSED) ok = make_weight_map(&h->tm_fc3, h->w.w_fc3, d, 3 * d);
    if (!ok) { delete h; return fail(EAGLE_ERR_CUDA, "cuTensorMapEncodeTiled failed (weights must be 16-byte aligned)"); }
  }
  size_t total = 0;
  carve(h, nullptr, &total);
  if (fault_injected("alloc")) {
    delete h;
    return fail(EAGLE_ERR_OOM, "workspace of %zu bytes (failure injected by EAGLE_FAULT=alloc)", total);
  }
  if (cudaMalloc(&h->ws, total) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return fail(EAGLE_ERR_OOM, "workspace of %zu bytes", total);
  }
  h->ws_bytes = total;
  carve(h, static_cast<char*>(h->ws), &total);
  if ((e = cudaMemset(h->ws, 0, h->ws_bytes)) != cudaSuccess) {
    cudaFree(h->ws);
    delete h;
    return fail(EAGLE_ERR_CUDA, "cudaMemset: %s", cudaGetErrorString(e));
  }
  // rotary tables: angle = pos * theta^(-2j/hd), evaluated in double
  {
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
      return fail(EAGLE_ERR_CUDA, "rope table upload");
    }
  }
  if ((e = cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking)) != cudaSuccess) {
    cudaFree(h->ws);
    delete h;
    return fail(EAGLE_ERR_CUDA, "cudaStreamCreate: %s", cudaGetErrorString(e));
  }
  h->launches = 1 + (c.feat_kind == EAGLE_FEAT_FUSED ? 1 : 0) + (h->tc ? 9 : 8) * c.depth + 1;
  if (h->tc && c.feat_kind == EAGLE_FEAT_FUSED && fc3_by_tma(h, c.max_batch)) h->launches += 1;   // fc3's operand copy
  if (h->tc)   // LM heads over more than 128 rows run as several launches (at max_batch), and
               // those over many rows add one select launch each
    for (int s = 0; s < h->D; ++s) {
      const int N = c.max_batch * h->rows[s], parts = ceil_div(N, MAX_ROWS_PER_BLOCK);
      // the LM head (+ a select per launch when it stores logits); up to 256 rows run as one
      // launch of CTA pairs
      const int launches = N <= 2 * MAX_ROWS_PER_BLOCK ? 1 : parts;
      h->launches += launches - 1 + (N >= h->lm_logits_min_rows && lm_select_parts(c.vocab) > 0 ? launches : 0);
    }
  *out = h;
  return EAGLE_OK;
}

extern "C" void eagle_draft_destroy(eagle_draft_t* h) {
  if (!h) return;
  if (h->graph) cudaGraphExecDestroy(h->graph);
  for (cudaEvent_t e : h->ev_pool) cudaEventDestroy(e);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  if (h->ws) cudaFree(h->ws);
  delete h;
}

extern "C" const char* eagle_draft_last_error(void) { return g_last_error.c_str(); }

// Lets the other translation units of the library report through eagle_draft_last_error().
void eagle::set_last_error(const char* msg) { g_last_error = msg; }

extern "C" eagle_status_t eagle_draft_query(const eagle_draft_t* h, eagle_draft_info_t* info) {
  if (!h || !info) return fail(EAGLE_ERR_INVALID_ARG, "null argument");
  info->slots = h->S;
  info->generated = h->gen;
  info->rows = h->R;
  info->n_max = h->n_max;
  info->k_max = h->k_max;
  info->f_max = h->f_max;
  info->launches_per_tree = h->launches;
  info->tensor_core_gemm = h->tc ? 1 : 0;
  info->workspace_bytes = static_cast<int64_t>(h->ws_bytes);
  return EAGLE_OK;
}

extern "C" eagle_status_t eagle_draft_check(eagle_draft_t* h, uint32_t* word) {
  if (!h) return fail(EAGLE_ERR_INVALID_ARG, "null handle");
  CU(cudaDeviceSynchronize());
  unsigned w = 0;
  CU(cudaMemcpy(&w, h->err, sizeof(unsigned), cudaMemcpyDeviceToHost));
  if (word) *word = w;
  if (w) {
    CU(cudaMemset(h->err, 0, sizeof(unsigned)));
    if (w & DEVERR_TIMEOUT) {
      // a GEMM CTA that gave up never arrived on its split tiles' counters: clear them (and
      // the expansion's) so that the next call starts from zero
      CU(cudaMemset(h->counters, 0, sizeof(int) * 16384));
      CU(cudaMemset(h->exp_counters, 0, sizeof(int) * h->cfg.max_batch));
    }
    return fail(EAGLE_ERR_DEVICE, "device error word 0x%x", w);
  }
  return EAGLE_OK;
}

extern "C" eagle_status_t eagle_draft_set_wait_limit(eagle_draft_t* h, int64_t cycles) {
  if (!h || cycles < 0) return fail(EAGLE_ERR_INVALID_ARG, "null handle or negative limit");
  if (h->wait_limit != cycles && h->graph) {   // the limit is a kernel argument of the cached graph
    cudaGraphExecDestroy(h->graph);
    h->graph = nullptr;
  }
  h->wait_limit = cycles;
  return EAGLE_OK;
}


// ------------------------------------------------------------- GEMM setup
static GemmPlan base_plan(eagle_draft* h, const CUtensorMap& tm0, const CUtensorMap* tm1, const void* w0,
                          const void* w1, int M, int K, int m_split) {
  GemmPlan p = gemm_plan(h->tc, tm0, tm1, w0, w1, M, K, m_split, h->part, h->counters, h->err);
  p.args.wait_limit = h->wait_limit;
  return p;
}

// split-K scratch of one rank of a CTA pair (the buffer holds two)
static size_t part_half() { return static_cast<size_t>(num_sms() / 2) * 2 * MAX_ROWS_PER_BLOCK * BM; }

static eagle_status_t run_gemm(eagle_draft* h, GemmPlan& p, int N, cudaStream_t st, int kind) {
  const EpiKind ek = static_cast<EpiKind>(p.args.e.kind);
  if (p.tc && p.args.b_tma && N > MAX_ROWS_PER_BLOCK && N <= 2 * MAX_ROWS_PER_BLOCK &&
      (ek == EPI_STORE || ek == EPI_QKV || ek == EPI_SWIGLU || ek == EPI_LOGITS)) {
    // up to 256 rows: one launch of CTA pairs, each weight stage loaded once for both halves
    GemmPlan q = p;
    if (plan_gemm_pair(q, N, part_half())) {
      ProfScope ps(h, kind, st);
      CU(launch_gemm(q, st, h->use_pdl && !h->profiling));
      return EAGLE_OK;
    }
  }
  if (!plan_gemm(p, N)) return fail(EAGLE_ERR_UNSUPPORTED, "GEMM M=%d K=%d N=%d does not fit", p.args.M, p.args.K, N);
  ProfScope ps(h, kind, st);
  CU(launch_gemm(p, st, h->use_pdl && !h->profiling));
  return EAGLE_OK;
}

static LmPartials lm_partials(eagle_draft* h, int N);
static LmPartials lm_partials(eagle_draft* h, int N, bool via_logits);

// Sampled drafting of the LM head's top-k: per-request seeds, rows per request and depth.
struct SampleArgs {
  const unsigned long long* seeds = nullptr;
  int rows = 1, depth = 0;
};

static void set_sampling(EpiArgs& e, const SampleArgs& sa, int row0) {
  e.seeds = sa.seeds;
  e.sample_rows = sa.rows;
  e.sample_depth = sa.depth;
  e.sample_row0 = row0;
}

static bool lm_via_logits(const eagle_draft* h, const uint16_t* a_hl, int N) {
  return h->logits && a_hl && N >= h->lm_logits_min_rows;
}

static eagle_status_t lm_head(eagle_draft* h, const float* a, const uint16_t* a_hl, int N, int topk,
                              cudaStream_t st, const SampleArgs& sa = SampleArgs()) {
  const eagle_draft_config_t& c = h->cfg;
  if (lm_via_logits(h, a_hl, N)) {
    const LmPartials lm = lm_partials(h, N, true);
    if (N > MAX_ROWS_PER_BLOCK && N <= 2 * MAX_ROWS_PER_BLOCK) {
      // one launch of CTA pairs storing the logits of all rows (the LM head streamed once),
      // then the select kernel over them
      GemmPlan p = base_plan(h, h->tm_lm, nullptr, h->w.w_lm, nullptr, c.vocab, c.d, c.vocab);
      tma_operand(p, a_hl);
      p.args.e.kind = EPI_LOGITS;
      p.args.e.logits = h->logits;
      eagle_status_t r = run_gemm(h, p, N, st, EAGLE_K_LMHEAD);
      if (r != EAGLE_OK) return r;
      ProfScope ps(h, EAGLE_K_LM_SELECT, st);
      CU(launch_lm_select(h->logits, N, c.vocab, topk, sa.seeds, sa.rows, sa.depth, 0, lm, st,
                          h->use_pdl && !h->profiling));
      return EAGLE_OK;
    }
    // launches of <= 128 rows (double-buffered accumulators) that store the logits, each
    // followed by the select kernel over its rows
    const int parts = ceil_div(N, MAX_ROWS_PER_BLOCK), per = ceil_div(N, parts);
    for (int r0 = 0; r0 < N; r0 += per) {
      const int n = std::min(per, N - r0);
      GemmPlan p = base_plan(h, h->tm_lm, nullptr, h->w.w_lm, nullptr, c.vocab, c.d, c.vocab);
      tma_operand(p, a_hl + 2 * static_cast<size_t>(r0) * c.d);
      EpiArgs& e = p.args.e;
      e.kind = EPI_LOGITS;
      e.logits = h->logits + static_cast<size_t>(r0) * c.vocab;
      eagle_status_t r = run_gemm(h, p, n, st, EAGLE_K_LMHEAD);
      if (r != EAGLE_OK) return r;
      ProfScope ps(h, EAGLE_K_LM_SELECT, st);
      CU(launch_lm_select(h->logits + static_cast<size_t>(r0) * c.vocab, n, c.vocab, topk, sa.seeds, sa.rows,
                          sa.depth, r0, lm, st, h->use_pdl && !h->profiling));
    }
    return EAGLE_OK;
  }
  if (a_hl && N > MAX_ROWS_PER_BLOCK) {
    // More rows than one TMEM accumulator pair holds: launches of <= 128 rows each, so the
    // accumulators stay double-buffered (the top-k epilogue of one tile overlaps the next
    // tile's MMAs); the partials of each launch land at its rows' offsets.
    const int parts = ceil_div(N, MAX_ROWS_PER_BLOCK), per = ceil_div(N, parts);
    const long long T = ceil_div(c.vocab, BM), G = lm_partials(h, N).G;
    for (int r0 = 0; r0 < N; r0 += per) {
      const int n = std::min(per, N - r0);
      GemmPlan p = base_plan(h, h->tm_lm, nullptr, h->w.w_lm, nullptr, c.vocab, c.d, c.vocab);
      p.args.b.mode = B_F32;
      p.args.b.x = a + static_cast<size_t>(r0) * c.d;
      p.args.b.ldx = c.d;
      tma_operand(p, a_hl + 2 * static_cast<size_t>(r0) * c.d);
      EpiArgs& e = p.args.e;
      e.kind = EPI_LMHEAD;
      e.lm_max = h->lm_max + r0 * T;
      e.lm_sum = h->lm_sum + r0 * T;
      e.lm_val = h->lm_val + r0 * G * topk;
      e.lm_id = h->lm_id + r0 * G * topk;
      e.topk = topk;
      set_sampling(e, sa, r0);
      eagle_status_t r = run_gemm(h, p, n, st, EAGLE_K_LMHEAD);
      if (r != EAGLE_OK) return r;
    }
    return EAGLE_OK;
  }
  GemmPlan p = base_plan(h, h->tm_lm, nullptr, h->w.w_lm, nullptr, c.vocab, c.d, c.vocab);
  p.args.b.mode = B_F32;
  p.args.b.x = a;
  p.args.b.ldx = c.d;
  if (a_hl) tma_operand(p, a_hl);
  EpiArgs& e = p.args.e;
  e.kind = EPI_LMHEAD;
  e.lm_max = h->lm_max;
  e.lm_sum = h->lm_sum;
  e.lm_val = h->lm_val;
  e.lm_id = h->lm_id;
  e.topk = topk;
  set_sampling(e, sa, 0);
  return run_gemm(h, p, N, st, EAGLE_K_LMHEAD);
}

static LmPartials lm_partials(eagle_draft* h, int N, bool via_logits) {
  LmPartials lm;
  lm.poison_if = nullptr;   // the handle reports kernel-side problems through eagle_draft_check
  lm.max = h->lm_max;
  lm.sum = h->lm_sum;
  lm.val = h->lm_val;
  lm.id = h->lm_id;
  if (via_logits) {   // one list and one log-sum-exp state per vocabulary part
    lm.T = lm.G = lm_select_parts(h->cfg.vocab);
    return lm;
  }
  lm.T = ceil_div(h->cfg.vocab, BM);
  lm.G = h->tc ? std::min<long long>(num_sms(), static_cast<long long>(ceil_div(h->cfg.vocab, BM)) * ceil_div(h->cfg.d, BK))
               : ceil_div(h->cfg.vocab, BM);
  (void)N;
  return lm;
}

static LmPartials lm_partials(eagle_draft* h, int N) { return lm_partials(h, N, false); }

// ------------------------------------------------------- the launch sequence
static eagle_status_t enqueue_tree(eagle_draft* h, const eagle_draft_inputs_t* in, const eagle_draft_outputs_t* out,
                                   const eagle_draft_trace_t* trc, cudaStream_t st) {
  const eagle_draft_config_t& c = h->cfg;
  const int B = in->B, d = c.d, hq = c.n_heads * c.head_dim, ff = c.d_ff;
  const bool pdl = h->use_pdl && !h->profiling;
  TreeArgs t;
  memset(&t, 0, sizeof(t));
  t.B = B;
  t.depth = h->D;
  t.tree_kind = c.tree_kind == EAGLE_TREE_STATIC ? 1 : 2;
  t.k = c.k;
  t.m = c.m;
  t.slots = h->S;
  for (int s = 0; s < h->D; ++s) {
    t.kids[s] = h->kids[s];
    t.rows[s] = h->rows[s];
  }
  for (int s = 0; s <= h->D; ++s) {
    t.row_base[s] = h->row_base[s];
    t.node_base[s] = h->node_base[s];
  }
  t.tree_rows = h->R;
  t.max_nodes = h->max_nodes;
  t.max_prefix = c.max_prefix;
  t.vocab = c.vocab;
  t.root_tok = in->root_tok;
  t.cu_seqlens = in->cu_seqlens;
  t.seeds = reinterpret_cast<const unsigned long long*>(in->seeds);
  t.node_tok = h->node_tok;
  t.node_parent = h->node_parent;
  t.node_depth = h->node_depth;
  t.node_row = h->node_row;
  t.node_logv = h->node_logv;
  t.n_eff = h->n_eff;
  t.frontier = h->frontier;
  t.slot_mask = h->slot_mask;
  t.exp_counters = h->exp_counters;
  t.exp_v = h->exp_v;
  t.exp_tok = h->exp_tok;
  t.err = h->err;
  {
    ProfScope ps(h, EAGLE_K_INIT, st);
    CU(launch_tree_init(t, h->meta[0], st, pdl));
  }

  const float* feat0 = static_cast<const float*>(in->root_feat);
  if (c.feat_kind == EAGLE_FEAT_FUSED) {
    // EAGLE-3: g = FC([l; m; h]) for the verified position of every request
    GemmPlan p = base_plan(h, h->tm_fc3, nullptr, h->w.w_fc3, nullptr, d, 3 * d, d);
    if (h->tc && fc3_by_tma(h, B)) {
      // the rows' operand copy (bf16: hi = the value, lo = 0) in fc's operand buffer (fc's
      // own copy overwrites it after this GEMM), then a TMA operand like every other GEMM
      p.args.b.mode = B_BF16;
      p.args.b.xb = static_cast<const uint16_t*>(in->root_feat);
      {
        ProfScope ps(h, EAGLE_K_FC_OPERAND, st);
        CU(launch_bf16_operand(static_cast<const uint16_t*>(in->root_feat), B, 3 * d, 3 * d, h->fc_hl, st, pdl));
      }
      tma_operand(p, h->fc_hl, h->gemm_occ2);
    } else if (h->tc) {
      p.args.b.mode = B_BF16;
      p.args.b.xb = static_cast<const uint16_t*>(in->root_feat);
    } else {
      p.args.b.mode = B_F32;
      p.args.b.x = static_cast<const float*>(in->root_feat);
    }
    p.args.b.ldx = 3 * d;
    p.args.e = epi_store(h->g_root, d, nullptr, 0, nullptr, 0);
    eagle_status_t r = run_gemm(h, p, B, st, EAGLE_K_FC3);
    if (r != EAGLE_OK) return r;
    feat0 = h->g_root;
  }

  const size_t nmax = h->n_max;
  for (int s = 1; s <= h->D; ++s) {
    const int rows = h->rows[s - 1], N = B * rows;
    const RowMeta& cur = h->meta[(s - 1) & 1];
    const RowMeta& nxt = h->meta[s & 1];
    const float* a_prev = s == 1 ? feat0 : h->a[(s - 2) & 1];
    float* a_cur = h->a[(s - 1) & 1];
    eagle_status_t r;
    // fc over [feat ; emb(tok)]
    {
      GemmPlan p = base_plan(h, h->tm_fc, nullptr, h->w.w_fc, nullptr, d, 2 * d, d);
      if (h->tc) {
        // the rows' operand copy (gather + hi/lo split) once, then a TMA operand like
        // every other projection
        FcOperandArgs fo;
        fo.N = N;
        fo.d = d;
        fo.vocab = c.vocab;
        fo.row_feat = cur.feat;
        fo.row_tok = cur.tok;
        fo.feat = s == 1 ? a_prev : nullptr;
        fo.ldf = d;
        fo.feat_hl = s == 1 ? nullptr : h->a_hl;
        fo.emb = static_cast<const uint16_t*>(h->w.embed);
        fo.out = h->fc_hl;
        {
          ProfScope ps(h, EAGLE_K_FC_OPERAND, st);
          CU(launch_fc_operand(fo, st, pdl));
        }
        tma_operand(p, h->fc_hl, h->gemm_occ2);
      } else {
        BSrc& b = p.args.b;
        b.mode = B_FC;
        b.x = a_prev;
        b.ldx = d;
        b.split = d;
        b.row_feat = cur.feat;
        b.row_tok = cur.tok;
        b.emb = h->w.embed;
        b.emb_bf16 = 0;
      }
      p.args.e = epi_store(h->h, d, nullptr, 0, h->ss_h, static_cast<int>(nmax));
      if (h->tc) write_operand(p.args.e, h->xa_hl, d, h->w.attn_norm);
      if ((r = run_gemm(h, p, N, st, EAGLE_K_FC)) != EAGLE_OK) return r;
    }
    // RMSNorm + QKV + rotary
    {
      const int qkv = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
      GemmPlan p = base_plan(h, h->tm_qkv, nullptr, h->w.w_qkv, nullptr, qkv, d, qkv);
      BSrc& b = p.args.b;
      b.mode = B_NORM;
      b.x = h->h;
      b.ldx = d;
      b.ss = h->ss_h;
      b.ss_tiles = ceil_div(d, BM);
      b.ss_ld = static_cast<int>(nmax);
      b.gamma = h->w.attn_norm;
      b.eps = c.rms_eps;
      b.dnorm = d;
      EpiArgs& e = p.args.e;
      memset(&e, 0, sizeof(e));
      e.kind = EPI_QKV;
      e.q = h->q;
      e.tk = h->tk;
      e.tv = h->tv;
      e.row_req = cur.req;
      e.row_slot = cur.slot;
      e.row_pos = cur.pos;
      e.rope_cos = h->rope_cos;
      e.rope_sin = h->rope_sin;
      e.max_pos = h->max_pos;
      e.Hq = c.n_heads;
      e.Hkv = c.n_kv_heads;
      e.hd = c.head_dim;
      e.tree_rows = h->R;
      if (h->tc) {
        tma_operand(p, h->xa_hl, h->gemm_occ2);
        factored_norm(e, h->ss_h, ceil_div(d, BM), static_cast<int>(nmax), d, c.rms_eps);
      }
      if ((r = run_gemm(h, p, N, st, EAGLE_K_QKV)) != EAGLE_OK) return r;
    }
    // tree-masked attention
    {
      AttnArgs a;
      memset(&a, 0, sizeof(a));
      a.q = h->q;
      a.k_cache = in->k_cache;
      a.v_cache = in->v_cache;
      a.cache_bf16 = h->tc ? 1 : 0;
      a.cu_seqlens = in->cu_seqlens;
      a.n_eff = h->n_eff;
      a.max_prefix = c.max_prefix;
      a.tk = h->tk;
      a.tv = h->tv;
      a.row_mask = cur.mask;
      a.rows_per_req = rows;
      a.tree_rows = h->R;
      a.tree_upto = h->row_base[s];
      a.B = B;
      a.Hq = c.n_heads;
      a.Hkv = c.n_kv_heads;
      a.hd = c.head_dim;
      a.max_splits = h->max_splits;
      a.out = h->o;
      a.out_hl = h->tc ? h->o_hl : nullptr;
      a.kv_keep = h->kv_keep;
      a.wait_limit = h->wait_limit;
      a.err = h->err;
      ProfScope ps(h, EAGLE_K_ATTN, st);
      if (s == std::min(2, h->D) && fault_injected("launch"))
        return fail(EAGLE_ERR_CUDA, "launch_attention failed: injected by EAGLE_FAULT=launch (depth %d)", s);
      CU(launch_attention(a, st, pdl));
    }
    // O projection + residual
    {
      GemmPlan p = base_plan(h, h->tm_o, nullptr, h->w.w_o, nullptr, d, hq, d);
      p.args.b.mode = B_F32;
      p.args.b.x = h->o;
      p.args.b.ldx = hq;
      p.args.e = epi_store(h->y, d, h->h, d, h->ss_y, static_cast<int>(nmax));
      if (h->tc) {
        tma_operand(p, h->o_hl, h->gemm_occ2);
        write_operand(p.args.e, h->xm_hl, d, h->w.mlp_norm);
      }
      if ((r = run_gemm(h, p, N, st, EAGLE_K_OPROJ)) != EAGLE_OK) return r;
    }
    // RMSNorm + gate | up; the tensor-core path emits silu(g) * u directly
    {
      GemmPlan p = h->tc ? base_plan(h, h->tm_gate, &h->tm_up, nullptr, nullptr, 2 * ff, d, 2 * ff)
                         : base_plan(h, h->tm_gate, &h->tm_up, h->w.w_gate, h->w.w_up, 2 * ff, d, ff);
      BSrc& b = p.args.b;
      b.mode = B_NORM;
      b.x = h->y;
      b.ldx = d;
      b.ss = h->ss_y;
      b.ss_tiles = ceil_div(d, BM);
      b.ss_ld = static_cast<int>(nmax);
      b.gamma = h->w.mlp_norm;
      b.eps = c.rms_eps;
      b.dnorm = d;
      if (h->tc) {
        p.args.a_pair = 1;
        p.args.e = epi_store(nullptr, ff, nullptr, 0, nullptr, 0);
        p.args.e.kind = EPI_SWIGLU;
        tma_operand(p, h->xm_hl, h->gemm_occ2);
        factored_norm(p.args.e, h->ss_y, ceil_div(d, BM), static_cast<int>(nmax), d, c.rms_eps);
        write_operand(p.args.e, h->s_hl, ff, nullptr);
      } else {
        p.args.e = epi_store(h->gu, 2 * ff, nullptr, 0, nullptr, 0);
      }
      if ((r = run_gemm(h, p, N, st, EAGLE_K_GATEUP)) != EAGLE_OK) return r;
    }
    // down projection of silu(g) * u + residual -> the next feature
    {
      GemmPlan p = base_plan(h, h->tm_down, nullptr, h->w.w_down, nullptr, d, ff, d);
      BSrc& b = p.args.b;
      if (h->tc) {
        tma_operand(p, h->s_hl, h->gemm_occ2);
      } else {
        b.mode = B_SWIGLU;
        b.x = h->gu;
        b.ldx = 2 * ff;
        b.split = ff;
      }
      p.args.e = epi_store(a_cur, d, h->y, d, nullptr, 0);
      if (h->tc) write_operand(p.args.e, h->a_hl, d, nullptr);
      if ((r = run_gemm(h, p, N, st, EAGLE_K_DOWN)) != EAGLE_OK) return r;
    }
    // frozen LM head: online log-sum-exp + top-k partials
    SampleArgs sa;
    sa.seeds = t.seeds;
    sa.rows = rows;
    sa.depth = s;
    if ((r = lm_head(h, a_cur, h->tc ? h->a_hl : nullptr, N, h->kids[s - 1], st, sa)) != EAGLE_OK) return r;
    // children, values, next frontier
    {
      ExpandTrace tr;
      memset(&tr, 0, sizeof(tr));
      tr.k_max = h->k_max;
      if (trc) {
        const size_t o = static_cast<size_t>(s - 1) * nmax;
        if (trc->children) tr.children = trc->children + o * h->k_max;
        if (trc->child_logp) tr.child_logp = trc->child_logp + o * h->k_max;
        if (trc->lse) tr.lse = trc->lse + o;
        if (trc->frontier) tr.frontier = trc->frontier + static_cast<size_t>(s - 1) * c.max_batch * h->f_max;
      }
      tr.f_max = h->f_max;
      ProfScope ps(h, EAGLE_K_EXPAND, st);
      CU(launch_expand(t, s, lm_partials(h, N, lm_via_logits(h, h->tc ? h->a_hl : nullptr, N)), cur, nxt, tr, st,
                       pdl));
    }
    if (trc) {
      const size_t o = static_cast<size_t>(s - 1) * nmax;
      if (trc->h) CU(cudaMemcpyAsync(trc->h + o * d, h->h, sizeof(float) * N * d, cudaMemcpyDeviceToDevice, st));
      if (trc->q) CU(cudaMemcpyAsync(trc->q + o * hq, h->q, sizeof(float) * N * hq, cudaMemcpyDeviceToDevice, st));
      if (trc->attn) CU(cudaMemcpyAsync(trc->attn + o * hq, h->o, sizeof(float) * N * hq, cudaMemcpyDeviceToDevice, st));
      if (trc->y) CU(cudaMemcpyAsync(trc->y + o * d, h->y, sizeof(float) * N * d, cudaMemcpyDeviceToDevice, st));
      if (trc->a) CU(cudaMemcpyAsync(trc->a + o * d, a_cur, sizeof(float) * N * d, cudaMemcpyDeviceToDevice, st));
    }
  }
  OutArgs o;
  o.tokens = out->tokens;
  o.parents = out->parents;
  o.positions = out->positions;
  o.logv = out->logv;
  o.mask = out->mask;
  o.final_nodes = trc ? trc->final_nodes : nullptr;
  {
    ProfScope ps(h, EAGLE_K_RERANK, st);
    CU(launch_rerank(t, o, st, pdl));
  }
  if (trc && (trc->tree_k || trc->tree_v)) {
    const size_t n = static_cast<size_t>(B) * h->R * c.n_kv_heads * c.head_dim;
    if (trc->tree_k) CU(cudaMemcpyAsync(trc->tree_k, h->tk, n * 4, cudaMemcpyDeviceToDevice, st));
    if (trc->tree_v) CU(cudaMemcpyAsync(trc->tree_v, h->tv, n * 4, cudaMemcpyDeviceToDevice, st));
  }
  return EAGLE_OK;
}

extern "C" eagle_status_t eagle_draft_tree(eagle_draft_t* h, const eagle_draft_inputs_t* in,
                                           const eagle_draft_outputs_t* out, const eagle_draft_trace_t* trc,
                                           void* stream) {
  if (!h || !in || !out) return fail(EAGLE_ERR_INVALID_ARG, "null argument");
  if (in->B < 1 || in->B > h->cfg.max_batch) return fail(EAGLE_ERR_INVALID_ARG, "B=%d outside 1..%d", in->B, h->cfg.max_batch);
  if (!in->root_feat || !in->root_tok || !in->cu_seqlens || (h->cfg.max_prefix > 0 && (!in->k_cache || !in->v_cache)))
    return fail(EAGLE_ERR_INVALID_ARG, "null input pointer");
  if (!out->tokens || !out->parents || !out->positions || !out->logv || !out->mask)
    return fail(EAGLE_ERR_INVALID_ARG, "null output pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (h->profiling && !trc) {
    // one-off graph holding the kernels and their event-record nodes: the GPU runs the
    // kernels back to back, so the events time the kernels and not the host in between
    CU(cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal));
    eagle_status_t r = enqueue_tree(h, in, out, nullptr, h->cap_stream);
    cudaGraph_t g = nullptr;
    cudaError_t ec = cudaStreamEndCapture(h->cap_stream, &g);
    if (r != EAGLE_OK) {
      if (g) cudaGraphDestroy(g);
      return r;
    }
    if (ec != cudaSuccess) return fail(EAGLE_ERR_CUDA, "stream capture: %s", cudaGetErrorString(ec));
    cudaGraphExec_t ge = nullptr;
    ec = cudaGraphInstantiate(&ge, g, 0);
    cudaGraphDestroy(g);
    if (ec != cudaSuccess) return fail(EAGLE_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(ec));
    ec = cudaGraphLaunch(ge, st);
    cudaGraphExecDestroy(ge);
    if (ec != cudaSuccess) return fail(EAGLE_ERR_CUDA, "graph launch: %s", cudaGetErrorString(ec));
    return EAGLE_OK;
  }
  if (trc || !h->use_graph) return enqueue_tree(h, in, out, trc, st);
  std::vector<const void*> key = {reinterpret_cast<const void*>(static_cast<intptr_t>(in->B)), in->root_feat,
                                  in->root_tok, in->k_cache, in->v_cache, in->cu_seqlens, in->seeds, out->tokens,
                                  out->parents, out->positions, out->logv, out->mask};
  if (!h->graph || key != h->graph_key) {
    if (h->graph) {
      cudaGraphExecDestroy(h->graph);
      h->graph = nullptr;
    }
    CU(cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeThreadLocal));
    eagle_status_t r = enqueue_tree(h, in, out, nullptr, h->cap_stream);
    cudaGraph_t g = nullptr;
    cudaError_t ec = cudaStreamEndCapture(h->cap_stream, &g);
    if (r != EAGLE_OK) {
      if (g) cudaGraphDestroy(g);
      return r;
    }
    if (ec != cudaSuccess) return fail(EAGLE_ERR_CUDA, "stream capture: %s", cudaGetErrorString(ec));
    ec = cudaGraphInstantiate(&h->graph, g, 0);
    cudaGraphDestroy(g);
    if (ec != cudaSuccess) {
      h->graph = nullptr;
      return fail(EAGLE_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(ec));
    }
    h->graph_key = key;
  }
  CU(cudaGraphLaunch(h->graph, st));
  return EAGLE_OK;
}

extern "C" eagle_status_t eagle_draft_lm_head_topk(eagle_draft_t* h, const float* a, int32_t N, int32_t k,
                                                   int32_t* ids, float* logp, float* lse, void* stream) {
  if (!h || !a || !ids || !logp || !lse) return fail(EAGLE_ERR_INVALID_ARG, "null argument");
  if (N < 1 || N > h->n_max) return fail(EAGLE_ERR_INVALID_ARG, "N=%d outside 1..%d", N, h->n_max);
  if (k < 1 || k > KMAX) return fail(EAGLE_ERR_INVALID_ARG, "k=%d outside 1..%d", k, KMAX);
  if (reinterpret_cast<uintptr_t>(a) % 16) return fail(EAGLE_ERR_INVALID_ARG, "a must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  eagle_status_t r = lm_head(h, a, nullptr, N, k, st);
  if (r != EAGLE_OK) return r;
  ProfScope ps(h, EAGLE_K_MERGE, st);
  CU(launch_lm_merge(lm_partials(h, N), N, k, ids, logp, lse, st, h->use_pdl && !h->profiling));
  return EAGLE_OK;
}

extern "C" eagle_status_t eagle_draft_profile(eagle_draft_t* h, int32_t enable) {
  if (!h) return fail(EAGLE_ERR_INVALID_ARG, "null handle");
  h->profiling = enable != 0;
  return EAGLE_OK;
}

extern "C" eagle_status_t eagle_draft_profile_read(eagle_draft_t* h, float* ms, int32_t* launches) {
  if (!h || !ms || !launches) return fail(EAGLE_ERR_INVALID_ARG, "null argument");
  for (int i = 0; i < EAGLE_K_COUNT; ++i) {
    ms[i] = 0.f;
    launches[i] = 0;
  }
  if (h->ev_used) CU(cudaEventSynchronize(h->ev_pool[h->ev_used - 1]));
  for (size_t i = 0; i < h->ev_kind.size(); ++i) {
    float t = 0.f;
    CU(cudaEventElapsedTime(&t, h->ev_pool[2 * i], h->ev_pool[2 * i + 1]));
    ms[h->ev_kind[i]] += t;
    launches[h->ev_kind[i]] += 1;
  }
  h->ev_used = 0;
  h->ev_kind.clear();
  return EAGLE_OK;
}

extern "C" const char* eagle_draft_kernel_name(int32_t kind) {
  return (kind >= 0 && kind < EAGLE_K_COUNT) ? kKernelNames[kind] : "?";
}
