// Host-side declarations shared by the translation units of the library.
#pragma once

#include "common.cuh"

namespace eagle {

// Message returned by eagle_draft_last_error() on this thread.
void set_last_error(const char* msg);

// ----------------------------------------------------------------- GEMM
struct GemmPlan {
  bool tc = false;               // tcgen05 mainloop (bf16 weights) or SIMT (f32 weights)
  CUtensorMap tm0, tm1;          // weight maps (tc): rows [0, m_split) and [m_split, M)
  CUtensorMap tmB;               // activation operand copy (tc, args.b_tma)
  const uint16_t* b_hl = nullptr;  // its base: bf16 [2 N][K], rows 2r / 2r+1 = hi / lo of row r
  const float* w0f = nullptr;    // f32 weights (simt)
  const float* w1f = nullptr;
  GemmArgs args{};
  int grid = 0, grid_y = 1;
  size_t smem = 0;
  int occ = 1;                   // tc with TMA operand: 2 = two CTAs per SM (smaller ring)
  bool stream_k = false;         // force the stream-K schedule (no per-tile CTA clusters)
  // pair: clusters of two CTAs sharing the weight stream, rank 1 on the rows of args1 / tmB1
  bool pair = false;
  GemmArgs args1{};
  CUtensorMap tmB1;
};

// Plans GEMM p over N > 128 rows (TMA operand, STORE / QKV / SWIGLU / LOGITS epilogue) as one
// launch of CTA pairs: rank 0 on the first ceil(N/2) rows, rank 1 on the rest, each weight
// stage loaded once for both.  `part_half` floats of split-K scratch and 8192 counters apart
// per rank.  Returns false when the shape does not fit.
bool plan_gemm_pair(GemmPlan& p, int N, size_t part_half);

// Allow `func` the device's opt-in maximum of dynamic shared memory (minus its static use).
cudaError_t allow_max_smem(const void* func, size_t* granted = nullptr);
size_t max_dyn_smem(const void* func);

bool make_weight_map(CUtensorMap* tm, const void* w, int M, int K, int box_rows = BM);
// 3-D map over a bf16 prefix cache [tokens][Hkv][128]: boxes of 64 tokens x 64 dims of one
// KV head, 128-byte swizzle (the attention kernel's key / value tiles).
bool make_kv_map(CUtensorMap* tm, const void* cache, long long tokens, int Hkv);

// A GEMM over weights [M][K] (rows [0, m_split) from map / pointer 0, the rest from 1),
// with the caller's split-K scratch, arrival counters and device error word.
GemmPlan gemm_plan(bool tc, const CUtensorMap& tm0, const CUtensorMap* tm1, const void* w0, const void* w1,
                   int M, int K, int m_split, float* part, int* counters, unsigned* err);
// EPI_STORE epilogue: out = acc (+ resid); per-tile sums of squares into ss (nullable).
EpiArgs epi_store(float* out, int ldo, const float* resid, int ldr, float* ss, int ss_ld);
// Operand tile loaded by TMA from a bf16 hi/lo copy written by the producing kernel.
inline void tma_operand(GemmPlan& p, const uint16_t* hl, bool shared_sm = false) {
  p.args.b.mode = B_TMA;
  p.args.b_tma = 1;
  p.b_hl = hl;
  p.occ = shared_sm ? 2 : 1;
}
// The producing epilogue also writes the next GEMM's operand copy (value * gamma).
inline void write_operand(EpiArgs& e, uint16_t* hl, int ld, const float* gamma) {
  e.hl = hl;
  e.hl_ld = ld;
  e.hl_gamma = gamma;
}
// The consumer applies the RMSNorm row scale in its epilogue (per-tile sums of squares).
inline void factored_norm(EpiArgs& e, const float* ss, int tiles, int ld, int d, float eps) {
  e.nss = ss;
  e.nss_tiles = tiles;
  e.nss_ld = ld;
  e.nss_d = d;
  e.nss_eps = eps;
}
int num_sms();
int gemm_active_clusters(int S);
bool plan_gemm(GemmPlan& p, int N);
cudaError_t gemm_setup_attributes();
cudaError_t launch_gemm(const GemmPlan& p, cudaStream_t st, bool pdl);

// ------------------------------------------------------------ attention
struct AttnArgs {
  const float* q;           // [N][Hq*hd] rotated queries of this depth's rows
  const void* k_cache;      // [sum n][Hkv][hd] prefix keys (post-RoPE), bf16 or f32
  const void* v_cache;
  int cache_bf16;
  const int* cu_seqlens;    // [B+1]
  const int* n_eff;         // [B] validated prefix lengths
  int max_prefix;           // cu_seqlens lengths are clamped to [0, max_prefix]
  const float* tk;          // [B][tree_rows][Hkv][hd] rotated keys of tree rows
  const float* tv;
  const unsigned long long* row_mask;  // [N] ancestor-or-self bits over request-local rows
  int rows_per_req;         // rows of this depth per request
  int tree_rows;            // request-local row capacity
  int tree_upto;            // rows that exist so far (through this depth)
  int B, Hq, Hkv, hd;
  int max_splits;           // prefix chunks + 1 (tree chunk) of the longest request
  int row_groups;           // > 1: a request's rows run as this many groups of rows_per_group
  int rows_per_group;       // (tensor-core kernel only; 0 / 1 = one group)
  float* out;               // [N][Hq*hd]
  uint16_t* out_hl;         // [2N][Hq*hd] bf16 hi / lo rows of out (operand of the O projection)
  int kv_keep;              // tensor-core kernel: prefix tiles loaded with the L2 evict-last hint
                            // (0: evict-first; set when every request's prefix fits in L2 at once)
  long long wait_limit;     // tensor-core kernel: clock cycles a bounded wait may take (0: ~1 s)
  unsigned* err;            // tensor-core kernel: device error word (DEVERR_TIMEOUT)
};
size_t attn_smem_bytes(int qv, int hd);
size_t attn_merge_capacity(int qv, int hd);
cudaError_t attn_setup_attributes();
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t st, bool pdl);
// Largest rows_per_group the tensor-core kernel takes for Hq / Hkv query heads per KV head.
int attn_rows_per_group(int Hq, int Hkv);

// --------------------------------------------------------- tree kernels
struct TreeArgs {
  int B, depth, tree_kind, k, m, slots;
  int kids[EAGLE_MAX_DEPTH_INTERNAL];       // children per row at each depth
  int rows[EAGLE_MAX_DEPTH_INTERNAL];       // rows per request at each depth
  int row_base[EAGLE_MAX_DEPTH_INTERNAL + 1];
  int node_base[EAGLE_MAX_DEPTH_INTERNAL + 1];
  int tree_rows;            // R: rows per request over all depths
  int max_nodes;            // generated + 1 (root)
  int max_prefix;
  int vocab;
  // inputs
  const int* root_tok;
  const int* cu_seqlens;
  const unsigned long long* seeds;   // [B] sampled drafting, or null (greedy top-k)
  // node table [B][max_nodes]
  int* node_tok;
  int* node_parent;
  int* node_depth;
  int* node_row;            // request-local row that generated the node
  float* node_logv;
  // per-request state
  int* n_eff;               // [B]
  int* frontier;            // [B][64] node ids of the current frontier
  unsigned long long* slot_mask;  // [B][tree_rows] ancestor-or-self bits of every row
  int* exp_counters;        // [B] rows of the depth finished (zero between depths)
  float* exp_v;             // [B][256] values of the depth's children
  int* exp_tok;             // [B][256] their tokens
  unsigned* err;
};

// Row metadata of one depth (N = B * rows rows).
struct RowMeta {
  int* req;                 // request
  int* slot;                // request-local row id
  int* pos;                 // position id n_b + depth
  int* tok;                 // input token
  int* feat;                // feature row (index into the previous feature buffer)
  int* node;                // tree node the row expands
  unsigned long long* mask; // ancestor-or-self bits
  float* v;                 // path value V of the node
};

struct LmPartials {
  float* max;               // [N][T] per vocabulary tile
  float* sum;               // [N][T]
  float* val;               // [N][G][k] per CTA
  int* id;                  // [N][G][k]
  int G;                    // CTAs that wrote top-k partials
  int T;                    // vocabulary tiles
  const unsigned* poison_if;  // standalone merge: when this device word is non-zero (a kernel of
                              // the call gave up), every output row is poisoned instead of merged
};

struct OutArgs {
  int* tokens;
  int* parents;
  int* positions;
  float* logv;
  unsigned char* mask;
  int* final_nodes;         // trace (nullable)
};

struct ExpandTrace {
  int* children;            // [N][k_max] (nullable)
  float* child_logp;
  float* lse;               // [N]
  int* frontier;            // [B][f_max]
  int k_max;
  int f_max;
};

cudaError_t tree_setup_attributes();
cudaError_t launch_tree_init(const TreeArgs& t, const RowMeta& rows0, cudaStream_t st, bool pdl);

// The fc GEMM's tensor-core operand for one depth: row n = [feature of row row_feat[n] ;
// embedding of token row_tok[n]] as bf16 hi (row 2n) and lo (row 2n+1) parts, [2N][2d].
// The feature comes from an fp32 matrix (the roots) or from the previous depth's operand
// copy (already hi/lo); an embedding is exact in bf16 (lo = 0).
struct FcOperandArgs {
  int N, d, vocab;
  const int* row_feat;
  const int* row_tok;
  const float* feat;          // [*][ldf] fp32, or null
  int ldf;
  const uint16_t* feat_hl;    // [2 *][d] hi / lo rows, or null
  const uint16_t* emb;        // [V][d] bf16
  uint16_t* out;              // [2N][2d]
};
cudaError_t launch_fc_operand(const FcOperandArgs& a, cudaStream_t st, bool pdl);
// The operand copy of N bf16 rows x [N][K] (stride ldx; K, ldx multiples of 8): out [2N][K],
// row 2n = row n of x, row 2n + 1 = zeros (a bf16 value has no low-order part).
cudaError_t launch_bf16_operand(const uint16_t* x, int N, int K, int ldx, uint16_t* out, cudaStream_t st, bool pdl);
cudaError_t launch_expand(const TreeArgs& t, int s, const LmPartials& lm, const RowMeta& cur,
                          const RowMeta& next, const ExpandTrace& tr, cudaStream_t st, bool pdl);
cudaError_t launch_rerank(const TreeArgs& t, const OutArgs& o, cudaStream_t st, bool pdl);
cudaError_t launch_lm_merge(const LmPartials& lm, int N, int k, int* ids, float* logp, float* lse,
                            cudaStream_t st, bool pdl);
// LM head over many rows, second half: the rows' stored logits [N][vocab] -> per (row, part)
// log-sum-exp state and top-k keys (logit, or logit + Gumbel noise with seeds), written at
// rows row0.. of `lm` (G = T = lm_select_parts(vocab)).  N rows of this launch.
int lm_select_parts(int vocab);
cudaError_t launch_lm_select(const float* logits, int N, int vocab, int k, const unsigned long long* seeds,
                             int sample_rows, int sample_depth, int row0, const LmPartials& lm, cudaStream_t st,
                             bool pdl);

}  // namespace eagle
