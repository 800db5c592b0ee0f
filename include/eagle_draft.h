/*
 * eagle_draft.h - C ABI of the GB300 draft-tree expansion step for EAGLE-style
 * speculative decoding (EAGLE-1 static tree, EAGLE-2 expand-and-rerank dynamic
 * tree, EAGLE-3 fused-feature input).
 *
 * What one call computes (sources: four pages on EAGLE):
 *   - the draft recurrence x = [feat ; emb(tok)] -> fc (2d -> d) -> one decoder
 *     layer over the verified-prefix KV cache -> frozen LM head
 *     ("The recurrence, written out", aicassindra.com tm_eagle_deep; "The Mechanism",
 *     stable-lab "EAGLE: Drafting in Feature Space");
 *   - at each of `depth` sequential steps every frontier node gets its top-k children
 *     by draft probability; path value V = sum of log confidences along the path
 *     ("EAGLE-2 - context-aware dynamic tree", zackli.ai "Speculative Decoding Deep
 *     Dive III"; "EAGLE-2: expand and rerank", aicassindra.com);
 *   - static trees (EAGLE-1) expand every node with a fixed per-depth branching
 *     ("Drafting a Tree, Not a Chain", stable-lab); dynamic trees keep the top-k nodes
 *     of each depth as the next frontier and, after the last depth, the top-m of all
 *     generated nodes;
 *   - EAGLE-3: the root feature is g = FC([l; m; h]) (3d -> d); later steps feed back the
 *     draft's own output a ("EAGLE-3 - free representation + training-time test +
 *     feature fusion", zackli.ai; "Multi-layer feature fusion", aicassindra.com);
 *   - the emitted tree: token ids, parent slots, position ids and the ancestor-only
 *     attention mask ("Tree attention in one verification pass", aicassindra.com).
 *
 * Names follow the pages' notation: B requests, n verified prefix length, depth =
 * gamma, k branching, m kept nodes, d hidden size, vocab = |V|.
 *
 * Memory: every pointer below is a DEVICE pointer unless marked host.  Weights are
 * borrowed for the lifetime of the handle; inputs, outputs and trace buffers for the
 * duration of the call (the call is stream-ordered: they must stay valid until the
 * stream reaches the end of the call).  The handle owns its device workspace.
 * Errors: functions return eagle_status_t; eagle_draft_last_error() gives a
 * thread-local message.  Kernel-side problems (a prefix longer than max_prefix, a
 * wait that ran out) are recorded in a device error word that eagle_draft_check()
 * reads after synchronising.  Calls on one handle must not overlap on the GPU.
 * Tests of the error paths: EAGLE_FAULT=alloc in the environment makes eagle_draft_create's
 * workspace allocation fail (EAGLE_ERR_OOM, nothing allocated); EAGLE_FAULT=launch makes a
 * launch in the middle of eagle_draft_tree fail (EAGLE_ERR_CUDA).
 */
#ifndef EAGLE_DRAFT_H
#define EAGLE_DRAFT_H

#include <stdint.h>
#include <stddef.h>

#if defined(__GNUC__)
#define EAGLE_API __attribute__((visibility("default")))
#else
#define EAGLE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  EAGLE_OK = 0,
  EAGLE_ERR_INVALID_ARG = 1,   /* null pointer, size out of range, B > max_batch, ... */
  EAGLE_ERR_UNSUPPORTED = 2,   /* shape outside what the kernels implement */
  EAGLE_ERR_OOM = 3,           /* workspace allocation failed */
  EAGLE_ERR_CUDA = 4,          /* a CUDA runtime / driver call failed */
  EAGLE_ERR_DEVICE = 5         /* the device error word is set (see eagle_draft_check) */
} eagle_status_t;

typedef enum { EAGLE_DTYPE_F32 = 0, EAGLE_DTYPE_BF16 = 1 } eagle_dtype_t;
typedef enum { EAGLE_TREE_STATIC = 1, EAGLE_TREE_DYNAMIC = 2 } eagle_tree_kind_t;
typedef enum { EAGLE_FEAT_F = 1, EAGLE_FEAT_FUSED = 3 } eagle_feat_kind_t;

#define EAGLE_MAX_DEPTH 16

/* Device error word bits (eagle_draft_check). */
#define EAGLE_DEVERR_TIMEOUT     0x1u   /* a bounded wait inside a kernel ran out */
#define EAGLE_DEVERR_PREFIX      0x2u   /* a request's prefix length was < 0 or > max_prefix */
#define EAGLE_DEVERR_TOKEN       0x4u   /* a root token was outside [0, vocab) (treated as 0) */
#define EAGLE_DEVERR_SELECT      0x8u   /* a row had fewer than k valid next-token candidates
                                           (non-finite logits); the missing children get token 0 */

typedef struct {
  int32_t d;            /* hidden size; d % 128 == 0 for bf16 weights */
  int32_t n_heads;      /* query heads Hq */
  int32_t n_kv_heads;   /* key/value heads Hkv; Hq % Hkv == 0 (grouped-query attention) */
  int32_t head_dim;     /* hd: 128 for bf16 weights, 64 or 128 for f32 */
  int32_t d_ff;         /* SwiGLU hidden size */
  int32_t vocab;        /* |V| */
  float   rms_eps;      /* RMSNorm epsilon */
  float   rope_theta;   /* rotary base: inv_freq_i = theta^(-2i/hd), rotate-half pairs (i, i+hd/2) */
  int32_t dtype;        /* eagle_dtype_t of the weights, embedding table and KV cache */
  int32_t tree_kind;    /* eagle_tree_kind_t */
  int32_t feat_kind;    /* eagle_feat_kind_t */
  int32_t depth;        /* gamma: sequential draft steps, 1..EAGLE_MAX_DEPTH */
  int32_t k;            /* dynamic: children per expanded node and frontier width, 1..16 */
  int32_t m;            /* dynamic: nodes kept by the rerank (static trees keep all) */
  int32_t branching[EAGLE_MAX_DEPTH]; /* static: children per node at depth 1..depth, 1..16 */
  int32_t max_batch;    /* workspace sizing: largest B a call may pass */
  int32_t max_prefix;   /* workspace sizing: largest prefix length n_b a call may pass */
  int32_t flags;        /* EAGLE_FLAG_*; 0 = CUDA-graph replay and programmatic dependent launch */
} eagle_draft_config_t;

#define EAGLE_FLAG_NO_GRAPH 0x1   /* enqueue the kernels directly on every call */
#define EAGLE_FLAG_NO_PDL   0x2   /* plain stream order between kernels */
#define EAGLE_FLAG_GEMM_TWO_CTA 0x4 /* stream-K GEMMs with a TMA operand run two CTAs per SM (a smaller
                                       ring each) instead of one per SM with the full register file */

/* Weights, stored [out, in] row-major in `dtype` (the norm gains are always f32).
 * w_qkv stacks the query rows, then the key rows, then the value rows.
 * w_fc multiplies [feat ; emb(tok)] (the feature first).  w_fc3 (EAGLE-3 only) multiplies
 * [l ; m ; h].  w_lm is the frozen LM head [vocab, d]; embed the frozen table [vocab, d]. */
typedef struct {
  const void*  embed;      /* [vocab, d] */
  const void*  w_fc;       /* [d, 2d] */
  const void*  w_fc3;      /* [d, 3d] or NULL unless feat_kind == EAGLE_FEAT_FUSED */
  const float* attn_norm;  /* [d] */
  const void*  w_qkv;      /* [(Hq + 2 Hkv) hd, d] */
  const void*  w_o;        /* [d, Hq hd] */
  const float* mlp_norm;   /* [d] */
  const void*  w_gate;     /* [d_ff, d] */
  const void*  w_up;       /* [d_ff, d] */
  const void*  w_down;     /* [d, d_ff] */
  const void*  w_lm;       /* [vocab, d] */
} eagle_draft_weights_t;

/* One call's inputs (device).  The prefix KV cache is the draft layer's own cache of
 * the verified positions, packed over requests and already rotated (post-RoPE). */
typedef struct {
  int32_t        B;          /* requests, 1..max_batch */
  const void*    root_feat;  /* EAGLE-1/2: f32 [B, d] target feature f; EAGLE-3: `dtype` [B, 3d] = [l;m;h] */
  const int32_t* root_tok;   /* [B] the token sampled from f (the tree root) */
  const void*    k_cache;    /* `dtype` [sum n_b, Hkv, hd] */
  const void*    v_cache;    /* `dtype` [sum n_b, Hkv, hd] */
  const int32_t* cu_seqlens; /* [B + 1], cu_seqlens[0] = 0, n_b = cu_seqlens[b+1] - cu_seqlens[b] */
  const uint64_t* seeds;     /* [B] or NULL.  NULL: greedy drafting (each node's k most likely tokens).
                                Set: sampled drafting ("EAGLE-1 - autoregressive feature drafting",
                                zackli.ai: the draft samples t-hat ~ p-hat): a node's k children are k
                                tokens drawn without replacement from the draft's distribution, the top-k
                                of log p + Gumbel noise.  The noise of token t of frontier slot i at depth s
                                of request b is -log(-log U), U = (x + 1/2) / 2^32 with x word
                                (t mod 128) / 32 of Philox4x32-10(counter = (32 (t / 128) + t mod 32, i, s,
                                0), key = seeds[b] as (low, high) 32-bit words).  Children are then kept in
                                draw order (largest perturbed value first) instead of token order; path
                                values add the unperturbed log-probabilities. */
} eagle_draft_inputs_t;

/* Outputs (device).  S = kept + 1 slots per request (eagle_draft_info_t.slots):
 * slot 0 is the root (token root_tok, parent -1, position n_b, logv 0); slots 1.. are the
 * kept nodes in generation order (depth, then the parent's frontier slot, then token id -
 * draw order when sampling), so a parent always precedes its children. */
typedef struct {
  int32_t* tokens;     /* [B, S] */
  int32_t* parents;    /* [B, S] parent slot, -1 for the root */
  int32_t* positions;  /* [B, S] n_b + depth */
  float*   logv;       /* [B, S] path value V = sum of log draft probabilities */
  uint8_t* mask;       /* [B, S, S] mask[b][i][j] = 1 iff slot j is an ancestor of slot i or i itself */
} eagle_draft_outputs_t;

/* Optional per-depth intermediates for parity testing (any member may be NULL).
 * N_max = max_batch * max rows per depth; rows of depth s (0-based) sit at
 * [s][b * rows_s + i]; dimensions per row as named. */
typedef struct {
  float*   h;           /* [depth][N_max][d]       fc output */
  float*   q;           /* [depth][N_max][Hq*hd]   queries after rotation */
  float*   attn;        /* [depth][N_max][Hq*hd]   attention output */
  float*   y;           /* [depth][N_max][d]       after O-proj + residual */
  float*   a;           /* [depth][N_max][d]       layer output (next feature f' / latent a) */
  float*   lse;         /* [depth][N_max]          log-sum-exp of the row's logits */
  int32_t* children;    /* [depth][N_max][k_max]   children token ids (ascending; draw order when sampling) */
  float*   child_logp;  /* [depth][N_max][k_max]   their log-probabilities */
  int32_t* frontier;    /* [depth][max_batch][f_max] node ids expanded at the next depth */
  int32_t* final_nodes; /* [max_batch][S]          node id of every emitted slot */
  float*   tree_k;      /* [max_batch][R][Hkv][hd] rotated keys of every row (R rows per request) */
  float*   tree_v;      /* [max_batch][R][Hkv][hd] */
} eagle_draft_trace_t;

typedef struct {
  int32_t slots;            /* S = kept + 1 */
  int32_t generated;        /* nodes generated per request */
  int32_t rows;             /* R: draft-layer rows per request over all depths */
  int32_t n_max;            /* max_batch * max rows per depth */
  int32_t k_max;            /* max children per row over depths */
  int32_t f_max;            /* max rows per request at one depth */
  int32_t launches_per_tree;/* kernels one eagle_draft_tree launches */
  int32_t tensor_core_gemm; /* 1 when the GEMMs run on tcgen05 (bf16 weights) */
  int64_t workspace_bytes;
} eagle_draft_info_t;

typedef struct eagle_draft eagle_draft_t;

/* Validates the config, allocates the workspace, builds the TMA descriptors of the
 * weights and the rotary tables.  The current CUDA device must be the one holding the
 * weights.  Returns EAGLE_ERR_UNSUPPORTED for shapes the kernels do not implement:
 * bf16 needs d, d_ff, vocab, (Hq+2Hkv)hd multiples of 128 and hd == 128; every config
 * needs at most 64 rows per request, at most 63 kept nodes, k and branching <= 16. */
EAGLE_API eagle_status_t eagle_draft_create(const eagle_draft_config_t* cfg,
                                  const eagle_draft_weights_t* weights,
                                  eagle_draft_t** out_handle);

/* Enqueues one draft-tree expansion on `stream` (a cudaStream_t; NULL = legacy default
 * stream) and returns.  Without a trace the launches are replayed from a CUDA graph
 * captured on the first call with the same B and pointers.  `trace` may be NULL. */
EAGLE_API eagle_status_t eagle_draft_tree(eagle_draft_t* handle,
                                const eagle_draft_inputs_t* inputs,
                                const eagle_draft_outputs_t* outputs,
                                const eagle_draft_trace_t* trace,
                                void* stream);

/* One launch of the fused LM-head kernel (frozen LM head + online log-softmax + per-row
 * top-k, ties to the lower token id; no [rows x |V|] logits are written) followed by the
 * cross-CTA merge, on the handle's weights and workspace.
 * a: f32 [N, d] device; N <= n_max; k <= 16.
 * Outputs (device): ids int32 [N, k] sorted by descending logit, logp f32 [N, k],
 * lse f32 [N].  This is the kernel the tree step launches at depths of up to 16 rows;
 * from 17 rows the step's LM head stores the rows' logits and a select kernel takes the
 * log-sum-exp and top-k per 1024-token part instead. */
EAGLE_API eagle_status_t eagle_draft_lm_head_topk(eagle_draft_t* handle, const float* a, int32_t N,
                                        int32_t k, int32_t* ids, float* logp, float* lse,
                                        void* stream);

/* Allocation-free variant of eagle_draft_lm_head_topk, with no handle.  The pages on
 * EAGLE have no counterpart: this exists for callers that cannot call cudaMalloc - e.g.
 * a serving engine that reserved nearly all device memory for its own pools at start-up,
 * or a latency-critical loop where an allocation would synchronise the device.  The
 * same LM-head and merge kernels run, but their scratch (split-K partial tiles, arrival
 * counters, per-tile log-sum-exp and per-CTA top-k partials) lives in one 4 MiB
 * file-scope device array that every GPU loading the library holds until exit; the call
 * allocates nothing.
 * w_lm: bf16 [vocab, d]; a: f32 [N, d]; ids int32 [N, k] (descending logit, ties to the
 * lower id), logp f32 [N, k], lse f32 [N]; all device pointers, 16-byte aligned.
 * Limits (EAGLE_ERR_INVALID_ARG beyond them, message in eagle_draft_last_error()):
 * 1 <= N <= 16, 1 <= k <= 16, vocab and d multiples of 128 with vocab <= 131072 and
 * d <= 16384; EAGLE_ERR_UNSUPPORTED on a device with more than 192 SMs.
 * The first call on a device looks up the array's device address and sets the kernels'
 * shared-memory limits (make that first call before any stream capture).  Every call
 * shares the array and clears the parts that must start at zero; calls whose kernels
 * overlap on the GPU (other streams, other threads) race on it and give wrong results.
 * Kernel-side errors: with no handle to hold a device error word, they show in the
 * outputs.  If a bounded wait inside the LM-head kernel runs out, every row of the call
 * comes back as id -1 with NaN logp and lse; a row with fewer than k finite logits gets
 * id -1 in the places it could not fill. */
EAGLE_API eagle_status_t eagle_lm_head_topk_noalloc(const void* w_lm, int32_t vocab, int32_t d,
                                                    const float* a, int32_t N, int32_t k,
                                                    int32_t* ids, float* logp, float* lse,
                                                    void* stream);

/* Kernel kinds reported by the profiler. */
typedef enum {
  EAGLE_K_INIT = 0, EAGLE_K_FC3 = 1, EAGLE_K_FC = 2, EAGLE_K_QKV = 3, EAGLE_K_ATTN = 4,
  EAGLE_K_OPROJ = 5, EAGLE_K_GATEUP = 6, EAGLE_K_DOWN = 7, EAGLE_K_LMHEAD = 8,
  EAGLE_K_EXPAND = 9, EAGLE_K_RERANK = 10, EAGLE_K_MERGE = 11, EAGLE_K_FC_OPERAND = 12, EAGLE_K_LM_SELECT = 13,
  EAGLE_K_COUNT = 14
} eagle_kernel_kind_t;

/* Profiling mode (enable != 0): every later eagle_draft_tree call (without a trace)
 * captures its kernels into a one-off CUDA graph, without programmatic dependent launch,
 * with a CUDA event recorded before and after each kernel, and replays it on the call's
 * stream (eagle_draft_lm_head_topk records its events directly on the stream).  eagle_draft_profile_read() synchronises, returns per
 * kind the summed kernel time in ms (host array ms[EAGLE_K_COUNT]) and the number of
 * launches (host array launches[EAGLE_K_COUNT]), and clears the records.  Disabling
 * returns to graph replay. */
EAGLE_API eagle_status_t eagle_draft_profile(eagle_draft_t* handle, int32_t enable);
EAGLE_API eagle_status_t eagle_draft_profile_read(eagle_draft_t* handle, float* ms, int32_t* launches);
/* Short name of a kernel kind ("lm_head", ...); "?" outside the range. */
EAGLE_API const char* eagle_draft_kernel_name(int32_t kind);

/* Sizes of the handle's buffers (host struct). */
EAGLE_API eagle_status_t eagle_draft_query(const eagle_draft_t* handle, eagle_draft_info_t* info);

/* Synchronises the device and returns EAGLE_ERR_DEVICE if the device error word is set
 * (its bits in *word if word != NULL, host), EAGLE_ERR_CUDA on a sticky CUDA error, and
 * EAGLE_OK otherwise.  Clears the word. */
EAGLE_API eagle_status_t eagle_draft_check(eagle_draft_t* handle, uint32_t* word);

/* Sets how long (clock cycles) each bounded wait inside the GEMM kernels may take before the
 * kernel gives up, sets EAGLE_DEVERR_TIMEOUT, lets its own copies and MMAs finish and returns;
 * 0 restores the default (about one second).  A short limit makes the waits run out on purpose,
 * for tests of that path: eagle_draft_check then reports the timeout, and clears the state a
 * CTA that gave up leaves behind, so the next call on the handle is whole again. */
EAGLE_API eagle_status_t eagle_draft_set_wait_limit(eagle_draft_t* handle, int64_t cycles);

/* Frees the workspace and the handle.  NULL is accepted. */
EAGLE_API void eagle_draft_destroy(eagle_draft_t* handle);

/* ------------------------------------------------------------------------------------
 * Verification side: the target's one pass over an emitted tree ("Tree attention in one
 * verification pass", aicassindra.com tm_eagle_deep) and greedy acceptance ("How
 * speculative decoding works", kaushalya.io, steps "target verification" / "output of the
 * round"; "Acceptance length under a tree", aicassindra.com).
 *
 * The target is one Llama-style decoder layer (RMSNorm, QKV, rotary, grouped-query
 * attention, O, RMSNorm, SwiGLU MLP) with its own weights, between the frozen embedding
 * and the frozen LM head, with a final RMSNorm before the LM head.  Every slot of the
 * tree is one row: token tokens[b][i] at position positions[b][i], attending to the
 * request's whole verified prefix (the target's own post-RoPE cache) and to the slots j
 * with mask[b][i][j] = 1 (its ancestors and itself).  The result per slot is the target's
 * most likely next token after that slot's path (ties to the lower id), its
 * log-probability and the log-sum-exp of the logits.  No [slots x |V|] logits are stored.
 * bf16 weights and cache, head_dim 128 only.
 * ------------------------------------------------------------------------------------ */
typedef struct {
  int32_t d, n_heads, n_kv_heads, head_dim, d_ff, vocab;  /* as in eagle_draft_config_t */
  float   rms_eps, rope_theta;
  int32_t dtype;        /* EAGLE_DTYPE_BF16 */
  int32_t max_batch;    /* largest B a call may pass */
  int32_t max_slots;    /* largest S (slots per request, root included); <= 64, max_batch * max_slots <= 256 */
  int32_t max_prefix;   /* largest prefix length n_b; positions must be < max_prefix + max_slots + 1 */
  int32_t flags;        /* EAGLE_FLAG_NO_PDL or 0 */
} eagle_verify_config_t;

/* Target weights (device, bf16 [out, in] row-major; gains f32), borrowed for the handle's
 * lifetime.  embed and w_lm are the frozen tables the draft shares with the target. */
typedef struct {
  const void*  embed;       /* [vocab, d] */
  const float* attn_norm;   /* [d] */
  const void*  w_qkv;       /* [(Hq + 2 Hkv) hd, d] */
  const void*  w_o;         /* [d, Hq hd] */
  const float* mlp_norm;    /* [d] */
  const void*  w_gate;      /* [d_ff, d] */
  const void*  w_up;        /* [d_ff, d] */
  const void*  w_down;      /* [d, d_ff] */
  const float* final_norm;  /* [d] */
  const void*  w_lm;        /* [vocab, d] */
} eagle_verify_weights_t;

/* One call's inputs (device): the emitted tree as eagle_draft_tree writes it, and the
 * target's verified-prefix cache, packed like the draft's. */
typedef struct {
  int32_t        B;            /* requests, 1..max_batch */
  int32_t        S;            /* slots per request, 1..max_slots */
  const int32_t* tokens;       /* [B, S] */
  const int32_t* positions;    /* [B, S] */
  const uint8_t* mask;         /* [B, S, S] 1 = slot j is visible to slot i (ancestor or self) */
  const int32_t* parents;      /* [B, S] parent slot (-1 for the root); needed only for acceptance */
  const void*    k_cache;      /* bf16 [sum n_b, Hkv, hd] target keys, post-RoPE */
  const void*    v_cache;      /* bf16 [sum n_b, Hkv, hd] */
  const int32_t* cu_seqlens;   /* [B + 1] */
} eagle_verify_inputs_t;

/* Outputs (device; any of them may be NULL, acceptance runs when accept_len is set). */
typedef struct {
  int32_t* top_id;        /* [B, S] the target's most likely next token after slot i's path */
  float*   top_logp;      /* [B, S] its log-probability */
  float*   lse;           /* [B, S] log-sum-exp of the slot's logits */
  float*   hidden;        /* [B, S, d] layer output before the final norm */
  float*   logits;        /* [B, S, vocab] the target's logits per slot (input of eagle_speculative_accept) */
  int32_t* accept_len;    /* [B] accepted draft tokens (root excluded) */
  int32_t* accept_slots;  /* [B, S] the accepted slots in path order, -1 after accept_len */
  int32_t* correction;    /* [B] the target's most likely token after the accepted path */
} eagle_verify_outputs_t;

typedef struct eagle_verify eagle_verify_t;

/* Validates the shapes, allocates the workspace (owned by the handle), builds the weights'
 * TMA descriptors and the rotary tables.  EAGLE_ERR_UNSUPPORTED outside bf16 / head_dim
 * 128 / multiples of 128 / the slot limits above. */
EAGLE_API eagle_status_t eagle_verify_create(const eagle_verify_config_t* cfg, const eagle_verify_weights_t* weights,
                                             eagle_verify_t** out_handle);
/* Enqueues one verification pass (and, with accept_len set, the greedy acceptance walk)
 * on `stream`.  Stream-ordered and asynchronous; kernel-side problems (a token outside
 * [0, vocab), a position past the rotary table, a parent that does not precede its slot)
 * set the handle's device error word, read by eagle_verify_check. */
EAGLE_API eagle_status_t eagle_verify_tree(eagle_verify_t* handle, const eagle_verify_inputs_t* inputs,
                                           const eagle_verify_outputs_t* outputs, void* stream);
/* Synchronises; EAGLE_ERR_DEVICE (bits in *word) if the device error word is set, then clears it. */
EAGLE_API eagle_status_t eagle_verify_check(eagle_verify_t* handle, uint32_t* word);
EAGLE_API void eagle_verify_destroy(eagle_verify_t* handle);

/* ------------------------------------------------------------------------------------
 * DFlash block-parallel draft ("DFlash-1: parallel block + KV injection", zackli.ai
 * "Speculative Decoding Deep Dive III"; "DFlash" card and algorithm sketch, kaushalya.io).
 * Per request, the block [E(anchor), E(MASK) x gamma] (rows at positions n_b .. n_b + gamma)
 * runs through n_layers draft layers in one pass: each Llama-style layer takes queries from
 * the block's hidden states and keys / values from [the layer's injected context ; the block]
 * - the target's fused context features of the verified prefix, projected by the layer, are
 * its extra KV memory - with attention bidirectional inside the block.  A final RMSNorm and
 * the frozen shared LM head give each mask row's draft distribution; the call returns its
 * top-k tokens (ties to the lower id), their log-probabilities and the log-sum-exp.  The
 * injected keys / values are a per-layer cache the caller keeps (keys rotated at the prefix
 * positions), like the draft's own KV cache of the EAGLE step.  bf16, head_dim 128.
 * ------------------------------------------------------------------------------------ */
typedef struct {
  int32_t d, n_heads, n_kv_heads, head_dim, d_ff, vocab;  /* as in eagle_draft_config_t */
  float   rms_eps, rope_theta;
  int32_t dtype;        /* EAGLE_DTYPE_BF16 */
  int32_t n_layers;     /* draft layers, 1..16 */
  int32_t gamma;        /* mask slots per block, 1..63 */
  int32_t k;            /* tokens kept per mask slot, 1..16 */
  int32_t mask_token;   /* the MASK row of the shared embedding table */
  int32_t max_batch;    /* largest B; max_batch * (gamma + 1) <= 256 */
  int32_t max_prefix;   /* largest prefix n_b */
  int32_t flags;        /* EAGLE_FLAG_NO_PDL or 0 */
} eagle_dflash_config_t;

/* Weights (device, bf16 [out, in] row-major; gains f32), borrowed for the handle's lifetime.
 * The per-layer members are HOST arrays of n_layers device pointers (copied at create). */
typedef struct {
  const void*  embed;                /* [vocab, d] frozen, shared with the target */
  const void*  w_lm;                 /* [vocab, d] frozen, shared with the target */
  const float* final_norm;           /* [d] */
  const float* const* attn_norm;     /* [n_layers] -> [d] */
  const void* const*  w_qkv;         /* [n_layers] -> [(Hq + 2 Hkv) hd, d] */
  const void* const*  w_o;           /* [n_layers] -> [d, Hq hd] */
  const float* const* mlp_norm;      /* [n_layers] -> [d] */
  const void* const*  w_gate;        /* [n_layers] -> [d_ff, d] */
  const void* const*  w_up;          /* [n_layers] -> [d_ff, d] */
  const void* const*  w_down;        /* [n_layers] -> [d, d_ff] */
} eagle_dflash_weights_t;

typedef struct {
  int32_t        B;            /* requests, 1..max_batch */
  const int32_t* anchor;       /* [B] the verified anchor token of each block */
  const void* const* ctx_k;    /* HOST array [n_layers] of device bf16 [sum n_b, Hkv, hd] injected keys */
  const void* const* ctx_v;    /* HOST array [n_layers] of device bf16 [sum n_b, Hkv, hd] injected values */
  const int32_t* cu_seqlens;   /* [B + 1] */
} eagle_dflash_inputs_t;

typedef struct {
  int32_t* tokens;   /* [B, gamma, k] the draft's top-k tokens of each mask slot (best first) */
  float*   logp;     /* [B, gamma, k] their log-probabilities */
  float*   lse;      /* [B, gamma] log-sum-exp of each mask slot's logits */
  float*   hidden;   /* [B, gamma + 1, d] (nullable) the last layer's output, anchor row included */
} eagle_dflash_outputs_t;

typedef struct eagle_dflash eagle_dflash_t;

EAGLE_API eagle_status_t eagle_dflash_create(const eagle_dflash_config_t* cfg, const eagle_dflash_weights_t* weights,
                                             eagle_dflash_t** out_handle);
/* Enqueues one block-parallel draft on `stream`; stream-ordered, asynchronous.  An anchor or
 * mask token outside [0, vocab) or a prefix longer than max_prefix sets the device error word
 * (eagle_dflash_check). */
EAGLE_API eagle_status_t eagle_dflash_draft(eagle_dflash_t* handle, const eagle_dflash_inputs_t* inputs,
                                            const eagle_dflash_outputs_t* outputs, void* stream);
EAGLE_API eagle_status_t eagle_dflash_check(eagle_dflash_t* handle, uint32_t* word);
EAGLE_API void eagle_dflash_destroy(eagle_dflash_t* handle);

/* Multi-round speculative sampling over emitted trees ("Speculative Decoding Deep Dive III",
 * zackli.ai, EAGLE-1: tree attention plus multi-round speculative sampling; "How speculative
 * decoding works", kaushalya.io: accept a drafted token with probability min(1, p/q), else draw
 * from the renormalised residual max(0, p - q)).  Per request, from the root, the children of
 * the current slot are tried in slot order (the draw order of sampled drafting): child x is
 * accepted when U * q(x) < p(x); on rejection the target becomes norm(max(0, p - q)) and x leaves
 * the proposal (q restricted to the untried tokens, renormalised).  The walk moves to an accepted
 * child; where none is accepted (or at a leaf) one token is drawn from the current target by
 * Gumbel-max, and the walk ends.  p and q at slot u are the softmax of the target's and the
 * draft's logits there (the draft's are those u's children were drawn from).  Random numbers:
 * Philox4x32-10 keyed by seeds[b]: trying child slot c uses U = (x + 1/2) / 2^32, x word 0 of
 * counter (c, 0, 0, 2); the token drawn at slot u after r rejections takes the Gumbel noise of
 * word (t mod 128) / 32 of counter (32 (t / 128) + t mod 32, u, r, 1) for token t.
 * Device pointers: tokens, parents [B, S] int32 (as eagle_draft_tree emits them; S <= 64);
 * logits_target, logits_draft [B, S, vocab] f32; seeds [B] uint64; outputs accept_len [B],
 * accept_slots [B, S] (accepted slots in path order, -1 after), correction [B] (the drawn
 * token).  *err_word (device, caller-owned) gets EAGLE_DEVERR_TOKEN for a token outside
 * [0, vocab) or a parent that does not precede its slot, EAGLE_DEVERR_SELECT when no token had
 * positive probability.  Allocates nothing; stream-ordered. */
EAGLE_API eagle_status_t eagle_speculative_accept(int32_t B, int32_t S, int32_t vocab, const int32_t* tokens,
                                                  const int32_t* parents, const float* logits_target,
                                                  const float* logits_draft, const uint64_t* seeds,
                                                  int32_t* accept_len, int32_t* accept_slots, int32_t* correction,
                                                  uint32_t* err_word, void* stream);

/* Thread-local description of the last error (never NULL). */
EAGLE_API const char* eagle_draft_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* EAGLE_DRAFT_H */
