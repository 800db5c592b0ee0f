"""Float64 CPU oracle of the DFlash block-parallel draft.

TEST INFRASTRUCTURE.  Only the tests may import or run this module; no product code does.
Plain numpy in float64, built from the primitives of ``oracle.eagle_oracle`` (which shares
no code with the CUDA library).

What is computed ("DFlash-1: parallel block + KV injection", zackli.ai "Speculative
Decoding Deep Dive III"; "DFlash" card and algorithm sketch, kaushalya.io):

* the block: the verified anchor token followed by gamma mask slots,
  [E(anchor), E(MASK), ..., E(MASK)], drafted in one parallel pass;
* every draft layer attends with queries from the block's hidden states H_d and keys /
  values [W_K H_ctx ; W_K H_d], [W_V H_ctx ; W_V H_d]: the target's fused context features
  H_ctx of the verified prefix are injected as extra KV memory in every layer;
  attention is bidirectional inside the block;
* draft logits through the frozen shared LM head, q_t = softmax(W_LM h_t); the gamma mask
  rows give the drafted block.

Readings where the pages are silent (listed in the design notes):
* the block is gamma + 1 rows (anchor + gamma masks) at positions n, ..., n + gamma after a
  prefix of n; the mask rows' outputs are the draft, the anchor row's is not used;
* each layer's injected keys / values of the prefix, W_K H_ctx and W_V H_ctx (keys rotated
  at the prefix positions), are a per-layer cache that the draft step reads, like the
  prefix KV cache of the EAGLE draft; its refresh for newly verified rows is not part of
  the step;
* a draft layer is a Llama-style layer (RMSNorm, QKV, rotary, grouped-query attention, O
  with residual, RMSNorm, SwiGLU with residual); the stack ends in a final RMSNorm before
  the LM head; MASK is one token id of the shared embedding table;
* the draft takes the top-k tokens of each mask row (k = 1: the greedy block).

Parity: pinned by ``tests/test_oracle_dflash.py`` (a separately written torch stack with
library attention; invariance of the context under permutation; identity layers in closed
form; the anchor-only and context-free cases; bidirectionality).
"""
from __future__ import annotations

import numpy as np

from .eagle_oracle import as_f64, gqa_attention, linear, log_softmax, rms_norm, rope, silu, top_k


def dflash_block(cfg: dict, W: dict, anchor: int, n_prefix: int, ctx_k, ctx_v, k: int = 1) -> dict:
    """One request's block-parallel draft.

    W: ``embed``, ``w_lm``, ``final_norm`` and ``layers``, a list of per-layer dicts
    (``attn_norm``, ``w_qkv``, ``w_o``, ``mlp_norm``, ``w_gate``, ``w_up``, ``w_down``);
    ctx_k / ctx_v: per layer, the injected context keys / values [n_prefix, Hkv, hd]
    (keys rotated at positions 0..n_prefix-1).  cfg: d, n_heads, n_kv_heads, head_dim,
    rms_eps, rope_theta, gamma, mask_token.
    Returns the per-layer hidden states, the block's log-probabilities [gamma + 1, |V|],
    the top-k tokens of every mask row and their log-probabilities."""
    Hq, Hkv, hd = cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    eps, theta, g = cfg["rms_eps"], cfg["rope_theta"], cfg["gamma"]
    rows = g + 1
    tokens = np.array([anchor] + [cfg["mask_token"]] * g, dtype=np.int64)
    pos = n_prefix + np.arange(rows)
    x = as_f64(np.asarray(W["embed"])[tokens])
    hidden = [x]
    for l, L in enumerate(W["layers"]):
        qkv = linear(rms_norm(x, L["attn_norm"], eps), L["w_qkv"])
        q = rope(qkv[:, :Hq * hd].reshape(rows, Hq, hd), pos[:, None], theta)
        kb = rope(qkv[:, Hq * hd:(Hq + Hkv) * hd].reshape(rows, Hkv, hd), pos[:, None], theta)
        vb = qkv[:, (Hq + Hkv) * hd:].reshape(rows, Hkv, hd)
        K = np.concatenate([as_f64(ctx_k[l]), kb])          # injected context, then the block
        V = np.concatenate([as_f64(ctx_v[l]), vb])
        attn = np.stack([gqa_attention(q[i], K, V) for i in range(rows)])   # every row sees all
        y = x + linear(attn.reshape(rows, Hq * hd), L["w_o"])
        yn = rms_norm(y, L["mlp_norm"], eps)
        x = y + linear(silu(linear(yn, L["w_gate"])) * linear(yn, L["w_up"]), L["w_down"])
        hidden.append(x)
    logp, lse = log_softmax(linear(rms_norm(x, W["final_norm"], eps), W["w_lm"]))
    picks, margins = [], []
    for i in range(1, rows):
        sel, margin = top_k(logp[i], k)
        picks.append(sel)
        margins.append(margin)
    picks = np.stack(picks)
    return dict(hidden=hidden, logp=logp, lse=lse, tokens=picks,
                token_logp=np.take_along_axis(logp[1:], picks, axis=1), margins=np.array(margins))


def dflash_draft(cfg: dict, W: dict, inp: dict, k: int = 1) -> list:
    """Every request of a call: inp has ``anchor`` [B], ``cu_seqlens`` [B+1] and the
    per-layer packed context caches ``ctx_k`` / ``ctx_v`` ([L][sum n_b, Hkv, hd])."""
    cu = np.asarray(inp["cu_seqlens"], dtype=np.int64)
    out = []
    for b in range(len(cu) - 1):
        lo, hi = cu[b], cu[b + 1]
        out.append(dflash_block(cfg, W, int(inp["anchor"][b]), int(hi - lo),
                                [c[lo:hi] for c in inp["ctx_k"]], [c[lo:hi] for c in inp["ctx_v"]], k))
    return out
