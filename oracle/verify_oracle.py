"""Float64 CPU oracle of the verification side of an EAGLE draft tree.

TEST INFRASTRUCTURE.  Only the tests may import or run this module; no product code
does.  Plain numpy in float64, the primitives of ``oracle.eagle_oracle`` (which shares no
code with the CUDA library) and library matmul; nothing here is fused or reordered.

What is computed (sources are the four pages on EAGLE):

* Tree attention in one verification pass ("Tree attention in one verification pass",
  aicassindra.com tm_eagle_deep): the emitted tree's nodes are flattened into one
  sequence after the verified prefix; each node attends to the prefix and to its own
  ancestors and itself only (the emitted ancestor mask), at position id prefix length +
  depth.  One pass of the target gives, for every node, the target's next-token
  distribution conditioned on exactly that node's path.
* Greedy acceptance ("How speculative decoding works", steps "target verification" and
  "output of the round", kaushalya.io; "Acceptance length under a tree",
  aicassindra.com): at temperature 0 a drafted token passes when it equals the target's
  most likely next token after its parent's path.  Verification keeps the deepest path
  whose every token passes, and the target's most likely token after that path is
  emitted as the correction (bonus) token.

Readings where the pages are silent (listed in the design notes): the synthetic target
is one Llama-style decoder layer with the draft's head shapes, its own weights, the
frozen embedding and LM head it shares with the draft, and a final RMSNorm before the LM
head; the most likely token breaks ties to the lower token id; siblings carry distinct
tokens (the draft's top-k), so at most one child of a node can pass.

Parity: pinned by ``tests/test_oracle_verify.py`` (one masked pass against a separate
causal pass per root-to-node path; acceptance against enumeration of every node's path).
"""
from __future__ import annotations

import numpy as np

from .eagle_oracle import as_f64, gqa_attention, linear, log_softmax, rms_norm, rope, silu


def target_rows(cfg: dict, Wt: dict, embed, w_lm, tokens, pos, attend) -> dict:
    """One pass of the synthetic target (embedding, one decoder layer, final norm, LM head)
    over a set of rows.

    tokens [N] token ids; pos [N] position ids; ``attend(i, k_i, v_i)`` returns the (K, V)
    stacks [L, Hkv, hd] that row i sees (its own k_i / v_i included).  Returns a dict of
    per-row intermediates, ``logp`` [N, |V|] the target's next-token log-probabilities.
    """
    Hq, Hkv, hd = cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    eps, theta = cfg["rms_eps"], cfg["rope_theta"]
    tokens = np.asarray(tokens, dtype=np.int64)
    N = len(tokens)
    x = as_f64(np.asarray(embed)[tokens])                          # frozen embedding rows
    qkv = linear(rms_norm(x, Wt["attn_norm"], eps), Wt["w_qkv"])
    q = rope(qkv[:, :Hq * hd].reshape(N, Hq, hd), np.asarray(pos)[:, None], theta)
    k = rope(qkv[:, Hq * hd:(Hq + Hkv) * hd].reshape(N, Hkv, hd), np.asarray(pos)[:, None], theta)
    v = qkv[:, (Hq + Hkv) * hd:].reshape(N, Hkv, hd)
    attn = np.empty((N, Hq, hd))
    for i in range(N):
        Ki, Vi = attend(i, k, v)
        attn[i] = gqa_attention(q[i], Ki, Vi)
    y = x + linear(attn.reshape(N, Hq * hd), Wt["w_o"])
    yn = rms_norm(y, Wt["mlp_norm"], eps)
    hidden = y + linear(silu(linear(yn, Wt["w_gate"])) * linear(yn, Wt["w_up"]), Wt["w_down"])
    logp, lse = log_softmax(linear(rms_norm(hidden, Wt["final_norm"], eps), w_lm))
    return dict(k=k, v=v, hidden=hidden, logp=logp, lse=lse)


def verify_tree(cfg: dict, Wt: dict, W: dict, tokens, positions, mask, k_prefix, v_prefix) -> dict:
    """The target's pass over one request's emitted tree.

    tokens / positions [S] and mask [S, S] (mask[i, j] = 1 iff slot j is an ancestor of
    slot i or i itself) as the draft step emits them; k_prefix / v_prefix [n, Hkv, hd]
    the target's verified-prefix cache.  Row i attends to the whole prefix and to the
    slots its mask row marks.
    """
    mask = np.asarray(mask).astype(bool)
    Kp, Vp = as_f64(k_prefix), as_f64(v_prefix)

    def attend(i, k, v):
        sel = np.nonzero(mask[i])[0]
        return np.concatenate([Kp, k[sel]]), np.concatenate([Vp, v[sel]])

    return target_rows(cfg, Wt, W["embed"], W["w_lm"], tokens, positions, attend)


def target_path(cfg: dict, Wt: dict, W: dict, path_tokens, n_prefix: int, k_prefix, v_prefix) -> dict:
    """The target run causally over one token sequence after the prefix: row r (token r of
    the path, at position n_prefix + r) attends to the prefix and to rows 0..r."""
    Kp, Vp = as_f64(k_prefix), as_f64(v_prefix)
    pos = n_prefix + np.arange(len(path_tokens))

    def attend(i, k, v):
        return np.concatenate([Kp, k[:i + 1]]), np.concatenate([Vp, v[:i + 1]])

    return target_rows(cfg, Wt, W["embed"], W["w_lm"], path_tokens, pos, attend)


def most_likely(logp_row) -> int:
    """The most likely token; ties to the lower token id."""
    row = np.asarray(logp_row)
    return int(np.flatnonzero(row == row.max())[0])


def greedy_accept(tokens, parents, logp) -> dict:
    """Greedy (temperature 0) acceptance over one emitted tree.

    tokens / parents [S] (slot 0 the root, parent -1); logp [S, |V|] the target's
    next-token log-probabilities per slot.  From the root, the child whose token is the
    target's most likely next token is accepted and the walk continues from it; the walk
    stops at a slot with no such child.  Returns the accepted slots (root excluded), their
    tokens, and the correction token (the most likely token after the last accepted slot).
    """
    tokens = np.asarray(tokens)
    parents = np.asarray(parents)
    children = {}
    for s in range(1, len(tokens)):
        children.setdefault(int(parents[s]), []).append(s)
    u, accepted = 0, []
    while True:
        want = most_likely(logp[u])
        nxt = [c for c in children.get(u, []) if int(tokens[c]) == want]
        if not nxt:
            break
        u = nxt[0]
        accepted.append(u)
    return dict(slots=accepted, tokens=[int(tokens[s]) for s in accepted],
                correction=most_likely(logp[u]), length=len(accepted))
