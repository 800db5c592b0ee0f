"""Float64 CPU oracle of the EAGLE draft-tree expansion step.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import or run this module; the product path never does.  It
shares no code with the CUDA library: plain numpy, float64 throughout, library
matmul as the only building block beyond elementwise numpy.

What is computed (sources are the four pages on EAGLE):

* The draft recurrence ("The recurrence, written out", aicassindra.com tm_eagle_deep;
  "The Mechanism" equation, stable-lab "EAGLE: Drafting in Feature Space";
  "EAGLE-1 - autoregressive feature drafting" inference equation, zackli.ai
  "Speculative Decoding Deep Dive III"):
      x = [feat ; emb(tok)]            (2d)
      h = fc(x)                        (2d -> d)
      a = DecoderLayer(h, cache)       (the predicted next feature f', or EAGLE-3's latent a)
      p = softmax(LMHead(a))           (the frozen target LM head)
  The decoder layer is one Llama-style layer: RMSNorm, QKV projection, rotary
  embedding, grouped-query attention over the verified-prefix KV cache plus the
  KV of the node's own tree ancestors, output projection with residual, RMSNorm,
  SwiGLU MLP with residual.
* EAGLE-3 input ("EAGLE-3 - free representation ..." and "Multi-layer feature
  fusion"): at the verified position the feature is g = FC([l; m; h]) (3d -> d);
  later steps feed back the draft's own output a.
* Trees: a static tree expands every node with a fixed per-depth branching
  ("Drafting a Tree, Not a Chain", stable-lab); the EAGLE-2 dynamic tree expands,
  at each depth, the top-k nodes of that depth by path value
  V = sum of log draft confidences along the path (product of confidences,
  "EAGLE-2 - context-aware dynamic tree", zackli.ai; "EAGLE-2: expand and rerank",
  aicassindra.com), giving each its top-k children; after the last depth the
  rerank keeps the top-m of all generated nodes by V.
* Output: tokens, parent slots, position ids (prefix length + depth) and the
  ancestor-only attention mask ("Tree attention in one verification pass",
  aicassindra.com).

Readings where the pages are silent (each listed in the design notes):
rotate-half RoPE with inv_freq = theta^(-2i/hd); no biases; no final norm before the
LM head; children of one node ordered by token id; ties broken by lower token id
(top-k) or lower generation index (frontier, rerank); frontier and emitted nodes
kept in generation order; the root row sits at position n_b.

Parity: pinned by tests under ``tests/test_oracle_*`` (closed forms, library
routines, brute-force enumeration, hand-worked fixtures in ``tests/golden``).
"""
from __future__ import annotations

import numpy as np

MARGIN_TOL = 1e-3


# --------------------------------------------------------------------------- basics
def as_f64(a) -> np.ndarray:
    """Exact upcast: uint16 arrays are bfloat16 bit patterns, float arrays are widened."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y = x W^T with W stored [out, in]; W is upcast exactly to float64 in row blocks."""
    x = np.asarray(x, dtype=np.float64)
    M, K = w.shape
    out = np.empty((x.shape[0], M), dtype=np.float64)
    step = max(1, (1 << 24) // K)
    for m0 in range(0, M, step):
        out[:, m0:m0 + step] = x @ as_f64(w[m0:m0 + step]).T
    return out


def rms_norm(x: np.ndarray, gamma, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * gamma over the last axis."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * as_f64(gamma)


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    i = np.arange(head_dim // 2, dtype=np.float64)
    return theta ** (-2.0 * i / head_dim)


def rope(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """Rotate-half rotary embedding of x[..., hd] at integer position(s) pos.

    Pair (i, i + hd/2) is rotated by the angle pos * theta^(-2i/hd).
    ``pos`` broadcasts against x's leading axes.
    """
    hd = x.shape[-1]
    half = hd // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None] * rope_inv_freq(hd, theta)
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def gqa_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """softmax(q K^T / sqrt(hd)) V for every query head; q [Hq, hd], K/V [L, Hkv, hd].

    Query head j reads KV head j // (Hq / Hkv).
    """
    Hq, hd = q.shape
    rep = Hq // K.shape[1]
    out = np.empty_like(q)
    for j in range(Hq):
        s = K[:, j // rep, :] @ q[j] / np.sqrt(hd)
        p = np.exp(s - s.max())
        out[j] = (p / p.sum()) @ V[:, j // rep, :]
    return out


def log_softmax(logits: np.ndarray):
    """(log-probabilities, log-sum-exp) over the last axis."""
    mx = logits.max(axis=-1, keepdims=True)
    lse = mx + np.log(np.sum(np.exp(logits - mx), axis=-1, keepdims=True))
    return logits - lse, lse[..., 0]


# ------------------------------------------------------------------ top-k selection
def top_k(values: np.ndarray, k: int, keys: np.ndarray | None = None):
    """The k largest values, ties to the smaller key (default: the index).

    Returns (indices in selection order, boundary margin = v_(k) - v_(k+1)).
    """
    values = np.asarray(values, dtype=np.float64)
    keys = np.arange(len(values)) if keys is None else np.asarray(keys)
    order = np.lexsort((keys, -values))
    margin = float(values[order[k - 1]] - values[order[k]]) if len(values) > k else np.inf
    return order[:k], margin


def is_valid_top_k(values: np.ndarray, chosen, k: int, tol: float) -> bool:
    """True when ``chosen`` is a top-k of ``values`` up to ``tol`` (sets that differ from
    the exact one only by near-ties are accepted)."""
    values = np.asarray(values, dtype=np.float64)
    chosen = np.asarray(chosen, dtype=np.int64)
    if len(chosen) != k or len(np.unique(chosen)) != k:
        return False
    if np.any(chosen < 0) or np.any(chosen >= len(values)):
        return False
    if len(values) == k:
        return True
    rest = np.ones(len(values), bool)
    rest[chosen] = False
    return bool(values[chosen].min() >= values[rest].max() - tol)


# --------------------------------------------------------------- the draft layer
def decoder_rows(cfg: dict, W: dict, x_in: np.ndarray, pos: np.ndarray, attend):
    """One pass of fc + decoder layer + LM head over a batch of rows.

    x_in [N, 2d] = [feat ; emb(tok)]; pos [N] position ids; ``attend(i, k_i, v_i)``
    returns the (K, V) stacks [L, Hkv, hd] that row i sees (prefix + tree ancestors,
    its own k_i/v_i included).  Returns a dict of per-row intermediates.
    """
    d, Hq, Hkv, hd = cfg["d"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    eps, theta = cfg["rms_eps"], cfg["rope_theta"]
    N = x_in.shape[0]
    h = linear(x_in, W["w_fc"])                                   # fc: 2d -> d
    qkv = linear(rms_norm(h, W["attn_norm"], eps), W["w_qkv"])
    q = qkv[:, :Hq * hd].reshape(N, Hq, hd)
    k = qkv[:, Hq * hd:(Hq + Hkv) * hd].reshape(N, Hkv, hd)
    v = qkv[:, (Hq + Hkv) * hd:].reshape(N, Hkv, hd)
    q = rope(q, pos[:, None], theta)
    k = rope(k, pos[:, None], theta)
    attn = np.empty((N, Hq, hd))
    for i in range(N):
        Ki, Vi = attend(i, k[i], v[i])
        attn[i] = gqa_attention(q[i], Ki, Vi)
    o = attn.reshape(N, Hq * hd)
    y = h + linear(o, W["w_o"])                                   # O-proj + residual
    yn = rms_norm(y, W["mlp_norm"], eps)
    s = silu(linear(yn, W["w_gate"])) * linear(yn, W["w_up"])     # SwiGLU
    a = y + linear(s, W["w_down"])                                # down-proj + residual
    logits = linear(a, W["w_lm"])                                 # frozen LM head
    logp, lse = log_softmax(logits)
    return dict(h=h, q=q, k=k, v=v, attn=o, y=y, a=a, logp=logp, lse=lse)


# ------------------------------------------------------------------- tree builder
class _Req:
    """Per-request tree state.  Node 0 is the root; generated nodes follow in
    generation order (depth, frontier slot of the parent, token id)."""

    def __init__(self, n_prefix: int, root_tok: int):
        self.n = int(n_prefix)
        self.tok = [int(root_tok)]
        self.parent = [-1]
        self.depth = [0]
        self.logv = [0.0]
        self.src_row = [-1]      # row whose LM head generated the node
        self.rows = []           # dicts: node, pos, anc (row ids incl. self) + network state
        self.frontier = [0]      # node ids expanded at the next depth

    def path(self, u: int):
        """Tokens from the root's child down to node u (the root's path is empty)."""
        out = []
        while u > 0:
            out.append(self.tok[u])
            u = self.parent[u]
        return tuple(reversed(out))


def _choose(values, k, keys, forced, tol, log, what, ordered=False):
    """Exact top-k, or the forced choice when it is a valid top-k up to tol.

    With ``ordered`` the order of the choice is part of the decision (sampled children are
    kept in draw order, and a child's slot picks the noise its own row draws later): a
    forced choice must then also list its values in descending order up to tol."""
    exact, margin = top_k(values, k, keys)
    if forced is None:
        return exact, margin
    forced = np.asarray(forced, dtype=np.int64)
    if ordered:
        if np.array_equal(forced, exact):
            return exact, margin
        if is_valid_top_k(values, forced, k, tol) and \
                bool(np.all(values[forced[:-1]] >= values[forced[1:]] - tol)):
            log["forced"].append(what)
            return forced, margin
        log["mismatch"].append(what)
        return exact, margin
    if set(forced.tolist()) == set(exact.tolist()):
        return exact, margin
    if is_valid_top_k(values, forced, k, tol):
        log["forced"].append(what)
        return forced, margin
    log["mismatch"].append(what)
    return exact, margin


def expand_tree(cfg: dict, n_prefix, root_tok, step, force: dict | None = None,
                tol: float = MARGIN_TOL, seeds=None):
    """Static or EAGLE-2 dynamic tree expansion, independent of the network.

    ``step(s, reqs, rows)`` runs the draft model on the rows of depth s and returns
    log-probabilities [N_s, |V|] plus a dict of per-row extras; ``rows`` lists
    (request, node, row id) in row order.  Before the call each request's
    ``rows`` list already holds the new rows (node, pos, anc).

    ``force`` (optional) carries another implementation's decisions so the two can be
    compared through near-ties: ``force["children"][s]`` [N_s, k_s] tokens per row,
    ``force["frontier"][s]`` [B, F] node ids, ``force["final"]`` [B, m] node ids.
    A forced choice is adopted only when it is a valid top-k up to ``tol``; otherwise
    the oracle keeps its own and records a mismatch.

    ``seeds`` (optional, one 64-bit seed per request) switches to sampled drafting
    ("EAGLE-1 - autoregressive feature drafting", zackli.ai: the draft samples its next
    token from p-hat): a row's children are k tokens drawn without replacement from its
    distribution, the top-k of log p + Gumbel noise (``oracle.sampling``), kept in draw
    order; path values still add the unperturbed log-probabilities.
    """
    from . import sampling
    D = cfg["depth"]
    static = cfg["tree"] == "static"
    reqs = [_Req(n, t) for n, t in zip(n_prefix, root_tok)]
    log = {"forced": [], "mismatch": [], "margins": []}
    traces = []
    for s in range(1, D + 1):
        kids = cfg["branching"][s - 1] if static else cfg["k"]
        # ---- rows of this depth: one per frontier node, batched over requests
        rows = []
        for b, r in enumerate(reqs):
            for u in r.frontier:
                anc = ([] if u == 0 else list(r.rows[r.src_row[u]]["anc"])) + [len(r.rows)]
                rows.append((b, u, len(r.rows)))
                r.rows.append(dict(node=u, pos=r.n + r.depth[u], anc=anc))
        logp, extra = step(s, reqs, rows)

        # ---- children: top-k tokens of each row, kept in token-id order
        children, child_logp = [], []
        for i, (b, u, rid) in enumerate(rows):
            r = reqs[b]
            forced = None if force is None else force["children"][s][i]
            key = logp[i]
            if seeds is not None:           # draw order: largest perturbed value first
                key = logp[i] + sampling.gumbel(len(logp[i]), r.frontier.index(u), s, int(seeds[b]))
            sel, margin = _choose(key, kids, None, forced, tol, log, ("children", s, i),
                                  ordered=seeds is not None)
            log["margins"].append(("children", s, i, margin))
            if seeds is None:
                sel = np.sort(sel)
            children.append(sel)
            child_logp.append(logp[i][sel])
            for t in sel:
                r.tok.append(int(t))
                r.parent.append(u)
                r.depth.append(s)
                r.logv.append(r.logv[u] + float(logp[i][t]))
                r.src_row.append(rid)

        # ---- next frontier: every child (static) or the top-k of this depth by V
        frontiers = []
        if s < D:
            for b, r in enumerate(reqs):
                new = np.array([j for j in range(len(r.tok)) if r.depth[j] == s])
                if static:
                    r.frontier = new.tolist()
                else:
                    forced = None if force is None else force["frontier"][s][b]
                    forced_pos = None
                    if forced is not None:
                        idx = {int(g): p for p, g in enumerate(new)}
                        forced_pos = [idx.get(int(g), -1) for g in forced]
                    vals = np.array([r.logv[j] for j in new])
                    sel, margin = _choose(vals, cfg["k"], new, forced_pos, tol, log,
                                          ("frontier", s, b))
                    log["margins"].append(("frontier", s, b, margin))
                    r.frontier = np.sort(new[sel]).tolist()
                frontiers.append(list(r.frontier))
        traces.append(dict(rows=rows, tokens=np.array([reqs[b].tok[u] for b, u, _ in rows]),
                           pos=np.array([reqs[b].rows[rid]["pos"] for b, _, rid in rows]),
                           children=np.stack(children), child_logp=np.stack(child_logp),
                           frontier=frontiers, **extra))

    # ---- rerank: keep the top-m generated nodes by V, emit in generation order
    result = []
    for b, r in enumerate(reqs):
        gen = np.arange(1, len(r.tok))
        if static:
            keep = gen
        else:
            forced = None if force is None else force["final"][b]
            forced_pos = None if forced is None else [int(g) - 1 for g in forced]
            vals = np.array([r.logv[j] for j in gen])
            sel, margin = _choose(vals, cfg["m"], gen, forced_pos, tol, log, ("final", b))
            log["margins"].append(("final", b, margin))
            keep = np.sort(gen[sel])
        result.append(emit(r, keep))
    return dict(requests=result, trace=traces, log=log, reqs=reqs)


def emit(r: _Req, keep) -> dict:
    """Slot 0 = root, slots 1.. = kept nodes in generation order; parents as slots,
    positions = prefix length + depth, mask[i, j] = 1 iff slot j is an ancestor of
    slot i or i itself."""
    slots = [0] + [int(g) for g in keep]
    slot_of = {g: i for i, g in enumerate(slots)}
    S = len(slots)
    mask = np.zeros((S, S), np.uint8)
    for i, g in enumerate(slots):
        j = g
        while j != -1:                  # walk up: ancestor-or-self
            mask[i, slot_of[j]] = 1
            j = r.parent[j]
    return dict(
        tokens=np.array([r.tok[g] for g in slots], np.int64),
        parents=np.array([-1] + [slot_of[r.parent[g]] for g in slots[1:]], np.int64),
        positions=np.array([r.n + r.depth[g] for g in slots], np.int64),
        logv=np.array([r.logv[g] for g in slots]),
        mask=mask,
        node_ids=np.array(slots, np.int64),
        n_generated=len(r.tok) - 1,
    )


def draft_tree(cfg: dict, W: dict, inp: dict, force: dict | None = None,
               tol: float = MARGIN_TOL):
    """The whole draft-tree step for every request, float64 (see ``expand_tree``)."""
    cu = np.asarray(inp["cu_seqlens"], dtype=np.int64)
    B = len(cu) - 1
    Kc, Vc = as_f64(inp["k_cache"]), as_f64(inp["v_cache"])
    emb = W["embed"]
    # root feature: the target feature f, or EAGLE-3's fused g = FC([l;m;h])
    root_feat = as_f64(inp["root_feat"])
    if cfg["feat"] == "fused":
        root_feat = linear(root_feat, W["w_fc3"])

    def step(s, reqs, rows):
        feats, toks, pos = [], [], []
        for b, u, rid in rows:
            r = reqs[b]
            feats.append(root_feat[b] if u == 0 else r.rows[r.src_row[u]]["a"])
            toks.append(r.tok[u])
            pos.append(r.rows[rid]["pos"])
        x_in = np.concatenate([np.stack(feats), as_f64(emb[np.asarray(toks)])], axis=1)

        def attend(i, k_i, v_i):
            b, _, rid = rows[i]
            r = reqs[b]
            row = r.rows[rid]
            row["k"], row["v"] = k_i, v_i
            tk = np.stack([r.rows[j]["k"] for j in row["anc"]])
            tv = np.stack([r.rows[j]["v"] for j in row["anc"]])
            lo, hi = cu[b], cu[b + 1]
            return np.concatenate([Kc[lo:hi], tk]), np.concatenate([Vc[lo:hi], tv])

        out = decoder_rows(cfg, W, x_in, np.asarray(pos), attend)
        for i, (b, _, rid) in enumerate(rows):
            reqs[b].rows[rid]["a"] = out["a"][i]
        logp = out.pop("logp")
        return logp, out

    res = expand_tree(cfg, cu[1:] - cu[:-1], inp["root_tok"], step, force, tol, inp.get("seeds"))
    res["root_feat"] = root_feat
    return res


def fused_feature(W: dict, lmh) -> np.ndarray:
    """EAGLE-3 g = FC([l; m; h]) for [B, 3d] inputs."""
    return linear(as_f64(lmh), W["w_fc3"])


def lm_head_top_k(a, w_lm, k: int):
    """Teacher-forced LM-head decision: log-softmax of W_lm a and its top-k (by token id)."""
    logp, lse = log_softmax(linear(np.atleast_2d(as_f64(a)), w_lm))
    sel = [np.sort(top_k(row, k)[0]) for row in logp]
    return np.stack(sel), logp, lse
