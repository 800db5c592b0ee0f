"""Pins for the oracle's tree logic and the whole draft step (CPU only).

Each check compares the oracle against something other than itself: hand-worked
fixtures, brute-force enumeration, a separately written chain recurrence built from
torch library routines, closed forms of degenerate inputs, and the head-size count
printed on the pages.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import eagle_oracle as O
from eagle_speculative_decoding_03_gb300 import configs, synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _run(cfg):
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    return W, I, O.draft_tree(synth.oracle_cfg(cfg), W, I)


@pytest.fixture(scope="module")
def small_runs():
    return {n: _run(configs.get(n)) for n in ("small_dyn", "small_static", "small_fused", "small_f32")}


# ----------------------------------------------------------------- golden fixture
def _scripted_step(fx):
    table = {k: np.log(np.array(v)) for k, v in fx["probs_by_path"].items()}
    default = np.log(np.array(fx["probs_default"]))

    def step(s, reqs, rows):
        lp = [table.get(",".join(map(str, reqs[b].path(u))), default) for b, u, _ in rows]
        return np.stack(lp), {}
    return step


@pytest.mark.parametrize("case", range(4))
def test_golden_expand_rerank(case):
    fx = json.load(open(os.path.join(GOLDEN, "expand_rerank_tiny.json")))
    c = fx["cases"][case]
    cfg = dict(tree=c["tree"], depth=c["depth"], k=c.get("k", 0), m=c.get("m", 0),
               branching=tuple(c.get("branching", ())))
    res = O.expand_tree(cfg, [fx["n_prefix"]], [fx["root_tok"]], _scripted_step(fx))
    r = res["requests"][0]
    assert r["tokens"].tolist() == c["tokens"]
    assert r["parents"].tolist() == c["parents"]
    assert r["positions"].tolist() == [fx["n_prefix"] + dd for dd in c["depths"]]
    np.testing.assert_allclose(np.exp(r["logv"]), c["values"], rtol=1e-12)
    S = len(c["tokens"])
    want = np.zeros((S, S), np.uint8)
    for i, anc in enumerate(c["ancestors"]):
        want[i, anc] = 1
    assert np.array_equal(r["mask"], want)


# ------------------------------------------------------------------- node counts
def test_node_counts():
    assert configs.get("eagle1_static").generated_per_request() == 36
    assert [configs.get(n).generated_per_request() for n in ("eagle2_b1", "eagle2_b32", "eagle3_b8")] \
        == [510, 328, 610]


def test_node_counts_formula():
    for name in ("eagle2_b1", "eagle2_b32", "eagle3_b8"):
        c = configs.get(name)
        assert c.generated_per_request() == c.k + (c.depth - 1) * c.k ** 2
    c = configs.get("eagle1_static")
    assert sum(int(np.prod(c.branching[:j + 1])) for j in range(c.depth)) == 36
    assert [c.rows_at(s) for s in range(1, 6)] == [1, 4, 8, 8, 8]


def test_generated_counts_match(small_runs):
    for name, (_, _, res) in small_runs.items():
        cfg = configs.get(name)
        for r in res["requests"]:
            assert r["n_generated"] == cfg.generated_per_request()
            assert len(r["tokens"]) == cfg.kept_per_request() + 1


# ---------------------------------------------------- head size on the pages
def test_head_parameter_count():
    """fc adds 2d^2 and the decoder layer about 12d^2 ('What is actually in the head')."""
    c = configs.get("eagle1_static")
    d = c.d
    fc = 2 * d * d
    layer = c.qkv_dim * d + d * c.attn_dim + 3 * d * c.d_ff
    assert fc == 2 * d ** 2
    assert abs(layer / d ** 2 - 12) < 0.1


# ---------------------------------------------- chain recurrence (k = 1) pin
def _chain_reference(cfg, W, I):
    """The written recurrence x=[f; emb(t)] -> fc -> layer -> LM head, rolled forward
    greedily with plain causal attention over [prefix, earlier draft positions]; torch
    float64 library routines only."""
    T = lambda a: torch.from_numpy(O.as_f64(a))
    d, Hq, Hkv, hd = cfg.d, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    n = int(I["cu_seqlens"][1])
    Ks, Vs = T(I["k_cache"][:n]), T(I["v_cache"][:n])
    f, t = T(I["root_feat"][0]), int(I["root_tok"][0])
    inv = cfg.rope_theta ** (-torch.arange(hd // 2, dtype=torch.float64) * 2 / hd)

    def rot(x, pos):   # complex-multiplication form of the rotation
        z = torch.complex(x[..., :hd // 2], x[..., hd // 2:]) * torch.polar(torch.ones_like(inv), pos * inv)
        return torch.cat([z.real, z.imag], -1)

    toks, logv, feats = [], [0.0], []
    for step in range(cfg.depth):
        pos = n + step
        h = torch.cat([f, T(W["embed"][t])]) @ T(W["w_fc"]).T
        x = F.rms_norm(h, (d,), T(W["attn_norm"]), cfg.rms_eps)
        qkv = x @ T(W["w_qkv"]).T
        q = rot(qkv[:Hq * hd].view(Hq, hd), pos)
        k = rot(qkv[Hq * hd:(Hq + Hkv) * hd].view(1, Hkv, hd), pos)
        v = qkv[(Hq + Hkv) * hd:].view(1, Hkv, hd)
        Ks, Vs = torch.cat([Ks, k]), torch.cat([Vs, v])
        rep = Hq // Hkv
        att = F.scaled_dot_product_attention(
            q[:, None], Ks.permute(1, 0, 2).repeat_interleave(rep, 0),
            Vs.permute(1, 0, 2).repeat_interleave(rep, 0))[:, 0].reshape(-1)
        y = h + att @ T(W["w_o"]).T
        z = F.rms_norm(y, (d,), T(W["mlp_norm"]), cfg.rms_eps)
        a = y + (F.silu(z @ T(W["w_gate"]).T) * (z @ T(W["w_up"]).T)) @ T(W["w_down"]).T
        lp = torch.log_softmax(a @ T(W["w_lm"]).T, -1)
        t = int(torch.argmax(lp))
        toks.append(t)
        logv.append(logv[-1] + float(lp[t]))
        feats.append(a.numpy())
        f = a
    return toks, np.array(logv), feats


def _chain_along_path(cfg, W, I, b, tokens):
    """The written recurrence run causally along one token path of request b:
    step j feeds [feature of step j-1 ; emb(tokens[j])] (the root feature at j = 0:
    f, or EAGLE-3's FC([l;m;h])) through fc and the layer at position n_b + j, with
    plain causal attention over [prefix of b, steps 0..j].  torch float64 library
    routines only; nothing is shared with the oracle but the upcast.  Returns the
    per-step h, rotated q, attention output, layer output a and log-sum-exp."""
    T = lambda a: torch.from_numpy(O.as_f64(a))
    d, Hq, Hkv, hd = cfg.d, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    lo, hi = int(I["cu_seqlens"][b]), int(I["cu_seqlens"][b + 1])
    n = hi - lo
    Ks, Vs = T(I["k_cache"][lo:hi]), T(I["v_cache"][lo:hi])
    f = T(I["root_feat"][b])
    if cfg.feat == "fused":
        f = T(W["w_fc3"]) @ f
    inv = cfg.rope_theta ** (-torch.arange(hd // 2, dtype=torch.float64) * 2 / hd)

    def rot(x, pos):
        z = torch.complex(x[..., :hd // 2], x[..., hd // 2:]) * torch.polar(torch.ones_like(inv), pos * inv)
        return torch.cat([z.real, z.imag], -1)

    out = []
    for j, t in enumerate(tokens):
        pos = n + j
        h = torch.cat([f, T(W["embed"][int(t)])]) @ T(W["w_fc"]).T
        x = F.rms_norm(h, (d,), T(W["attn_norm"]), cfg.rms_eps)
        qkv = x @ T(W["w_qkv"]).T
        q = rot(qkv[:Hq * hd].view(Hq, hd), pos)
        k = rot(qkv[Hq * hd:(Hq + Hkv) * hd].view(1, Hkv, hd), pos)
        v = qkv[(Hq + Hkv) * hd:].view(1, Hkv, hd)
        Ks, Vs = torch.cat([Ks, k]), torch.cat([Vs, v])
        rep = Hq // Hkv
        att = F.scaled_dot_product_attention(
            q[:, None], Ks.permute(1, 0, 2).repeat_interleave(rep, 0),
            Vs.permute(1, 0, 2).repeat_interleave(rep, 0))[:, 0].reshape(-1)
        y = h + att @ T(W["w_o"]).T
        z = F.rms_norm(y, (d,), T(W["mlp_norm"]), cfg.rms_eps)
        a = y + (F.silu(z @ T(W["w_gate"]).T) * (z @ T(W["w_up"]).T)) @ T(W["w_down"]).T
        lse = torch.logsumexp(a @ T(W["w_lm"]).T, -1)
        out.append(dict(h=h.numpy(), q=q.numpy(), attn=att.numpy(), a=a.numpy(), lse=float(lse)))
        f = a
    return out


def _assert_rows_follow_their_paths(cfg, W, I, res):
    """Every tree row equals the causal chain re-run along its own root-to-node path."""
    checked = 0
    for s, tr in enumerate(res["trace"], 1):
        for i, (b, u, rid) in enumerate(tr["rows"]):
            req = res["reqs"][b]
            path = (req.tok[0],) + req.path(u)           # the root token, then the path to u
            assert len(path) == s
            last = _chain_along_path(cfg, W, I, b, path)[-1]
            for key in ("h", "q", "attn", "a"):
                got = tr[key][i].reshape(-1)
                np.testing.assert_allclose(got, last[key].reshape(-1), rtol=1e-11, atol=1e-11,
                                           err_msg=f"{cfg.name} depth {s} row {i} {key}")
            np.testing.assert_allclose(tr["lse"][i], last["lse"], rtol=1e-12, atol=1e-11)
            checked += 1
    return checked


@pytest.mark.parametrize("name", ["small_dyn", "small_static", "small_fused", "tiny16"])
def test_every_tree_row_equals_the_chain_along_its_path(name, small_runs):
    """Ancestor-only tree attention ('Tree attention in one verification pass'): a row of
    a branching tree sees the prefix and its ancestors' KV only, so it must equal the
    plain recurrence ('The recurrence, written out') run causally along its own path.
    A sibling or cousin leaking into a row's KV, or a row reading the wrong source row's
    ancestors, breaks this."""
    if name == "tiny16":
        cfg = TINY
        W, I, res = _run(cfg)
    else:
        cfg = configs.get(name)
        W, I, res = small_runs[name]
    assert _assert_rows_follow_their_paths(cfg, W, I, res) == sum(len(t["rows"]) for t in res["trace"])


def test_chain_recurrence_k1():
    cfg = configs.get("tiny_chain")
    W, I, res = _run(cfg)
    toks, logv, feats = _chain_reference(cfg, W, I)
    r = res["requests"][0]
    assert r["tokens"][1:].tolist() == toks
    assert r["parents"].tolist() == [-1, 0, 1, 2, 3]
    np.testing.assert_allclose(r["logv"], logv, rtol=1e-12)
    for s, a in enumerate(feats):
        np.testing.assert_allclose(res["trace"][s]["a"][0], a, rtol=1e-11, atol=1e-12)


# ------------------------------------------------------ mask, values, positions
def test_mask_is_brute_force_ancestor_relation(small_runs):
    for _, (_, _, res) in small_runs.items():
        for r in res["requests"]:
            S = len(r["tokens"])
            for i in range(S):
                anc, j = set(), i
                while j != -1:
                    anc.add(j)
                    j = r["parents"][j]
                assert set(np.nonzero(r["mask"][i])[0].tolist()) == anc
                assert all(r["parents"][i] < i for i in range(1, S))


def test_values_are_products_of_confidences(small_runs):
    """exp(V) equals the product of softmax probabilities along the path."""
    for name, (W, I, res) in small_runs.items():
        rows_prob = {}
        for s, tr in enumerate(res["trace"], 1):
            logits = torch.from_numpy(tr["a"]) @ torch.from_numpy(O.as_f64(W["w_lm"])).T
            probs = torch.softmax(logits, -1).numpy()
            for i, (b, u, rid) in enumerate(tr["rows"]):
                rows_prob[(b, rid)] = probs[i]
        for b, req in enumerate(res["reqs"]):
            for g in range(1, len(req.tok)):
                p, j = 1.0, g
                while j > 0:
                    p *= rows_prob[(b, req.src_row[j])][req.tok[j]]
                    j = req.parent[j]
                np.testing.assert_allclose(np.exp(req.logv[g]), p, rtol=1e-10)


def test_positions_are_prefix_plus_depth(small_runs):
    for _, (_, I, res) in small_runs.items():
        n = np.diff(I["cu_seqlens"])
        for b, r in enumerate(res["requests"]):
            depth = np.array([res["reqs"][b].depth[g] for g in r["node_ids"]])
            assert np.array_equal(r["positions"], n[b] + depth)


def test_rerank_is_sorted_selection_and_ancestor_closed(small_runs):
    for name, (_, _, res) in small_runs.items():
        cfg = configs.get(name)
        if cfg.tree != "dynamic":
            continue
        for b, r in enumerate(res["requests"]):
            req = res["reqs"][b]
            gen = list(range(1, len(req.tok)))
            full = sorted(gen, key=lambda g: (-req.logv[g], g))[:cfg.m]
            assert sorted(full) == r["node_ids"][1:].tolist()
            kept = set(r["node_ids"].tolist())
            assert all(req.parent[g] in kept for g in kept if g)


# ----------------------------------- frontier = global top-k, rerank = best subset
TINY = configs.DraftConfig(
    name="tiny16", d=64, n_heads=2, n_kv_heads=1, head_dim=32, d_ff=96, vocab=16,
    rms_eps=1e-6, rope_theta=1e4, dtype="f32", tree="dynamic", depth=3, k=3, m=6,
    B=2, prefix=(3, 9), seed=3001, gamma_jitter=0.2)


def test_frontier_is_global_top_k_over_node_token_pairs():
    cfg = TINY
    W, I, res = _run(cfg)
    for s, tr in enumerate(res["trace"][:-1], 1):
        logits = torch.from_numpy(tr["a"]) @ torch.from_numpy(O.as_f64(W["w_lm"])).T
        lp = torch.log_softmax(logits, -1).numpy()
        for b, req in enumerate(res["reqs"]):
            pairs = []
            for i, (bb, u, rid) in enumerate(tr["rows"]):
                if bb == b:
                    pairs += [(req.logv[u] + lp[i, t], i, t) for t in range(cfg.vocab)]
            best = sorted(pairs, key=lambda p: (-p[0], p[1], p[2]))[:cfg.k]
            got = {(req.src_row[g], req.tok[g]) for g in tr["frontier"][b]}
            want = {(tr["rows"][i][2], t) for _, i, t in best}
            assert got == want


def test_rerank_is_best_ancestor_closed_subset():
    cfg = TINY.with_(k=2, m=5, seed=3002, B=3)
    W, I, res = _run(cfg)
    for b, req in enumerate(res["reqs"]):
        gen = range(1, len(req.tok))
        assert len(gen) == 10
        best, best_set = -np.inf, None
        for sub in itertools.combinations(gen, cfg.m):
            s = set(sub)
            if any(req.parent[g] not in s and req.parent[g] != 0 for g in s):
                continue
            v = sum(req.logv[g] for g in s)
            if v > best:
                best, best_set = v, s
        assert best_set == set(res["requests"][b]["node_ids"][1:].tolist())


# -------------------------------------------------------------- degenerate cases
def test_zero_lm_head_is_uniform_and_breaks_ties_by_index():
    cfg = TINY.with_(k=2, m=4, B=1, seed=3003)
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    W["w_lm"] = np.zeros_like(W["w_lm"])
    res = O.draft_tree(synth.oracle_cfg(cfg), W, I)
    r = res["requests"][0]
    # every child has log p = -ln|V|: children are tokens 0,1; the frontier and the
    # rerank keep the lowest generation indices
    assert r["tokens"][1:].tolist() == [0, 1, 0, 1]
    assert r["parents"].tolist() == [-1, 0, 0, 1, 1]
    np.testing.assert_allclose(r["logv"], [0, -np.log(16), -np.log(16), -2 * np.log(16), -2 * np.log(16)],
                               rtol=1e-14)


def test_depth_one_tree():
    cfg = TINY.with_(depth=1, k=4, m=3, seed=3004)
    W, I, res = _run(cfg)
    for b, r in enumerate(res["requests"]):
        assert r["parents"].tolist() == [-1, 0, 0, 0]
        lp = res["trace"][0]["child_logp"][b]
        assert sorted(r["logv"][1:].tolist(), reverse=True) == sorted(lp.tolist(), reverse=True)[:3]


def test_eagle3_root_row_uses_fused_feature(small_runs):
    cfg = configs.get("small_fused")
    W, I, res = small_runs["small_fused"]
    T = lambda a: torch.from_numpy(O.as_f64(a))
    g = T(I["root_feat"]) @ T(W["w_fc3"]).T                       # g = FC([l; m; h])
    x = torch.cat([g, T(W["embed"][I["root_tok"]])], 1)
    h = x @ T(W["w_fc"]).T
    np.testing.assert_allclose(res["trace"][0]["h"], h.numpy(), rtol=1e-12, atol=1e-12)
    # later rows read the draft's own output a of the parent row
    tr1, tr0 = res["trace"][1], res["trace"][0]
    b, u, rid = tr1["rows"][0]
    parent_row = res["reqs"][b].src_row[u]
    x1 = torch.cat([torch.from_numpy(tr0["a"][parent_row]), T(W["embed"][res["reqs"][b].tok[u]])])
    np.testing.assert_allclose(tr1["h"][0], (x1 @ T(W["w_fc"]).T).numpy(), rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------- forced mode
def test_force_mode_accepts_near_ties_and_flags_real_mismatches():
    cfg = configs.get("small_dyn")
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    ocfg = synth.oracle_cfg(cfg)
    base = O.draft_tree(ocfg, W, I)
    force = {"children": {s + 1: tr["children"] for s, tr in enumerate(base["trace"])},
             "frontier": {s + 1: tr["frontier"] for s, tr in enumerate(base["trace"][:-1])},
             "final": [r["node_ids"][1:] for r in base["requests"]]}
    same = O.draft_tree(ocfg, W, I, force=force)
    assert same["log"]["forced"] == [] and same["log"]["mismatch"] == []
    for a, b in zip(same["requests"], base["requests"]):
        assert np.array_equal(a["tokens"], b["tokens"])
    # a wrong child set is flagged, never adopted
    bad = dict(force, children=dict(force["children"]))
    ch = bad["children"][1].copy()
    ch[0, 0] = (ch[0, 0] + 1) % cfg.vocab if (ch[0, 0] + 1) % cfg.vocab not in ch[0] else ch[0, 0]
    bad["children"][1] = ch
    res = O.draft_tree(ocfg, W, I, force=bad, tol=1e-9)
    if not np.array_equal(ch, force["children"][1]):
        assert ("children", 1, 0) in res["log"]["mismatch"]
