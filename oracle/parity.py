"""Compare a draft tree computed elsewhere against the float64 oracle.

TEST INFRASTRUCTURE (see eagle_oracle.py).  Takes plain numpy arrays; imports nothing
but numpy and the oracle.

Bar (per the step's definition):
  * token ids, parents, positions and the mask must match exactly, except where the
    oracle's own top-k / frontier / rerank boundary margin is below ``margin`` in log
    probability: there the other side's choice is accepted when it is a valid top-k up
    to ``margin`` (reported as "forced", not failed);
  * features (fc output, queries, attention output, post-attention residual, layer
    output) within max relative error ``tol_feat`` = max|x - x_ref| / max|x_ref|;
  * path values V and children log-probabilities within absolute ``tol_v``.
"""
from __future__ import annotations

import numpy as np

from . import eagle_oracle as O


def rel_err(x, ref) -> float:
    x, ref = np.asarray(x, np.float64), np.asarray(ref, np.float64)
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(x - ref)) / den) if den > 0 else float(np.max(np.abs(x)))


def compare(ocfg: dict, W: dict, I: dict, out: dict, trace: dict | None, S: int,
            tol_feat: float = 2e-2, tol_v: float = 1e-2, margin: float = O.MARGIN_TOL,
            f_max: int | None = None):
    """``out``: tokens/parents/positions/logv [B,S], mask [B,S,S]; ``trace`` (optional):
    the per-depth arrays of eagle_draft_trace_t as numpy.  Returns a report dict."""
    B = len(I["root_tok"])
    D = ocfg["depth"]
    static = ocfg["tree"] == "static"
    force = None
    if trace is not None:
        kids = [ocfg["branching"][s] if static else ocfg["k"] for s in range(D)]
        rows = [1]
        for s in range(1, D):
            rows.append(rows[-1] * kids[s - 1] if static else ocfg["k"])
        force = {"children": {}, "frontier": {}, "final": [trace["final_nodes"][b][1:S] for b in range(B)]}
        for s in range(1, D + 1):
            N = B * rows[s - 1]
            force["children"][s] = trace["children"][s - 1][:N, :kids[s - 1]]
            if s < D and not static:
                force["frontier"][s] = [trace["frontier"][s - 1][b][:rows[s]] for b in range(B)]
    ora = O.draft_tree(ocfg, W, I, force=force, tol=margin)
    errs, stats = [], {}
    if ora["log"]["mismatch"]:
        errs.append(f"decisions differ beyond the {margin} margin: {ora['log']['mismatch'][:8]}")
    for b, r in enumerate(ora["requests"]):
        for key in ("tokens", "parents", "positions"):
            if not np.array_equal(np.asarray(out[key][b][:S], np.int64), r[key]):
                errs.append(f"request {b}: {key} differ: {np.asarray(out[key][b][:S]).tolist()} vs {r[key].tolist()}")
        if not np.array_equal(np.asarray(out["mask"][b][:S, :S]), r["mask"]):
            errs.append(f"request {b}: mask differs")
        dv = float(np.max(np.abs(np.asarray(out["logv"][b][:S], np.float64) - r["logv"])))
        stats["logv"] = max(stats.get("logv", 0.0), dv)
    if stats.get("logv", 0.0) > tol_v:
        errs.append(f"logv off by {stats['logv']:.3g} > {tol_v}")
    if trace is not None:
        for s, tr in enumerate(ora["trace"]):
            N = len(tr["rows"])
            for key in ("h", "q", "attn", "y", "a"):
                ref = tr[key].reshape(N, -1)
                got = np.asarray(trace[key][s][:N]).reshape(N, -1)
                e = rel_err(got, ref)
                stats[key] = max(stats.get(key, 0.0), e)
            kk = tr["children"].shape[1]
            dl = float(np.max(np.abs(np.asarray(trace["child_logp"][s][:N, :kk], np.float64) - tr["child_logp"])))
            stats["child_logp"] = max(stats.get("child_logp", 0.0), dl)
            dse = float(np.max(np.abs(np.asarray(trace["lse"][s][:N], np.float64) - tr["lse"])))
            stats["lse"] = max(stats.get("lse", 0.0), dse)
        for key in ("h", "q", "attn", "y", "a"):
            if stats[key] > tol_feat:
                errs.append(f"{key}: max relative error {stats[key]:.3g} > {tol_feat}")
        for key in ("child_logp", "lse"):
            if stats[key] > tol_v:
                errs.append(f"{key}: max abs error {stats[key]:.3g} > {tol_v}")
        # tree K/V of every row (rotated keys, values)
        for b, req in enumerate(ora["reqs"]):
            for rid, row in enumerate(req.rows):
                for key, tk in (("k", "tree_k"), ("v", "tree_v")):
                    e = rel_err(np.asarray(trace[tk][b][rid]), row[key])
                    stats["tree_" + key] = max(stats.get("tree_" + key, 0.0), e)
        for key in ("tree_k", "tree_v"):
            if stats.get(key, 0.0) > tol_feat:
                errs.append(f"{key}: max relative error {stats[key]:.3g} > {tol_feat}")
    near = [m for m in ora["log"]["margins"] if m[-1] < margin]
    return {"ok": not errs, "errors": errs, "stats": stats, "forced": ora["log"]["forced"],
            "near_ties": near, "oracle": ora}


def _force_from_trace(ocfg: dict, trace: dict, B: int, S: int) -> dict:
    """Another implementation's decisions, read from its trace (see O.expand_tree)."""
    D = ocfg["depth"]
    static = ocfg["tree"] == "static"
    kids = [ocfg["branching"][s] if static else ocfg["k"] for s in range(D)]
    rows = [1]
    for s in range(1, D):
        rows.append(rows[-1] * kids[s - 1] if static else ocfg["k"])
    force = {"children": {}, "frontier": {}, "final": [trace["final_nodes"][b][1:S] for b in range(B)]}
    for s in range(1, D + 1):
        force["children"][s] = trace["children"][s - 1][:B * rows[s - 1], :kids[s - 1]]
        if s < D and not static:
            force["frontier"][s] = [trace["frontier"][s - 1][b][:rows[s]] for b in range(B)]
    return force


def compare_teacher_forced(ocfg: dict, W: dict, I: dict, out: dict, trace: dict, S: int,
                           tol_feat: float = 2e-2, tol_v: float = 1e-2, margin: float = O.MARGIN_TOL):
    """Every request of a batched run, depth by depth, with the other side's inputs.

    At each depth the oracle runs the fc + decoder layer (float64) on the rows the other
    side ran: the parent row's feature is the other side's layer output of the previous
    depth (the root feature, or FC([l;m;h]), at depth 1), the token is its chosen child,
    and attention reads the prefix plus the keys / values of the row's ancestors that the
    oracle computed at the earlier depths.  Its outputs (h, rotated q, attention output,
    residual, layer output) must match within ``tol_feat``.  The LM head, log-softmax,
    children, frontier and rerank are then taken by the oracle from the other side's layer
    output, so errors never compound across depths; tree structure must match exactly
    (near-ties below ``margin`` forced), values within ``tol_v``."""
    B = len(I["root_tok"])
    cu = np.asarray(I["cu_seqlens"], dtype=np.int64)
    Kc, Vc = O.as_f64(I["k_cache"]), O.as_f64(I["v_cache"])
    root_feat = O.as_f64(I["root_feat"])
    if ocfg["feat"] == "fused":
        root_feat = O.linear(root_feat, W["w_fc3"])
    force = _force_from_trace(ocfg, trace, B, S)
    stats, errs = {}, []

    def step(s, reqs, rows):
        N = len(rows)
        feats, toks, pos = [], [], []
        for b, u, rid in rows:
            r = reqs[b]
            if u == 0:
                feats.append(root_feat[b])
            else:   # the other side's layer output of the row that generated u
                src = r.src_row[u]
                feats.append(np.asarray(trace["a"][s - 2][r.rows[src]["gpu_row"]], np.float64))
            toks.append(r.tok[u])
            pos.append(r.rows[rid]["pos"])
        for i, (b, u, rid) in enumerate(rows):
            reqs[b].rows[rid]["gpu_row"] = i
        x_in = np.concatenate([np.stack(feats), O.as_f64(W["embed"][np.asarray(toks)])], axis=1)

        def attend(i, k_i, v_i):
            b, _, rid = rows[i]
            r = reqs[b]
            row = r.rows[rid]
            row["k"], row["v"] = k_i, v_i
            tk = np.stack([r.rows[j]["k"] for j in row["anc"]])
            tv = np.stack([r.rows[j]["v"] for j in row["anc"]])
            lo, hi = cu[b], cu[b + 1]
            return np.concatenate([Kc[lo:hi], tk]), np.concatenate([Vc[lo:hi], tv])

        ref = O.decoder_rows(ocfg, W, x_in, np.asarray(pos), attend)
        for key in ("h", "q", "attn", "y", "a"):
            got = np.asarray(trace[key][s - 1][:N]).reshape(N, -1)
            stats[key] = max(stats.get(key, 0.0), rel_err(got, ref[key].reshape(N, -1)))
        a_other = np.asarray(trace["a"][s - 1][:N], np.float64)
        logp, lse = O.log_softmax(O.linear(a_other, W["w_lm"]))
        stats["lse"] = max(stats.get("lse", 0.0),
                           float(np.max(np.abs(np.asarray(trace["lse"][s - 1][:N], np.float64) - lse))))
        return logp, {"lse": lse}

    res = O.expand_tree(ocfg, cu[1:] - cu[:-1], I["root_tok"], step, force, margin)
    if res["log"]["mismatch"]:
        errs.append(f"decisions differ beyond the {margin} margin: {res['log']['mismatch'][:8]}")
    for b, r in enumerate(res["requests"]):
        for key in ("tokens", "parents", "positions"):
            if not np.array_equal(np.asarray(out[key][b][:S], np.int64), r[key]):
                errs.append(f"request {b}: {key} differ")
        if not np.array_equal(np.asarray(out["mask"][b][:S, :S]), r["mask"]):
            errs.append(f"request {b}: mask differs")
        if not np.array_equal(np.asarray(trace["final_nodes"][b][:S], np.int64), r["node_ids"]):
            errs.append(f"request {b}: emitted node ids differ")
        stats["logv"] = max(stats.get("logv", 0.0),
                            float(np.max(np.abs(np.asarray(out["logv"][b][:S], np.float64) - r["logv"]))))
    for s, tr in enumerate(res["trace"]):
        N = len(tr["rows"])
        kk = tr["children"].shape[1]
        if not np.array_equal(np.asarray(trace["children"][s][:N, :kk], np.int64), tr["children"]):
            errs.append(f"depth {s + 1}: children differ")
        stats["child_logp"] = max(stats.get("child_logp", 0.0), float(np.max(np.abs(
            np.asarray(trace["child_logp"][s][:N, :kk], np.float64) - tr["child_logp"]))))
    for key in ("h", "q", "attn", "y", "a"):
        if stats.get(key, 0.0) > tol_feat:
            errs.append(f"{key}: max relative error {stats[key]:.3g} > {tol_feat}")
    for key in ("lse", "logv", "child_logp"):
        if stats.get(key, 0.0) > tol_v:
            errs.append(f"{key}: max abs error {stats[key]:.3g} > {tol_v}")
    near = [m for m in res["log"]["margins"] if m[-1] < margin]
    return {"ok": not errs, "errors": errs, "stats": stats, "forced": res["log"]["forced"],
            "near_ties": near, "requests": B}
