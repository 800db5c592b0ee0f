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
