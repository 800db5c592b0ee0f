"""CPU checks of the teacher-forced all-requests comparison (oracle/parity.py): it
accepts the oracle's own run laid out like the library's trace, and it flags a wrong
feature, a wrong child token and a wrong emitted parent in any request."""
import numpy as np
import pytest

from oracle import eagle_oracle as O, parity
from eagle_speculative_decoding_03_gb300 import configs, synth


def _as_trace(cfg, res):
    """The oracle's run in the layout of eagle_draft_trace_t (plus the outputs)."""
    B, D = cfg.B, cfg.depth
    R = [cfg.rows_at(s) for s in range(1, D + 1)]
    n_max, k_max = B * max(R), max(cfg.children_at(s) for s in range(1, D + 1))
    S = cfg.kept_per_request() + 1
    hq = cfg.n_heads * cfg.head_dim
    tr = {key: np.zeros((D, n_max, w)) for key, w in (("h", cfg.d), ("q", hq), ("attn", hq), ("y", cfg.d),
                                                         ("a", cfg.d))}
    tr["lse"] = np.zeros((D, n_max))
    tr["children"] = np.full((D, n_max, k_max), -1, np.int64)
    tr["child_logp"] = np.zeros((D, n_max, k_max))
    tr["frontier"] = np.full((D, B, max(R)), -1, np.int64)
    for s, t in enumerate(res["trace"]):
        N = len(t["rows"])
        for key in ("h", "q", "attn", "y", "a"):
            tr[key][s, :N] = t[key].reshape(N, -1)
        tr["lse"][s, :N] = t["lse"]
        kk = t["children"].shape[1]
        tr["children"][s, :N, :kk] = t["children"]
        tr["child_logp"][s, :N, :kk] = t["child_logp"]
        for b, f in enumerate(t["frontier"]):
            tr["frontier"][s, b, :len(f)] = f
    tr["final_nodes"] = np.stack([r["node_ids"] for r in res["requests"]])
    out = {key: np.stack([r[key] for r in res["requests"]]) for key in ("tokens", "parents", "positions", "logv",
                                                                         "mask")}
    return out, tr, S


@pytest.fixture(scope="module", params=["small_dyn", "small_static", "small_fused"])
def run(request):
    cfg = configs.get(request.param)
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    res = O.draft_tree(synth.oracle_cfg(cfg), W, I)
    return cfg, W, I, res


def test_accepts_the_oracles_own_run(run):
    cfg, W, I, res = run
    out, tr, S = _as_trace(cfg, res)
    rep = parity.compare_teacher_forced(synth.oracle_cfg(cfg), W, I, out, tr, S)
    assert rep["ok"], rep["errors"]
    assert rep["requests"] == cfg.B
    assert max(rep["stats"][k] for k in ("h", "q", "attn", "y", "a")) < 1e-12


def test_flags_a_wrong_feature_in_the_last_request(run):
    cfg, W, I, res = run
    out, tr, S = _as_trace(cfg, res)
    R = cfg.rows_at(2)
    tr["y"][1, (cfg.B - 1) * R] *= 1.1          # depth 2, first row of the last request
    rep = parity.compare_teacher_forced(synth.oracle_cfg(cfg), W, I, out, tr, S)
    assert not rep["ok"] and any(e.startswith("y:") for e in rep["errors"])


def test_flags_a_wrong_child_or_parent(run):
    cfg, W, I, res = run
    out, tr, S = _as_trace(cfg, res)
    bad = dict(tr, children=tr["children"].copy())
    row = (cfg.B - 1) * cfg.rows_at(2)
    c = bad["children"][1, row]
    taken = set(c.tolist())
    c[0] = next(t for t in range(cfg.vocab) if t not in taken)
    rep = parity.compare_teacher_forced(synth.oracle_cfg(cfg), W, I, out, bad, S, margin=1e-9)
    assert not rep["ok"]
    out2 = dict(out, parents=out["parents"].copy())
    out2["parents"][cfg.B - 1, -1] = 0 if out2["parents"][cfg.B - 1, -1] != 0 else 1
    rep = parity.compare_teacher_forced(synth.oracle_cfg(cfg), W, I, out2, tr, S)
    assert not rep["ok"] and any("parents" in e for e in rep["errors"])
