"""End-to-end GPU parity of the draft-tree step through the C ABI against the float64
oracle: tree structure bit-exact (near-ties within 1e-3 reported), features within 2e-2
relative, path values within 1e-2."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from eagle_speculative_decoding_03_gb300 import binding as eb, configs, synth
from oracle import parity
from tests.gpu_util import run_tree


@pytest.fixture(scope="module")
def lib():
    from eagle_speculative_decoding_03_gb300 import build
    build.build()
    return eb.load()


SMALL = ["tiny_chain", "small_f32", "small_dyn", "small_static", "small_fused", "small_max", "small_wide", "small_pairs"]


@pytest.mark.parametrize("name", SMALL)
def test_tree_parity_small(lib, name):
    cfg = configs.get(name)
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    d, out, tr = run_tree(cfg, W, I)
    rep = parity.compare(synth.oracle_cfg(cfg), W, I, out, tr, d.info["slots"])
    print(name, {k: f"{v:.2e}" for k, v in rep["stats"].items()}, "forced:", rep["forced"])
    assert rep["ok"], rep["errors"]


@pytest.mark.parametrize("name", ["small_max", "small_wide"])
def test_tree_parity_fused_lm_epilogue_many_rows(lib, name, monkeypatch):
    # depths of 24 to 96 rows normally store the logits for the select kernel; with the
    # crossover raised the LM head keeps its multi-chunk log-sum-exp + top-k epilogue
    monkeypatch.setenv("EAGLE_LM_LOGITS_MIN_ROWS", "100000")
    cfg = configs.get(name)
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    d, out, tr = run_tree(cfg, W, I)
    rep = parity.compare(synth.oracle_cfg(cfg), W, I, out, tr, d.info["slots"])
    assert rep["ok"], rep["errors"]


@pytest.mark.parametrize("name", ["small_dyn", "small_static", "small_fused", "small_max", "small_wide"])
def test_tree_parity_attention_128_key_tiles(lib, name, monkeypatch):
    # launches whose CTAs walk few tiles keep 64-key tiles; force the 128-key instance over
    # the small cases' ragged prefixes (3 to 200 keys: partial, shifted and single tiles)
    monkeypatch.setenv("EAGLE_ATTN_TILE", "128")
    cfg = configs.get(name)
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    d, out, tr = run_tree(cfg, W, I)
    rep = parity.compare(synth.oracle_cfg(cfg), W, I, out, tr, d.info["slots"])
    assert rep["ok"], rep["errors"]


def test_partial_batch_and_empty_prefix_128_key_tiles(lib, monkeypatch):
    monkeypatch.setenv("EAGLE_ATTN_TILE", "128")
    cfg = configs.get("small_dyn")
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg, B=2, seed_offset=5)
    n1 = int(I["cu_seqlens"][2] - I["cu_seqlens"][1])
    I["k_cache"], I["v_cache"] = I["k_cache"][-n1:], I["v_cache"][-n1:]
    I["cu_seqlens"] = np.array([0, 0, n1], np.int32)
    d, out, tr = run_tree(cfg, W, I, max_batch=3)
    rep = parity.compare(synth.oracle_cfg(cfg), W, I, out, tr, d.info["slots"])
    assert rep["ok"], rep["errors"]


@pytest.mark.parametrize("name", ["small_dyn", "small_static", "small_fused"])
def test_graph_replay_matches_direct_launch(lib, name):
    cfg = configs.get(name)
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    d, out_trace, _ = run_tree(cfg, W, I, trace=True)
    _, out_graph, _ = run_tree(cfg, W, I, trace=False, handle=d)
    _, out_graph2, _ = run_tree(cfg, W, I, trace=False, handle=d)
    _, out_plain, _ = run_tree(cfg, W, I, trace=False, flags=eb.FLAG_NO_GRAPH | eb.FLAG_NO_PDL)
    for k in out_trace:
        assert np.array_equal(out_trace[k], out_graph[k]), k
        assert np.array_equal(out_graph[k], out_graph2[k]), k
        assert np.array_equal(out_graph[k], out_plain[k]), k


def test_partial_batch_and_empty_prefix(lib):
    cfg = configs.get("small_dyn")
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg, B=2, seed_offset=5)
    # request 0 has no verified prefix at all: it attends to its tree rows only
    n1 = int(I["cu_seqlens"][2] - I["cu_seqlens"][1])
    I["k_cache"], I["v_cache"] = I["k_cache"][-n1:], I["v_cache"][-n1:]
    I["cu_seqlens"] = np.array([0, 0, n1], np.int32)
    d, out, tr = run_tree(cfg, W, I, max_batch=3)
    rep = parity.compare(synth.oracle_cfg(cfg), W, I, out, tr, d.info["slots"])
    assert rep["ok"], rep["errors"]
    assert out["positions"][0][0] == 0


def test_zero_lm_head_ties(lib):
    cfg = configs.get("small_dyn")
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    W["w_lm"] = np.zeros_like(W["w_lm"])
    d, out, tr = run_tree(cfg, W, I)
    rep = parity.compare(synth.oracle_cfg(cfg), W, I, out, tr, d.info["slots"])
    assert rep["ok"], rep["errors"]
    assert rep["forced"] == []
    # all children are tokens 0..k-1; the frontier and the rerank keep the lowest node ids
    assert out["tokens"][0][1:cfg.k + 1].tolist() == list(range(cfg.k))


@pytest.mark.parametrize("name", ["small_wide", "small_pairs"])
def test_select_kernel_ties(lib, name):
    # depths of 96 / 192 rows store the logits for the select kernel; an LM head of zeros but
    # one row makes every part a run of equal keys (the radix fallback: the lowest ids win),
    # with token 5 above or below the ties depending on the row
    cfg = configs.get(name)
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    w = np.zeros_like(W["w_lm"])
    w[5] = W["w_lm"][5]
    W["w_lm"] = w
    d, out, tr = run_tree(cfg, W, I)
    rep = parity.compare(synth.oracle_cfg(cfg), W, I, out, tr, d.info["slots"])
    assert rep["ok"], rep["errors"]
    # the select decisions are exact (equal keys: lowest ids); the frontier and the rerank may
    # meet path values equal in float64 but not in float32, forced within the margin
    assert [f for f in rep["forced"] if f[0] == "children"] == []
    kids = out["tokens"][:, 1:cfg.k + 1]
    assert all(set(r.tolist()) <= {0, 1, 2, 3, 4, 5} for r in kids)


def test_prefix_longer_than_max_prefix_is_reported(lib):
    cfg = configs.get("small_dyn")
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    d = eb.EagleDraft(cfg, eb.device_weights(W), max_prefix=16)
    d.tree(eb.device_inputs(I))
    with pytest.raises(eb.EagleError) as ei:
        d.check()
    assert ei.value.status == eb.EAGLE_ERR_DEVICE
    d.check()   # the word was cleared


def test_out_of_range_root_token_is_reported(lib):
    cfg = configs.get("small_dyn")
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    I["root_tok"] = I["root_tok"].copy()
    I["root_tok"][1] = cfg.vocab + 5
    d = eb.EagleDraft(cfg, eb.device_weights(W))
    d.tree(eb.device_inputs(I))
    with pytest.raises(eb.EagleError) as ei:
        d.check()
    assert ei.value.status == eb.EAGLE_ERR_DEVICE and "0x4" in str(ei.value)


def test_non_finite_logits_are_reported_and_stay_in_bounds(lib):
    # an LM head of NaNs: no row has a valid next-token candidate; the library flags it
    # in the device error word and every emitted index stays inside its table
    cfg = configs.get("small_dyn")
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    W["w_lm"] = np.full_like(W["w_lm"], 0x7FC0)          # bf16 quiet NaN
    d = eb.EagleDraft(cfg, eb.device_weights(W))
    out = {k: v.cpu().numpy() for k, v in d.tree(eb.device_inputs(I)).items()}
    with pytest.raises(eb.EagleError) as ei:
        d.check()
    assert ei.value.status == eb.EAGLE_ERR_DEVICE and "0x8" in str(ei.value)
    S = d.info["slots"]
    assert ((out["tokens"] >= 0) & (out["tokens"] < cfg.vocab)).all()
    assert ((out["parents"] >= -1) & (out["parents"] < S)).all()
    assert set(np.unique(out["mask"])) <= {0, 1}


def test_invalid_batch_rejected(lib):
    cfg = configs.get("small_dyn")
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    d = eb.EagleDraft(cfg, eb.device_weights(W), max_batch=2)
    with pytest.raises(eb.EagleError) as ei:
        d.tree(eb.device_inputs(I))
    assert ei.value.status == eb.EAGLE_ERR_INVALID_ARG
