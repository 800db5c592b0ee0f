"""GPU parity of sampled drafting through the C ABI ("EAGLE-1 - autoregressive feature
drafting", zackli.ai: the draft samples t-hat ~ p-hat).  With per-request seeds a node's
children are k tokens drawn without replacement from the draft's distribution (the top-k of
log p + Gumbel noise from Philox4x32-10), in draw order; the float64 oracle draws the same
noise from its own Philox.  Same bar as greedy drafting: structure exact except near-ties
of the perturbed values below 1e-3, features 2e-2, values 1e-2."""
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


def _seeds(B, base):
    return np.array([(base * 0x9E3779B97F4A7C15 + 0x1234567 * (b + 1)) % 2 ** 64 for b in range(B)], np.uint64)


@pytest.mark.parametrize("name", ["small_dyn", "small_static", "small_fused", "small_max", "small_f32", "small_wide", "small_pairs"])
def test_sampled_tree_matches_oracle(lib, name):
    cfg = configs.get(name)
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    I["seeds"] = _seeds(cfg.B, 7)
    d, out, tr = run_tree(cfg, W, I)
    rep = parity.compare(synth.oracle_cfg(cfg), W, I, out, tr, d.info["slots"])
    print(name, {k: f"{v:.2e}" for k, v in rep["stats"].items()}, "forced:", rep["forced"])
    assert rep["ok"], rep["errors"]


def test_seeds_change_the_tree_and_repeat_exactly(lib):
    cfg = configs.get("small_dyn")
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    d = eb.EagleDraft(cfg, eb.device_weights(W))
    greedy = {k: v.cpu().numpy() for k, v in d.tree(eb.device_inputs(I)).items()}
    trees = []
    for base in (1, 2, 1):
        I2 = dict(I, seeds=_seeds(cfg.B, base))
        trees.append({k: v.cpu().numpy() for k, v in d.tree(eb.device_inputs(I2)).items()})
    d.check()
    for k in trees[0]:
        assert np.array_equal(trees[0][k], trees[2][k]), k          # same seeds, same tree
    assert not np.array_equal(trees[0]["tokens"], trees[1]["tokens"])
    assert not np.array_equal(trees[0]["tokens"], greedy["tokens"])
    # graph replay without seeds is still the greedy tree
    again = {k: v.cpu().numpy() for k, v in d.tree(eb.device_inputs(I)).items()}
    for k in greedy:
        assert np.array_equal(greedy[k], again[k]), k


@pytest.mark.slow
def test_sampled_tree_full_size_eagle2_b1(lib):
    cfg = configs.get("eagle2_b1")
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    I["seeds"] = _seeds(1, 3)
    d, out, tr = run_tree(cfg, W, I)
    rep = parity.compare(synth.oracle_cfg(cfg), W, I, out, tr, d.info["slots"])
    print("eagle2_b1 sampled", {k: f"{v:.2e}" for k, v in rep["stats"].items()}, "forced:", rep["forced"])
    assert rep["ok"], rep["errors"]
