"""GPU parity of the fused LM-head kernel (frozen LM head + online log-softmax + top-k),
called through the C ABI, against the float64 oracle on the same inputs."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from eagle_speculative_decoding_03_gb300 import binding as eb, configs, synth
from oracle import eagle_oracle as O


@pytest.fixture(scope="module")
def lib():
    from eagle_speculative_decoding_03_gb300 import build
    build.build()
    return eb.load()


def _check_topk(a, w_lm, ids, logp, lse, k, margin=1e-3):
    lp_ref, lse_ref = O.log_softmax(O.linear(a, w_lm))
    np.testing.assert_allclose(lse, lse_ref, atol=1e-3, rtol=0)
    forced = 0
    for n in range(a.shape[0]):
        exact, mg = O.top_k(lp_ref[n], k)
        if set(ids[n].tolist()) != set(exact.tolist()):
            assert O.is_valid_top_k(lp_ref[n], ids[n], k, margin), (n, ids[n], exact, mg)
            forced += 1
        np.testing.assert_allclose(logp[n], lp_ref[n][ids[n]], atol=1e-3, rtol=0)
        assert np.all(np.diff(logp[n]) <= 0), "ids are returned by descending logit"
    return forced


@pytest.mark.parametrize("name,N,k", [("small_dyn", 10, 8), ("small_dyn", 1, 1), ("small_dyn", 37, 16),
                                      ("small_f32", 5, 3)])
def test_lm_head_topk_small(lib, name, N, k):
    cfg = configs.get(name)
    W = synth.make_weights(cfg)
    rng = np.random.default_rng(N * 100 + k)
    a = (rng.standard_normal((N, cfg.d)) * 1.17).astype(np.float32)
    rows = max(cfg.rows_at(s) for s in range(1, cfg.depth + 1))
    d = eb.EagleDraft(cfg, eb.device_weights(W), max_batch=-(-N // rows))
    ids, logp, lse = d.lm_head_topk(torch.from_numpy(a).cuda(), k)
    d.check()
    _check_topk(a, W["w_lm"], ids.cpu().numpy(), logp.cpu().numpy(), lse.cpu().numpy(), k)


def test_lm_head_all_ties_pick_lowest_ids(lib):
    cfg = configs.get("small_dyn")
    W = synth.make_weights(cfg)
    W["w_lm"] = np.zeros_like(W["w_lm"])
    a = np.random.default_rng(1).standard_normal((6, cfg.d)).astype(np.float32)
    d = eb.EagleDraft(cfg, eb.device_weights(W))
    ids, logp, lse = d.lm_head_topk(torch.from_numpy(a).cuda(), 7)
    d.check()
    assert np.array_equal(ids.cpu().numpy(), np.tile(np.arange(7), (6, 1)))
    np.testing.assert_allclose(lse.cpu().numpy(), np.log(cfg.vocab), rtol=1e-6)


@pytest.mark.slow
def test_lm_head_topk_llama3_shape(lib):
    """The LM head of the Llama-3-8B-shaped head (|V| = 128256, d = 4096), 10 rows, k = 10:
    the launch the B=1 dynamic tree makes at every depth."""
    base = configs.get("eagle2_b1")
    cfg = base.with_(d_ff=128, n_heads=1, n_kv_heads=1)   # only the LM head matters here
    W = synth.make_weights(cfg)
    a = (np.random.default_rng(3).standard_normal((10, cfg.d)) * 1.17).astype(np.float32)
    d = eb.EagleDraft(cfg, eb.device_weights(W), max_batch=1, max_prefix=16)
    ids, logp, lse = d.lm_head_topk(torch.from_numpy(a).cuda(), 10)
    d.check()
    _check_topk(a, W["w_lm"], ids.cpu().numpy(), logp.cpu().numpy(), lse.cpu().numpy(), 10)
