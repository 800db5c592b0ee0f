"""The allocation-free LM-head top-k (eagle_lm_head_topk_noalloc).

Some callers cannot allocate device memory: a serving engine that reserved almost all
of HBM for its own pools at start-up, or a latency-critical loop where cudaMalloc would
synchronise the device.  For them the library offers a handle-less variant of the LM-head
top-k whose scratch lives in a file-scope device array.  These checks call it through the
C ABI twice in a row (the array keeps the previous call's contents) and compare it with
the handle-based entry point eagle_draft_lm_head_topk on the same inputs.
"""
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


def _same_result(ref, got, lp_ref, k):
    ids_r, logp_r, lse_r = (t.cpu().numpy() for t in ref)
    ids_g, logp_g, lse_g = (t.cpu().numpy() for t in got)
    np.testing.assert_allclose(lse_g, lse_r, atol=1e-3, rtol=0)
    for n in range(ids_r.shape[0]):
        if not np.array_equal(ids_g[n], ids_r[n]):
            # only a near-tie (within the 1e-3 margin the parity tests use) may reorder ids
            assert O.is_valid_top_k(lp_ref[n], ids_g[n], k, 1e-3), (n, ids_g[n], ids_r[n])
        np.testing.assert_allclose(logp_g[n], lp_ref[n][ids_g[n]], atol=1e-3, rtol=0)
    np.testing.assert_allclose(np.sort(logp_g, axis=1), np.sort(logp_r, axis=1), atol=1e-3, rtol=0)


@pytest.mark.parametrize("name,N,k", [("small_dyn", 10, 8), ("small_fused", 16, 5)])
def test_noalloc_matches_handle_entry_point_twice(lib, name, N, k):
    cfg = configs.get(name)
    W = synth.make_weights(cfg)
    dW = eb.device_weights(W)
    rng = np.random.default_rng(N + 7 * k)
    a_np = (rng.standard_normal((N, cfg.d)) * synth.FEATURE_RMS).astype(np.float32)
    a = torch.from_numpy(a_np).cuda()
    lp_ref, _ = O.log_softmax(O.linear(a_np, W["w_lm"]))

    rows = max(cfg.rows_at(s) for s in range(1, cfg.depth + 1))
    handle = eb.EagleDraft(cfg, dW, max_batch=-(-N // rows))
    ref = handle.lm_head_topk(a, k)
    handle.check()
    for _ in range(2):
        got = eb.lm_head_topk_noalloc(dW["w_lm"], a, k)
        torch.cuda.synchronize()
        _same_result(ref, got, lp_ref, k)
    handle.close()


@pytest.mark.slow
def test_noalloc_llama3_vocab_matches_handle_entry_point_twice(lib):
    """The Llama-3-8B-shaped LM head (|V| = 128256, d = 4096: 1002 vocabulary tiles over the
    full SM grid), N = 16 rows, k = 16: the largest launch the array is laid out for."""
    base = configs.get("eagle2_b1")
    cfg = base.with_(d_ff=128, n_heads=1, n_kv_heads=1, k=16, m=16, depth=2)   # only the LM head matters
    W = synth.make_weights(cfg)
    dW = eb.device_weights(W)
    N, k = 16, 16
    a_np = (np.random.default_rng(11).standard_normal((N, cfg.d)) * synth.FEATURE_RMS).astype(np.float32)
    a = torch.from_numpy(a_np).cuda()
    lp_ref, _ = O.log_softmax(O.linear(a_np, W["w_lm"]))
    handle = eb.EagleDraft(cfg, dW, max_batch=1, max_prefix=16)
    ref = handle.lm_head_topk(a, k)
    handle.check()
    for _ in range(2):
        got = eb.lm_head_topk_noalloc(dW["w_lm"], a, k)
        torch.cuda.synchronize()
        _same_result(ref, got, lp_ref, k)
    handle.close()


def test_noalloc_allocates_nothing(lib):
    cfg = configs.get("small_dyn")
    dW = eb.device_weights(synth.make_weights(cfg))
    a = torch.randn(4, cfg.d, device="cuda")
    eb.lm_head_topk_noalloc(dW["w_lm"], a, 3)       # first call: set-up on this device
    torch.cuda.synchronize()
    ids = torch.empty((4, 3), dtype=torch.int32, device="cuda")
    logp = torch.empty((4, 3), dtype=torch.float32, device="cuda")
    lse = torch.empty((4,), dtype=torch.float32, device="cuda")
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        st = lib.eagle_lm_head_topk_noalloc(dW["w_lm"].data_ptr(), cfg.vocab, cfg.d, a.data_ptr(), 4, 3,
                                            ids.data_ptr(), logp.data_ptr(), lse.data_ptr(), None)
        assert st == eb.EAGLE_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_noalloc_rejects_sizes_beyond_its_maximum(lib):
    cfg = configs.get("small_dyn")
    dW = eb.device_weights(synth.make_weights(cfg))
    for N, k in ((17, 4), (4, 17)):
        a = torch.randn(N, cfg.d, device="cuda")
        with pytest.raises(eb.EagleError) as ei:
            eb.lm_head_topk_noalloc(dW["w_lm"], a, k)
        assert ei.value.status == eb.EAGLE_ERR_INVALID_ARG
        assert "noalloc" in str(ei.value)
