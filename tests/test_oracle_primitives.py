"""Pins for the oracle's building blocks: closed forms, invariants, and special cases
that reduce to a library routine (torch / scipy in float64)."""
import itertools

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

from oracle import eagle_oracle as O
from eagle_speculative_decoding_03_gb300 import synth

RNG = np.random.default_rng(7)


def test_bf16_upcast_matches_torch():
    x = RNG.standard_normal(4096).astype(np.float32) * 37.0
    bits = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16)                 # torch rounds to nearest even
    assert np.array_equal(bits, ref.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(O.as_f64(bits), ref.to(torch.float64).numpy())


def test_linear_matches_full_matmul_across_row_blocks():
    K = 1 << 17                                                   # row block = 128 rows
    w = synth.f32_to_bf16_bits(RNG.standard_normal((300, K)).astype(np.float32))
    x = RNG.standard_normal((3, K))
    ref = torch.from_numpy(x) @ torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).double().T
    np.testing.assert_allclose(O.linear(x, w), ref.numpy(), rtol=1e-12, atol=1e-9)


def test_rms_norm_closed_form_and_library():
    g = RNG.standard_normal(64)
    c, eps = -2.5, 1e-6
    np.testing.assert_allclose(O.rms_norm(np.full(64, c), g, eps), g * c / np.sqrt(c * c + eps),
                               rtol=1e-14)
    x = RNG.standard_normal((5, 64)) * 3
    y = O.rms_norm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-13)
    ref = F.rms_norm(torch.from_numpy(x), (64,), weight=torch.from_numpy(g), eps=eps)
    np.testing.assert_allclose(O.rms_norm(x, g, eps), ref.numpy(), rtol=1e-12)


def test_rope_hand_example():
    # hd = 4, theta = 100: inv_freq = [1, 0.1]; pair (0, 2) turns by pos, pair (1, 3) by pos/10
    e0, e1 = np.eye(4)[0], np.eye(4)[1]
    np.testing.assert_allclose(O.rope(e0, 1, 100.0), [np.cos(1), 0, np.sin(1), 0], atol=1e-15)
    np.testing.assert_allclose(O.rope(e1, 3, 100.0), [0, np.cos(.3), 0, np.sin(.3)], atol=1e-15)


def _rope_complex(x, pos, theta):
    """Independent form: (x_i + i x_{i+hd/2}) * exp(i pos theta^(-2i/hd))."""
    hd = x.shape[-1]
    z = x[..., :hd // 2] + 1j * x[..., hd // 2:]
    z = z * np.exp(1j * pos * theta ** (-np.arange(hd // 2) * 2.0 / hd))
    return np.concatenate([z.real, z.imag], axis=-1)


def test_rope_invariants():
    q, k = RNG.standard_normal(128), RNG.standard_normal(128)
    for theta in (1e4, 5e5):
        np.testing.assert_allclose(O.rope(q, 0, theta), q, rtol=0, atol=0)
        np.testing.assert_allclose(np.linalg.norm(O.rope(q, 4099, theta)), np.linalg.norm(q), rtol=1e-13)
        np.testing.assert_allclose(O.rope(q, 777, theta), _rope_complex(q, 777, theta), atol=1e-12)
        np.testing.assert_allclose(O.rope(O.rope(q, 300, theta), 45, theta), O.rope(q, 345, theta),
                                   atol=1e-11)
        # q.k after rotation depends only on the position difference
        a = O.rope(q, 2050, theta) @ O.rope(k, 2047, theta)
        b = O.rope(q, 13, theta) @ O.rope(k, 10, theta)
        np.testing.assert_allclose(a, b, rtol=1e-10)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (8, 2), (6, 1)])
def test_gqa_attention_matches_sdpa(Hq, Hkv):
    L, hd = 37, 64
    q = RNG.standard_normal((Hq, hd))
    K = RNG.standard_normal((L, Hkv, hd))
    V = RNG.standard_normal((L, Hkv, hd))
    rep = Hq // Hkv
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(rep, 0)   # [Hq, L, hd]
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(rep, 0)
    ref = F.scaled_dot_product_attention(torch.from_numpy(q)[:, None, :], kt, vt)[:, 0, :]
    np.testing.assert_allclose(O.gqa_attention(q, K, V), ref.numpy(), rtol=1e-12, atol=1e-13)


def test_gqa_equals_mha_with_repeated_heads():
    q = RNG.standard_normal((8, 32))
    K, V = RNG.standard_normal((9, 2, 32)), RNG.standard_normal((9, 2, 32))
    mha = O.gqa_attention(q, np.repeat(K, 4, axis=1), np.repeat(V, 4, axis=1))
    np.testing.assert_allclose(O.gqa_attention(q, K, V), mha, rtol=1e-14)


def test_log_softmax_matches_scipy():
    x = RNG.standard_normal((3, 5000)) * 3 + 40
    lp, lse = O.log_softmax(x)
    np.testing.assert_allclose(lp, scipy.special.log_softmax(x, axis=1), rtol=1e-13, atol=1e-12)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(x, axis=1), rtol=1e-14)
    np.testing.assert_allclose(np.exp(lp).sum(axis=1), 1.0, rtol=1e-13)


def test_silu_matches_torch():
    x = RNG.standard_normal(1000) * 6
    np.testing.assert_allclose(O.silu(x), F.silu(torch.from_numpy(x)).numpy(), rtol=1e-14)


def test_top_k_brute_force_with_ties():
    vals = np.array([1.0, 3.0, 3.0, 2.0, 3.0, 0.5, 2.0])
    for k in range(1, len(vals) + 1):
        best = max(itertools.combinations(range(len(vals)), k),
                   key=lambda c: (sum(vals[list(c)]), [-i for i in sorted(c)]))
        sel, _ = O.top_k(vals, k)
        assert sorted(sel.tolist()) == sorted(best)
    sel, margin = O.top_k(vals, 2)
    assert sel.tolist() == [1, 2] and margin == 0.0
    sel, margin = O.top_k(vals, 3, keys=np.array([9, 8, 7, 6, 5, 4, 3]))
    assert sorted(sel.tolist()) == [1, 2, 4] and margin == 1.0


def test_valid_top_k_tolerance():
    vals = np.array([5.0, 4.0, 3.9995, 1.0])
    assert O.is_valid_top_k(vals, [0, 1], 2, 1e-3)
    assert O.is_valid_top_k(vals, [0, 2], 2, 1e-3)       # a near-tie swap is accepted
    assert not O.is_valid_top_k(vals, [0, 3], 2, 1e-3)
    assert not O.is_valid_top_k(vals, [0, 0], 2, 1e-3)
