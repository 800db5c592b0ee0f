"""Pins for the DFlash block-parallel draft oracle (oracle/dflash_oracle.py), CPU only.

* A separately written torch float64 stack ("DFlash-1: parallel block + KV injection",
  zackli.ai: Q from the block, K / V = [injected context ; block], bidirectional inside the
  block) built from library routines (rms_norm, complex-number rotary, non-causal
  scaled_dot_product_attention, silu) equals the oracle.
* Attention treats the injected context as a set: permuting its rows changes nothing.
* Identity layers (W_o = W_down = 0) leave every row at its embedding: the mask rows' logits
  are W_lm RMSNorm(E(MASK)) in closed form, the same for every mask row.
* Bidirectionality: the first mask row depends on the last slot of the block.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import dflash_oracle as D, eagle_oracle as O
from eagle_speculative_decoding_03_gb300 import configs, synth

CFG = configs.DFLASH["small_dflash"]


@pytest.fixture(scope="module")
def setup():
    W, I = synth.make_dflash_weights(CFG), synth.make_dflash_inputs(CFG)
    return W, I, D.dflash_draft(synth.dflash_oracle_cfg(CFG), W, I, k=CFG.k)


def _torch_block(cfg, W, anchor, ctx_k, ctx_v, n, mask_tok):
    T = lambda a: torch.from_numpy(O.as_f64(a))
    Hq, Hkv, hd, g = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.gamma
    toks = [anchor] + [mask_tok] * g
    x = T(W["embed"][np.array(toks)])
    inv = cfg.rope_theta ** (-torch.arange(hd // 2, dtype=torch.float64) * 2 / hd)
    pos = (n + torch.arange(g + 1, dtype=torch.float64))[:, None, None]

    def rot(t):
        z = torch.complex(t[..., :hd // 2], t[..., hd // 2:]) * torch.polar(torch.ones_like(inv), pos * inv)
        return torch.cat([z.real, z.imag], -1)

    for l, L in enumerate(W["layers"]):
        h = F.rms_norm(x, (cfg.d,), T(L["attn_norm"]), cfg.rms_eps) @ T(L["w_qkv"]).T
        q = rot(h[:, :Hq * hd].view(-1, Hq, hd))
        k = rot(h[:, Hq * hd:(Hq + Hkv) * hd].view(-1, Hkv, hd))
        v = h[:, (Hq + Hkv) * hd:].view(-1, Hkv, hd)
        K = torch.cat([T(ctx_k[l]), k]).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        V = torch.cat([T(ctx_v[l]), v]).permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)
        att = F.scaled_dot_product_attention(q.permute(1, 0, 2), K, V).permute(1, 0, 2).reshape(g + 1, -1)
        y = x + att @ T(L["w_o"]).T
        z = F.rms_norm(y, (cfg.d,), T(L["mlp_norm"]), cfg.rms_eps)
        x = y + (F.silu(z @ T(L["w_gate"]).T) * (z @ T(L["w_up"]).T)) @ T(L["w_down"]).T
    return torch.log_softmax(F.rms_norm(x, (cfg.d,), T(W["final_norm"]), cfg.rms_eps) @ T(W["w_lm"]).T, -1).numpy()


def test_block_equals_a_separate_torch_stack(setup):
    W, I, res = setup
    cu = I["cu_seqlens"]
    for b, r in enumerate(res):
        lo, hi = int(cu[b]), int(cu[b + 1])
        ref = _torch_block(CFG, W, int(I["anchor"][b]), [c[lo:hi] for c in I["ctx_k"]],
                           [c[lo:hi] for c in I["ctx_v"]], hi - lo, CFG.mask_id)
        np.testing.assert_allclose(r["logp"], ref, rtol=1e-11, atol=1e-11)
        want = np.stack([np.sort(O.top_k(ref[i], CFG.k)[0]) for i in range(1, CFG.gamma + 1)])
        assert np.array_equal(np.sort(r["tokens"], axis=1), want)


def test_context_is_a_set(setup):
    W, I, res = setup
    cu = I["cu_seqlens"]
    b = 2
    lo, hi = int(cu[b]), int(cu[b + 1])
    perm = np.random.default_rng(0).permutation(hi - lo)
    r2 = D.dflash_block(synth.dflash_oracle_cfg(CFG), W, int(I["anchor"][b]), hi - lo,
                        [c[lo:hi][perm] for c in I["ctx_k"]], [c[lo:hi][perm] for c in I["ctx_v"]], CFG.k)
    np.testing.assert_allclose(r2["logp"], res[b]["logp"], rtol=1e-10, atol=1e-12)


def test_identity_layers_give_the_embedding_logits():
    W, I = synth.make_dflash_weights(CFG), synth.make_dflash_inputs(CFG)
    for L in W["layers"]:
        L["w_o"] = np.zeros_like(L["w_o"])
        L["w_down"] = np.zeros_like(L["w_down"])
    r = D.dflash_draft(synth.dflash_oracle_cfg(CFG), W, I, k=1)[0]
    e = O.as_f64(W["embed"][CFG.mask_id])
    xn = e / np.sqrt(np.mean(e * e) + CFG.rms_eps) * O.as_f64(W["final_norm"])
    logits = O.as_f64(W["w_lm"]) @ xn
    want = logits - (logits.max() + np.log(np.exp(logits - logits.max()).sum()))
    for i in range(1, CFG.gamma + 1):
        np.testing.assert_allclose(r["logp"][i], want, rtol=1e-11, atol=1e-11)


def test_empty_context_and_bidirectional_block():
    W = synth.make_dflash_weights(CFG)
    cfgd = synth.dflash_oracle_cfg(CFG)
    kvs = (0, CFG.n_kv_heads, CFG.head_dim)
    empty = [np.zeros(kvs, np.uint16)] * CFG.layers
    r = D.dflash_block(cfgd, W, 5, 0, empty, empty, 1)
    np.testing.assert_allclose(r["logp"], _torch_block(CFG, W, 5, empty, empty, 0, CFG.mask_id),
                               rtol=1e-11, atol=1e-11)
    # a block [anchor, MASK] against [anchor, token 7]: the anchor row reads the slot after it
    # (bidirectional inside the block; a causal stack would leave row 0 unchanged)
    masked = D.dflash_block(dict(cfgd, gamma=1), W, 5, 0, empty, empty, 1)
    other = D.dflash_block(dict(cfgd, gamma=1, mask_token=7), W, 5, 0, empty, empty, 1)
    assert np.max(np.abs(other["logp"][0] - masked["logp"][0])) > 1e-3
