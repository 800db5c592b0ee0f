"""Pins of the verification-side oracle (oracle/verify_oracle.py), CPU only.

* One masked pass over the emitted tree must give every node the same next-token
  distribution as running the target causally over that node's own root-to-node path
  (the property the tree mask and depth positions exist for: "Tree attention in one
  verification pass", aicassindra.com) — checked on trees the draft oracle emits and on
  a hand-built tree.
* Greedy acceptance must equal the deepest node whose every path token is the target's
  most likely next token, found by enumerating every node ("Acceptance length under a
  tree", aicassindra.com; "How speculative decoding works", kaushalya.io).
"""
import numpy as np
import pytest

from eagle_speculative_decoding_03_gb300 import configs, synth
from oracle import eagle_oracle as O
from oracle import verify_oracle as VO


def _draft_trees(name):
    cfg = configs.get(name)
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    res = O.draft_tree(synth.oracle_cfg(cfg), W, I)
    return cfg, W, I, res["requests"]


def _prefix(I, T, b):
    lo, hi = int(I["cu_seqlens"][b]), int(I["cu_seqlens"][b + 1])
    return hi - lo, T["k_cache"][lo:hi], T["v_cache"][lo:hi]


def _path_slots(parents, s):
    out = []
    while s != -1:
        out.append(s)
        s = int(parents[s])
    return out[::-1]


@pytest.mark.parametrize("name", ["small_dyn", "small_static"])
def test_one_masked_pass_equals_a_causal_pass_per_path(name):
    cfg, W, I, trees = _draft_trees(name)
    ocfg = synth.oracle_cfg(cfg)
    Wt = synth.make_target(cfg)
    T = synth.make_target_cache(cfg, I)
    for b, tr in enumerate(trees):
        n, kp, vp = _prefix(I, T, b)
        one = VO.verify_tree(ocfg, Wt, W, tr["tokens"], tr["positions"], tr["mask"], kp, vp)
        for s in range(len(tr["tokens"])):
            path = _path_slots(tr["parents"], s)
            ref = VO.target_path(ocfg, Wt, W, tr["tokens"][path], n, kp, vp)
            np.testing.assert_allclose(one["logp"][s], ref["logp"][-1], rtol=0, atol=1e-11)
            np.testing.assert_allclose(one["hidden"][s], ref["hidden"][-1], rtol=1e-12, atol=1e-12)


def test_hand_built_tree_and_empty_prefix():
    # root -> (1, 2); 1 -> (3); 3 -> (4): slots in generation order, parents as slots
    cfg = configs.get("small_dyn")
    ocfg = synth.oracle_cfg(cfg)
    W, Wt = synth.make_weights(cfg), synth.make_target(cfg)
    tokens = np.array([7, 11, 5, 11, 3])
    parents = np.array([-1, 0, 0, 1, 3])
    depth = np.array([0, 1, 1, 2, 3])
    mask = np.zeros((5, 5), np.uint8)
    for i in range(5):
        for j in _path_slots(parents, i):
            mask[i, j] = 1
    empty = np.zeros((0, cfg.n_kv_heads, cfg.head_dim), np.float32)
    one = VO.verify_tree(ocfg, Wt, W, tokens, depth, mask, empty, empty)
    for s in range(5):
        ref = VO.target_path(ocfg, Wt, W, tokens[_path_slots(parents, s)], 0, empty, empty)
        np.testing.assert_allclose(one["logp"][s], ref["logp"][-1], rtol=0, atol=1e-11)
    # siblings do not see each other: slot 2's row is the same with slot 1 removed
    keep = [0, 2]
    sub = VO.verify_tree(ocfg, Wt, W, tokens[keep], depth[keep], mask[np.ix_(keep, keep)], empty, empty)
    np.testing.assert_allclose(sub["logp"][1], one["logp"][2], rtol=0, atol=1e-11)
    # distributions are normalised
    np.testing.assert_allclose(np.exp(one["logp"]).sum(axis=1), 1.0, rtol=0, atol=1e-12)


def _accept_by_enumeration(tokens, parents, logp):
    """The deepest slot whose every path token is the most likely one after its parent."""
    best = 0
    for s in range(1, len(tokens)):
        path = _path_slots(parents, s)
        if all(int(tokens[c]) == VO.most_likely(logp[p]) for p, c in zip(path[:-1], path[1:])):
            if len(path) - 1 > len(_path_slots(parents, best)) - 1:
                best = s
    return best


@pytest.mark.parametrize("name", ["small_dyn", "small_static"])
def test_greedy_acceptance_is_the_deepest_passing_path(name):
    cfg, W, I, trees = _draft_trees(name)
    ocfg = synth.oracle_cfg(cfg)
    Wt = synth.make_target(cfg)
    T = synth.make_target_cache(cfg, I)
    rng = np.random.default_rng(5)
    for b, tr in enumerate(trees):
        n, kp, vp = _prefix(I, T, b)
        logp = VO.verify_tree(ocfg, Wt, W, tr["tokens"], tr["positions"], tr["mask"], kp, vp)["logp"]
        # the real target's distributions, and ones rigged so that a random node's whole
        # path passes (acceptance of a random target is almost always empty)
        rigged = logp.copy()
        s = int(rng.integers(1, len(tr["tokens"])))
        path = _path_slots(tr["parents"], s)
        for p, c in zip(path[:-1], path[1:]):
            rigged[p, int(tr["tokens"][c])] = rigged[p].max() + 1.0
        for lp in (logp, rigged):
            got = VO.greedy_accept(tr["tokens"], tr["parents"], lp)
            deepest = _accept_by_enumeration(tr["tokens"], tr["parents"], lp)
            want = _path_slots(tr["parents"], deepest)[1:]
            assert got["slots"] == want
            assert got["correction"] == VO.most_likely(lp[deepest])
        assert VO.greedy_accept(tr["tokens"], tr["parents"], rigged)["length"] >= len(path) - 1


def test_greedy_acceptance_ties_and_chain():
    # uniform target: the most likely token is 0 everywhere, so only token-0 children pass
    tokens = np.array([9, 0, 4, 0, 2])
    parents = np.array([-1, 0, 0, 1, 3])
    logp = np.full((5, 8), -np.log(8.0))
    got = VO.greedy_accept(tokens, parents, logp)
    assert got["slots"] == [1, 3] and got["tokens"] == [0, 0] and got["correction"] == 0
    # a chain whose every token is predicted is accepted whole, correction from its leaf
    chain_tok = np.array([1, 2, 3, 4])
    chain_par = np.array([-1, 0, 1, 2])
    lp = np.full((4, 6), -5.0)
    for s, t in enumerate([2, 3, 4, 5]):
        lp[s, t] = -0.1
    got = VO.greedy_accept(chain_tok, chain_par, lp)
    assert got["slots"] == [1, 2, 3] and got["correction"] == 5 and got["length"] == 3


def test_target_layer_depends_on_position_differences_only():
    # rotary embedding on both q and k: shifting every position (empty prefix) leaves the
    # output unchanged; rotating only one side would not
    cfg = configs.get("small_dyn")
    ocfg = synth.oracle_cfg(cfg)
    W, Wt = synth.make_weights(cfg), synth.make_target(cfg)
    empty = np.zeros((0, cfg.n_kv_heads, cfg.head_dim), np.float32)
    toks = np.array([3, 17, 17, 250, 4095])
    a = VO.target_path(ocfg, Wt, W, toks, 0, empty, empty)["logp"]
    b = VO.target_path(ocfg, Wt, W, toks, 777, empty, empty)["logp"]
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-10)


def test_target_layer_without_branches_is_the_normed_embedding_through_the_head():
    # with the attention and MLP output projections zeroed the layer is the identity on the
    # residual stream: logits = W_lm (RMSNorm(E[tok]) * final gain), written out here with
    # plain numpy and scipy's log-softmax
    scipy_special = pytest.importorskip("scipy.special")
    cfg = configs.get("small_dyn")
    ocfg = synth.oracle_cfg(cfg)
    W, Wt = synth.make_weights(cfg), dict(synth.make_target(cfg))
    Wt["w_o"] = np.zeros_like(Wt["w_o"])
    Wt["w_down"] = np.zeros_like(Wt["w_down"])
    empty = np.zeros((0, cfg.n_kv_heads, cfg.head_dim), np.float32)
    toks = np.array([1, 2, 3])
    got = VO.target_path(ocfg, Wt, W, toks, 5, empty, empty)["logp"]
    e = synth.bf16_bits_to_f32(W["embed"][toks]).astype(np.float64)
    normed = e / np.sqrt((e * e).mean(axis=1, keepdims=True) + cfg.rms_eps) * Wt["final_norm"].astype(np.float64)
    logits = normed @ synth.bf16_bits_to_f32(W["w_lm"]).astype(np.float64).T
    np.testing.assert_allclose(got, scipy_special.log_softmax(logits, axis=1), rtol=0, atol=1e-10)
