"""Pins for the oracle's sampling parts (oracle/sampling.py), CPU only.

* Philox4x32-10 against its published known-answer vectors (tests/golden).
* Gumbel-top-k drafting ("EAGLE-1 - autoregressive feature drafting", zackli.ai: the
  draft samples t-hat from p-hat): over many seeds the first child's frequencies match the
  softmax, and ordered pairs match sampling without replacement, p_i p_j / (1 - p_i).
* Multi-round speculative sampling over a tree: exact enumeration of the rule's output
  distribution equals the target's distribution when the children were drawn in order
  without replacement from the draft's; the oracle's own sampler, run over many seeds on
  small trees, reproduces the target's distribution (chi-square); degenerate cases."""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import sampling as SP

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_philox_known_answers():
    kat = json.load(open(os.path.join(GOLDEN, "philox4x32_10_kat.json")))
    for v in kat["vectors"]:
        c = [int(x, 16) for x in v["ctr"]]
        k = [int(x, 16) for x in v["key"]]
        out = SP.philox4x32_10([c[0]], [c[1]], [c[2]], [c[3]], k[0], k[1])
        assert [f"{int(w[0]):08x}" for w in out] == v["out"]


def test_uniform_stays_inside_open_interval_and_gumbel_is_finite():
    x = np.array([0, 1, 2 ** 31, 2 ** 32 - 2, 2 ** 32 - 1], dtype=np.uint64)
    g = SP.gumbel_from_words(x)
    assert np.all(np.isfinite(g))
    assert np.all(np.diff(g) > 0)                       # monotone in the word
    # G = -log(-log U) for U = (x + 1/2) / 2^32 where the direct form is accurate
    u = (x[1:3].astype(np.float64) + 0.5) / 2 ** 32
    np.testing.assert_allclose(g[1:3], -np.log(-np.log(u)), rtol=1e-12)


def _chi2(counts, probs):
    n = counts.sum()
    e = n * probs
    return float(((counts - e) ** 2 / e).sum())


# chi-square 0.9999 quantiles for 1..4 degrees of freedom
CHI2_9999 = {1: 15.14, 2: 18.42, 3: 21.11, 4: 23.51, 5: 25.74, 11: 35.0}


@pytest.mark.parametrize("logits", [[0.3, -0.4], [1.0, 0.0, -1.0, 2.0, 0.5]])
def test_gumbel_top1_frequencies_match_softmax(logits):
    lp = np.array(logits) - np.log(np.exp(logits).sum())
    n = 20000
    counts = np.zeros(len(lp))
    for seed in range(n):
        sel, _, _ = SP.draw_children(lp, 1, 0, 1, seed * 7919 + 3)
        counts[sel[0]] += 1
    assert _chi2(counts, np.exp(lp)) < CHI2_9999[len(lp) - 1]


def test_gumbel_top2_pairs_match_sampling_without_replacement():
    lp = np.log(np.array([0.4, 0.3, 0.2, 0.1]))
    p = np.exp(lp)
    pairs = list(itertools.permutations(range(4), 2))
    want = np.array([p[i] * p[j] / (1 - p[i]) for i, j in pairs])
    counts = np.zeros(len(pairs))
    for seed in range(20000):
        sel, key, _ = SP.draw_children(lp, 2, 3, 2, 1000003 + seed)
        assert key[sel[0]] >= key[sel[1]]               # draw order
        counts[pairs.index((int(sel[0]), int(sel[1])))] += 1
    assert _chi2(counts, want) < CHI2_9999[11]


# ------------------------------------------------- the acceptance rule, by enumeration
def _exact_first_token(p, q, n):
    """Distribution of the first emitted token when n children are drawn in order without
    replacement from q and tried in that order (independent of the oracle's code)."""
    V = len(p)
    out = np.zeros(V)
    for seq in itertools.permutations(range(V), n):
        pr, avail = 1.0, 1.0
        for x in seq:                                     # P(this draw sequence)
            pr *= q[x] / avail
            avail -= q[x]
        if pr == 0:
            continue
        pc, qm, reach = p.copy(), q.copy(), 1.0
        for x in seq:
            qi = qm / qm.sum()
            acc = min(1.0, pc[x] / qi[x])
            out[x] += pr * reach * acc
            reach *= 1 - acc
            res = np.maximum(pc - qi, 0)
            if res.sum() > 0:
                pc = res / res.sum()
            qm[x] = 0.0
        out += pr * reach * pc
    return out


@pytest.mark.parametrize("n", [1, 2, 3])
def test_rule_preserves_the_target_distribution_exactly(n):
    rng = np.random.default_rng(n)
    for _ in range(5):
        p = rng.dirichlet(np.ones(4))
        q = rng.dirichlet(np.ones(4))
        np.testing.assert_allclose(_exact_first_token(p, q, n), p, atol=1e-12)


def test_oracle_residual_chain_matches_the_rule():
    """All drafted tokens impossible under the target: every child is rejected, and the
    oracle's per-trial proposal probabilities and final target follow the rule."""
    p = np.array([0.0, 0.0, 0.5, 0.3, 0.2])
    q = np.array([0.3, 0.25, 0.1, 0.15, 0.2])
    tokens, parents = [9, 0, 1], [-1, 0, 0]
    res = SP.speculative_accept(tokens, parents, np.log(np.maximum(p, 1e-300))[None].repeat(3, 0),
                                np.log(q)[None].repeat(3, 0), seed=5)
    assert res["length"] == 0 and [t["accepted"] for t in res["trials"]] == [False, False]
    np.testing.assert_allclose([t["q"] for t in res["trials"]], [0.3, 0.25 / 0.7], rtol=1e-12)
    r1 = np.maximum(p - q, 0)
    r1 /= r1.sum()
    q2 = q.copy()
    q2[0] = 0
    q2 /= q2.sum()
    r2 = np.maximum(r1 - q2, 0)
    r2 /= r2.sum()
    np.testing.assert_allclose(res["final_target"], r2, rtol=1e-12, atol=1e-15)
    assert res["correction"] in (2, 3, 4) and res["rejections_at_end"] == 2


def test_equal_distributions_accept_the_first_child():
    lp = np.log(np.array([0.1, 0.2, 0.3, 0.4]))
    for seed in range(50):
        res = SP.speculative_accept([0, 3, 1], [-1, 0, 0], lp[None].repeat(3, 0), lp[None].repeat(3, 0), seed)
        assert res["slots"][:1] == [1]


def test_sampler_reproduces_the_target_on_small_trees():
    """Root with two children drawn from q_root (without replacement), the first child with
    one child of its own drawn from q_c: over many seeds the first emitted token follows
    p_root, and given the first child was accepted, the second follows p_c."""
    rng = np.random.default_rng(42)
    V = 4
    p_root, q_root = rng.dirichlet(np.ones(V)), rng.dirichlet(np.ones(V))
    p_c, q_c = rng.dirichlet(np.ones(V)), rng.dirichlet(np.ones(V))
    first, second = np.zeros(V), {}
    for seed in range(12000):
        kids, _, _ = SP.draw_children(np.log(q_root), 2, 0, 1, 77 + 2 * seed)
        g, _, _ = SP.draw_children(np.log(q_c), 1, 0, 2, 78 + 2 * seed)
        tokens = [0, int(kids[0]), int(kids[1]), int(g[0])]
        parents = [-1, 0, 0, 1]
        lp = np.log(np.stack([p_root, p_c, p_root, p_root]))   # slot 2 and 3 are not expanded here
        lq = np.log(np.stack([q_root, q_c, q_root, q_root]))
        lp[3] = np.log(p_root)
        res = SP.speculative_accept(tokens, parents, lp, lq, seed)
        emitted = res["tokens"] + [res["correction"]]
        first[emitted[0]] += 1
        if res["slots"][:1] == [1]:
            second.setdefault(0, np.zeros(V))[emitted[1]] += 1
    assert _chi2(first, p_root) < CHI2_9999[V - 1]
    assert _chi2(second[0], p_c) < CHI2_9999[V - 1]


def test_sampled_children_compare_their_draw_order():
    """In sampled drafting the draw order is part of the decision (a child's slot picks the
    noise of its own row later): the other side's order is adopted at a near-tie of the
    perturbed values and is a mismatch beyond it; the greedy comparison ignores order."""
    from oracle.eagle_oracle import _choose
    v = np.array([0.1, 2.0, 1.0, 1.0 + 4e-4, -3.0, 0.5])
    def run(forced, ordered):
        log = {"forced": [], "mismatch": [], "margins": []}
        sel, _ = _choose(v, 3, None, forced, 1e-3, log, "w", ordered=ordered)
        return sel.tolist(), log
    assert run([1, 3, 2], True) == ([1, 3, 2], {"forced": [], "mismatch": [], "margins": []})
    sel, log = run([1, 2, 3], True)               # swapped within 4e-4: adopted
    assert sel == [1, 2, 3] and log["forced"] == ["w"] and not log["mismatch"]
    sel, log = run([2, 1, 3], True)               # 1.0 drawn before 2.0: a real difference
    assert sel == [1, 3, 2] and log["mismatch"] == ["w"]
    sel, log = run([2, 1, 3], False)              # greedy: the set decides
    assert sel == [1, 3, 2] and not log["mismatch"] and not log["forced"]
