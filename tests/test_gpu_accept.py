"""GPU parity of multi-round speculative sampling over emitted trees (eagle_speculative_accept)
against the float64 oracle (oracle/sampling.py), on the same float32 logits and seeds.

Bar: accepted slots and the drawn token equal the oracle's, except for a request where a
decision of the oracle is a near-tie (an acceptance test within 1e-5 relative of its boundary,
or a drawn token whose Gumbel-max margin is below 1e-3): there the GPU's walk is checked to be
a valid one (reported, not failed)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from eagle_speculative_decoding_03_gb300 import binding as eb, configs, synth
from oracle import eagle_oracle as O, sampling as SP


@pytest.fixture(scope="module")
def lib():
    from eagle_speculative_decoding_03_gb300 import build
    build.build()
    return eb.load()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _near_tie(res):
    for t in res["trials"]:
        if abs(t["u"] * t["q"] - t["p"]) <= 1e-5 * max(t["p"], t["q"], 1e-30):
            return True
    return res["margin"] < 1e-3


def _check(tokens, parents, lp, lq, seeds, got):
    """lp / lq: float32 logits [B,S,V]; got: the GPU outputs (numpy)."""
    near = []
    for b in range(tokens.shape[0]):
        ref = SP.speculative_accept(tokens[b], parents[b], O.log_softmax(lp[b].astype(np.float64))[0],
                                    O.log_softmax(lq[b].astype(np.float64))[0], int(seeds[b]))
        L = int(got["accept_len"][b])
        slots = got["accept_slots"][b][:L].tolist()
        assert (got["accept_slots"][b][L:] == -1).all()
        if _near_tie(ref):
            near.append(b)
            prev = 0
            for s in slots:                                # still a path down from the root
                assert parents[b][s] == prev
                prev = s
            continue
        assert slots == ref["slots"], (b, slots, ref["slots"])
        assert int(got["correction"][b]) == ref["correction"], (b, int(got["correction"][b]), ref["correction"])
    return near


def _random_trees(rng, B, S, V, lq):
    """Random trees (a parent precedes its child); a slot's children are tokens drawn without
    replacement from the draft distribution at the parent (Gumbel-top-k, draw order)."""
    tokens = np.zeros((B, S), np.int32)
    parents = np.full((B, S), -1, np.int32)
    for b in range(B):
        par = [-1] + [int(rng.integers(0, i)) for i in range(1, S)]
        for u in range(S):
            kids = [c for c in range(1, S) if par[c] == u]
            if kids:
                lpq = O.log_softmax(lq[b, u].astype(np.float64))[0]
                sel, _, _ = SP.draw_children(lpq, len(kids), u, 1, 1000 + 97 * b)
                for c, t in zip(kids, sel):
                    tokens[b, c] = int(t)
        parents[b] = par
        tokens[b, 0] = int(rng.integers(0, V))
    return tokens, parents


@pytest.mark.parametrize("V,S,scale", [(1000, 16, 1.0), (1000, 40, 0.3), (128256, 24, 0.5)])
def test_speculative_accept_matches_oracle(lib, V, S, scale):
    rng = np.random.default_rng(V + S)
    B = 4
    lp = (rng.standard_normal((B, S, V)) * 3).astype(np.float32)
    lq = (lp + rng.standard_normal((B, S, V)) * scale).astype(np.float32)   # a draft close to the target
    tokens, parents = _random_trees(rng, B, S, V, lq)
    seeds = np.array([0x9E3779B97F4A7C15 * (b + 3) % 2 ** 64 for b in range(B)], np.uint64)
    tree = {"tokens": _dev(tokens), "parents": _dev(parents)}
    out = eb.speculative_accept(tree, _dev(lp), _dev(lq), _dev(seeds.view(np.int64)))
    torch.cuda.synchronize()
    got = {k: v.cpu().numpy() for k, v in out.items()}
    assert got["err"][0] == 0
    near = _check(tokens, parents, lp, lq, seeds, got)
    print(V, S, "accepted", got["accept_len"].tolist(), "near-ties:", near)


def test_equal_target_and_draft_accept_the_first_children(lib):
    rng = np.random.default_rng(5)
    B, S, V = 2, 12, 500
    lp = (rng.standard_normal((B, S, V)) * 2).astype(np.float32)
    tokens, parents = _random_trees(rng, B, S, V, lp)
    seeds = np.array([11, 12], np.uint64)
    out = eb.speculative_accept({"tokens": _dev(tokens), "parents": _dev(parents)}, _dev(lp), _dev(lp),
                                _dev(seeds.view(np.int64)))
    got = {k: v.cpu().numpy() for k, v in out.items()}
    for b in range(B):   # U < 1 = p/q: the walk follows first children down to a leaf
        u, want = 0, []
        while True:
            kids = [c for c in range(1, S) if parents[b][c] == u]
            if not kids:
                break
            u = kids[0]
            want.append(u)
        assert got["accept_slots"][b][:got["accept_len"][b]].tolist() == want


def test_draft_verify_accept_end_to_end(lib):
    """A sampled draft tree on the GPU, the target's logits from the verification pass, the
    draft's logits at each slot from the draft's own layer outputs: GPU acceptance equals the
    oracle's on the same arrays."""
    cfg = configs.get("small_dyn")
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    I["seeds"] = np.array([5, 6, 7], np.uint64)
    Wt, Ct = synth.make_target(cfg), synth.make_target_cache(cfg, I)
    dW = eb.device_weights(W)
    d = eb.EagleDraft(cfg, dW)
    tr = d.alloc_trace()
    out = d.tree(eb.device_inputs(I), trace=tr)
    d.check()
    S = d.info["slots"]
    tree = {k: out[k].contiguous() for k in ("tokens", "positions", "parents", "mask")}
    v = eb.EagleVerify(cfg, eb.device_weights(Wt), dW, max_batch=cfg.B, max_slots=S)
    res = v.verify(tree, eb.device_weights(Ct), _dev(I["cu_seqlens"]), accept=False, logits=True)
    v.check()
    lp = res["logits"].cpu().numpy()
    # the draft's logits at slot u: its LM head on the layer output of the row that expanded u
    fn = tr["final_nodes"].cpu().numpy()
    front = tr["frontier"].cpu().numpy()
    a = tr["a"].cpu().numpy()
    pos = out["positions"].cpu().numpy()
    R = [cfg.rows_at(s) for s in range(1, cfg.depth + 1)]
    lq = lp.copy()                                          # slots never expanded: no children
    for b in range(cfg.B):
        for u in range(S):
            depth = int(pos[b, u] - pos[b, 0])
            if depth >= cfg.depth:
                continue
            if depth == 0:
                row = b * R[0]
            else:
                f = front[depth - 1, b, :R[depth]].tolist()
                if fn[b, u] not in f:
                    continue
                row = b * R[depth] + f.index(fn[b, u])
            lq[b, u] = O.linear(a[depth, row][None].astype(np.float64), W["w_lm"])[0].astype(np.float32)
    seeds = np.array([21, 22, 23], np.uint64)
    acc = eb.speculative_accept(tree, _dev(lp), _dev(lq), _dev(seeds.view(np.int64)))
    got = {k: v.cpu().numpy() for k, v in acc.items()}
    assert got["err"][0] == 0
    near = _check(out["tokens"].cpu().numpy(), out["parents"].cpu().numpy(), lp, lq, seeds, got)
    print("end to end: accepted", got["accept_len"].tolist(), "near-ties:", near)
    v.close()
    d.close()
