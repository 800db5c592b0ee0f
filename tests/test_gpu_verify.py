"""GPU parity of the verification side through the C ABI: the target's one masked pass over
an emitted draft tree ("Tree attention in one verification pass", aicassindra.com) and
greedy acceptance ("How speculative decoding works", kaushalya.io), against the float64
oracle (oracle/verify_oracle.py).

Bar: per slot, the target's most likely next token bit-exact, except where the oracle's
own top-1 / top-2 margin is below 1e-3 in log-probability (there the GPU's token must be
within 1e-3 of the best: reported as forced); its log-probability and the log-sum-exp
within 1e-2; the layer output within 2e-2 max-relative; acceptance (accepted slots,
correction token) equal to the oracle's greedy walk."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from eagle_speculative_decoding_03_gb300 import binding as eb, configs, synth
from oracle import eagle_oracle as O, verify_oracle as VO
from oracle.parity import rel_err


@pytest.fixture(scope="module")
def lib():
    from eagle_speculative_decoding_03_gb300 import build
    build.build()
    return eb.load()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _setup(cfg):
    """Draft tree on the GPU, then the target's inputs."""
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    Wt, Ct = synth.make_target(cfg), synth.make_target_cache(cfg, I)
    dW = eb.device_weights(W)
    d = eb.EagleDraft(cfg, dW)
    out = d.tree(eb.device_inputs(I))
    d.check()
    S = d.info["slots"]
    d.close()
    tree = {k: out[k].contiguous() for k in ("tokens", "positions", "parents", "mask")}
    v = eb.EagleVerify(cfg, eb.device_weights(Wt), dW, max_batch=cfg.B, max_slots=S)
    cache = eb.device_weights(Ct)
    return W, I, Wt, Ct, tree, v, cache, S


def _oracle(cfg, W, I, Wt, Ct, tree_np):
    cu = I["cu_seqlens"]
    refs = []
    for b in range(cfg.B):
        lo, hi = int(cu[b]), int(cu[b + 1])
        refs.append(VO.verify_tree(synth.oracle_cfg(cfg), Wt, W, tree_np["tokens"][b], tree_np["positions"][b],
                                   tree_np["mask"][b], Ct["k_cache"][lo:hi], Ct["v_cache"][lo:hi]))
    return refs


def _walk(tokens, parents, top):
    """The greedy walk on given per-slot most likely tokens (for forced near-ties)."""
    u, acc = 0, []
    while True:
        nxt = [j for j in range(1, len(tokens)) if parents[j] == u and tokens[j] == top[u]]
        if not nxt:
            return acc, int(top[u])
        u = nxt[0]
        acc.append(u)


def _compare(cfg, res, refs, tree_np, margin=1e-3):
    got = {k: v.cpu().numpy() for k, v in res.items()}
    forced, stats = [], {"hidden": 0.0, "logp": 0.0, "lse": 0.0}
    for b, ref in enumerate(refs):
        S = len(tree_np["tokens"][b])
        if "hidden" in got:
            stats["hidden"] = max(stats["hidden"], rel_err(got["hidden"][b], ref["hidden"]))
        for i in range(S):
            lp = ref["logp"][i]
            top = VO.most_likely(lp)
            gid = int(got["top_id"][b, i])
            if gid != top:
                srt = np.sort(lp)[::-1]
                assert srt[0] - srt[1] < margin and lp[gid] >= lp[top] - margin, (b, i, gid, top)
                forced.append((b, i))
            stats["logp"] = max(stats["logp"], abs(float(got["top_logp"][b, i]) - lp[gid]))
            stats["lse"] = max(stats["lse"], abs(float(got["lse"][b, i]) - float(ref["lse"][i])))
        if "accept_len" in got:
            L = int(got["accept_len"][b])
            slots = got["accept_slots"][b][:L].tolist()
            assert (got["accept_slots"][b][L:] == -1).all()
            if not [f for f in forced if f[0] == b]:
                acc = VO.greedy_accept(tree_np["tokens"][b], tree_np["parents"][b], ref["logp"])
                assert slots == acc["slots"], (b, slots, acc["slots"])
                assert int(got["correction"][b]) == acc["correction"]
            else:
                want, corr = _walk(tree_np["tokens"][b], tree_np["parents"][b], got["top_id"][b])
                assert slots == want and int(got["correction"][b]) == corr
    assert stats["hidden"] <= 2e-2 and stats["logp"] <= 1e-2 and stats["lse"] <= 1e-2, stats
    return stats, forced


# a variant of small_dyn whose 21 slots x 8 query heads per KV head exceed one CTA's 128
# query vectors: the attention splits each request's slots into two query groups
GROUPED = configs.get("small_dyn").with_(name="small_dyn_gq8", n_heads=16, n_kv_heads=2, m=20)


@pytest.mark.parametrize("cfg", [configs.get("small_dyn"), configs.get("small_static"), configs.get("small_fused"),
                                 GROUPED], ids=lambda c: c.name)
def test_verify_matches_oracle(lib, cfg):
    W, I, Wt, Ct, tree, v, cache, S = _setup(cfg)
    res = v.verify(tree, cache, _dev(I["cu_seqlens"]), accept=True, hidden=True)
    v.check()
    tree_np = {k: t.cpu().numpy() for k, t in tree.items()}
    stats, forced = _compare(cfg, res, _oracle(cfg, W, I, Wt, Ct, tree_np), tree_np)
    print(cfg.name, {k: f"{x:.2e}" for k, x in stats.items()}, "forced:", forced)
    v.close()


def test_verify_accepts_a_rigged_deepest_path(lib):
    """Rewrite the tokens along the deepest root-to-leaf path so each is the target's most
    likely token after its parent (siblings moved off it): the whole path is accepted."""
    cfg = configs.get("small_dyn")
    W, I, Wt, Ct, tree, v, cache, S = _setup(cfg)
    cu = _dev(I["cu_seqlens"])
    tok = tree["tokens"].cpu().numpy().copy()
    par = tree["parents"].cpu().numpy()
    pos = tree["positions"].cpu().numpy()
    for b in range(cfg.B):
        leaf = int(np.argmax(pos[b]))          # a deepest slot
        path = []
        j = leaf
        while j > 0:
            path.append(j)
            j = int(par[b][j])
        path = path[::-1]
        for j in path:
            tree["tokens"] = _dev(tok)
            top = v.verify(tree, cache, cu, accept=False)["top_id"].cpu().numpy()
            want = int(top[b][par[b][j]])
            for sib in range(1, S):            # siblings keep distinct tokens
                if sib != j and par[b][sib] == par[b][j] and tok[b][sib] == want:
                    used = set(tok[b][par[b] == par[b][j]].tolist())
                    tok[b][sib] = next(t for t in range(cfg.vocab) if t not in used and t != want)
            tok[b][j] = want
    tree["tokens"] = _dev(tok)
    res = v.verify(tree, cache, cu, accept=True)
    v.check()
    tree_np = {k: t.cpu().numpy() for k, t in tree.items()}
    _, forced = _compare(cfg, res, _oracle(cfg, W, I, Wt, Ct, tree_np), tree_np)
    depth = pos - pos[:, :1]
    for b in range(cfg.B):
        if not [f for f in forced if f[0] == b]:
            assert int(res["accept_len"][b]) == int(depth[b].max())
    v.close()


def test_verify_reports_bad_tokens_and_parents(lib):
    cfg = configs.get("small_dyn")
    W, I, Wt, Ct, tree, v, cache, S = _setup(cfg)
    cu = _dev(I["cu_seqlens"])
    bad = dict(tree)
    t = tree["tokens"].clone()
    t[0, 1] = cfg.vocab + 3
    bad["tokens"] = t
    v.verify(bad, cache, cu)
    with pytest.raises(eb.EagleError) as ei:
        v.check()
    assert ei.value.status == eb.EAGLE_ERR_DEVICE and "0x4" in str(ei.value)
    bad = dict(tree)
    p = tree["parents"].clone()
    p[1, 2] = 5                       # a parent after its child
    bad["parents"] = p
    v.verify(bad, cache, cu)
    with pytest.raises(eb.EagleError):
        v.check()
    v.check()                          # cleared
    v.close()


@pytest.mark.slow
def test_verify_full_size_eagle2_b1(lib):
    """The Llama-3-8B-shaped head with its 61-slot tree (2 query groups of the attention),
    prefix 2048."""
    cfg = configs.get("eagle2_b1")
    W, I, Wt, Ct, tree, v, cache, S = _setup(cfg)
    res = v.verify(tree, cache, _dev(I["cu_seqlens"]), accept=True, hidden=True)
    v.check()
    tree_np = {k: t.cpu().numpy() for k, t in tree.items()}
    stats, forced = _compare(cfg, res, _oracle(cfg, W, I, Wt, Ct, tree_np), tree_np)
    print("eagle2_b1 verify", {k: f"{x:.2e}" for k, x in stats.items()}, "forced:", forced)
    v.close()
