"""Helpers shared by the GPU tests: run the CUDA path on seeded inputs."""
import numpy as np

from eagle_speculative_decoding_03_gb300 import binding as eb


def run_tree(cfg, W, I, flags=0, trace=True, max_batch=None, max_prefix=None, handle=None):
    """Build a handle (unless given), run one tree; returns (handle, outputs, trace) as numpy."""
    d = handle or eb.EagleDraft(cfg, eb.device_weights(W), max_batch=max_batch,
                                max_prefix=max_prefix, flags=flags)
    dI = eb.device_inputs(I)
    tr = d.alloc_trace() if trace else None
    out = d.tree(dI, trace=tr)
    d.check()
    np_out = {k: v.cpu().numpy() for k, v in out.items()}
    np_tr = {k: v.cpu().numpy() for k, v in tr.items()} if tr is not None else None
    return d, np_out, np_tr


def rows_per_depth(cfg):
    """Rows (frontier nodes) per request at each depth 1..D."""
    return [cfg.rows_at(s) for s in range(1, cfg.depth + 1)]


def select_requests(cfg, I, out, tr, reqs):
    """Inputs, outputs and trace of a batched run restricted to the requests ``reqs``.

    Requests of one draft-tree call are independent (each attends to its own prefix and
    its own tree rows), so a subset can be checked against the oracle on its own."""
    reqs = list(reqs)
    cu = I["cu_seqlens"]
    lens = [int(cu[b + 1] - cu[b]) for b in reqs]
    sub = {"root_feat": I["root_feat"][reqs], "root_tok": I["root_tok"][reqs],
           "cu_seqlens": np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)}
    if "seeds" in I:
        sub["seeds"] = I["seeds"][reqs]
    for key in ("k_cache", "v_cache"):
        sub[key] = np.concatenate([I[key][int(cu[b]):int(cu[b + 1])] for b in reqs], axis=0)
    o = {k: v[reqs] for k, v in out.items()}
    if tr is None:
        return sub, o, None
    t = {}
    R = rows_per_depth(cfg)
    for key in ("h", "q", "attn", "y", "a", "lse", "children", "child_logp"):
        per = []
        for s in range(cfg.depth):
            idx = np.concatenate([np.arange(b * R[s], (b + 1) * R[s]) for b in reqs])
            x = tr[key][s][idx]
            pad = np.zeros((tr[key].shape[1] - len(idx),) + x.shape[1:], x.dtype)
            per.append(np.concatenate([x, pad]))
        t[key] = np.stack(per)
    t["frontier"] = tr["frontier"][:, reqs]
    for key in ("final_nodes", "tree_k", "tree_v"):
        t[key] = tr[key][reqs]
    return sub, o, t
