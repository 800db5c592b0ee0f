"""GPU parity at the full workload sizes, through the C ABI, in the launch configuration
the benchmark times (graph replay with programmatic dependent launch).

The oracle follows every request of a call independently, so for the batched workloads
it checks a sample of requests (the shortest and the longest prefix, and one between)
against the same rows of the full-batch GPU run, and then every request teacher-forced:
at each depth the oracle runs the layer on the GPU's own inputs and takes the LM head,
children, frontier and rerank from the GPU's layer output.  Tolerances are those of the small
parity tests: structure exact except near-ties below 1e-3 in log probability, features
2e-2 relative, path values 1e-2 absolute."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from eagle_speculative_decoding_03_gb300 import binding as eb, configs, synth
from oracle import parity
from tests.gpu_util import run_tree, select_requests


@pytest.fixture(scope="module")
def lib():
    from eagle_speculative_decoding_03_gb300 import build
    build.build()
    return eb.load()


def _sample(I, n):
    lens = np.diff(I["cu_seqlens"])
    order = np.argsort(lens, kind="stable")
    pick = [int(order[0]), int(order[-1]), int(order[len(order) // 2])]
    return sorted(set(pick))[:n]


@pytest.mark.parametrize("name,n_req", [("eagle2_b1", 1), ("eagle1_static", 1), ("eagle2_b32", 3),
                                        ("eagle3_b8", 1)])
def test_tree_parity_full_size(lib, name, n_req):
    cfg = configs.get(name)
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    d = eb.EagleDraft(cfg, eb.device_weights(W))
    dI = eb.device_inputs(I)
    out_g = {k: v.cpu().numpy() for k, v in d.tree(dI).items()}   # graph replay, as timed
    d.check()
    d2, out, tr = run_tree(cfg, W, I, handle=d)                   # the same call with a trace
    for k in out:
        assert np.array_equal(out[k], out_g[k]), k
    reqs = list(range(cfg.B)) if cfg.B <= n_req else _sample(I, n_req)
    sI, sout, str_ = select_requests(cfg, I, out, tr, reqs)
    rep = parity.compare(synth.oracle_cfg(cfg), W, sI, sout, str_, d.info["slots"])
    print(name, reqs, {k: f"{v:.2e}" for k, v in rep["stats"].items()}, "forced:", rep["forced"])
    assert rep["ok"], rep["errors"]
    if cfg.B > 1:
        # every request (past the first 128-row LM-head chunk too), depth by depth on the
        # GPU's own inputs: layer outputs, LM-head decisions, frontier, rerank and emit
        rep = parity.compare_teacher_forced(synth.oracle_cfg(cfg), W, I, out, tr, d.info["slots"])
        print(name, "all", rep["requests"], "requests (teacher-forced)",
              {k: f"{v:.2e}" for k, v in rep["stats"].items()}, "forced:", len(rep["forced"]))
        assert rep["ok"], rep["errors"]
        assert rep["requests"] == cfg.B
    d.close()
