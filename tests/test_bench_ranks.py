"""bench.py's multi-rank path on CPU: world size 2 over gloo.

Requests are independent, so `bench.py` under torchrun runs one replica per GPU and the
only cross-rank steps are the barriers around the timed region and the max over ranks of
its time.  These checks run that host logic with two gloo ranks (no GPU): both ranks get
the slowest rank's time, the whole-job rate counts every rank's units, every rank draws
its own inputs but the same weights, and the reference arm prints from rank 0 only.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as tdist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402
from eagle_speculative_decoding_03_gb300 import configs, synth  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [3.0, 5.0][rank]                     # rank 1 is the slow one
    tdist.barrier()
    ms = bench.max_over_ranks(local_ms, True, device="cpu")
    value = bench.job_throughput(world, 60, ms)
    tdist.barrier()
    tdist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ms": ms, "value": value}, f)


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for g in got:
        assert g["ms"] == 5.0                       # the max, on both ranks
        assert g["value"] == pytest.approx(2 * 60 / 5e-3)


def test_one_rank_is_the_identity():
    assert bench.max_over_ranks(7.5, False) == 7.5
    assert bench.job_throughput(1, 60, 2.0) == pytest.approx(30000.0)


def test_replicas_draw_their_own_inputs_and_share_the_weights():
    cfg = configs.get("small_dyn")
    w0, w1 = synth.make_weights(cfg), synth.make_weights(cfg)
    for k in w0:
        if w0[k] is not None:
            np.testing.assert_array_equal(w0[k], w1[k])
    i0, i1 = synth.make_inputs(cfg, seed_offset=0), synth.make_inputs(cfg, seed_offset=1)
    assert not np.array_equal(i0["root_feat"], i1["root_feat"])
    np.testing.assert_array_equal(synth.make_inputs(cfg, seed_offset=1)["root_feat"], i1["root_feat"])


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    args = bench.argparse.Namespace(gpus=2, steps=1, warmup=0, impl="reference", workload="small_dyn",
                                    no_cpu_baseline=False, no_b32=True)
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args) == 0
    assert buf.getvalue() == ""


def test_reference_arm_line_keeps_the_contract(monkeypatch):
    args = bench.argparse.Namespace(gpus=1, steps=1, warmup=0, impl="reference", workload="small_dyn",
                                    no_cpu_baseline=False, no_b32=True)
    monkeypatch.setenv("RANK", "0")
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args) == 0
    lines = buf.getvalue().strip().splitlines()
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


@pytest.mark.parametrize("name", ["small_dyn", "small_static", "small_fused"])
def test_reference_step_times_the_oracles_own_depth2_rows(name):
    """The reference arm's timed draft step is the oracle's own depth-2 step: same rows,
    tokens, features and attention (its layer outputs equal the whole-tree oracle's)."""
    from oracle import eagle_oracle as O
    cfg = configs.get(name)
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    st = bench.OracleStep(cfg, W, I)
    assert st.rows == cfg.B * cfg.rows_at(2)
    full = O.draft_tree(synth.oracle_cfg(cfg), W, I)["trace"][1]

    def attend(i, k_i, v_i):
        _, k0, v0, lo, hi = st.meta[i]
        return (np.concatenate([st.Kc[lo:hi], k0[None], k_i[None]]),
                np.concatenate([st.Vc[lo:hi], v0[None], v_i[None]]))

    x_in = np.concatenate([st.x_feat, O.as_f64(W["embed"][st.toks])], axis=1)
    out = O.decoder_rows(st.ocfg, W, x_in, st.pos, attend)
    np.testing.assert_allclose(out["a"], full["a"], rtol=1e-12, atol=1e-12)
    assert st.run() > 0
