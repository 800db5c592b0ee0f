"""Failure paths on the GPU that need no fault: a bounded wait that runs out (the kernels give
up, report it in the device error word and leave the handle usable), and host-side failures
injected with EAGLE_FAULT (an allocation that fails, a launch that fails part-way through a
tree).  After each, a normal call on the same handle gives the same tree as a clean handle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from eagle_speculative_decoding_03_gb300 import binding as eb, configs, synth


@pytest.fixture(scope="module")
def lib():
    from eagle_speculative_decoding_03_gb300 import build
    build.build()
    return eb.load()


@pytest.fixture(scope="module")
def setup(lib):
    cfg = configs.get("small_dyn")
    W, I = synth.make_weights(cfg), synth.make_inputs(cfg)
    dW, dI = eb.device_weights(W), eb.device_inputs(I)
    clean = eb.EagleDraft(cfg, dW)
    ref = {k: v.cpu().numpy() for k, v in clean.tree(dI).items()}
    clean.check()
    clean.close()
    return cfg, dW, dI, ref


def _same(out, ref):
    for k in ref:
        assert np.array_equal(out[k].cpu().numpy(), ref[k]), k


@pytest.mark.parametrize("flags", [0, eb.FLAG_NO_GRAPH])
def test_bounded_wait_runs_out_and_the_handle_recovers(setup, flags):
    cfg, dW, dI, ref = setup
    d = eb.EagleDraft(cfg, dW, flags=flags)
    d.set_wait_limit(64)          # clock cycles: any wait not met at once runs out
    d.tree(dI)
    with pytest.raises(eb.EagleError) as ei:
        d.check()
    assert ei.value.status == eb.EAGLE_ERR_DEVICE
    assert int(str(ei.value).split("0x")[-1], 16) & eb.DEVERR_TIMEOUT
    d.set_wait_limit(0)           # the default again
    out = d.tree(dI)
    d.check()
    _same(out, ref)
    d.close()


def test_injected_allocation_failure_allocates_nothing(setup, monkeypatch):
    cfg, dW, dI, _ = setup
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    monkeypatch.setenv("EAGLE_FAULT", "alloc")
    with pytest.raises(eb.EagleError) as ei:
        eb.EagleDraft(cfg, dW)
    assert ei.value.status == eb.EAGLE_ERR_OOM and "EAGLE_FAULT" in str(ei.value)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


@pytest.mark.parametrize("flags", [0, eb.FLAG_NO_GRAPH])
def test_injected_launch_failure_then_a_whole_tree(setup, monkeypatch, flags):
    cfg, dW, dI, ref = setup
    d = eb.EagleDraft(cfg, dW, flags=flags)
    monkeypatch.setenv("EAGLE_FAULT", "launch")
    with pytest.raises(eb.EagleError) as ei:
        d.tree(dI)
    assert ei.value.status == eb.EAGLE_ERR_CUDA
    monkeypatch.delenv("EAGLE_FAULT")
    torch.cuda.synchronize()
    out = d.tree(dI)
    d.check()
    _same(out, ref)
    d.close()
