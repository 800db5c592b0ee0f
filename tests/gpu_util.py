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
