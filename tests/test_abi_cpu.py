"""CPU checks of the C-ABI library: it builds, loads, exports every function that
include/eagle_draft.h declares, and rejects invalid arguments before any GPU work."""
import ctypes as C
import os
import re

import pytest

from eagle_speculative_decoding_03_gb300 import binding as eb, configs

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "eagle_draft.h")


@pytest.fixture(scope="module")
def lib():
    from eagle_speculative_decoding_03_gb300 import build
    build.build()
    return eb.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"EAGLE_API\s+[\w\s\*]*?\b(eagle_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    fns = declared_functions()
    for f in ("eagle_draft_create", "eagle_draft_tree", "eagle_draft_destroy", "eagle_draft_last_error"):
        assert f in fns


def test_library_exports_every_declared_symbol(lib):
    for f in declared_functions():
        assert hasattr(lib, f), f


def _weights_dummy():
    w = eb.Weights()
    for n, _ in eb.Weights._fields_:
        setattr(w, n, 256)   # never dereferenced: validation fails first
    return w


@pytest.mark.parametrize("mutate,status", [
    (dict(d=0), eb.EAGLE_ERR_INVALID_ARG),
    (dict(n_heads=3, n_kv_heads=2), eb.EAGLE_ERR_INVALID_ARG),
    (dict(depth=0), eb.EAGLE_ERR_INVALID_ARG),
    (dict(depth=17), eb.EAGLE_ERR_INVALID_ARG),
    (dict(k=17), eb.EAGLE_ERR_INVALID_ARG),
    (dict(head_dim=96), eb.EAGLE_ERR_UNSUPPORTED),
    (dict(d=4000), eb.EAGLE_ERR_UNSUPPORTED),
    (dict(vocab=1000), eb.EAGLE_ERR_UNSUPPORTED),
    (dict(max_batch=0), eb.EAGLE_ERR_INVALID_ARG),
])
def test_create_rejects_invalid_config(lib, mutate, status):
    c = eb.make_config(configs.get("eagle2_b1"))
    for k, v in mutate.items():
        setattr(c, k, v)
    h = C.c_void_p()
    st = lib.eagle_draft_create(C.byref(c), C.byref(_weights_dummy()), C.byref(h))
    assert st == status, lib.eagle_draft_last_error()
    assert not h.value
    assert lib.eagle_draft_last_error()


def test_create_rejects_null_weights(lib):
    c = eb.make_config(configs.get("eagle2_b1"))
    w = _weights_dummy()
    w.w_lm = None
    h = C.c_void_p()
    assert lib.eagle_draft_create(C.byref(c), C.byref(w), C.byref(h)) == eb.EAGLE_ERR_INVALID_ARG
    assert b"null weight" in lib.eagle_draft_last_error()


def test_null_handles(lib):
    assert lib.eagle_draft_tree(None, None, None, None, None) == eb.EAGLE_ERR_INVALID_ARG
    assert lib.eagle_draft_lm_head_topk(None, None, 1, 1, None, None, None, None) == eb.EAGLE_ERR_INVALID_ARG
    assert lib.eagle_draft_query(None, None) == eb.EAGLE_ERR_INVALID_ARG
    assert lib.eagle_draft_check(None, None) == eb.EAGLE_ERR_INVALID_ARG
    lib.eagle_draft_destroy(None)


STRUCTS = [("eagle_draft_config_t", "Config"), ("eagle_draft_weights_t", "Weights"),
           ("eagle_draft_inputs_t", "Inputs"), ("eagle_draft_outputs_t", "Outputs"),
           ("eagle_draft_trace_t", "Trace"), ("eagle_draft_info_t", "Info"),
           ("eagle_verify_config_t", "VerifyConfig"), ("eagle_verify_weights_t", "VerifyWeights"),
           ("eagle_verify_inputs_t", "VerifyInputs"), ("eagle_verify_outputs_t", "VerifyOutputs"),
           ("eagle_dflash_config_t", "DFlashConfigC"), ("eagle_dflash_weights_t", "DFlashWeights"),
           ("eagle_dflash_inputs_t", "DFlashInputs"), ("eagle_dflash_outputs_t", "DFlashOutputs")]


def test_struct_layout_matches_header(tmp_path):
    """Every struct the binding passes has the header's size and field offsets (the header
    compiled by the host C compiler)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    lines = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HEADER}"', "int main(void) {"]
    for cname, pyname in STRUCTS:
        lines.append(f'  printf("{pyname} size %zu\\n", sizeof({cname}));')
        for f, _ in getattr(eb, pyname)._fields_:
            lines.append(f'  printf("{pyname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("  return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, str(src), "-o", str(exe)], check=True)
    got = [x for x in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n") if x]
    assert len(got) == sum(1 + len(getattr(eb, p)._fields_) for _, p in STRUCTS)
    for line in got:
        pyname, field, value = line.split()
        cls = getattr(eb, pyname)
        want = C.sizeof(cls) if field == "size" else getattr(cls, field).offset
        assert int(value) == want, (pyname, field, value, want)


def test_noalloc_binding_rejects_wrong_dtypes(lib):
    """The allocation-free LM-head entry point reads w_lm as bf16 and a as float32; the
    binding rejects anything else before the call (no GPU needed to see it)."""
    import torch
    w32 = torch.zeros((256, 128), dtype=torch.float32)
    w16 = torch.zeros((256, 128), dtype=torch.bfloat16)
    a32 = torch.zeros((2, 128), dtype=torch.float32)
    for w, a in ((w32, a32), (w16, a32.double()), (w16, torch.zeros((2, 64), dtype=torch.float32))):
        with pytest.raises(eb.EagleError) as ei:
            eb.lm_head_topk_noalloc(w, a, 2)
        assert ei.value.status == eb.EAGLE_ERR_INVALID_ARG
