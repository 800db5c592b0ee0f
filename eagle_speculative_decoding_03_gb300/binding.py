"""ctypes binding of libeagle_draft.so (include/eagle_draft.h).

Argument marshalling only: every step of the draft tree runs in the library's CUDA
kernels.  torch is used for device memory and streams; tensors are passed as raw
pointers.  ``load()`` raises if the library has not been built.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from .configs import DraftConfig

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libeagle_draft.so")

EAGLE_OK, EAGLE_ERR_INVALID_ARG, EAGLE_ERR_UNSUPPORTED, EAGLE_ERR_OOM, EAGLE_ERR_CUDA, EAGLE_ERR_DEVICE = range(6)
DTYPE_F32, DTYPE_BF16 = 0, 1
TREE_STATIC, TREE_DYNAMIC = 1, 2
FEAT_F, FEAT_FUSED = 1, 3
FLAG_NO_GRAPH, FLAG_NO_PDL, FLAG_GEMM_TWO_CTA = 1, 2, 4
MAX_DEPTH = 16
KERNEL_KINDS = 14
DEVERR_TIMEOUT, DEVERR_PREFIX, DEVERR_TOKEN, DEVERR_SELECT = 1, 2, 4, 8


class Config(C.Structure):
    _fields_ = [("d", C.c_int32), ("n_heads", C.c_int32), ("n_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("d_ff", C.c_int32), ("vocab", C.c_int32),
                ("rms_eps", C.c_float), ("rope_theta", C.c_float), ("dtype", C.c_int32),
                ("tree_kind", C.c_int32), ("feat_kind", C.c_int32), ("depth", C.c_int32),
                ("k", C.c_int32), ("m", C.c_int32), ("branching", C.c_int32 * MAX_DEPTH),
                ("max_batch", C.c_int32), ("max_prefix", C.c_int32), ("flags", C.c_int32)]


class Weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("embed", "w_fc", "w_fc3", "attn_norm", "w_qkv", "w_o",
                                         "mlp_norm", "w_gate", "w_up", "w_down", "w_lm")]


class Inputs(C.Structure):
    _fields_ = [("B", C.c_int32), ("root_feat", C.c_void_p), ("root_tok", C.c_void_p),
                ("k_cache", C.c_void_p), ("v_cache", C.c_void_p), ("cu_seqlens", C.c_void_p),
                ("seeds", C.c_void_p)]


class Outputs(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("tokens", "parents", "positions", "logv", "mask")]


TRACE_FIELDS = ("h", "q", "attn", "y", "a", "lse", "children", "child_logp", "frontier",
                "final_nodes", "tree_k", "tree_v")


class Trace(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in TRACE_FIELDS]


class Info(C.Structure):
    _fields_ = [("slots", C.c_int32), ("generated", C.c_int32), ("rows", C.c_int32),
                ("n_max", C.c_int32), ("k_max", C.c_int32), ("f_max", C.c_int32),
                ("launches_per_tree", C.c_int32), ("tensor_core_gemm", C.c_int32),
                ("workspace_bytes", C.c_int64)]


class VerifyConfig(C.Structure):
    _fields_ = [("d", C.c_int32), ("n_heads", C.c_int32), ("n_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("d_ff", C.c_int32), ("vocab", C.c_int32),
                ("rms_eps", C.c_float), ("rope_theta", C.c_float), ("dtype", C.c_int32),
                ("max_batch", C.c_int32), ("max_slots", C.c_int32), ("max_prefix", C.c_int32),
                ("flags", C.c_int32)]


class VerifyWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("embed", "attn_norm", "w_qkv", "w_o", "mlp_norm", "w_gate",
                                         "w_up", "w_down", "final_norm", "w_lm")]


class VerifyInputs(C.Structure):
    _fields_ = [("B", C.c_int32), ("S", C.c_int32)] + \
        [(n, C.c_void_p) for n in ("tokens", "positions", "mask", "parents", "k_cache", "v_cache", "cu_seqlens")]


VERIFY_OUTPUTS = ("top_id", "top_logp", "lse", "hidden", "logits", "accept_len", "accept_slots", "correction")


class VerifyOutputs(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in VERIFY_OUTPUTS]


class DFlashConfigC(C.Structure):
    _fields_ = [("d", C.c_int32), ("n_heads", C.c_int32), ("n_kv_heads", C.c_int32),
                ("head_dim", C.c_int32), ("d_ff", C.c_int32), ("vocab", C.c_int32),
                ("rms_eps", C.c_float), ("rope_theta", C.c_float), ("dtype", C.c_int32),
                ("n_layers", C.c_int32), ("gamma", C.c_int32), ("k", C.c_int32), ("mask_token", C.c_int32),
                ("max_batch", C.c_int32), ("max_prefix", C.c_int32), ("flags", C.c_int32)]


class DFlashWeights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("w_lm", C.c_void_p), ("final_norm", C.c_void_p)] + \
        [(n, C.POINTER(C.c_void_p)) for n in ("attn_norm", "w_qkv", "w_o", "mlp_norm", "w_gate", "w_up", "w_down")]


class DFlashInputs(C.Structure):
    _fields_ = [("B", C.c_int32), ("anchor", C.c_void_p), ("ctx_k", C.POINTER(C.c_void_p)),
                ("ctx_v", C.POINTER(C.c_void_p)), ("cu_seqlens", C.c_void_p)]


class DFlashOutputs(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("tokens", "logp", "lse", "hidden")]


_lib = None


def load(path: str = LIB_PATH):
    """Load the library (once) and declare the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first (python -m "
                           "eagle_speculative_decoding_03_gb300.build)")
    lib = C.CDLL(path)
    P = C.c_void_p
    lib.eagle_draft_create.argtypes = [C.POINTER(Config), C.POINTER(Weights), C.POINTER(P)]
    lib.eagle_draft_create.restype = C.c_int
    lib.eagle_draft_tree.argtypes = [P, C.POINTER(Inputs), C.POINTER(Outputs), C.POINTER(Trace), P]
    lib.eagle_draft_tree.restype = C.c_int
    lib.eagle_draft_lm_head_topk.argtypes = [P, P, C.c_int32, C.c_int32, P, P, P, P]
    lib.eagle_draft_lm_head_topk.restype = C.c_int
    lib.eagle_draft_query.argtypes = [P, C.POINTER(Info)]
    lib.eagle_draft_query.restype = C.c_int
    lib.eagle_draft_check.argtypes = [P, C.POINTER(C.c_uint32)]
    lib.eagle_draft_check.restype = C.c_int
    lib.eagle_draft_set_wait_limit.argtypes = [P, C.c_int64]
    lib.eagle_draft_set_wait_limit.restype = C.c_int
    lib.eagle_draft_destroy.argtypes = [P]
    lib.eagle_draft_destroy.restype = None
    lib.eagle_draft_profile.argtypes = [P, C.c_int32]
    lib.eagle_draft_profile.restype = C.c_int
    lib.eagle_draft_profile_read.argtypes = [P, C.POINTER(C.c_float), C.POINTER(C.c_int32)]
    lib.eagle_draft_profile_read.restype = C.c_int
    lib.eagle_draft_kernel_name.argtypes = [C.c_int32]
    lib.eagle_draft_kernel_name.restype = C.c_char_p
    lib.eagle_lm_head_topk_noalloc.argtypes = [P, C.c_int32, C.c_int32, P, C.c_int32, C.c_int32, P, P, P, P]
    lib.eagle_lm_head_topk_noalloc.restype = C.c_int
    lib.eagle_verify_create.argtypes = [C.POINTER(VerifyConfig), C.POINTER(VerifyWeights), C.POINTER(P)]
    lib.eagle_verify_create.restype = C.c_int
    lib.eagle_verify_tree.argtypes = [P, C.POINTER(VerifyInputs), C.POINTER(VerifyOutputs), P]
    lib.eagle_verify_tree.restype = C.c_int
    lib.eagle_verify_check.argtypes = [P, C.POINTER(C.c_uint32)]
    lib.eagle_verify_check.restype = C.c_int
    lib.eagle_verify_destroy.argtypes = [P]
    lib.eagle_verify_destroy.restype = None
    lib.eagle_dflash_create.argtypes = [C.POINTER(DFlashConfigC), C.POINTER(DFlashWeights), C.POINTER(P)]
    lib.eagle_dflash_create.restype = C.c_int
    lib.eagle_dflash_draft.argtypes = [P, C.POINTER(DFlashInputs), C.POINTER(DFlashOutputs), P]
    lib.eagle_dflash_draft.restype = C.c_int
    lib.eagle_dflash_check.argtypes = [P, C.POINTER(C.c_uint32)]
    lib.eagle_dflash_check.restype = C.c_int
    lib.eagle_dflash_destroy.argtypes = [P]
    lib.eagle_dflash_destroy.restype = None
    lib.eagle_speculative_accept.argtypes = [C.c_int32, C.c_int32, C.c_int32, P, P, P, P, P, P, P, P, P, P]
    lib.eagle_speculative_accept.restype = C.c_int
    lib.eagle_draft_last_error.argtypes = []
    lib.eagle_draft_last_error.restype = C.c_char_p
    _lib = lib
    return lib


class EagleError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"eagle status {status}: {msg}")
        self.status = status


def _check(status: int):
    if status != EAGLE_OK:
        raise EagleError(status, load().eagle_draft_last_error().decode())


def make_config(cfg: DraftConfig, max_batch: int | None = None, max_prefix: int | None = None,
                flags: int = 0) -> Config:
    c = Config()
    c.d, c.n_heads, c.n_kv_heads, c.head_dim = cfg.d, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    c.d_ff, c.vocab, c.rms_eps, c.rope_theta = cfg.d_ff, cfg.vocab, cfg.rms_eps, cfg.rope_theta
    c.dtype = DTYPE_BF16 if cfg.dtype == "bf16" else DTYPE_F32
    c.tree_kind = TREE_STATIC if cfg.tree == "static" else TREE_DYNAMIC
    c.feat_kind = FEAT_FUSED if cfg.feat == "fused" else FEAT_F
    c.depth, c.k, c.m = cfg.depth, cfg.k, cfg.m
    for i, b in enumerate(cfg.branching):
        c.branching[i] = b
    c.max_batch = cfg.B if max_batch is None else max_batch
    c.max_prefix = cfg.prefix[1] if max_prefix is None else max_prefix
    c.flags = flags
    return c


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def device_weights(W: dict, device="cuda"):
    """numpy weights (bf16 as uint16 bits) -> device tensors (bf16 kept as int16 bits;
    uint64 seeds kept as int64 bits)."""
    import torch
    out = {}
    for k, v in W.items():
        arr = v.view(np.int16) if v.dtype == np.uint16 else v.view(np.int64) if v.dtype == np.uint64 else v
        out[k] = torch.from_numpy(np.ascontiguousarray(arr)).to(device)
    return out


def device_inputs(I: dict, device="cuda"):
    return device_weights(I, device)


def lm_head_topk_noalloc(w_lm, a, k: int, stream=None):
    """LM-head top-k without a handle and without any device allocation inside the
    library (for callers that cannot allocate); outputs are allocated here by torch.
    The library reads w_lm as bf16 and a as float32: other dtypes are rejected here.
    If a kernel of the call gave up, every row comes back as id -1 and NaN logp / lse."""
    import torch
    if w_lm.dtype not in (torch.bfloat16, torch.int16) or w_lm.dim() != 2:
        raise EagleError(EAGLE_ERR_INVALID_ARG, "noalloc: w_lm must be a 2-D bf16 tensor (or its int16 bits)")
    if a.dtype != torch.float32 or a.dim() != 2 or a.shape[1] != w_lm.shape[1]:
        raise EagleError(EAGLE_ERR_INVALID_ARG, "noalloc: a must be float32 [N, d] with d = w_lm.shape[1]")
    if not (w_lm.is_contiguous() and a.is_contiguous()):
        raise EagleError(EAGLE_ERR_INVALID_ARG, "noalloc: w_lm and a must be contiguous")
    N, d = int(a.shape[0]), int(a.shape[1])
    ids = torch.empty((N, k), dtype=torch.int32, device=a.device)
    logp = torch.empty((N, k), dtype=torch.float32, device=a.device)
    lse = torch.empty((N,), dtype=torch.float32, device=a.device)
    st = None if stream is None else stream.cuda_stream
    _check(load().eagle_lm_head_topk_noalloc(_ptr(w_lm), int(w_lm.shape[0]), d, _ptr(a), N, k,
                                             _ptr(ids), _ptr(logp), _ptr(lse), st))
    return ids, logp, lse


class EagleDraft:
    """One handle of the C library bound to device weights (torch tensors)."""

    def __init__(self, cfg: DraftConfig, dW: dict, max_batch: int | None = None,
                 max_prefix: int | None = None, flags: int = 0):
        lib = load()
        self.cfg = cfg
        self._dW = dW  # keep the weights alive
        w = Weights(**{n: _ptr(dW.get(n)) for n, _ in Weights._fields_})
        self._ccfg = make_config(cfg, max_batch, max_prefix, flags)
        h = C.c_void_p()
        _check(lib.eagle_draft_create(C.byref(self._ccfg), C.byref(w), C.byref(h)))
        self.h = h
        info = Info()
        _check(lib.eagle_draft_query(self.h, C.byref(info)))
        self.info = {n: getattr(info, n) for n, _ in Info._fields_}

    def close(self):
        if getattr(self, "h", None):
            load().eagle_draft_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def alloc_outputs(self, B: int, device="cuda"):
        import torch
        S = self.info["slots"]
        return {"tokens": torch.empty((B, S), dtype=torch.int32, device=device),
                "parents": torch.empty((B, S), dtype=torch.int32, device=device),
                "positions": torch.empty((B, S), dtype=torch.int32, device=device),
                "logv": torch.empty((B, S), dtype=torch.float32, device=device),
                "mask": torch.empty((B, S, S), dtype=torch.uint8, device=device)}

    def alloc_trace(self, device="cuda"):
        import torch
        c, i = self.cfg, self.info
        D, N, k = c.depth, i["n_max"], i["k_max"]
        Bm, hq = self._ccfg.max_batch, c.n_heads * c.head_dim
        f = dict(dtype=torch.float32, device=device)
        n = dict(dtype=torch.int32, device=device)
        return {"h": torch.zeros((D, N, c.d), **f), "q": torch.zeros((D, N, hq), **f),
                "attn": torch.zeros((D, N, hq), **f), "y": torch.zeros((D, N, c.d), **f),
                "a": torch.zeros((D, N, c.d), **f), "lse": torch.zeros((D, N), **f),
                "children": torch.full((D, N, k), -1, **n), "child_logp": torch.zeros((D, N, k), **f),
                "frontier": torch.full((D, Bm, i["f_max"]), -1, **n),
                "final_nodes": torch.full((Bm, i["slots"]), -1, **n),
                "tree_k": torch.zeros((Bm, i["rows"], c.n_kv_heads, c.head_dim), **f),
                "tree_v": torch.zeros((Bm, i["rows"], c.n_kv_heads, c.head_dim), **f)}

    def tree(self, dI: dict, out: dict | None = None, trace: dict | None = None, stream=None):
        """Enqueue one draft tree; returns the output tensors (device)."""
        B = int(dI["root_tok"].shape[0])
        out = self.alloc_outputs(B, dI["root_tok"].device) if out is None else out
        inp = Inputs(B=B, root_feat=_ptr(dI["root_feat"]), root_tok=_ptr(dI["root_tok"]),
                     k_cache=_ptr(dI["k_cache"]), v_cache=_ptr(dI["v_cache"]),
                     cu_seqlens=_ptr(dI["cu_seqlens"]), seeds=_ptr(dI.get("seeds")))
        o = Outputs(**{n: _ptr(out[n]) for n, _ in Outputs._fields_})
        tr = None if trace is None else C.byref(Trace(**{n: _ptr(trace.get(n)) for n in TRACE_FIELDS}))
        st = None if stream is None else stream.cuda_stream
        _check(load().eagle_draft_tree(self.h, C.byref(inp), C.byref(o), tr, st))
        return out

    def lm_head_topk(self, a, k: int, stream=None):
        import torch
        N = int(a.shape[0])
        ids = torch.empty((N, k), dtype=torch.int32, device=a.device)
        logp = torch.empty((N, k), dtype=torch.float32, device=a.device)
        lse = torch.empty((N,), dtype=torch.float32, device=a.device)
        st = None if stream is None else stream.cuda_stream
        _check(load().eagle_draft_lm_head_topk(self.h, _ptr(a), N, k, _ptr(ids), _ptr(logp), _ptr(lse), st))
        return ids, logp, lse

    def profile(self, enable: bool):
        _check(load().eagle_draft_profile(self.h, 1 if enable else 0))

    def profile_read(self) -> dict:
        """{kernel name: (total ms, launches)} since the last read (synchronises)."""
        ms = (C.c_float * KERNEL_KINDS)()
        n = (C.c_int32 * KERNEL_KINDS)()
        _check(load().eagle_draft_profile_read(self.h, ms, n))
        lib = load()
        return {lib.eagle_draft_kernel_name(i).decode(): (ms[i], n[i]) for i in range(KERNEL_KINDS) if n[i]}

    def set_wait_limit(self, cycles: int):
        _check(load().eagle_draft_set_wait_limit(self.h, int(cycles)))

    def check(self) -> int:
        """Synchronise; raise on a device error word or CUDA error."""
        w = C.c_uint32(0)
        st = load().eagle_draft_check(self.h, C.byref(w))
        if st != EAGLE_OK:
            raise EagleError(st, load().eagle_draft_last_error().decode())
        return w.value


class EagleVerify:
    """Handle of the target's verification pass over emitted trees (bf16 target layer)."""

    def __init__(self, cfg: DraftConfig, dWt: dict, dW: dict, max_batch: int, max_slots: int,
                 max_prefix: int | None = None, flags: int = 0):
        lib = load()
        self.cfg = cfg
        self._keep = (dWt, dW)
        c = VerifyConfig(d=cfg.d, n_heads=cfg.n_heads, n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim,
                         d_ff=cfg.d_ff, vocab=cfg.vocab, rms_eps=cfg.rms_eps, rope_theta=cfg.rope_theta,
                         dtype=DTYPE_BF16 if cfg.dtype == "bf16" else DTYPE_F32, max_batch=max_batch,
                         max_slots=max_slots, max_prefix=cfg.prefix[1] if max_prefix is None else max_prefix,
                         flags=flags)
        w = VerifyWeights(embed=_ptr(dW["embed"]), w_lm=_ptr(dW["w_lm"]),
                          **{n: _ptr(dWt[n]) for n in ("attn_norm", "w_qkv", "w_o", "mlp_norm", "w_gate",
                                                       "w_up", "w_down", "final_norm")})
        h = C.c_void_p()
        _check(lib.eagle_verify_create(C.byref(c), C.byref(w), C.byref(h)))
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            load().eagle_verify_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def verify(self, tree: dict, cache: dict, cu_seqlens, accept: bool = True, hidden: bool = False,
               logits: bool = False, stream=None) -> dict:
        """tree: device tensors tokens / positions / parents [B,S] int32 and mask [B,S,S] uint8
        (as eagle_draft_tree emits them); cache: the target's k_cache / v_cache."""
        import torch
        B, S = (int(x) for x in tree["tokens"].shape)
        dev = tree["tokens"].device
        out = {"top_id": torch.empty((B, S), dtype=torch.int32, device=dev),
               "top_logp": torch.empty((B, S), dtype=torch.float32, device=dev),
               "lse": torch.empty((B, S), dtype=torch.float32, device=dev)}
        if hidden:
            out["hidden"] = torch.empty((B, S, self.cfg.d), dtype=torch.float32, device=dev)
        if logits:
            out["logits"] = torch.empty((B, S, self.cfg.vocab), dtype=torch.float32, device=dev)
        if accept:
            out["accept_len"] = torch.empty((B,), dtype=torch.int32, device=dev)
            out["accept_slots"] = torch.empty((B, S), dtype=torch.int32, device=dev)
            out["correction"] = torch.empty((B,), dtype=torch.int32, device=dev)
        inp = VerifyInputs(B=B, S=S, tokens=_ptr(tree["tokens"]), positions=_ptr(tree["positions"]),
                           mask=_ptr(tree["mask"]), parents=_ptr(tree.get("parents")),
                           k_cache=_ptr(cache["k_cache"]), v_cache=_ptr(cache["v_cache"]),
                           cu_seqlens=_ptr(cu_seqlens))
        o = VerifyOutputs(**{n: _ptr(out.get(n)) for n in VERIFY_OUTPUTS})
        st = None if stream is None else stream.cuda_stream
        _check(load().eagle_verify_tree(self.h, C.byref(inp), C.byref(o), st))
        return out

    def check(self) -> int:
        w = C.c_uint32(0)
        st = load().eagle_verify_check(self.h, C.byref(w))
        if st != EAGLE_OK:
            raise EagleError(st, load().eagle_draft_last_error().decode())
        return w.value


def speculative_accept(tree: dict, logits_target, logits_draft, seeds, stream=None) -> dict:
    """Multi-round speculative sampling over emitted trees (device tensors): tokens / parents
    [B,S] int32, logits [B,S,V] float32, seeds [B] (int64 bits of the uint64 seeds).
    Returns accept_len [B], accept_slots [B,S], correction [B] and the error word [1]."""
    import torch
    B, S = (int(x) for x in tree["tokens"].shape)
    V = int(logits_target.shape[-1])
    if logits_target.dtype != torch.float32 or logits_draft.dtype != torch.float32:
        raise EagleError(EAGLE_ERR_INVALID_ARG, "speculative_accept: logits must be float32")
    if tuple(logits_target.shape) != (B, S, V) or tuple(logits_draft.shape) != (B, S, V):
        raise EagleError(EAGLE_ERR_INVALID_ARG, "speculative_accept: logits must be [B, S, vocab]")
    dev = tree["tokens"].device
    out = {"accept_len": torch.empty((B,), dtype=torch.int32, device=dev),
           "accept_slots": torch.empty((B, S), dtype=torch.int32, device=dev),
           "correction": torch.empty((B,), dtype=torch.int32, device=dev),
           "err": torch.zeros((1,), dtype=torch.int32, device=dev)}
    st = None if stream is None else stream.cuda_stream
    _check(load().eagle_speculative_accept(B, S, V, _ptr(tree["tokens"]), _ptr(tree["parents"]),
                                           _ptr(logits_target.contiguous()), _ptr(logits_draft.contiguous()),
                                           _ptr(seeds), _ptr(out["accept_len"]), _ptr(out["accept_slots"]),
                                           _ptr(out["correction"]), _ptr(out["err"]), st))
    return out


def _ptr_array(ts):
    return (C.c_void_p * len(ts))(*[_ptr(t) for t in ts])


def device_dflash_weights(W: dict, device="cuda") -> dict:
    """DFlash weights (synth.make_dflash_weights) -> device tensors; per-layer lists kept."""
    top = device_weights({k: W[k] for k in ("embed", "w_lm", "final_norm")}, device)
    top["layers"] = [device_weights(L, device) for L in W["layers"]]
    return top


class EagleDFlash:
    """Handle of the DFlash block-parallel draft (bf16)."""

    def __init__(self, cfg, dW: dict, max_batch: int | None = None, max_prefix: int | None = None,
                 flags: int = 0):
        lib = load()
        self.cfg = cfg
        self._keep = dW
        c = DFlashConfigC(d=cfg.d, n_heads=cfg.n_heads, n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim,
                          d_ff=cfg.d_ff, vocab=cfg.vocab, rms_eps=cfg.rms_eps, rope_theta=cfg.rope_theta,
                          dtype=DTYPE_BF16 if cfg.dtype == "bf16" else DTYPE_F32, n_layers=cfg.layers,
                          gamma=cfg.gamma, k=cfg.k, mask_token=cfg.mask_id,
                          max_batch=cfg.B if max_batch is None else max_batch,
                          max_prefix=cfg.prefix[1] if max_prefix is None else max_prefix, flags=flags)
        L = dW["layers"]
        self._arrays = {n: _ptr_array([l[n] for l in L]) for n in
                        ("attn_norm", "w_qkv", "w_o", "mlp_norm", "w_gate", "w_up", "w_down")}
        w = DFlashWeights(embed=_ptr(dW["embed"]), w_lm=_ptr(dW["w_lm"]), final_norm=_ptr(dW["final_norm"]),
                          **{n: C.cast(a, C.POINTER(C.c_void_p)) for n, a in self._arrays.items()})
        h = C.c_void_p()
        _check(lib.eagle_dflash_create(C.byref(c), C.byref(w), C.byref(h)))
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            load().eagle_dflash_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def draft(self, dI: dict, hidden: bool = False, stream=None) -> dict:
        """dI: anchor [B] int32, cu_seqlens [B+1], ctx_k / ctx_v lists of per-layer caches."""
        import torch
        B = int(dI["anchor"].shape[0])
        g, k, dev = self.cfg.gamma, self.cfg.k, dI["anchor"].device
        out = {"tokens": torch.empty((B, g, k), dtype=torch.int32, device=dev),
               "logp": torch.empty((B, g, k), dtype=torch.float32, device=dev),
               "lse": torch.empty((B, g), dtype=torch.float32, device=dev)}
        if hidden:
            out["hidden"] = torch.empty((B, g + 1, self.cfg.d), dtype=torch.float32, device=dev)
        ck, cv = _ptr_array(dI["ctx_k"]), _ptr_array(dI["ctx_v"])
        inp = DFlashInputs(B=B, anchor=_ptr(dI["anchor"]), ctx_k=C.cast(ck, C.POINTER(C.c_void_p)),
                           ctx_v=C.cast(cv, C.POINTER(C.c_void_p)), cu_seqlens=_ptr(dI["cu_seqlens"]))
        o = DFlashOutputs(**{n: _ptr(out.get(n)) for n in ("tokens", "logp", "lse", "hidden")})
        st = None if stream is None else stream.cuda_stream
        _check(load().eagle_dflash_draft(self.h, C.byref(inp), C.byref(o), st))
        return out

    def check(self) -> int:
        w = C.c_uint32(0)
        st = load().eagle_dflash_check(self.h, C.byref(w))
        if st != EAGLE_OK:
            raise EagleError(st, load().eagle_draft_last_error().decode())
        return w.value
