"""Seeded synthetic weights and inputs for the draft-tree step.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic.  Its arrays feed both the CUDA path and the float64 oracle.

Recipe (every tensor ~ N(0, sigma^2) unless stated):
  * frozen token embedding E [|V|, d]: sigma = 1 (the same scale as the feature f);
  * fc [d, 2d]: sigma^2 = 1/(2d); EAGLE-3 FC [d, 3d]: 1/(3d); qkv [(Hq+2Hkv)hd, d]: 1/d;
    o [d, Hq hd]: 1/(Hq hd); gate/up [ff, d]: 1/d; down [d, ff]: 1/ff  (N(0, 1/fan_in));
  * LM head [|V|, d]: sigma = logit_std / (FEATURE_RMS * sqrt(d)).  Under this recipe the
    draft output a has rms ~ FEATURE_RMS = 1.17 (the fc output has unit variance and the
    SwiGLU branch adds ~0.36 of variance), so the logits come out with std ~ logit_std;
  * RMSNorm gains: 1 + gamma_jitter * N(0,1) (unit gains when gamma_jitter = 0);
  * root feature f [B, d] ~ N(0,1) (EAGLE-1/2) or [l;m;h] [B, 3d] ~ N(0,1) (EAGLE-3);
  * root token ~ U[0, |V|); prefix lengths n_b ~ U[lo, hi];
  * verified-prefix KV cache, packed [sum n_b, Hkv, hd], post-RoPE, N(0,1).

Weights are stored ``[out, in]`` row-major; bf16 tensors are returned as uint16 bit
patterns (round-to-nearest-even from an fp32 draw), fp32 tensors as float32.
Generation is chunked: chunk ``i`` of tensor ``t`` draws from
PCG64(SeedSequence([seed, t, i])), so the result does not depend on thread count.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .configs import DraftConfig

_CHUNK = 1 << 22
FEATURE_RMS = 1.17

WEIGHT_NAMES = ("embed", "w_fc", "w_fc3", "attn_norm", "w_qkv", "w_o", "mlp_norm",
                "w_gate", "w_up", "w_down", "w_lm")


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the uint16 bit pattern."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + (((u >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(32, os.cpu_count() or 1))


def normal(shape, key, scale=1.0, dtype="f32", offset=0.0) -> np.ndarray:
    """offset + scale * N(0,1), drawn in fp32, stored as float32 or bf16 bits."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def work(i):
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([*key, i])))
        x = rng.standard_normal(hi - lo, dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        if offset != 0.0:
            x += np.float32(offset)
        out[lo:hi] = f32_to_bf16_bits(x) if dtype == "bf16" else x

    if nchunks <= 1:
        for i in range(nchunks):
            work(i)
    else:
        with ThreadPoolExecutor(min(_threads(), nchunks)) as ex:
            list(ex.map(work, range(nchunks)))
    return out.reshape(shape)


def make_weights(cfg: DraftConfig) -> dict:
    d, V, ff, hd = cfg.d, cfg.vocab, cfg.d_ff, cfg.head_dim
    s, dt = cfg.seed, cfg.dtype
    W = {
        "embed": normal((V, d), (s, 1), 1.0, dt),
        "w_fc": normal((d, 2 * d), (s, 2), (1.0 / (2 * d)) ** 0.5, dt),
        "attn_norm": normal((d,), (s, 4), cfg.gamma_jitter, "f32", 1.0) if cfg.gamma_jitter
        else np.ones(d, np.float32),
        "w_qkv": normal((cfg.qkv_dim, d), (s, 5), (1.0 / d) ** 0.5, dt),
        "w_o": normal((d, cfg.attn_dim), (s, 6), (1.0 / cfg.attn_dim) ** 0.5, dt),
        "mlp_norm": normal((d,), (s, 7), cfg.gamma_jitter, "f32", 1.0) if cfg.gamma_jitter
        else np.ones(d, np.float32),
        "w_gate": normal((ff, d), (s, 8), (1.0 / d) ** 0.5, dt),
        "w_up": normal((ff, d), (s, 9), (1.0 / d) ** 0.5, dt),
        "w_down": normal((d, ff), (s, 10), (1.0 / ff) ** 0.5, dt),
        "w_lm": normal((V, d), (s, 11), cfg.logit_std / (FEATURE_RMS * d ** 0.5), dt),
    }
    if cfg.feat == "fused":
        W["w_fc3"] = normal((d, 3 * d), (s, 3), (1.0 / (3 * d)) ** 0.5, dt)
    return W


def make_inputs(cfg: DraftConfig, B: int | None = None, seed_offset: int = 0) -> dict:
    """Per-request inputs of one draft-tree call."""
    B = cfg.B if B is None else B
    s = cfg.seed + 7919 * seed_offset
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([s, 20])))
    lo, hi = cfg.prefix
    n = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    cu = np.zeros(B + 1, np.int32)
    cu[1:] = np.cumsum(n)
    tok = rng.integers(0, cfg.vocab, size=B).astype(np.int32)
    total = int(cu[-1])
    kv_shape = (total, cfg.n_kv_heads, cfg.head_dim)
    if cfg.feat == "fused":
        root = normal((B, 3 * cfg.d), (s, 21), 1.0, "bf16")
    else:
        root = normal((B, cfg.d), (s, 21), 1.0, "f32")
    return {
        "root_feat": root,
        "root_tok": tok,
        "cu_seqlens": cu,
        "k_cache": normal(kv_shape, (s, 22), 1.0, cfg.dtype),
        "v_cache": normal(kv_shape, (s, 23), 1.0, cfg.dtype),
    }


def oracle_cfg(cfg: DraftConfig) -> dict:
    """The plain-dict view of a config that the oracle takes."""
    return dict(d=cfg.d, n_heads=cfg.n_heads, n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim,
                d_ff=cfg.d_ff, vocab=cfg.vocab, rms_eps=cfg.rms_eps, rope_theta=cfg.rope_theta,
                tree=cfg.tree, depth=cfg.depth, k=cfg.k, m=cfg.m,
                branching=tuple(cfg.branching), feat=cfg.feat)


# ------------------------------------------------- verification side (synthetic target)
def make_target(cfg: DraftConfig) -> dict:
    """One synthetic target decoder layer for the tree-verification pass.

    The same head shapes as the draft layer, its own weights, and a final RMSNorm gain.
    The target's frozen embedding and LM head are the draft's (``make_weights``): the
    draft reuses the target's tables.
    """
    d, ff, s, dt = cfg.d, cfg.d_ff, cfg.seed, cfg.dtype

    def gain(key):
        if cfg.gamma_jitter:
            return normal((d,), (s, key), cfg.gamma_jitter, "f32", 1.0)
        return np.ones(d, np.float32)

    return {
        "attn_norm": gain(40),
        "w_qkv": normal((cfg.qkv_dim, d), (s, 41), (1.0 / d) ** 0.5, dt),
        "w_o": normal((d, cfg.attn_dim), (s, 42), (1.0 / cfg.attn_dim) ** 0.5, dt),
        "mlp_norm": gain(43),
        "w_gate": normal((ff, d), (s, 44), (1.0 / d) ** 0.5, dt),
        "w_up": normal((ff, d), (s, 45), (1.0 / d) ** 0.5, dt),
        "w_down": normal((d, ff), (s, 46), (1.0 / ff) ** 0.5, dt),
        "final_norm": gain(47),
    }


def make_target_cache(cfg: DraftConfig, inp: dict, seed_offset: int = 0) -> dict:
    """The target layer's verified-prefix KV cache, packed like the draft's (same
    ``cu_seqlens``), post-RoPE, N(0,1)."""
    s = cfg.seed + 7919 * seed_offset
    shape = (int(inp["cu_seqlens"][-1]), cfg.n_kv_heads, cfg.head_dim)
    return {"k_cache": normal(shape, (s, 48), 1.0, cfg.dtype),
            "v_cache": normal(shape, (s, 49), 1.0, cfg.dtype)}


# -------------------------------------------------- DFlash block-parallel draft
LAYER_NAMES = ("attn_norm", "w_qkv", "w_o", "mlp_norm", "w_gate", "w_up", "w_down")


def make_dflash_weights(cfg) -> dict:
    """Per-layer weights of the draft stack (the recipe of ``make_weights``), the final
    RMSNorm gain, the frozen embedding and the frozen LM head.  The LM head reads a
    normalised state (rms ~ 1), so its scale is logit_std / sqrt(d)."""
    d, V, ff, s, dt = cfg.d, cfg.vocab, cfg.d_ff, cfg.seed, cfg.dtype

    def gain(key):
        if cfg.gamma_jitter:
            return normal((d,), (s, key), cfg.gamma_jitter, "f32", 1.0)
        return np.ones(d, np.float32)

    layers = []
    for l in range(cfg.layers):
        base = 100 + 10 * l
        layers.append({
            "attn_norm": gain(base),
            "w_qkv": normal((cfg.qkv_dim, d), (s, base + 1), (1.0 / d) ** 0.5, dt),
            "w_o": normal((d, cfg.attn_dim), (s, base + 2), (1.0 / cfg.attn_dim) ** 0.5, dt),
            "mlp_norm": gain(base + 3),
            "w_gate": normal((ff, d), (s, base + 4), (1.0 / d) ** 0.5, dt),
            "w_up": normal((ff, d), (s, base + 5), (1.0 / d) ** 0.5, dt),
            "w_down": normal((d, ff), (s, base + 6), (1.0 / ff) ** 0.5, dt),
        })
    return {"embed": normal((V, d), (s, 1), 1.0, dt),
            "w_lm": normal((V, d), (s, 11), cfg.logit_std / d ** 0.5, dt),
            "final_norm": gain(12), "layers": layers}


def make_dflash_inputs(cfg, B: int | None = None, seed_offset: int = 0) -> dict:
    """Anchor tokens, prefix lengths and every layer's injected context keys / values of the
    verified prefix (packed [sum n_b, Hkv, hd], keys post-RoPE, N(0,1))."""
    B = cfg.B if B is None else B
    s = cfg.seed + 7919 * seed_offset
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([s, 20])))
    lo, hi = cfg.prefix
    n = rng.integers(lo, hi + 1, size=B).astype(np.int32)
    cu = np.zeros(B + 1, np.int32)
    cu[1:] = np.cumsum(n)
    anchor = rng.integers(0, cfg.vocab - 1, size=B).astype(np.int32)
    shape = (int(cu[-1]), cfg.n_kv_heads, cfg.head_dim)
    return {"anchor": anchor, "cu_seqlens": cu,
            "ctx_k": [normal(shape, (s, 60 + 2 * l), 1.0, cfg.dtype) for l in range(cfg.layers)],
            "ctx_v": [normal(shape, (s, 61 + 2 * l), 1.0, cfg.dtype) for l in range(cfg.layers)]}


def dflash_oracle_cfg(cfg) -> dict:
    return dict(d=cfg.d, n_heads=cfg.n_heads, n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim,
                rms_eps=cfg.rms_eps, rope_theta=cfg.rope_theta, gamma=cfg.gamma, mask_token=cfg.mask_id)
