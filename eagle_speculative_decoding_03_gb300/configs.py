"""Workload shapes for the EAGLE draft-tree expansion step.

Sizes only: no arithmetic of the method lives here.  Notation follows the pages:
``B`` batch of requests, ``n`` verified-prefix length, ``depth`` the number of
sequential draft steps (gamma), ``k`` top-k branching, ``m`` nodes kept by the
rerank, ``d`` hidden size, ``vocab`` = |V| (kaushalya.io, "Dimension key used
throughout"; zackli.ai "Speculative Decoding Deep Dive III", section "EAGLE-2 -
context-aware dynamic tree").
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional, Tuple


@dataclass(frozen=True)
class DraftConfig:
    name: str
    d: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    d_ff: int
    vocab: int
    rms_eps: float
    rope_theta: float
    dtype: str                 # weight / cache storage: "f32" or "bf16"
    tree: str                  # "static" (EAGLE-1) or "dynamic" (EAGLE-2 expand-and-rerank)
    depth: int                 # gamma: sequential draft steps
    k: int = 0                 # dynamic: children per expanded node and frontier width
    m: int = 0                 # dynamic: nodes kept by the rerank
    branching: Tuple[int, ...] = ()   # static: children per node at each depth
    feat: str = "f"            # "f" (EAGLE-1/2 target feature) or "fused" (EAGLE-3 g = FC([l;m;h]))
    B: int = 1
    prefix: Tuple[int, int] = (0, 0)  # verified prefix length n_b ~ U[lo, hi] (lo == hi: fixed n)
    seed: int = 1000
    logit_std: float = 3.0     # LM-head weight scale: logits of an N(0,1)-scale feature have this std
    gamma_jitter: float = 0.0  # RMSNorm gains 1 + jitter * N(0,1); 0 gives unit gains

    # ---- derived sizes -------------------------------------------------
    @property
    def qkv_dim(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def attn_dim(self) -> int:
        return self.n_heads * self.head_dim

    def children_at(self, s: int) -> int:
        """Children generated per expanded row at depth s (1-based)."""
        return self.branching[s - 1] if self.tree == "static" else self.k

    def rows_at(self, s: int) -> int:
        """Rows (forward passes of the draft layer) per request at depth s."""
        if s == 1:
            return 1
        if self.tree == "static":
            r = 1
            for j in range(s - 1):
                r *= self.branching[j]
            return r
        return self.k

    def generated_per_request(self) -> int:
        return sum(self.rows_at(s) * self.children_at(s) for s in range(1, self.depth + 1))

    def rows_per_request(self) -> int:
        return sum(self.rows_at(s) for s in range(1, self.depth + 1))

    def kept_per_request(self) -> int:
        """Tree nodes emitted besides the root (static trees keep every node)."""
        return self.generated_per_request() if self.tree == "static" else self.m

    def with_(self, **kw) -> "DraftConfig":
        return replace(self, **kw)


LLAMA3_8B_HEAD = dict(d=4096, n_heads=32, n_kv_heads=8, head_dim=128, d_ff=14336, vocab=128256,
                      rms_eps=1e-6, rope_theta=5e5, dtype="bf16")

CONFIGS = {
    # 1. tiny fp32 chain: k=1, depth 4, n=32
    "tiny_chain": DraftConfig(
        name="tiny_chain", d=256, n_heads=4, n_kv_heads=4, head_dim=64, d_ff=688, vocab=1024,
        rms_eps=1e-6, rope_theta=1e4, dtype="f32", tree="dynamic", depth=4, k=1, m=4,
        B=1, prefix=(32, 32), seed=1001),
    # 2. EAGLE-1 static tree [4,2,1,1,1] on a Llama-2-7B-shaped head, n=1024
    "eagle1_static": DraftConfig(
        name="eagle1_static", d=4096, n_heads=32, n_kv_heads=32, head_dim=128, d_ff=11008,
        vocab=32000, rms_eps=1e-6, rope_theta=1e4, dtype="bf16", tree="static", depth=5,
        branching=(4, 2, 1, 1, 1), B=1, prefix=(1024, 1024), seed=1002),
    # 3. EAGLE-2 dynamic tree k=10 depth 6 m=60, Llama-3-8B-shaped head, n=2048
    "eagle2_b1": DraftConfig(
        name="eagle2_b1", **LLAMA3_8B_HEAD, tree="dynamic", depth=6, k=10, m=60,
        B=1, prefix=(2048, 2048), seed=1003),
    # 4. batched serving B=32, k=8 depth 6 m=48, per-request prefix n_b ~ U[256, 4096]
    "eagle2_b32": DraftConfig(
        name="eagle2_b32", **LLAMA3_8B_HEAD, tree="dynamic", depth=6, k=8, m=48,
        B=32, prefix=(256, 4096), seed=1004),
    # 5. EAGLE-3 fusion, Llama-3-70B-shaped head, B=8, n=4096, k=10 depth 7 m=60
    "eagle3_b8": DraftConfig(
        name="eagle3_b8", d=8192, n_heads=64, n_kv_heads=8, head_dim=128, d_ff=28672,
        vocab=128256, rms_eps=1e-6, rope_theta=5e5, dtype="bf16", tree="dynamic", depth=7,
        k=10, m=60, feat="fused", B=8, prefix=(4096, 4096), seed=1005),
}

# Small shapes that still span several tiles of every kernel and leave ragged tails;
# the oracle finishes each in well under a second.
SMALL = {
    "small_dyn": DraftConfig(
        name="small_dyn", d=512, n_heads=4, n_kv_heads=2, head_dim=128, d_ff=1280, vocab=4096,
        rms_eps=1e-6, rope_theta=1e4, dtype="bf16", tree="dynamic", depth=3, k=4, m=10,
        B=3, prefix=(37, 301), seed=2001, gamma_jitter=0.1),
    "small_static": DraftConfig(
        name="small_static", d=256, n_heads=2, n_kv_heads=2, head_dim=128, d_ff=768, vocab=2048,
        rms_eps=1e-6, rope_theta=1e4, dtype="bf16", tree="static", depth=4, branching=(3, 2, 1, 1),
        B=2, prefix=(0, 129), seed=2002, gamma_jitter=0.1),
    "small_fused": DraftConfig(
        name="small_fused", d=512, n_heads=8, n_kv_heads=2, head_dim=128, d_ff=1024, vocab=3072,
        rms_eps=1e-6, rope_theta=5e5, dtype="bf16", tree="dynamic", depth=4, k=5, m=12,
        feat="fused", B=2, prefix=(200, 200), seed=2003, gamma_jitter=0.1),
    # the largest tree the boundary takes: k = 16, 16 rows x 16 children = 256 candidates per
    # request at each depth, 49 rows per request (one 64-bit row mask), m + 1 = 64 slots
    "small_max": DraftConfig(
        name="small_max", d=256, n_heads=2, n_kv_heads=1, head_dim=128, d_ff=640, vocab=2048,
        rms_eps=1e-6, rope_theta=1e4, dtype="bf16", tree="dynamic", depth=4, k=16, m=63,
        B=2, prefix=(1, 90), seed=2005, gamma_jitter=0.1),
    # 24 requests x 4 rows = 96 rows per depth: the LM head stores logits and a select kernel
    # takes the top-k, over a vocabulary of 33 select parts of 1024 keys (the last one ragged)
    "small_wide": DraftConfig(
        name="small_wide", d=256, n_heads=2, n_kv_heads=1, head_dim=128, d_ff=640, vocab=33152,
        rms_eps=1e-6, rope_theta=1e4, dtype="bf16", tree="dynamic", depth=3, k=4, m=10,
        B=24, prefix=(5, 60), seed=2007, gamma_jitter=0.1),
    # 48 requests x 4 rows = 192 rows per depth: GEMMs and the LM head run as CTA pairs sharing
    # the weight stream (two row blocks), the LM head stores logits for the select kernel
    "small_pairs": DraftConfig(
        name="small_pairs", d=256, n_heads=2, n_kv_heads=1, head_dim=128, d_ff=640, vocab=16384,
        rms_eps=1e-6, rope_theta=1e4, dtype="bf16", tree="dynamic", depth=3, k=4, m=10,
        B=48, prefix=(5, 40), seed=2008, gamma_jitter=0.1),
    "small_f32": DraftConfig(
        name="small_f32", d=192, n_heads=3, n_kv_heads=1, head_dim=64, d_ff=400, vocab=700,
        rms_eps=1e-6, rope_theta=1e4, dtype="f32", tree="dynamic", depth=3, k=3, m=7,
        B=2, prefix=(5, 70), seed=2004, gamma_jitter=0.1),
}

ALL = {**CONFIGS, **SMALL}


def get(name: str) -> DraftConfig:
    return ALL[name]


@dataclass(frozen=True)
class DFlashConfig:
    """A DFlash block-parallel draft ("DFlash-1: parallel block + KV injection", zackli.ai):
    ``layers`` draft layers, a block of the anchor plus ``gamma`` mask slots, the top-``k``
    tokens of each mask slot; the target's fused context is injected as per-layer KV."""
    name: str
    d: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    d_ff: int
    vocab: int
    rms_eps: float
    rope_theta: float
    dtype: str
    layers: int
    gamma: int
    k: int = 1
    B: int = 1
    prefix: Tuple[int, int] = (0, 0)
    seed: int = 1000
    logit_std: float = 3.0
    gamma_jitter: float = 0.0
    mask_token: int = -1       # -1: the last id of the table

    @property
    def mask_id(self) -> int:
        return self.vocab - 1 if self.mask_token < 0 else self.mask_token

    @property
    def qkv_dim(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim

    @property
    def attn_dim(self) -> int:
        return self.n_heads * self.head_dim

    def with_(self, **kw) -> "DFlashConfig":
        return replace(self, **kw)


DFLASH = {
    # the Llama-3-8B-shaped head as a 5-layer DFlash drafting a block of 16 ("A 5-layer DFlash
    # drafting 16"), prefix 2048, B=1
    "dflash_b1": DFlashConfig(name="dflash_b1", **LLAMA3_8B_HEAD, layers=5, gamma=16, k=1, B=1,
                              prefix=(2048, 2048), seed=1006),
    "small_dflash": DFlashConfig(
        name="small_dflash", d=512, n_heads=4, n_kv_heads=2, head_dim=128, d_ff=1280, vocab=4096,
        rms_eps=1e-6, rope_theta=1e4, dtype="bf16", layers=3, gamma=8, k=3, B=3, prefix=(37, 301),
        seed=2006, gamma_jitter=0.1),
}
