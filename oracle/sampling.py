"""Sampled drafting and speculative sampling for the float64 oracle.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg may import or run this module; no product code does.  It shares no
code with the CUDA library: plain numpy.

* Counter-based random numbers: Philox4x32-10 (J. Salmon, M. Moraes, R. Dror, D. Shaw,
  "Parallel random numbers: as easy as 1, 2, 3", SC 2011), written from its published
  definition: ten rounds; each round multiplies counter words 0 and 2 by the two round
  constants (high and low halves of the 64-bit products), XORs the high halves with the
  other two counter words and the key, and permutes; the key advances by the two Weyl
  constants between rounds.
* Sampled drafting ("EAGLE-1 - autoregressive feature drafting", zackli.ai: the draft
  samples its next token from p-hat; "The recurrence, written out", aicassindra.com):
  a node's k children are k tokens drawn without replacement from the draft's
  distribution, taken as the top-k of log p-hat + Gumbel noise (the Gumbel-top-k trick).

Readings (listed in the design notes):
* the noise of token t in row i (frontier slot) at depth s of request b is
  G = -log(-log U), U built from word ((t mod 128) div 32) of
  Philox4x32-10(counter = (32 * (t div 128) + t mod 32, i, s, 0), key = the request's
  64-bit seed as (low word, high word)), U = (x + 1/2) / 2^32, with -log U evaluated as
  -log1p(-(2^32 - 1/2 - x) / 2^32) so that U near 1 keeps its precision;
* temperature 1; the children's path values use the unperturbed log-probabilities.
"""
from __future__ import annotations

import numpy as np

M0, M1 = 0xD2511F53, 0xCD9E8D57          # round multipliers
W0, W1 = 0x9E3779B9, 0xBB67AE85          # key increments (Weyl sequence)
MASK32 = 0xFFFFFFFF


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox4x32 with 10 rounds over arrays of counters (uint32 words); returns 4 words."""
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & MASK32 for c in (c0, c1, c2, c3))
    k0 = np.uint64(int(k0) & MASK32)
    k1 = np.uint64(int(k1) & MASK32)
    for r in range(10):
        if r:
            k0 = np.uint64((int(k0) + W0) & MASK32)
            k1 = np.uint64((int(k1) + W1) & MASK32)
        p0 = np.uint64(M0) * c0            # < 2^64: exact in uint64
        p1 = np.uint64(M1) * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(MASK32)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(MASK32)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return tuple(x.astype(np.uint32) for x in (c0, c1, c2, c3))


def token_words(vocab: int, i: int, s: int, seed: int) -> np.ndarray:
    """The 32-bit word that token t (0..vocab-1) of row i at depth s draws (layout above)."""
    t = np.arange(vocab, dtype=np.int64)
    c0 = 32 * (t // 128) + t % 32
    word = (t % 128) // 32
    out = philox4x32_10(c0, np.full_like(c0, i), np.full_like(c0, s), np.zeros_like(c0),
                        seed & MASK32, (seed >> 32) & MASK32)
    return np.choose(word, out).astype(np.uint64)


def gumbel_from_words(x) -> np.ndarray:
    """G = -log(-log U), U = (x + 1/2) / 2^32, with -log U = -log1p(-(2^32 - 1/2 - x) / 2^32)."""
    x = np.asarray(x, dtype=np.float64)
    one_minus_u = (4294967296.0 - 0.5 - x) / 4294967296.0
    e = -np.log1p(-one_minus_u)            # = -log U > 0
    return -np.log(e)


def gumbel(vocab: int, i: int, s: int, seed: int) -> np.ndarray:
    return gumbel_from_words(token_words(vocab, i, s, seed))


# --------------------------------------------------------- speculative sampling (tree)
def accept_uniform(slot: int, seed: int) -> float:
    """The uniform that decides whether child slot `slot` is accepted:
    word 0 of Philox4x32-10(counter = (slot, 0, 0, 2), key = seed), U = (x + 1/2) / 2^32."""
    x = philox4x32_10([slot], [0], [0], [2], seed & MASK32, (seed >> 32) & MASK32)[0][0]
    return (float(x) + 0.5) / 4294967296.0


def correction_gumbel(vocab: int, u: int, r: int, seed: int) -> np.ndarray:
    """Gumbel noise for the token drawn at slot u after r rejected children: the drafting
    layout with counter words 1..3 = (u, r, 1)."""
    t = np.arange(vocab, dtype=np.int64)
    c0 = 32 * (t // 128) + t % 32
    word = (t % 128) // 32
    out = philox4x32_10(c0, np.full_like(c0, u), np.full_like(c0, r), np.ones_like(c0),
                        seed & MASK32, (seed >> 32) & MASK32)
    return gumbel_from_words(np.choose(word, out).astype(np.uint64))


def speculative_accept(tokens, parents, logp_target, logq_draft, seed: int) -> dict:
    """Multi-round speculative sampling over one emitted tree ("tree attention + multi-round
    speculative sampling", zackli.ai "Speculative Decoding Deep Dive III", EAGLE-1;
    "How speculative decoding works", kaushalya.io: accept a drafted token with
    probability min(1, p/q), otherwise draw from the renormalised residual).

    tokens / parents [S] (slot 0 the root); logp_target[u] the target's next-token
    log-probabilities after slot u's path; logq_draft[u] the draft's, from which u's
    children were drawn.  From the root, u's children are tried in slot order: child x is
    accepted when U * q(x) < p(x) (U = accept_uniform(slot)); on rejection the target
    becomes norm(max(0, p - q)) and x leaves the proposal (q restricted to the untried
    tokens, renormalised).  The walk moves to an accepted child; at a slot where no child
    is accepted (or a leaf) one token is drawn from the current target by Gumbel-max
    (correction_gumbel with the number of rejections there) and the walk ends.
    Returns the accepted slots, their tokens, the drawn token and per-trial records."""
    tokens = np.asarray(tokens, dtype=np.int64)
    parents = np.asarray(parents, dtype=np.int64)
    kids = {}
    for s in range(1, len(tokens)):
        kids.setdefault(int(parents[s]), []).append(s)
    u, accepted, trials = 0, [], []
    while True:
        p = np.exp(np.asarray(logp_target[u], dtype=np.float64))
        q = np.exp(np.asarray(logq_draft[u], dtype=np.float64))
        removed = 0.0                          # proposal mass of the rejected tokens
        nxt, r = None, 0
        for c in kids.get(u, []):
            x = int(tokens[c])
            qx = q[x] / (1.0 - removed)
            U = accept_uniform(c, seed)
            ok = U * qx < p[x]
            trials.append(dict(slot=c, token=x, u=U, p=float(p[x]), q=float(qx), accepted=bool(ok)))
            if ok:
                nxt = c
                break
            qcur = q / (1.0 - removed)
            res = np.maximum(p - qcur, 0.0)
            z = res.sum()
            if z > 0.0:                        # (z = 0 only when p == q, where x is always accepted)
                p = res / z
            removed += q[x]
            q[x] = 0.0
            r += 1
        if nxt is None:
            with np.errstate(divide="ignore"):
                score = np.where(p > 0.0, np.log(p), -np.inf) + correction_gumbel(len(p), u, r, seed)
            corr = int(np.argmax(score))
            srt = np.sort(score[np.isfinite(score)])[::-1]
            margin = float(srt[0] - srt[1]) if len(srt) > 1 else np.inf
            return dict(slots=accepted, tokens=[int(tokens[s]) for s in accepted], correction=corr,
                        length=len(accepted), trials=trials, rejections_at_end=r, margin=margin,
                        final_target=p)
        accepted.append(nxt)
        u = nxt


def draw_children(logp_row, k: int, i: int, s: int, seed: int):
    """k tokens drawn without replacement from exp(logp_row): the top-k of logp + Gumbel
    noise of row i at depth s, in draw order (largest perturbed value first, ties to the
    lower token id).  Returns (tokens in draw order, perturbed values, margin)."""
    from .eagle_oracle import top_k
    key = np.asarray(logp_row, dtype=np.float64) + gumbel(len(logp_row), i, s, seed)
    sel, margin = top_k(key, k)
    return sel, key, margin
