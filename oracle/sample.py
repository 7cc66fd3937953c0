"""Sampling beyond greedy for the final step: the oracle's definition
(TEST INFRASTRUCTURE ONLY; the package header's rule applies).

The pages stop at the next token; they name no sampler.  The plainest
temperature sampler is taken: the next token is a draw from
softmax(logits / T).  It is written as the Gumbel-max construction: with
independent standard Gumbel noise g_v, argmax_v (logits_v / T + g_v) is
distributed as softmax(logits / T) (Gumbel, "Statistical Theory of Extreme
Values", 1954; used for categorical sampling throughout the literature).
Every draw the method needs comes from a counter-based generator whose
published definition both sides implement on their own: Philox4x32-10
(Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
SC 2011, section 4 and its reference implementation's known-answer values).

Noise of vocabulary row v for the request in batch slot `slot` decoding
position `pos`, with seed s (64 bits):
    x = word 0 of Philox4x32-10(counter = (v, pos, slot, 0), key = (s mod 2^32, s >> 32))
    u = ((x >> 9) + 1/2) * 2^-23            (exact in float32, strictly inside (0, 1))
    g = -log(-log(u))
and the token is the lowest index among the maxima of the float32-rounded
keys logits / T + g (the kernel's precision for the decision).  T = 0 is
greedy decoding.

Nucleus (top-p) sampling restricts the draw to the nucleus: rows sorted by
logit (descending, lower index first among equal logits), the shortest
prefix whose softmax(logits / T) mass reaches p.  Gumbel-max over a subset
draws from the distribution renormalised to that subset, so the token is the
argmax of the same keys over the nucleus only.  p = 1 is plain temperature
sampling.
"""
from __future__ import annotations

import numpy as np
import torch

M0, M1 = 0xD2511F53, 0xCD9E8D57          # Philox4x32 multipliers
W0, W1 = 0x9E3779B9, 0xBB67AE85          # Weyl increments of the key
MASK = 0xFFFFFFFF


def philox4x32_10(ctr, key):
    """Philox4x32 with 10 rounds over arrays: ctr = (c0, c1, c2, c3) and
    key = (k0, k1), each an integer or a uint64 numpy array of 32-bit
    values.  Returns the four output words as uint64 arrays."""
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & np.uint64(MASK) for c in ctr)
    k0, k1 = (np.asarray(k, dtype=np.uint64) & np.uint64(MASK) for k in key)
    m0, m1, mask, sh = np.uint64(M0), np.uint64(M1), np.uint64(MASK), np.uint64(32)
    for r in range(10):
        if r > 0:                                   # the key moves on before every round but the first
            k0 = (k0 + np.uint64(W0)) & mask
            k1 = (k1 + np.uint64(W1)) & mask
        p0 = m0 * c0                                # 64-bit products of 32-bit words: exact
        p1 = m1 * c2
        hi0, lo0 = p0 >> sh, p0 & mask
        hi1, lo1 = p1 >> sh, p1 & mask
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def uniform(rows, pos: int, slot: int, seed: int) -> np.ndarray:
    """u in (0, 1) for vocabulary rows `rows` (float64, each exact in float32)."""
    v = np.asarray(rows, dtype=np.uint64)
    x = philox4x32_10((v, pos, slot, 0), (seed & MASK, (seed >> 32) & MASK))[0]
    return ((x >> np.uint64(9)).astype(np.float64) + 0.5) * 2.0 ** -23


def gumbel(rows, pos: int, slot: int, seed: int) -> np.ndarray:
    u = uniform(rows, pos, slot, seed)
    return -np.log(-np.log(u))


def sample_keys(logits: torch.Tensor, temperature: float, seed: int, slot: int, pos: int) -> torch.Tensor:
    """float64 keys logits / T + g over the whole vocabulary (T > 0)."""
    g = gumbel(np.arange(logits.shape[0]), pos, slot, seed)
    return logits.double() / temperature + torch.from_numpy(g)


def nucleus(logits: torch.Tensor, temperature: float, top_p: float) -> torch.Tensor:
    """Row indices of the nucleus for T > 0 and 0 < top_p <= 1 (float64 mass)."""
    l = logits.double()
    order = sorted(range(l.shape[0]), key=lambda v: (-float(l[v]), v))
    prob = torch.softmax(l / temperature, 0)
    mass, keep = 0.0, []
    for v in order:
        keep.append(v)
        mass += float(prob[v])
        if mass >= top_p:
            break
    return torch.tensor(keep, dtype=torch.long)


def sample_token(logits: torch.Tensor, temperature: float, seed: int, slot: int, pos: int,
                 top_p: float = 1.0) -> int:
    """The next token: greedy at T = 0, else the argmax of the float32 keys
    (lowest index on ties), over the nucleus when top_p < 1."""
    if temperature == 0:
        return int(torch.argmax(logits.to(torch.float32)))
    keys = sample_keys(logits, temperature, seed, slot, pos).to(torch.float32)
    if top_p >= 1.0:
        return int(torch.argmax(keys))
    rows = nucleus(logits, temperature, top_p)
    sub = keys[rows]
    best = float(sub.max())
    return int(rows[sub == best].min())
