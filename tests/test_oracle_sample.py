"""Pins of the oracle's temperature sampler (oracle/sample.py), CPU only.

- Philox4x32-10 against the known-answer values published with its
  reference implementation (tests/golden/philox4x32_10_kat.json);
- the uniforms sit strictly inside (0, 1) at both ends of the 32-bit range;
- draws over many positions follow softmax(logits / T) (chi-square), which
  pins the Gumbel transform's signs and the 1 / T scaling;
- a tiny temperature gives the greedy token, and distinct (slot, position)
  pairs draw distinct noise."""
import json
import math
import os

import numpy as np
import torch

from oracle import sample as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.json")


def test_philox_known_answers():
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        ctr = [int(x, 16) for x in c["counter"]]
        key = [int(x, 16) for x in c["key"]]
        out = [int(w) for w in S.philox4x32_10(ctr, key)]
        assert out == [int(x, 16) for x in c["out"]], c


def test_uniform_strictly_inside_unit_interval():
    # the generator's extreme outputs map to 2^-24 and 1 - 2^-24
    lo = ((np.uint64(0) >> np.uint64(9)).astype(np.float64) + 0.5) * 2.0 ** -23
    hi = ((np.uint64(0xFFFFFFFF) >> np.uint64(9)).astype(np.float64) + 0.5) * 2.0 ** -23
    assert lo == 2.0 ** -24 and hi == 1 - 2.0 ** -24
    u = S.uniform(np.arange(100000), pos=7, slot=3, seed=99)
    assert u.min() > 0 and u.max() < 1
    assert np.all(u.astype(np.float32).astype(np.float64) == u)      # exact in float32
    assert abs(u.mean() - 0.5) < 0.005


def test_draws_follow_softmax_of_scaled_logits():
    logits = torch.tensor([1.0, 0.2, -0.5, 2.0, 0.0], dtype=torch.float64)
    T = 1.3
    p = torch.softmax(logits / T, 0).numpy()
    n = 40000
    counts = np.zeros(5)
    for pos in range(n):
        counts[S.sample_token(logits, T, seed=2024, slot=pos % 3, pos=pos)] += 1
    chi2 = float(((counts - n * p) ** 2 / (n * p)).sum())
    assert chi2 < 25.0, (counts, n * p, chi2)      # 4 degrees of freedom: p-value ~ 5e-5
    # the same draws at T and at 2T differ: the scaling enters
    other = np.zeros(5)
    for pos in range(4000):
        other[S.sample_token(logits, 2 * T, seed=2024, slot=pos % 3, pos=pos)] += 1
    assert abs(other[3] / 4000 - torch.softmax(logits / (2 * T), 0)[3]) < 0.03


def test_tiny_temperature_is_greedy_and_noise_is_keyed():
    g = torch.Generator().manual_seed(5)
    logits = torch.randn(1000, generator=g, dtype=torch.float64) * 3
    for pos in range(20):
        assert S.sample_token(logits, 1e-6, seed=1, slot=0, pos=pos) == int(torch.argmax(logits))
    assert S.sample_token(logits, 0, seed=1, slot=0, pos=0) == int(torch.argmax(logits))
    a = S.gumbel(np.arange(64), pos=5, slot=0, seed=1)
    assert not np.array_equal(a, S.gumbel(np.arange(64), pos=6, slot=0, seed=1))
    assert not np.array_equal(a, S.gumbel(np.arange(64), pos=5, slot=1, seed=1))
    assert not np.array_equal(a, S.gumbel(np.arange(64), pos=5, slot=0, seed=2))
    assert not np.array_equal(a, S.gumbel(np.arange(64), pos=5, slot=0, seed=1 << 32))
    assert np.array_equal(a, S.gumbel(np.arange(64), pos=5, slot=0, seed=1))
    # the Gumbel law: mean = Euler-Mascheroni constant, variance = pi^2 / 6
    z = S.gumbel(np.arange(200000), pos=0, slot=0, seed=77)
    assert abs(z.mean() - 0.5772156649) < 0.01 and abs(z.var() - math.pi ** 2 / 6) < 0.03


def test_nucleus_is_the_shortest_prefix_reaching_p():
    g = torch.Generator().manual_seed(9)
    for trial in range(20):
        logits = torch.randn(12, generator=g, dtype=torch.float64) * 2
        logits[3] = logits[7]                       # an exact tie: the lower index comes first
        T = 0.5 + trial * 0.1
        p = 0.05 + 0.045 * trial
        rows = S.nucleus(logits, T, p).tolist()
        prob = torch.softmax(logits / T, 0)
        # brute force: the full order by (logit desc, index asc), then the shortest prefix with mass >= p
        order = sorted(range(12), key=lambda v: (-float(logits[v]), v))
        k = next(i for i in range(1, 13) if float(prob[order[:i]].sum()) >= p)
        assert rows == order[:k]
        assert float(prob[rows].sum()) >= p and (k == 1 or float(prob[rows[:-1]].sum()) < p)


def test_nucleus_draws_follow_the_renormalised_truncated_softmax():
    logits = torch.tensor([1.0, 0.2, -0.5, 2.0, 0.0, -1.0], dtype=torch.float64)
    T, p = 1.1, 0.8
    keep = S.nucleus(logits, T, p).tolist()
    prob = torch.softmax(logits / T, 0)
    want = np.zeros(6)
    want[keep] = (prob[keep] / prob[keep].sum()).numpy()
    n = 30000
    counts = np.zeros(6)
    for pos in range(n):
        counts[S.sample_token(logits, T, seed=5, slot=pos % 4, pos=pos, top_p=p)] += 1
    assert counts[[v for v in range(6) if v not in keep]].sum() == 0
    chi2 = float(sum((counts[v] - n * want[v]) ** 2 / (n * want[v]) for v in keep))
    assert chi2 < 25.0, (counts, n * want, chi2)


def test_nucleus_limits():
    g = torch.Generator().manual_seed(4)
    logits = torch.randn(300, generator=g, dtype=torch.float64)
    for pos in range(30):
        # a nucleus that is the whole vocabulary draws exactly the plain temperature sample
        assert S.sample_token(logits, 0.9, 3, 1, pos, top_p=1 - 1e-12) == S.sample_token(logits, 0.9, 3, 1, pos)
        # a vanishing nucleus is the greedy token
        assert S.sample_token(logits, 0.9, 3, 1, pos, top_p=1e-9) == int(torch.argmax(logits))
