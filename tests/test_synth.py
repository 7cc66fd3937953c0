"""Seeded input generator: determinism, distribution, paged placement, and
(on a GPU) identical bits from the host and device builds."""
import numpy as np
import pytest
import torch

import synth
from synth import TINY


def test_deterministic_and_offset_consistent():
    a = synth.normal((1000,), 0, "x")
    b = synth.normal((1000,), 0, "x")
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    c = synth.normal((400,), 0, "x", start=600)
    assert torch.equal(a[600:].view(torch.int16), c.view(torch.int16))
    d = synth.normal((1000,), 1, "x")
    e = synth.normal((1000,), 0, "y")
    assert not torch.equal(a, d) and not torch.equal(a, e)


def test_moments():
    x = synth.normal((2_000_000,), 0, "m", sigma=0.02).double()
    assert abs(x.mean().item()) < 1e-4
    assert abs(x.std().item() / 0.02 - 1) < 2e-3
    g = synth.normal((100_000,), 0, "g", mean=1.0).double()
    assert abs(g.mean().item() - 1) < 1e-3


def test_uniform_ints_range_and_mean():
    t = synth.uniform_ints(200_000, 4096, 0, "tok")
    assert int(t.min()) >= 0 and int(t.max()) < 4096
    assert abs(t.double().mean().item() / 2047.5 - 1) < 0.01


def test_kv_paged_placement_matches_logical_cpu():
    D = TINY
    n = 100
    pt = torch.from_numpy(synth.page_permutation(12, 0))
    pool = torch.zeros(12, D.n_kv_heads, D.head_dim, D.page_size, dtype=torch.bfloat16)
    synth.fill_kv_paged_(pool, pt, n, 0, synth.kv_name(3, 1, "K"))
    k, _ = synth.prior_kv(D, 0, 3, 1, n)
    for pos in range(n):
        got = pool[pt[pos // D.page_size], :, :, pos % D.page_size]
        assert torch.equal(got.view(torch.int16), k[pos].view(torch.int16))


def test_log_uniform_lengths_in_range():
    w = synth.workload("full_b8_long")
    assert len(w.ctx) == 8 and all(8192 <= c <= 262144 for c in w.ctx)
    w = synth.workload("full_b32_churn")
    assert len(w.ctx) == 32 and all(512 <= c <= 32768 for c in w.ctx)


@pytest.mark.gpu
def test_host_and_device_bits_identical():
    n = 3_000_003
    a = synth.normal((n,), 7, "cmp", start=(1 << 33) + 5)
    b = synth.normal((n,), 7, "cmp", start=(1 << 33) + 5, device="cuda").cpu()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    D = TINY
    pt = torch.from_numpy(synth.page_permutation(12, 0))
    pc = torch.zeros(12, D.n_kv_heads, D.head_dim, D.page_size, dtype=torch.bfloat16)
    pg = pc.cuda()
    synth.fill_kv_paged_(pc, pt, 150, 0, "kvcmp")
    synth.fill_kv_paged_(pg, pt.cuda(), 150, 0, "kvcmp")
    assert torch.equal(pc.view(torch.int16), pg.cpu().view(torch.int16))
