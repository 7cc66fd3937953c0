"""Pins for the oracle's building blocks, each against something other than
the oracle itself: closed forms, brute force on tiny inputs, library
routines, and invariants."""
import math
import random

import pytest
import torch

from oracle import decode as O

F64 = torch.float64


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_rne_matches_torch_float32_conversion():
    # For float32-representable inputs, direct RNE to bf16 equals torch's
    # float32 -> bfloat16 conversion (a library routine, RNE).
    g = torch.Generator().manual_seed(1)
    x32 = (torch.randn(20000, generator=g) * torch.exp(torch.randn(20000, generator=g) * 3)).float()
    ref = x32.to(torch.bfloat16).to(F64)
    assert torch.equal(O.bf16_rne(x32.to(F64)), ref)


def test_bf16_rne_ties_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties to the even mantissa (1).
    assert O.bf16_rne(torch.tensor([1 + 2 ** -8], dtype=F64)).item() == 1.0
    # 1 + 3*2^-8 is halfway between 1+2^-7 (odd) and 1+2^-6 (even).
    assert O.bf16_rne(torch.tensor([1 + 3 * 2 ** -8], dtype=F64)).item() == 1 + 2 ** -6
    # just above the halfway point rounds up
    assert O.bf16_rne(torch.tensor([1 + 2 ** -8 + 2 ** -30], dtype=F64)).item() == 1 + 2 ** -7
    assert O.bf16_rne(torch.tensor([-3.0], dtype=F64)).item() == -3.0


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_matches_library():
    g = torch.Generator().manual_seed(2)
    x = torch.randn(300, generator=g, dtype=F64)
    gamma = (1 + 0.02 * torch.randn(300, generator=g)).to(torch.bfloat16)
    ref = torch.nn.functional.rms_norm(x, (300,), weight=gamma.to(F64), eps=1e-6)
    assert torch.allclose(O.rmsnorm(x, gamma, 1e-6), ref, rtol=1e-14, atol=0)


def test_rmsnorm_constant_vector_gives_gain():
    gamma = torch.tensor([0.5, 1.0, 2.0, -1.0], dtype=torch.bfloat16)
    for c in (3.0, -0.25):
        y = O.rmsnorm(torch.full((4,), c, dtype=F64), gamma, 0.0)
        assert torch.allclose(y, math.copysign(1, c) * gamma.to(F64), rtol=1e-15)


# ---------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    v = torch.randn(3, 8, dtype=F64)
    assert torch.equal(O.rope(v, 0, 1e4), v)


def test_rope_closed_form_pairs_and_sign():
    # d = 4: pairs (0, 2) with inv_freq 1 and (1, 3) with inv_freq theta^(-1/2).
    theta, p = 100.0, 3
    e0 = torch.tensor([[1.0, 0, 0, 0]], dtype=F64)
    assert torch.allclose(O.rope(e0, p, theta), torch.tensor([[math.cos(p), 0, math.sin(p), 0]], dtype=F64))
    e1 = torch.tensor([[0, 1.0, 0, 0]], dtype=F64)
    w = p * theta ** -0.5
    assert torch.allclose(O.rope(e1, p, theta), torch.tensor([[0, math.cos(w), 0, math.sin(w)]], dtype=F64))
    e2 = torch.tensor([[0, 0, 1.0, 0]], dtype=F64)
    assert torch.allclose(O.rope(e2, p, theta), torch.tensor([[-math.sin(p), 0, math.cos(p), 0]], dtype=F64))


def test_rope_preserves_norm_and_is_relative():
    g = torch.Generator().manual_seed(3)
    q = torch.randn(1, 64, generator=g, dtype=F64)
    k = torch.randn(1, 64, generator=g, dtype=F64)
    assert torch.allclose(O.rope(q, 12345, 1e4).norm(), q.norm(), rtol=1e-13)
    a = (O.rope(q, 700, 1e4) * O.rope(k, 650, 1e4)).sum()
    b = (O.rope(q, 50, 1e4) * k).sum()
    assert abs(a - b) < 1e-10


# ---------------------------------------------------------------- attention

def _brute_attention(q, K, V):
    nq, d = q.shape
    T, nkv, _ = K.shape
    G = nq // nkv
    out = [[0.0] * d for _ in range(nq)]
    for h in range(nq):
        g = h // G
        s = [sum(float(q[h, i]) * float(K[t, g, i]) for i in range(d)) / math.sqrt(d) for t in range(T)]
        m = max(s)
        w = [math.exp(x - m) for x in s]
        z = sum(w)
        for i in range(d):
            out[h][i] = sum(w[t] * float(V[t, g, i]) for t in range(T)) / z
    return torch.tensor(out, dtype=F64)


def test_attention_brute_force_tiny():
    g = torch.Generator().manual_seed(4)
    q = torch.randn(6, 8, generator=g, dtype=F64)
    K = torch.randn(5, 3, 8, generator=g).to(torch.bfloat16)
    V = torch.randn(5, 3, 8, generator=g).to(torch.bfloat16)
    assert torch.allclose(O.gqa_attention(q, K, V), _brute_attention(q, K, V), rtol=1e-12, atol=1e-13)


def test_attention_single_token_returns_value():
    q = torch.randn(4, 16, dtype=F64)
    K = torch.randn(1, 2, 16).to(torch.bfloat16)
    V = torch.randn(1, 2, 16).to(torch.bfloat16)
    o = O.gqa_attention(q, K, V)
    assert torch.equal(o[0], V[0, 0].to(F64)) and torch.equal(o[3], V[0, 1].to(F64))


def test_attention_group_mapping_contiguous():
    # KV head g carries the constant value g + 1: head h must read group h // G.
    nq, nkv, d, T = 8, 2, 4, 7
    q = torch.randn(nq, d, dtype=F64)
    K = torch.randn(T, nkv, d).to(torch.bfloat16)
    V = torch.stack([torch.full((T, d), g + 1.0) for g in range(nkv)], dim=1).to(torch.bfloat16)
    o = O.gqa_attention(q, K, V)
    for h in range(nq):
        assert torch.allclose(o[h], torch.full((d,), h // (nq // nkv) + 1.0, dtype=F64), rtol=1e-14)


def test_attention_two_token_closed_form():
    d = 4
    q = torch.tensor([[2.0, 0, 0, 0]], dtype=F64)
    K = torch.tensor([[[1.0, 0, 0, 0]], [[0.0, 0, 0, 0]]]).to(torch.bfloat16)
    V = torch.tensor([[[1.0, 0, 0, 0]], [[0.0, 1.0, 0, 0]]]).to(torch.bfloat16)
    # s0 = 2/sqrt(4) = 1, s1 = 0
    p0 = math.e / (math.e + 1)
    o = O.gqa_attention(q, K, V)
    assert torch.allclose(o[0], torch.tensor([p0, 1 - p0, 0, 0], dtype=F64), rtol=1e-14)


def test_attention_key_order_invariant():
    g = torch.Generator().manual_seed(5)
    q = torch.randn(4, 16, generator=g, dtype=F64)
    K = torch.randn(33, 2, 16, generator=g).to(torch.bfloat16)
    V = torch.randn(33, 2, 16, generator=g).to(torch.bfloat16)
    perm = torch.randperm(33, generator=g)
    assert torch.allclose(O.gqa_attention(q, K, V), O.gqa_attention(q, K[perm], V[perm]), rtol=1e-12)


# ---------------------------------------------------------------- routing

def test_route_brute_force_and_gates():
    rng = random.Random(6)
    for _ in range(50):
        E, k = rng.choice([(8, 2), (16, 4), (128, 8)])
        r = torch.tensor([rng.gauss(0, 1) for _ in range(E)], dtype=F64)
        ids, gates, P = O.route(r, k)
        r32 = [float(x) for x in r.to(torch.float32)]
        want = sorted(range(E), key=lambda i: (-r32[i], i))[:k]
        assert ids == want
        assert abs(float(P.sum()) - 1) < 1e-12 and abs(float(gates.sum()) - 1) < 1e-12
        z = sum(math.exp(float(r[i])) for i in want)
        for j, i in enumerate(want):
            assert abs(float(gates[j]) - math.exp(float(r[i])) / z) < 1e-12


def test_route_ties_go_to_lower_index():
    r = torch.tensor([0.5, 1.0, 0.2, 1.0, 1.0, 0.9], dtype=F64)
    ids, gates, _ = O.route(r, 2)
    assert ids == [1, 3]
    assert torch.allclose(gates, torch.tensor([0.5, 0.5], dtype=F64))
    ids, _, _ = O.route(r, 4)
    assert ids == [1, 3, 4, 5]


def test_route_k_equals_E_is_plain_softmax():
    r = torch.randn(8, dtype=F64)
    ids, gates, P = O.route(r, 8)
    full = torch.softmax(r, dim=0)
    assert torch.allclose(gates, full[ids], rtol=1e-13)


def test_route_force_keeps_own_gates():
    r = torch.tensor([3.0, 2.0, 1.0, 0.0], dtype=F64)
    ids, gates, _ = O.route(r, 2, force=[0, 2])
    assert ids == [0, 2]
    assert abs(float(gates[0]) - math.exp(3) / (math.exp(3) + math.exp(1))) < 1e-14


# ---------------------------------------------------------------- SwiGLU expert

def test_silu_closed_form():
    z = torch.tensor([0.0, 1.0, -2.0, 30.0], dtype=F64)
    want = [0.0, 1 / (1 + math.exp(-1)), -2 / (1 + math.exp(2)), 30 / (1 + math.exp(-30))]
    assert torch.allclose(O.silu(z), torch.tensor(want, dtype=F64), rtol=1e-15)


def test_expert_brute_force_non_square():
    g = torch.Generator().manual_seed(7)
    H, F = 6, 4
    xn = torch.randn(H, generator=g, dtype=F64)
    wg = torch.randn(F, H, generator=g).to(torch.bfloat16)
    wu = torch.randn(F, H, generator=g).to(torch.bfloat16)
    wd = torch.randn(H, F, generator=g).to(torch.bfloat16)
    h = []
    for f in range(F):
        a = sum(float(wg[f, i]) * float(xn[i]) for i in range(H))
        b = sum(float(wu[f, i]) * float(xn[i]) for i in range(H))
        h.append(a / (1 + math.exp(-a)) * b)
    y = [sum(float(wd[o, f]) * h[f] for f in range(F)) for o in range(H)]
    assert torch.allclose(O.expert_ffn(xn, wg, wu, wd), torch.tensor(y, dtype=F64), rtol=1e-12)
