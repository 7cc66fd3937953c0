"""End-to-end pins of the oracle's decode step on small hand-built models with
non-square shapes (H != n_q*d), through special cases whose result is known
in closed form or by brute force, and through invariants."""
import math

import torch

from oracle import decode as O
from synth import Dims

F64 = torch.float64
BF = torch.bfloat16

D = Dims(n_layers=2, hidden=48, n_q_heads=4, n_kv_heads=2, head_dim=16, n_experts=4, top_k=2,
         expert_ffn=24, vocab=50)


class DictWeights:
    """Weight provider with random bf16 defaults and per-tensor overrides."""

    def __init__(self, dims, seed=0, over=None, **named):
        g = torch.Generator().manual_seed(seed)
        H, nq, nkv, d, E, F, V = (dims.hidden, dims.n_q_heads, dims.n_kv_heads, dims.head_dim,
                                  dims.n_experts, dims.expert_ffn, dims.vocab)
        r = lambda *s, sc=0.2: (torch.randn(*s, generator=g) * sc).to(BF)
        L = dims.n_layers
        self.t = {
            "embed": r(V, H, sc=1.0), "final_norm": (1 + r(H, sc=0.02).float()).to(BF), "lm_head": r(V, H),
        }
        for l in range(L):
            self.t[("attn_norm", l)] = (1 + r(H, sc=0.02).float()).to(BF)
            self.t[("ffn_norm", l)] = (1 + r(H, sc=0.02).float()).to(BF)
            self.t[("wq", l)] = r(nq * d, H)
            self.t[("wk", l)] = r(nkv * d, H)
            self.t[("wv", l)] = r(nkv * d, H)
            self.t[("wo", l)] = r(H, nq * d)
            self.t[("router", l)] = r(E, H)
            for e in range(E):
                self.t[("expert", l, e)] = (r(F, H), r(F, H), r(H, F))
        self.t.update(named)
        self.t.update(over or {})

    def embed_rows(self, toks):
        return self.t["embed"][list(toks)]

    def final_norm(self):
        return self.t["final_norm"]

    def lm_head(self):
        return self.t["lm_head"]

    def attn_norm(self, l):
        return self.t[("attn_norm", l)]

    def ffn_norm(self, l):
        return self.t[("ffn_norm", l)]

    def wq(self, l):
        return self.t[("wq", l)]

    def wk(self, l):
        return self.t[("wk", l)]

    def wv(self, l):
        return self.t[("wv", l)]

    def wo(self, l):
        return self.t[("wo", l)]

    def router(self, l):
        return self.t[("router", l)]

    def expert(self, l, e):
        return self.t[("expert", l, e)]


def prior_fn(dims, T, seed=11, perm=None):
    g = torch.Generator().manual_seed(seed)
    data = {l: (torch.randn(T, dims.n_kv_heads, dims.head_dim, generator=g).to(BF),
                torch.randn(T, dims.n_kv_heads, dims.head_dim, generator=g).to(BF))
            for l in range(dims.n_layers)}

    def f(rid, l, n):
        K, V = data[l]
        if perm is not None:
            K, V = K[perm], V[perm]
        return K[:n], V[:n]
    return f, data


def req(dims, T, **kw):
    f, data = prior_fn(dims, T, **kw)
    return O.OracleRequest(0, T, f, dims.n_layers), data


def dot(a, b):
    return sum(float(x) * float(y) for x, y in zip(a, b))


def test_prior_key_order_does_not_change_step():
    W = DictWeights(D)
    T = 19
    perm = torch.randperm(T, generator=torch.Generator().manual_seed(3))
    r1, _ = req(D, T)
    r2, _ = req(D, T, perm=perm)
    a = O.decode_step(W, D, r1, 5)
    b = O.decode_step(W, D, r2, 5)
    assert torch.allclose(a.logits, b.logits, rtol=1e-11, atol=1e-12)
    assert torch.allclose(a.hidden, b.hidden, rtol=1e-11, atol=1e-12)
    assert a.next_token == b.next_token


def test_zero_branches_leave_residual_and_give_plain_lm_head():
    over = {}
    for l in range(D.n_layers):
        over[("wo", l)] = torch.zeros(D.hidden, D.n_q_heads * D.head_dim, dtype=BF)
        for e in range(D.n_experts):
            wg, wu, _ = DictWeights(D).t[("expert", l, e)]
            over[("expert", l, e)] = (wg, wu, torch.zeros(D.hidden, D.expert_ffn, dtype=BF))
    W = DictWeights(D, over=over)
    r, _ = req(D, 9)
    tok = 17
    out = O.decode_step(W, D, r, tok)
    x = [float(v) for v in W.t["embed"][tok]]
    for l in range(D.n_layers):
        assert torch.equal(out.layers[l].x_out, torch.tensor(x, dtype=F64))
    ms = sum(v * v for v in x) / len(x)
    xf = [v / math.sqrt(ms + D.rms_eps) * float(gm) for v, gm in zip(x, W.t["final_norm"])]
    logits = [dot(W.t["lm_head"][i], xf) for i in range(D.vocab)]
    assert torch.allclose(out.logits, torch.tensor(logits, dtype=F64), rtol=1e-12, atol=1e-12)
    assert out.next_token == max(range(D.vocab), key=lambda i: (logits[i], -i))


def _const_embed_weights(c=0.75, over=None, **named):
    emb = torch.full((D.vocab, D.hidden), c, dtype=BF)
    return DictWeights(D, embed=emb, over=over, **named)


def test_zero_query_gives_uniform_attention_including_new_token():
    # Wq = 0 -> all scores equal -> o is the mean of the cached V rows plus
    # the new token's bf16-rounded v.  A constant embedding row c > 0 gives
    # rmsnorm(x) = gamma exactly.
    over = {("wq", l): torch.zeros(D.n_q_heads * D.head_dim, D.hidden, dtype=BF) for l in range(2)}
    W = _const_embed_weights(over=over)
    T = 13
    r, data = req(D, T)
    out = O.decode_step(W, D, r, 3)
    gamma = [float(v) for v in W.t[("attn_norm", 0)]]
    wv = W.t[("wv", 0)]
    d, G = D.head_dim, D.group
    v_new = [float(O.bf16_rne(torch.tensor(dot(wv[i], gamma), dtype=F64))) for i in range(D.n_kv_heads * d)]
    K0, V0 = data[0]
    o = []
    for h in range(D.n_q_heads):
        g = h // G
        for i in range(d):
            o.append((sum(float(V0[t, g, i]) for t in range(T)) + v_new[g * d + i]) / (T + 1))
    x = [0.75] * D.hidden
    x_mid = [x[j] + dot(W.t[("wo", 0)][j], o) for j in range(D.hidden)]
    assert torch.allclose(out.layers[0].x_mid, torch.tensor(x_mid, dtype=F64), rtol=1e-11, atol=1e-12)
    # the appended K row is the rotated, bf16-rounded key at position T
    wk = W.t[("wk", 0)]
    k_raw = torch.tensor([dot(wk[i], gamma) for i in range(D.n_kv_heads * d)], dtype=F64).view(2, d)
    half = d // 2
    k_rot = torch.empty_like(k_raw)
    for i in range(half):
        a = T * D.rope_theta ** (-2.0 * i / d)
        k_rot[:, i] = k_raw[:, i] * math.cos(a) - k_raw[:, i + half] * math.sin(a)
        k_rot[:, i + half] = k_raw[:, i + half] * math.cos(a) + k_raw[:, i] * math.sin(a)
    assert torch.allclose(r.appended_k[0][0], O.bf16_rne(k_rot), rtol=0, atol=0)


def test_second_step_attends_to_first_steps_value():
    over = {("wq", l): torch.zeros(D.n_q_heads * D.head_dim, D.hidden, dtype=BF) for l in range(2)}
    W = _const_embed_weights(over=over)
    T = 6
    r, data = req(D, T)
    O.decode_step(W, D, r, 3)
    v1 = r.appended_v[0][0]
    out2 = O.decode_step(W, D, r, 8)
    assert r.length == T + 2
    v2 = r.appended_v[0][1]
    V0 = data[0][1].to(F64)
    G, d = D.group, D.head_dim
    mean = (V0.sum(0) + v1 + v2) / (T + 2)                # [nkv, d]
    o = torch.cat([mean[h // G] for h in range(D.n_q_heads)])
    x_mid = torch.full((D.hidden,), 0.75, dtype=F64) + W.t[("wo", 0)].to(F64) @ o
    assert torch.allclose(out2.layers[0].x_mid, x_mid, rtol=1e-12)


def _brute_expert(wg, wu, wd, xn):
    F, H = wg.shape
    h = []
    for f in range(F):
        a = dot(wg[f], xn)
        h.append(a / (1 + math.exp(-a)) * dot(wu[f], xn))
    return [dot(wd[o], h) for o in range(H)]


def test_moe_gates_renormalise_over_selected_experts():
    # Identical experts: with k = 1 the single gate must be exactly 1 (a
    # missing renormalisation would give P_j < 1); with k = E the gates sum
    # to 1 and the mixture equals the one expert.
    for E, k in ((4, 1), (4, 4)):
        dims = Dims(1, 48, 4, 2, 16, E, k, 24, 50)
        base = DictWeights(dims)
        ex = base.t[("expert", 0, 0)]
        over = {("expert", 0, e): ex for e in range(E)}
        W = DictWeights(dims, over=over)
        r, _ = req(dims, 5)
        out = O.decode_step(W, dims, r, 4)
        tr = out.layers[0]
        assert abs(float(tr.gates.sum()) - 1.0) < 1e-14
        xn2 = O.rmsnorm(tr.x_mid, W.ffn_norm(0), dims.rms_eps)
        y = _brute_expert(*ex, [float(v) for v in xn2])
        assert torch.allclose(tr.x_out, tr.x_mid + torch.tensor(y, dtype=F64), rtol=1e-11, atol=1e-13)


def test_moe_weighted_sum_matches_brute_force():
    W = DictWeights(D)
    r, _ = req(D, 7)
    out = O.decode_step(W, D, r, 9)
    tr = out.layers[1]
    xn2 = [float(v) for v in O.rmsnorm(tr.x_mid, W.ffn_norm(1), D.rms_eps)]
    rl = [dot(W.t[("router", 1)][e], xn2) for e in range(D.n_experts)]
    sel = sorted(range(D.n_experts), key=lambda e: (-rl[e], e))[:D.top_k]
    z = sum(math.exp(rl[e]) for e in sel)
    x = [float(v) for v in tr.x_mid]
    for e in sel:
        y = _brute_expert(*W.t[("expert", 1, e)], xn2)
        x = [a + math.exp(rl[e]) / z * b for a, b in zip(x, y)]
    assert tr.experts == sel
    assert torch.allclose(tr.x_out, torch.tensor(x, dtype=F64), rtol=1e-11, atol=1e-12)


def test_greedy_ties_take_lower_index():
    over = {}
    for l in range(D.n_layers):
        over[("wo", l)] = torch.zeros(D.hidden, D.n_q_heads * D.head_dim, dtype=BF)
        for e in range(D.n_experts):
            wg, wu, _ = DictWeights(D).t[("expert", l, e)]
            over[("expert", l, e)] = (wg, wu, torch.zeros(D.hidden, D.expert_ffn, dtype=BF))
    lm = torch.zeros(D.vocab, D.hidden, dtype=BF)
    lm[7] = 1.0
    lm[3] = 1.0
    lm[20] = 0.5
    W = _const_embed_weights(lm_head=lm, over=over)
    r, _ = req(D, 4)
    out = O.decode_step(W, D, r, 1)
    assert float(out.logits[3]) == float(out.logits[7]) > float(out.logits[20])
    assert out.next_token == 3


def test_batch_is_independent_requests():
    W = DictWeights(D)
    a1, _ = req(D, 10, seed=1)
    b1, _ = req(D, 20, seed=2)
    a2, _ = req(D, 10, seed=1)
    b2, _ = req(D, 20, seed=2)
    ra = O.decode_step(W, D, a1, 4)
    O.decode_step(W, D, b1, 6)
    ra2 = O.decode_step(W, D, a2, 4)
    assert torch.equal(ra.logits, ra2.logits)


def _prior_scores_closed_form(q, K, pos, dims):
    """Scores of the rotated query against stored keys, written through the
    rotation angle instead of a rotated vector: for the rotate-half pair
    (i, i + d/2) with angle phi_i = pos * theta^(-2i/d),
      <R(phi) q, k> = sum_i (q_i k_i + q_j k_j) cos phi_i + (q_i k_j - q_j k_i) sin phi_i,
    j = i + d/2, scaled by 1/sqrt(d).  q [d] floats, K [T][d] floats."""
    d = len(q)
    half = d // 2
    out = []
    for k in K:
        s = 0.0
        for i in range(half):
            j = i + half
            phi = pos * dims.rope_theta ** (-2.0 * i / d)
            s += (q[i] * k[i] + q[j] * k[j]) * math.cos(phi) + (q[i] * k[j] - q[j] * k[i]) * math.sin(phi)
        out.append(s / math.sqrt(d))
    return out


def _x_mid_from_scores(W, x, data, T, scores_of, dims):
    """x + Wo o with o_h = sum_t p_t V_t over the T prior tokens and a new
    token whose key and value are zero (score 0, value 0)."""
    G, d = dims.group, dims.head_dim
    K0, V0 = data[0]
    o = []
    for h in range(dims.n_q_heads):
        g = h // G
        s = scores_of(h, [[float(v) for v in K0[t, g]] for t in range(T)])
        z = 1.0 + sum(math.exp(v) for v in s)              # the new token adds exp(0)
        for i in range(d):
            o.append(sum(math.exp(s[t]) * float(V0[t, g, i]) for t in range(T)) / z)
    return [x[r] + dot(W.t[("wo", 0)][r], o) for r in range(dims.hidden)]


def test_query_is_rotated_at_the_decode_position():
    # Non-zero Wq with Wk = Wv = 0: the new token scores 0 and carries a zero
    # value, so the layer-0 output depends on the query only through its
    # scores against the stored prior keys.  Those follow the closed form in
    # cos/sin of the decode position; an unrotated query, a query rotated one
    # position off, or the opposite rotation direction each give a different
    # x_mid (phi is linear in the position, so the opposite direction is
    # position -T), checked below so the pin cannot pass vacuously.
    zeros_k = torch.zeros(D.n_kv_heads * D.head_dim, D.hidden, dtype=BF)
    for T in (5, 11):
        over = {}
        for l in range(D.n_layers):
            over[("wk", l)] = zeros_k
            over[("wv", l)] = zeros_k
        W = DictWeights(D, seed=4, over=over)
        r, data = req(D, T, seed=12)
        tok = 6
        out = O.decode_step(W, D, r, tok)
        x = [float(v) for v in W.t["embed"][tok]]
        ms = sum(v * v for v in x) / len(x)
        xn = [v / math.sqrt(ms + D.rms_eps) * float(gm) for v, gm in zip(x, W.t[("attn_norm", 0)])]
        d = D.head_dim
        q = [dot(W.t[("wq", 0)][i], xn) for i in range(D.n_q_heads * d)]

        def at(pos):
            return lambda h, K: _prior_scores_closed_form(q[h * d:(h + 1) * d], K, pos, D)

        want = _x_mid_from_scores(W, x, data, T, at(T), D)
        got = out.layers[0].x_mid
        assert torch.allclose(got, torch.tensor(want, dtype=F64), rtol=1e-10, atol=1e-12)
        # the wrong readings are far away
        for wrong_pos in (0, T - 1, T + 1, -T):
            wrong = _x_mid_from_scores(W, x, data, T, at(wrong_pos), D)
            assert float((got - torch.tensor(wrong, dtype=F64)).abs().max()) > 1e-3
