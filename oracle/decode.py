"""Plain float64 CPU decode step (test infrastructure only; see package doc).

Readings of the pages taken here (the pages name the ops but print no
formulas; each reading is the plainest one the rest supports):
  * pre-norm residual decoder: x += Attn(rmsnorm(x)); x += MoE(rmsnorm(x));
    logits = W_lm rmsnorm(x) with a final gain; no biases, no QK-norm, no
    shared expert, untied embedding;
  * RMSNorm: x / sqrt(mean(x^2) + eps) * gamma;
  * RoPE: rotate-half pairs (i, i + d/2), inv_freq_i = theta^(-2i/d), applied
    to the new token's q and k at position = tokens already cached;
    prior cached K is taken as already rotated;
  * GQA: query head h reads KV head h // (n_q_heads / n_kv_heads);
  * attention over the cached tokens plus the new one (bf16-rounded K/V),
    scores scaled by 1/sqrt(head_dim), exact softmax;
  * router: softmax over all experts, top-k by logit (ties -> lower index),
    gates renormalised over the selected k;
  * expert: SwiGLU, h = silu(W_gate xn) * (W_up xn), y = W_down h;
    x += sum_j gate_j * y_j in rank order j = 0..k-1;
  * greedy next token = argmax of the logits, lowest index on ties.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Callable, Dict, List, Optional, Sequence

import torch

F64 = torch.float64


def widen(w: torch.Tensor) -> torch.Tensor:
    """bf16 (or any float) tensor -> float64, exact for bf16."""
    return w.to(F64)


def bf16_rne(x: torch.Tensor) -> torch.Tensor:
    """Round float64 values to the nearest bfloat16 (8 significant bits),
    ties to even, returned as float64.  Valid for normal-range values."""
    m, e = torch.frexp(x)                       # x = m * 2^e, 0.5 <= |m| < 1
    r = torch.round(m * 256.0)                  # torch.round: half to even
    return torch.ldexp(r, (e - 8).to(F64))


def rmsnorm(x: torch.Tensor, gamma: torch.Tensor, eps: float) -> torch.Tensor:
    return x / torch.sqrt((x * x).mean() + eps) * widen(gamma)


def rope(v: torch.Tensor, pos: int, theta: float) -> torch.Tensor:
    """Rotate rows of v [n, d] to position pos (rotate-half convention)."""
    d = v.shape[-1]
    half = d // 2
    i = torch.arange(half, dtype=F64)
    inv_freq = theta ** (-2.0 * i / d)
    ang = float(pos) * inv_freq
    c, s = torch.cos(ang), torch.sin(ang)
    a, b = v[..., :half], v[..., half:]
    return torch.cat([a * c - b * s, b * c + a * s], dim=-1)


def gqa_attention(q: torch.Tensor, K: torch.Tensor, V: torch.Tensor) -> torch.Tensor:
    """Decode attention of one token.  q [nq, d]; K, V [T, nkv, d] -> o [nq, d]."""
    nq, d = q.shape
    nkv = K.shape[1]
    G = nq // nkv
    o = torch.empty(nq, d, dtype=F64)
    for g in range(nkv):
        Kg, Vg = widen(K[:, g, :]), widen(V[:, g, :])
        qg = q[g * G:(g + 1) * G]                       # [G, d]
        s = (Kg @ qg.T) / math.sqrt(d)                   # [T, G]
        s = s - s.max(dim=0, keepdim=True).values
        p = torch.exp(s)
        p = p / p.sum(dim=0, keepdim=True)
        o[g * G:(g + 1) * G] = p.T @ Vg
    return o


def route(r: torch.Tensor, k: int, force: Optional[Sequence[int]] = None):
    """Top-k MoE routing.  r [E] float64 logits.

    Returns (ids in rank order, gates float64 [k], P = softmax(r)).  The
    selection is made on float32-rounded logits (the kernel's precision),
    descending, ties to the lower expert index.  ``force`` replaces the
    selection (used when a GPU choice inside a near-tie is adopted); gates
    always come from this function's own softmax."""
    P = torch.exp(r - r.max())
    P = P / P.sum()
    if force is None:
        r32 = r.to(torch.float32)
        order = torch.sort(r32, descending=True, stable=True).indices
        ids = [int(i) for i in order[:k]]
    else:
        ids = [int(i) for i in force]
    sel = P[ids]
    return ids, sel / sel.sum(), P


def silu(z: torch.Tensor) -> torch.Tensor:
    return z / (1.0 + torch.exp(-z))


def expert_ffn(xn, wg, wu, wd) -> torch.Tensor:
    h = silu(widen(wg) @ xn) * (widen(wu) @ xn)
    return widen(wd) @ h


# Prior-KV source: (rid, layer, n_tok) -> (K, V), each bf16 [n_tok, nkv, d].
PriorFn = Callable[[int, int, int], tuple]


@dataclass
class OracleRequest:
    """One request's decode state: prior context length plus the K/V rows the
    oracle itself appended (bf16 values held as float64), per layer."""
    rid: int
    prior_len: int
    prior: PriorFn
    n_layers: int
    appended_k: List[List[torch.Tensor]] = field(default_factory=list)
    appended_v: List[List[torch.Tensor]] = field(default_factory=list)

    def __post_init__(self):
        if not self.appended_k:
            self.appended_k = [[] for _ in range(self.n_layers)]
            self.appended_v = [[] for _ in range(self.n_layers)]

    @property
    def length(self) -> int:
        return self.prior_len + len(self.appended_k[0])

    def cache(self, layer: int):
        K0, V0 = self.prior(self.rid, layer, self.prior_len)
        K = widen(K0)
        V = widen(V0)
        if self.appended_k[layer]:
            K = torch.cat([K, torch.stack(self.appended_k[layer])])
            V = torch.cat([V, torch.stack(self.appended_v[layer])])
        return K, V


@dataclass
class LayerTrace:
    router_logits: torch.Tensor      # [E] float64
    experts: List[int]               # rank order
    gates: torch.Tensor              # [k] float64
    x_mid: torch.Tensor              # hidden after the attention residual
    x_out: torch.Tensor              # hidden after the MoE residual


@dataclass
class StepResult:
    logits: torch.Tensor             # [V] float64
    next_token: int
    layers: List[LayerTrace]

    @property
    def hidden(self) -> torch.Tensor:
        return torch.stack([t.x_out for t in self.layers])


def attention_block(W, dims, l: int, x: torch.Tensor, req: OracleRequest, pos: int) -> torch.Tensor:
    """x + Wo * Attn(rmsnorm(x)) for one request; appends this token's K/V."""
    nq, nkv, d = dims.n_q_heads, dims.n_kv_heads, dims.head_dim
    xn = rmsnorm(x, W.attn_norm(l), dims.rms_eps)
    q = (widen(W.wq(l)) @ xn).view(nq, d)
    k = (widen(W.wk(l)) @ xn).view(nkv, d)
    v = (widen(W.wv(l)) @ xn).view(nkv, d)
    q = rope(q, pos, dims.rope_theta)
    k = rope(k, pos, dims.rope_theta)
    K, V = req.cache(l)
    assert K.shape[0] == pos
    k_b, v_b = bf16_rne(k), bf16_rne(v)
    req.appended_k[l].append(k_b)
    req.appended_v[l].append(v_b)
    K = torch.cat([K, k_b[None]])
    V = torch.cat([V, v_b[None]])
    o = gqa_attention(q, K, V).reshape(nq * d)
    return x + widen(W.wo(l)) @ o


def moe_block(W, dims, l: int, x_mid: torch.Tensor, force: Optional[Sequence[int]] = None):
    """x_mid + sum_j gate_j * expert_j(rmsnorm(x_mid)); no side effects."""
    xn2 = rmsnorm(x_mid, W.ffn_norm(l), dims.rms_eps)
    r = widen(W.router(l)) @ xn2
    ids, gates, _ = route(r, dims.top_k, force)
    x_out = x_mid.clone()
    for j, e in enumerate(ids):
        wg, wu, wd = W.expert(l, e)
        x_out = x_out + gates[j] * expert_ffn(xn2, wg, wu, wd)
    return x_out, LayerTrace(r, ids, gates, x_mid, x_out)


def decode_layer(W, dims, l: int, x: torch.Tensor, req: OracleRequest, pos: int,
                 force: Optional[Sequence[int]] = None):
    """One transformer layer for one request; appends this token's K/V."""
    x_mid = attention_block(W, dims, l, x, req, pos)
    return moe_block(W, dims, l, x_mid, force)


def lm_head(W, dims, x: torch.Tensor):
    """Final RMSNorm, LM head and greedy argmax (float32 decision, lowest index on ties)."""
    xf = rmsnorm(x, W.final_norm(), dims.rms_eps)
    Wl = W.lm_head()
    logits = torch.cat([widen(Wl[i:i + 16384]) @ xf for i in range(0, Wl.shape[0], 16384)])
    nxt = int(torch.argmax(logits.to(torch.float32)))   # first index among equal maxima
    return logits, nxt


def decode_step(W, dims, req: OracleRequest, token: int,
                force: Optional[Dict[int, Sequence[int]]] = None) -> StepResult:
    """Decode one token for one request at position req.length."""
    pos = req.length
    x = widen(W.embed_rows([token])[0])
    traces = []
    for l in range(dims.n_layers):
        x, tr = decode_layer(W, dims, l, x, req, pos, None if force is None else force.get(l))
        traces.append(tr)
    logits, nxt = lm_head(W, dims, x)
    return StepResult(logits, nxt, traces)
