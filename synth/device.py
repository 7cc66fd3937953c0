"""Seeded synthetic model and paged KV cache placed on a CUDA device in the
layout the megakernel's C ABI takes (include/mk.h).

The values are the same generator streams ``SynthWeights`` reads on the
host; only their placement differs (grouped QKV rows, gate/up rows stacked
per expert, K/V scattered into shuffled pages).  Nothing here computes any
part of the decode step.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List

import numpy as np
import torch

from . import (KV_SIGMA, Dims, Workload, fill_kv_paged_, fill_normal_, first_token, kv_name, normal,
               page_permutation, wname)


class DeviceModel:
    """bf16 weights on `device`, per include/mk.h.

    wqkv[l] rows are grouped per KV head g: the G query heads of group g,
    then key head g, then value head g (rows taken from the logical wq, wk,
    wv streams).  w_gate_up[l][e] interleaves the gate and up rows: row 2f is
    gate row f, row 2f + 1 is up row f."""

    def __init__(self, D: Dims, seed: int = 0, device: str = "cuda"):
        self.D, self.seed = D, seed
        H, G, d, nkv = D.hidden, D.group, D.head_dim, D.n_kv_heads
        E, F, V, L = D.n_experts, D.expert_ffn, D.vocab, D.n_layers
        dev = device
        self.embed = normal((V, H), seed, "embed", device=dev)
        self.final_norm = normal((H,), seed, "final_norm", mean=1.0, device=dev)
        self.lm_head = normal((V, H), seed, "lm_head", device=dev)
        self.attn_norm, self.wqkv, self.wo, self.ffn_norm = [], [], [], []
        self.router, self.w_gate_up, self.w_down = [], [], []
        Rg = (G + 2) * d
        for l in range(L):
            self.attn_norm.append(normal((H,), seed, wname("attn_norm", l), mean=1.0, device=dev))
            w = torch.empty(nkv * Rg, H, dtype=torch.bfloat16, device=dev)
            for g in range(nkv):
                fill_normal_(w[g * Rg: g * Rg + G * d], seed, wname("wq", l), start=g * G * d * H)
                fill_normal_(w[g * Rg + G * d: g * Rg + (G + 1) * d], seed, wname("wk", l), start=g * d * H)
                fill_normal_(w[g * Rg + (G + 1) * d: (g + 1) * Rg], seed, wname("wv", l), start=g * d * H)
            self.wqkv.append(w)
            self.wo.append(normal((H, D.n_q_heads * d), seed, wname("wo", l), device=dev))
            self.ffn_norm.append(normal((H,), seed, wname("ffn_norm", l), mean=1.0, device=dev))
            # router stored transposed, [H, E] (values keyed by the logical [E, H] index)
            self.router.append(normal((E, H), seed, wname("router", l), device=dev).t().contiguous())
            gu = torch.empty(E, F, 2, H, dtype=torch.bfloat16, device=dev)
            tmp = torch.empty(F, H, dtype=torch.bfloat16, device=dev)
            for e in range(E):
                gu[e, :, 0].copy_(fill_normal_(tmp, seed, wname("gate", l), start=e * F * H))
                gu[e, :, 1].copy_(fill_normal_(tmp, seed, wname("up", l), start=e * F * H))
            self.w_gate_up.append(gu.view(E, 2 * F, H))
            # down projection stored transposed per expert, [E, F, H]: row f holds
            # the H output coefficients of ffn unit f (values keyed by the logical
            # [E, H, F] index, so the oracle's view is unchanged)
            wd = torch.empty(E, F, H, dtype=torch.bfloat16, device=dev)
            tmpd = torch.empty(H, F, dtype=torch.bfloat16, device=dev)
            for e in range(E):
                wd[e].copy_(fill_normal_(tmpd, seed, wname("down", l), start=e * H * F).t())
            self.w_down.append(wd)

    def weights(self) -> dict:
        return {"embed": self.embed, "final_norm": self.final_norm, "lm_head": self.lm_head,
                "attn_norm": self.attn_norm, "wqkv": self.wqkv, "wo": self.wo, "ffn_norm": self.ffn_norm,
                "router": self.router, "w_gate_up": self.w_gate_up, "w_down": self.w_down}

    def nbytes(self) -> int:
        ts = [self.embed, self.final_norm, self.lm_head]
        for k in ("attn_norm", "wqkv", "wo", "ffn_norm", "router", "w_gate_up", "w_down"):
            ts += getattr(self, k)
        return sum(t.numel() * t.element_size() for t in ts)


@dataclass
class Request:
    rid: int            # logical request id (keys its synthetic prior KV and first token)
    prior_len: int      # synthetic tokens cached before the first decode step
    length: int         # tokens cached now
    pages: List[int]    # physical pages, in position order


class PagedKV:
    """Per-layer KV page pools plus the host-side page bookkeeping of a batch:
    which physical pages each request holds (seeded shuffled free list).  A
    pool is bf16 [num_pages, nkv, 2, head_dim, page_size] (per page and KV head
    the K block, then the V block); k[l] and v[l] are views of its two halves."""

    def __init__(self, D: Dims, num_pages: int, max_pages: int, seed: int = 0, device: str = "cuda",
                 perm_salt: int = 0, poison: bool = False):
        self.D, self.seed, self.max_pages, self.num_pages = D, seed, max_pages, num_pages
        shape = (num_pages, D.n_kv_heads, 2, D.head_dim, D.page_size)   # pages hold [d, slot] blocks
        self.kv = [torch.empty(shape, dtype=torch.bfloat16, device=device) for _ in range(D.n_layers)]
        self.k = [t[:, :, 0] for t in self.kv]
        self.v = [t[:, :, 1] for t in self.kv]
        if poison:   # NaN everywhere no token was written: unused slots must never matter
            for t in self.kv:
                t.fill_(float("nan"))
        self.free = [int(x) for x in page_permutation(num_pages, seed, perm_salt)]
        self._rng = np.random.Generator(np.random.PCG64([seed, 7]))
        self.device = device

    def admit(self, rid: int, prior_len: int, reserve_tokens: int) -> Request:
        """Give a request pages for prior_len + reserve_tokens positions and
        write its synthetic prior K/V into them."""
        need = (prior_len + reserve_tokens + self.D.page_size - 1) // self.D.page_size
        if need > self.max_pages or need > len(self.free):
            raise RuntimeError("out of KV pages")
        pages = [self.free.pop() for _ in range(need)]
        pt = torch.tensor(pages, dtype=torch.int32, device=self.device)
        for l in range(self.D.n_layers):
            fill_kv_paged_(self.k[l], pt, prior_len, self.seed, kv_name(rid, l, "K"))
            fill_kv_paged_(self.v[l], pt, prior_len, self.seed, kv_name(rid, l, "V"))
        return Request(rid, prior_len, prior_len, pages)

    def release(self, req: Request) -> None:
        self.free.extend(req.pages)
        self._rng.shuffle(self.free)

    def page_table(self, reqs: List[Request]) -> List[int]:
        out = []
        for r in reqs:
            row = r.pages + [-1] * (self.max_pages - len(r.pages))
            out += row
        return out


def kv_pages_needed(D: Dims, ctx: List[int], steps: int, extra_requests: int = 0, extra_ctx: int = 0) -> int:
    ps = D.page_size
    n = sum((c + steps + ps) // ps + 1 for c in ctx)
    n += extra_requests * ((extra_ctx + steps + ps) // ps + 1)
    return n


def initial_tokens(w: Workload, rids: List[int]) -> List[int]:
    return [first_token(w.dims, w.seed, r) for r in rids]
