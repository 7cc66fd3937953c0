"""Shared GPU-vs-oracle machinery for the parity tests.

The GPU runs free; the oracle replays each step from the same input token
with its own KV cache.  Integer outputs must match exactly, except inside a
near-tie: an expert-set difference is excused when every swapped expert's
oracle logit is within 1e-3 of the oracle's k-th logit, and a greedy token
difference is excused when the oracle's logit of the GPU token is within 1e-3
of the maximum.  After an excused difference the oracle adopts the GPU's
choice (gates from its own softmax), so both trajectories stay aligned.
Unexcused mismatches must be zero.  Floating point: logits relative L2 <= 1e-2
and max-abs <= 5e-2; per-layer hidden states relative L2 <= 1e-2.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

import synth
from synth.device import DeviceModel, PagedKV, initial_tokens, kv_pages_needed

NEAR_TIE = 1e-3
NUCLEUS_MASS_TOL = 2e-3   # nucleus cut: mass tolerance between float32 (GPU) and float64 (oracle) masses
LOGIT_REL_L2 = 1e-2
LOGIT_MAX_ABS = 5e-2
HIDDEN_REL_L2 = 1e-2


def rel_l2(a: torch.Tensor, b: torch.Tensor) -> float:
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm().clamp_min(1e-30))


@dataclass
class StepRecord:
    tok_in: torch.Tensor          # [B] int
    next_tok: torch.Tensor        # [B]
    logits: Optional[torch.Tensor]  # [B, V] float32
    hidden: torch.Tensor          # [B, L, H]
    ids: torch.Tensor             # [B, L, k]
    rlog: torch.Tensor            # [B, L, E]
    rids: List[int]


class GpuRun:
    """A workload's model, paged cache and plan on cuda:0."""

    def __init__(self, wl: synth.Workload, steps: Optional[int] = None, model: Optional[DeviceModel] = None,
                 rids: Optional[List[int]] = None, perm_salt: int = 0, poison: bool = False,
                 extra_requests: int = 0, extra_ctx: int = 0, **plan_kw):
        from persistent_moe_decode_02_gb300 import mk
        D = wl.dims
        self.wl, self.D = wl, D
        self.steps = wl.steps if steps is None else steps
        self.model = model if model is not None else DeviceModel(D, wl.seed)
        ps = D.page_size
        max_pages = max((c + self.steps + 1 + ps - 1) // ps for c in wl.ctx + [extra_ctx]) + 1
        num_pages = kv_pages_needed(D, wl.ctx, self.steps, extra_requests, extra_ctx) + 4
        self.kv = PagedKV(D, num_pages, max_pages, wl.seed, perm_salt=perm_salt, poison=poison)
        rids = list(range(wl.batch)) if rids is None else rids
        self.reqs = [self.kv.admit(rid, c, self.steps + 1) for rid, c in zip(rids, wl.ctx)]
        self.next_rid = max(rids) + 1
        self.max_pages = max_pages
        self.plan = mk.Plan(D, self.model.weights(), self.kv.kv, [r.length for r in self.reqs],
                            self.kv.page_table(self.reqs), max_pages, **plan_kw)
        self.tokens = torch.tensor(initial_tokens(wl, [r.rid for r in self.reqs]), dtype=torch.int32,
                                   device="cuda")

    def step(self, capture: bool = True, logits: bool = True) -> StepRecord:
        from persistent_moe_decode_02_gb300 import mk
        D, B = self.D, len(self.reqs)
        tok_in = self.tokens.clone()
        lg = torch.empty(B, D.vocab, dtype=torch.float32, device="cuda") if logits else None
        nxt = torch.empty(B, dtype=torch.int32, device="cuda")
        rc = self.plan.step(self.tokens, nxt, lg)
        assert rc == 0, mk.status_string(rc)
        rec = None
        if capture:
            hid = torch.empty(B, D.n_layers, D.hidden, dtype=torch.float32, device="cuda")
            ids = torch.empty(B, D.n_layers, D.top_k, dtype=torch.int32, device="cuda")
            rl = torch.empty(B, D.n_layers, D.n_experts, dtype=torch.float32, device="cuda")
            self.plan.read_debug(mk.MK_DBG_HIDDEN, hid)
            self.plan.read_debug(mk.MK_DBG_EXPERT_IDS, ids)
            self.plan.read_debug(mk.MK_DBG_ROUTER_LOGITS, rl)
        st = self.plan.sync()
        assert st == 0, f"device status {st}: {mk.status_string(st)} {mk.lib().mk_last_error().decode()}"
        if capture:
            rec = StepRecord(tok_in.cpu(), nxt.cpu(), lg.cpu() if lg is not None else None, hid.cpu(),
                             ids.cpu().long(), rl.cpu(), [r.rid for r in self.reqs])
        for r in self.reqs:
            r.length += 1
        self.tokens = nxt
        return rec

    def churn(self, leave: int, join: int, join_ctx: int) -> list:
        """Continuous batching: the `leave` oldest requests finish, `join` new
        ones (fresh request ids) join at `join_ctx` cached tokens, and the plan
        is updated.  Returns the new requests."""
        for r in self.reqs[:leave]:
            self.kv.release(r)
        keep_tok = self.tokens[leave:]
        self.reqs = self.reqs[leave:]
        new = [self.kv.admit(self.next_rid + i, join_ctx, self.steps + 1) for i in range(join)]
        self.next_rid += join
        self.reqs += new
        new_tok = torch.tensor(initial_tokens(self.wl, [r.rid for r in new]), dtype=torch.int32, device="cuda")
        self.tokens = torch.cat([keep_tok, new_tok])
        self.plan.update([r.length for r in self.reqs], self.kv.page_table(self.reqs), self.max_pages)
        return new


@dataclass
class Report:
    steps: int = 0
    layers_checked: int = 0
    expert_excused: int = 0
    expert_unexcused: int = 0
    token_excused: int = 0
    token_unexcused: int = 0
    max_hidden_rel: float = 0.0
    max_logit_rel: float = 0.0
    max_logit_abs: float = 0.0
    notes: List[str] = field(default_factory=list)

    def assert_ok(self):
        assert self.expert_unexcused == 0 and self.token_unexcused == 0, self
        assert self.max_hidden_rel <= HIDDEN_REL_L2, self
        assert self.max_logit_rel <= LOGIT_REL_L2 and self.max_logit_abs <= LOGIT_MAX_ABS, self


def make_prior(D, seed, cache: bool):
    store: Dict = {}

    def prior(rid, l, n):
        key = (rid, l, n)
        if cache and key in store:
            return store[key]
        kv = synth.prior_kv(D, seed, rid, l, n)
        if cache:
            store[key] = kv
        return kv
    return prior


class OracleReplay:
    """Replays GPU steps for one request in the float64 oracle."""

    def __init__(self, wl: synth.Workload, rid: int, prior_len: int, W=None, cache_prior: bool = True,
                 n_layers: Optional[int] = None):
        from oracle import decode as O
        self.O = O
        self.D = wl.dims
        self.W = W if W is not None else synth.SynthWeights(self.D, wl.seed)
        self.L = self.D.n_layers if n_layers is None else n_layers
        self.req = O.OracleRequest(rid, prior_len, make_prior(self.D, wl.seed, cache_prior), self.D.n_layers)

    def step(self, rec: StepRecord, b: int, rep: Report, sampling: Optional[tuple] = None) -> None:
        """sampling = (temperature, seed, batch slot[, top_p]): the expected
        token is the oracle's temperature draw (oracle/sample.py), over the
        nucleus when top_p < 1, instead of the greedy one.  A difference is
        excused when the GPU token's oracle key is within NEAR_TIE of the
        largest key, or (top_p < 1) when it is the draw over a nucleus whose
        mass is within NUCLEUS_MASS_TOL of top_p."""
        O, D = self.O, self.D
        pos = self.req.length
        x = O.widen(self.W.embed_rows([int(rec.tok_in[b])])[0])
        for l in range(self.L):
            x_mid = O.attention_block(self.W, D, l, x, self.req, pos)
            x_out, tr = O.moe_block(self.W, D, l, x_mid)
            gpu_ids = [int(e) for e in rec.ids[b, l]]
            if set(gpu_ids) != set(tr.experts):
                r = tr.router_logits
                kth = float(torch.sort(r, descending=True).values[D.top_k - 1])
                swapped = set(gpu_ids) ^ set(tr.experts)
                if all(abs(float(r[e]) - kth) <= NEAR_TIE for e in swapped):
                    rep.expert_excused += 1
                else:
                    rep.expert_unexcused += 1
                    rep.notes.append(f"layer {l} pos {pos}: gpu {sorted(gpu_ids)} oracle {sorted(tr.experts)}")
                x_out, tr = O.moe_block(self.W, D, l, x_mid, force=gpu_ids)
            rep.max_hidden_rel = max(rep.max_hidden_rel, rel_l2(rec.hidden[b, l], x_out))
            rep.layers_checked += 1
            x = x_out
        if self.L < D.n_layers:
            # layers past L are not replayed: keep the appended-KV bookkeeping consistent
            for l in range(self.L, D.n_layers):
                self.req.appended_k[l].append(torch.zeros(D.n_kv_heads, D.head_dim, dtype=torch.float64))
                self.req.appended_v[l].append(torch.zeros(D.n_kv_heads, D.head_dim, dtype=torch.float64))
            rep.steps += 1
            return
        logits, nxt = O.lm_head(self.W, D, x)
        if rec.logits is not None:
            g = rec.logits[b].double()
            rep.max_logit_rel = max(rep.max_logit_rel, rel_l2(g, logits))
            rep.max_logit_abs = max(rep.max_logit_abs, float((g - logits).abs().max()))
        gt = int(rec.next_tok[b])
        score = logits
        allowed = None
        if sampling is not None:
            from oracle import sample as OS
            T, seed, slot = sampling[:3]
            top_p = sampling[3] if len(sampling) > 3 else 1.0
            score = OS.sample_keys(logits, T, seed, slot, pos)
            nxt = OS.sample_token(logits, T, seed, slot, pos, top_p=top_p)
            if top_p < 1.0:
                # the draw is over the nucleus; its cut depends on masses the
                # two sides compute in different precisions, so every cut
                # whose mass lies within NUCLEUS_MASS_TOL of top_p is allowed
                lo = OS.nucleus(logits, T, max(top_p - NUCLEUS_MASS_TOL, 1e-12)).shape[0]
                order = OS.nucleus(logits, T, min(top_p + NUCLEUS_MASS_TOL, 1.0)).tolist()
                keys32 = score.to(torch.float32)
                allowed = set()
                for n in range(lo, len(order) + 1):
                    sub = keys32[order[:n]]
                    best = float(sub.max())
                    allowed.add(min(v for v, k in zip(order[:n], sub.tolist()) if k == best))
                score = torch.full_like(score, -math.inf)
                score[order] = OS.sample_keys(logits, T, seed, slot, pos)[order]
        if gt != nxt:
            if allowed is not None and gt in allowed:
                rep.token_excused += 1
            elif float(score[gt]) >= float(score.max()) - NEAR_TIE:
                rep.token_excused += 1
            else:
                rep.token_unexcused += 1
                rep.notes.append(f"pos {pos}: gpu token {gt} oracle {nxt}")
        rep.steps += 1


def run_and_check(wl: synth.Workload, steps: int, oracle_steps: Optional[int] = None,
                  requests: Optional[List[int]] = None, n_layers: Optional[int] = None,
                  cache_prior: bool = True, poison: bool = False, **plan_kw) -> Report:
    """Run `steps` GPU steps, replay the first `oracle_steps` of the chosen
    requests in the oracle; returns the report (not yet asserted)."""
    run = GpuRun(wl, steps=steps, poison=poison, **plan_kw)
    oracle_steps = steps if oracle_steps is None else oracle_steps
    recs = [run.step(capture=(s < oracle_steps)) for s in range(steps)]
    requests = list(range(wl.batch)) if requests is None else requests
    rep = Report()
    W = synth.SynthWeights(wl.dims, wl.seed)
    for b in requests:
        rr = OracleReplay(wl, run.reqs[b].rid, wl.ctx[b], W=W, cache_prior=cache_prior, n_layers=n_layers)
        for s in range(oracle_steps):
            rr.step(recs[s], b, rep)
    run.plan.close()
    return rep


def run_churn_and_check(wl: synth.Workload, capacity: int, steps: int, leave: int, join: int, join_ctx: int,
                        sample: Optional[List[int]] = None, n_layers: Optional[int] = None,
                        cache_prior: bool = True, **plan_kw) -> Report:
    """Run `steps` GPU steps with `leave` requests finishing and `join` joining
    after each step (batch capacity `capacity`), then replay every request
    (or the request ids in `sample`) in the oracle over the steps it took part in."""
    run = GpuRun(wl, steps=steps, max_batch=capacity, extra_requests=join * steps, extra_ctx=join_ctx, **plan_kw)
    prior = {r.rid: r.prior_len for r in run.reqs}
    recs = []
    for s in range(steps):
        recs.append(run.step())
        if s + 1 < steps:
            for r in run.churn(leave, join, join_ctx):
                prior[r.rid] = join_ctx
    rep = Report()
    W = synth.SynthWeights(wl.dims, wl.seed)
    for rid in (sorted(prior) if sample is None else sample):
        rr = OracleReplay(wl, rid, prior[rid], W=W, cache_prior=cache_prior, n_layers=n_layers)
        for rec in recs:
            if rid in rec.rids:
                rr.step(rec, rec.rids.index(rid), rep)
    run.plan.close()
    return rep
