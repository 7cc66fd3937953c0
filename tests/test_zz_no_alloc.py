"""mk_decode_step_noalloc, the entry point for callers that cannot allocate
device memory when they decode (hosts that keep all device memory in their own
pool and forbid raw cudaMalloc inside their enqueue callbacks, allocator hooks
that would recurse, loops that cannot take cudaMalloc's implicit
synchronisation).  Its scratch is a fixed static device array inside libmk.so.

The test runs two decode steps in a row through it and through the plan-based
mk_decode_step on identical inputs and caches, and requires the same greedy
tokens and logits within the parity tolerances.  This file sorts last so a
stop-at-first-failure run has executed every other test before it."""
import dataclasses

import pytest
import torch

import synth
from synth.device import DeviceModel, PagedKV, initial_tokens, kv_pages_needed
from tests.gpu_util import LOGIT_MAX_ABS, LOGIT_REL_L2, rel_l2

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("ctx", [[128, 45], [300, 17, 160]])
def test_noalloc_matches_plan_step_on_two_calls(built, ctx):
    # batch 2, and batch 3 whose contexts split into several KV chunks per
    # (request, group) with a combine each (the plan runs batch 3 on the batch-8
    # instance's tensor cores, the no-alloc step on the batch-4 instance's CUDA
    # cores: the same tokens, logits within the parity tolerances)
    from persistent_moe_decode_02_gb300 import mk
    wl = dataclasses.replace(synth.workload("tiny"), ctx=ctx, steps=2)
    D = wl.dims
    model = DeviceModel(D, wl.seed)
    max_pages = max((c + 3 + D.page_size) // D.page_size for c in wl.ctx) + 1
    num_pages = kv_pages_needed(D, wl.ctx, 3) + 4

    def cache():
        kv = PagedKV(D, num_pages, max_pages, wl.seed)
        return kv, [kv.admit(b, c, 3) for b, c in enumerate(wl.ctx)]

    kv_a, reqs_a = cache()
    kv_b, reqs_b = cache()
    assert [r.pages for r in reqs_a] == [r.pages for r in reqs_b]
    pt = kv_a.page_table(reqs_a)
    lens = [r.length for r in reqs_a]
    plan = mk.Plan(D, model.weights(), kv_a.kv, lens, pt, max_pages)
    tok_a = torch.tensor(initial_tokens(wl, list(range(wl.batch))), dtype=torch.int32, device="cuda")
    tok_b = tok_a.clone()
    B = wl.batch
    for step in range(2):
        nxt_a = torch.empty(B, dtype=torch.int32, device="cuda")
        nxt_b = torch.empty(B, dtype=torch.int32, device="cuda")
        lg_a = torch.empty(B, D.vocab, device="cuda")
        lg_b = torch.empty(B, D.vocab, device="cuda")
        status = torch.full((4,), -99, dtype=torch.int32, device="cuda")
        assert plan.step(tok_a, nxt_a, lg_a) == mk.MK_OK
        assert plan.sync() == mk.MK_OK
        rc = mk.decode_step_noalloc(D, model.weights(), kv_b.kv, lens, pt, max_pages, tok_b, nxt_b,
                                    lg_b, status)
        assert rc == mk.MK_OK, mk.lib().mk_last_error()
        torch.cuda.synchronize()
        assert int(status[0]) == mk.MK_OK
        assert torch.equal(nxt_a, nxt_b), step
        assert rel_l2(lg_b.cpu(), lg_a.cpu().double()) <= LOGIT_REL_L2
        assert float((lg_b - lg_a).abs().max()) <= LOGIT_MAX_ABS
        lens = [n + 1 for n in lens]
        tok_a, tok_b = nxt_a, nxt_b
    plan.close()


def test_noalloc_rejects_oversized_step(built):
    # a context whose per-layer buffers exceed the static array is refused
    # with MK_ERR_CAPACITY before anything is enqueued
    from persistent_moe_decode_02_gb300 import mk
    D = synth.MID
    model_like = {"embed": torch.zeros(8, device="cuda"), "final_norm": torch.zeros(8, device="cuda"),
                  "lm_head": torch.zeros(8, device="cuda")}
    for k in ("attn_norm", "wqkv", "wo", "ffn_norm", "router", "w_gate_up", "w_down"):
        model_like[k] = [torch.zeros(8, device="cuda")] * D.n_layers
    # only the pool's page count is read before the refusal: a 65,536-page stand-in
    pools = [torch.zeros(1 << 16, 8, dtype=torch.bfloat16, device="cuda")]
    ctx = 600000
    pages = (ctx + D.page_size) // D.page_size
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = mk.decode_step_noalloc(D, model_like, pools * D.n_layers, [ctx], list(range(pages)), pages, tok, tok)
    assert rc == mk.MK_ERR_CAPACITY
    msg = mk.lib().mk_last_error().decode()
    assert "bytes of scratch" in msg and str(64 << 20) in msg, msg
