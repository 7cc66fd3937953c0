"""Host-only tests of the continuous-batching scheduler (mk_sched_*, no GPU).

The scheduler is driven with a fake model (the next token is a fixed function
of the request and its position) and compared step by step with a plain
Python restatement of the policy include/mk.h documents: pages reserved for
prompt + max_new - 1 positions at admission, first come first served with
head-of-line blocking, prompt tokens fed in order with their predictions
discarded except after the last one, retirement after max_new outputs or on
the end token, pages and slots freed at once, batch order kept.  With prefill
chunks a prompt may take several consecutive rows of a step: one row per
request first, then the spare rows to prompts in batch order, up to the chunk
size and the prompt's remaining tokens (above 8 rows a chunk ends at the next
multiple of 8)."""
import random

import pytest


@pytest.fixture(scope="module")
def mk():
    from persistent_moe_decode_02_gb300 import build, mk as m
    build.build()
    return m


def fake_next(rid: int, pos: int, vocab: int = 50) -> int:
    return (rid * 7919 + pos * 104729) % vocab


class PolicyModel:
    """The documented policy, restated independently of the C++."""

    def __init__(self, num_pages, ps, max_batch, max_pages, max_chunk=1):
        self.free, self.ps, self.max_batch, self.max_pages = num_pages, ps, max_batch, max_pages
        self.max_chunk = max_chunk
        self.queue, self.active, self.reqs = [], [], {}
        self.rows_of = []

    def submit(self, rid, prompt, max_new, eos):
        self.reqs[rid] = dict(prompt=list(prompt), max_new=max_new, eos=eos, out=[], len=0, done=False,
                              pages=-(-(len(prompt) + max_new - 1) // self.ps))
        self.queue.append(rid)

    def next(self):
        while self.queue and len(self.active) < self.max_batch and self.reqs[self.queue[0]]["pages"] <= self.free:
            rid = self.queue.pop(0)
            self.free -= self.reqs[rid]["pages"]
            self.active.append(rid)
        rows_of = [1] * len(self.active)
        spare = self.max_batch - len(self.active)
        for i, rid in enumerate(self.active):
            r = self.reqs[rid]
            extra = min(spare, min(self.max_chunk, len(r["prompt"]) - r["len"]) - 1)
            if extra > 0:
                rows_of[i] += extra
                spare -= extra
        batch, row = [], 0
        for i, rid in enumerate(self.active):
            if self.max_batch > 8:
                rows_of[i] = min(rows_of[i], 8 - row % 8)
            r = self.reqs[rid]
            for j in range(rows_of[i]):
                pos = r["len"] + j
                tok = r["prompt"][pos] if pos < len(r["prompt"]) else r["out"][-1]
                batch.append((rid, pos, tok))
                row += 1
        self.rows_of = rows_of
        return batch

    def commit(self, nxt):
        keep, row = [], 0
        for rid, n in zip(self.active, self.rows_of):
            r = self.reqs[rid]
            r["len"] += n
            row += n
            tok = nxt[row - 1]
            if r["len"] >= len(r["prompt"]):
                r["out"].append(tok)
                if len(r["out"]) >= r["max_new"] or (r["eos"] >= 0 and tok == r["eos"]):
                    r["done"] = True
            if r["done"]:
                self.free += r["pages"]
            else:
                keep.append(rid)
        self.active = keep


def drive(mk, num_pages, ps, max_batch, max_pages, requests, arrivals=None, max_steps=500, max_chunk=1):
    """Run scheduler and policy model side by side; returns the scheduler."""
    s = mk.Scheduler(num_pages, ps, max_batch, max_pages)
    if max_chunk > 1:
        s.set_prefill(max_chunk)
    ref = PolicyModel(num_pages, ps, max_batch, max_pages, max_chunk)
    arrivals = arrivals or {0: list(range(len(requests)))}
    step = 0
    prev = None
    prev_chunks = False
    while step < max_steps:
        for i in arrivals.get(step, []):
            rid, prompt, max_new, eos = requests[i]
            s.submit(rid, prompt, max_new, eos)
            ref.submit(rid, prompt, max_new, eos)
        b = s.next()
        want = ref.next()
        if b is None:
            assert want == []
            if step > max(arrivals):
                break
            step += 1
            continue
        assert list(zip(b["rids"], b["seq_lens"], b["tokens"])) == want
        chunks = max(ref.rows_of) > 1
        assert b["changed"] == (prev != b["rids"] or chunks or prev_chunks)
        prev, prev_chunks = b["rids"], chunks
        # chunk starts: each row points at the first row of its request
        first = {}
        for i, rid in enumerate(b["rids"]):
            first.setdefault(rid, i)
            assert b["chunk_first"][i] == first[rid]
            if max_batch > 8:
                assert first[rid] // 8 == i // 8          # a chunk stays inside one launch of 8 rows
        # page rows: a request's rows share its pages, distinct across requests
        rows = [b["page_table"][i * max_pages:(i + 1) * max_pages] for i in range(len(b["rids"]))]
        per_req = {}
        for rid, row in zip(b["rids"], rows):
            assert per_req.setdefault(rid, row) == row
        held = [p for row in per_req.values() for p in row if p >= 0]
        assert len(held) == len(set(held)) and all(0 <= p < num_pages for p in held)
        for rid, row in zip(b["rids"], rows):
            n = ref.reqs[rid]["pages"]
            assert all(p >= 0 for p in row[:n]) and all(p == -1 for p in row[n:])
        assert s.stats()["free_pages"] == ref.free
        nxt = [fake_next(rid, pos) for rid, pos, _ in want]
        before = s.stats()
        ahead = s.peek()                      # the prediction made while the step "runs"
        assert s.stats() == before            # peeking changes nothing
        s.commit(nxt)
        ref.commit(nxt)
        ends = any(r["eos"] >= 0 for r in ref.reqs.values())
        if not ends and step + 1 not in arrivals:
            # with no end token and no arrival the prediction is the next batch
            # (its rows and lengths: what the task list depends on; a decode
            # row's input token is unknown until the step ends)
            nb = s.peek()
            if ahead is None:
                assert nb is None
            else:
                for k in ("rids", "seq_lens", "page_table", "chunk_first"):
                    assert ahead[k] == nb[k], k
        step += 1
    for rid, r in ref.reqs.items():
        out, done = s.result(rid)
        assert (out, done) == (r["out"], r["done"]), rid
    return s, ref


def test_prompts_then_outputs_in_one_batch(mk):
    reqs = [(10, [1, 2, 3], 4, -1), (11, [5], 3, -1), (12, [7, 8, 9, 10, 11, 12], 2, -1)]
    s, ref = drive(mk, 64, 16, 4, 8, reqs)
    for rid, prompt, max_new, _ in reqs:
        out, done = s.result(rid)
        assert done and len(out) == max_new
        # the first output is the prediction after the last prompt token, then each output feeds the next step
        assert out[0] == fake_next(rid, len(prompt) - 1)
        assert all(out[i + 1] == fake_next(rid, len(prompt) + i) for i in range(max_new - 1))
    st = s.stats()
    assert st["queued"] == 0 and st["active"] == 0 and st["retired"] == 3 and st["free_pages"] == 64


@pytest.mark.parametrize("max_batch,max_chunk", [(4, 4), (4, 8), (12, 8), (8, 3)])
def test_prefill_chunks_follow_the_policy(mk, max_batch, max_chunk):
    rng = random.Random(17 + max_chunk)
    reqs = [(200 + i, [rng.randrange(50) for _ in range(rng.randrange(1, 30))], rng.randrange(1, 12), -1)
            for i in range(20)]
    arrivals = {0: list(range(6)), 4: list(range(6, 14)), 11: list(range(14, 20))}
    s, ref = drive(mk, 48, 4, max_batch, 16, reqs, arrivals, max_chunk=max_chunk)
    assert all(r["done"] for r in ref.reqs.values())
    assert s.stats()["free_pages"] == 48
    # prefill shortens the run: fewer steps than feeding one prompt token per step
    s1, _ = drive(mk, 48, 4, max_batch, 16, reqs, arrivals, max_chunk=1)
    assert s.stats()["steps"] < s1.stats()["steps"]


def test_prefill_setting_is_checked(mk):
    s = mk.Scheduler(16, 16, 4, 2)
    for bad in (0, 9):
        with pytest.raises(mk.MkError):
            s.set_prefill(bad)
    s.set_prefill(4)
    s.submit(1, [1, 2, 3, 4, 5, 6], 2)
    b = s.next()
    assert b["rids"] == [1] * 4 and b["seq_lens"] == [0, 1, 2, 3] and b["chunk_first"] == [0] * 4
    with pytest.raises(mk.MkError):
        s.set_prefill(2)                        # a batch is pending
    s.commit([0, 0, 0, 9])                      # no output yet: the prompt has 6 tokens
    assert s.result(1) == ([], False)
    b = s.next()
    assert b["seq_lens"] == [4, 5] and b["tokens"] == [5, 6]
    s.commit([0, 7])                            # the prediction after the last prompt token
    assert s.result(1) == ([7], False)


def test_slots_and_pages_limit_admission_fifo(mk):
    rng = random.Random(5)
    reqs = [(100 + i, [rng.randrange(50) for _ in range(rng.randrange(1, 26))], rng.randrange(1, 16), -1)
            for i in range(24)]
    arrivals = {0: list(range(8)), 3: list(range(8, 16)), 9: list(range(16, 24))}
    s, ref = drive(mk, 12, 4, 3, 16, reqs, arrivals)
    assert all(r["done"] for r in ref.reqs.values())
    assert s.stats()["free_pages"] == 12


def test_head_of_line_request_blocks_until_pages_free(mk):
    # 8 pages of 4 tokens: the second request needs all 8 and must wait for the first
    reqs = [(1, [3] * 5, 4, -1), (2, [4] * 20, 13, -1), (3, [5], 1, -1)]
    s = mk.Scheduler(8, 4, 4, 8)
    for r in reqs:
        s.submit(*r)
    b = s.next()
    assert b["rids"] == [1]          # request 2 needs 8 pages, 6 are free; request 3 waits behind it
    st = s.stats()
    assert st["queued"] == 2 and st["free_pages"] == 6
    s.commit([0])
    s, ref = drive(mk, 8, 4, 4, 8, reqs)
    assert all(r["done"] for r in ref.reqs.values())


def test_end_token_retires_early(mk):
    eos = fake_next(7, 2)              # the first output of request 7 (prompt of 3 tokens)
    reqs = [(7, [1, 1, 1], 10, eos), (8, [2, 2], 3, eos)]
    s, ref = drive(mk, 32, 16, 2, 4, reqs)
    out, done = s.result(7)
    assert done and out == [eos]


def test_abandon_repeats_the_batch(mk):
    s = mk.Scheduler(16, 16, 2, 2)
    s.submit(1, [4, 5], 3)
    b1 = s.next()
    assert b1["changed"]
    s.abandon()
    b2 = s.next()
    assert b2["changed"] and (b2["rids"], b2["seq_lens"], b2["tokens"]) == (b1["rids"], b1["seq_lens"], b1["tokens"])
    s.commit([9])
    b3 = s.next()
    assert not b3["changed"] and b3["seq_lens"] == [1] and b3["tokens"] == [5]


def test_errors(mk):
    s = mk.Scheduler(4, 16, 2, 2)
    s.submit(1, [1], 2)
    with pytest.raises(mk.MkError) as e:
        s.submit(1, [1], 2)                     # repeated id
    assert e.value.code == mk.MK_ERR_INVALID
    with pytest.raises(mk.MkError) as e:
        s.submit(2, [1] * 30, 4)                # 33 positions: 3 pages, a row holds 2
    assert e.value.code == mk.MK_ERR_CAPACITY
    for bad in ([], [-1]):
        with pytest.raises(mk.MkError) as e:
            s.submit(3, bad, 2)
        assert e.value.code == mk.MK_ERR_INVALID
    with pytest.raises(mk.MkError):
        s.submit(4, [1], 0)
    with pytest.raises(mk.MkError):
        s.commit([0])                           # nothing pending
    s.next()
    with pytest.raises(mk.MkError):
        s.next()                                # previous batch not committed
    s.commit([0])
    with pytest.raises(mk.MkError):
        s.forget(1)                             # not finished yet
    s.next()
    s.commit([0])
    assert s.result(1) == ([0, 0], True)
    s.forget(1)
    with pytest.raises(mk.MkError):
        s.result(1)
    with pytest.raises(mk.MkError):
        mk.Scheduler(0, 16, 1, 1)
    assert s.next() is None
