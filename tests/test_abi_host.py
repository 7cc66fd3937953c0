"""C ABI on the host (no GPU): the library loads, exports every symbol that
include/mk.h declares, rejects bad shapes, and its task planner produces
lists that cannot deadlock and whose counters all fire."""
import ctypes
import os
import re
from collections import defaultdict

import pytest
import torch

import synth
from synth import FULL, MID, TINY, Dims

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

T_QKV, T_ATTN, T_OPROJ, T_MOE, T_RED, T_LM, T_COMB = range(7)


@pytest.fixture(scope="module")
def mk(built):
    from persistent_moe_decode_02_gb300 import mk
    return mk


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mk.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mk_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(mk):
    names = declared_functions()
    assert set(names) == set(mk.EXPORTS)
    lib = ctypes.CDLL(mk.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(mk):
    for c in (0, -1, -2, -3, -4, -5):
        assert mk.status_string(c) and mk.status_string(c) != "unknown status"


def test_rejects_bad_shapes(mk):
    with pytest.raises(mk.MkError) as e:
        mk.inspect_tasks(Dims(2, 256, 6, 4, 64, 8, 2, 512, 4096), [10], 8)   # 6 % 4 != 0
    assert e.value.code == mk.MK_ERR_INVALID
    with pytest.raises(mk.MkError) as e:
        mk.inspect_tasks(Dims(2, 256, 4, 2, 96, 8, 2, 512, 4096), [10], 8)   # head_dim 96
    assert e.value.code == mk.MK_ERR_UNSUPPORTED
    with pytest.raises(mk.MkError) as e:
        mk.inspect_tasks(Dims(2, 256, 4, 2, 64, 8, 9, 512, 4096), [10], 8)   # top_k 9
    assert e.value.code in (mk.MK_ERR_INVALID, mk.MK_ERR_UNSUPPORTED)
    with pytest.raises(mk.MkError):
        mk.inspect_tasks(TINY, [5] * 9, 8)                                  # batch 9


def signals_per_step(D, B, tasks):
    """Counter -> number of increments one step makes (ticket counters count
    every producer; 'done' counters of ticket families fire once per group)."""
    L, nkv = D.n_layers, D.n_kv_heads
    # same layout as the device counter map
    base = {}
    c = 0
    for name, n in (("qkv", L * nkv), ("attn", L * B * nkv), ("combine", L), ("o", L),
                    ("rdone", L), ("gu", L), ("down", L), ("lm", 1)):
        base[name] = c
        c += n
    sig = defaultdict(int)
    for t in tasks.tolist():
        typ, l, a = t[0], t[1], t[2:10]
        if typ == T_QKV:
            sig[base["qkv"] + l * nkv + a[2]] += 1
        elif typ == T_ATTN:
            sig[base["attn"] + (l * B + a[0]) * nkv + a[1]] += 1
        elif typ == T_OPROJ:
            sig[base["o"] + l] += 1
        elif typ == T_MOE:
            sig[base["gu"] + l] += 1
        elif typ == T_RED:
            sig[base["down"] + l] += 1
        elif typ == T_LM:
            sig[base["lm"]] += 1
        elif typ == T_COMB:
            sig[base["combine"] + l] += 1
    for l in range(L):
        sig[base["rdone"] + l] = 1             # gate/up tile 0 publishes the routing table
    return sig, base


def emulate(tasks, cta_start, sig_fn):
    """Run the per-CTA lists in lock-free rounds: a CTA advances when its next
    task's wait is satisfied.  Returns the completion order or raises on deadlock."""
    C = len(cta_start) - 1
    pos = [cta_start[c] for c in range(C)]
    ctr = defaultdict(int)
    done = 0
    n = len(tasks)
    order = []
    while done < n:
        progressed = False
        for c in range(C):
            if pos[c] >= cta_start[c + 1]:
                continue
            t = tasks[pos[c]].tolist()
            wc, wn = t[10], t[11]
            if wc < 0 or ctr[wc] >= wn:
                for k in sig_fn(t):
                    ctr[k] += 1
                order.append(pos[c])
                pos[c] += 1
                done += 1
                progressed = True
        if not progressed:
            raise AssertionError(f"deadlock after {done} of {n} tasks")
    return order


@pytest.mark.parametrize("D,ctx,C", [(TINY, [128], 152), (TINY, [0, 15, 16, 300], 7), (MID, [4096], 152),
                                     (FULL, [8192], 152), (FULL, [100, 262144, 9000], 152), (TINY, [50], 1)])
def test_planner_lists_complete_without_deadlock(mk, D, ctx, C):
    tasks, cs = mk.inspect_tasks(D, ctx, C)
    B = len(ctx)
    assert cs[0] == 0 and cs[-1] == tasks.shape[0] and all(a <= b for a, b in zip(cs, cs[1:]))
    sig, base = signals_per_step(D, B, tasks)
    # every wait names a counter that reaches exactly its count in one step
    for t in tasks.tolist():
        if t[10] >= 0:
            assert sig[t[10]] == t[11], t
    L, nkv = D.n_layers, D.n_kv_heads

    def fires(t):
        typ, l, a = t[0], t[1], t[2:10]
        out = []
        if typ == T_QKV:
            out.append(base["qkv"] + l * nkv + a[2])
        elif typ == T_ATTN:
            out.append(base["attn"] + (l * B + a[0]) * nkv + a[1])
        elif typ == T_OPROJ:
            out.append(base["o"] + l)
        elif typ == T_MOE:
            out.append(base["gu"] + l)
        elif typ == T_RED:
            out.append(base["down"] + l)
        elif typ == T_COMB:
            out.append(base["combine"] + l)
        return out

    def fires_with_finishers(t):
        out = fires(t)
        if t[0] == T_MOE and t[2] == 0:
            out.append(base["rdone"] + t[1])
        return out

    order = emulate(tasks, cs, fires_with_finishers)
    assert len(order) == tasks.shape[0]
    # the attention chunks of each (request, group) cover its pages exactly once
    for b, c in enumerate(ctx):
        for g in range(nkv):
            ch = sorted((t[4], t[5]) for t in tasks.tolist() if t[0] == T_ATTN and t[1] == 0 and t[2] == b
                        and t[3] == g)
            assert ch[0][0] == 0 and ch[-1][1] == -1
            for (a0, a1), (b0, _) in zip(ch, ch[1:]):
                assert a1 == b0
    # row tiles cover their matrices exactly
    def cover(typ, n):
        rows = sorted((t[2], t[3]) for t in tasks.tolist() if t[0] == typ and t[1] == 0)
        assert rows[0][0] == 0 and rows[-1][1] == n
        assert all(x[1] == y[0] for x, y in zip(rows, rows[1:]))
    cover(T_QKV, D.n_kv_heads * (D.group + 2) * D.head_dim)
    cover(T_OPROJ, D.hidden)
    cover(T_RED, D.hidden)
    # the O tiles carry distinct router-partial indices 0 .. tiles - 1
    oi = sorted(t[4] for t in tasks.tolist() if t[0] == T_OPROJ and t[1] == 0)
    assert oi == list(range(len(oi)))
    lm = sorted((t[2], t[3]) for t in tasks.tolist() if t[0] == T_LM)
    assert lm[0][0] == 0 and lm[-1][1] == D.vocab
    # every query head of every (request, group) is combined exactly once, from
    # that pair's own partial slots
    for b in range(B):
        for g in range(nkv):
            comb = [t for t in tasks.tolist() if t[0] == T_COMB and t[1] == 0 and t[2] == b and t[3] == g]
            heads = sorted(h for t in comb for h in range(t[4], t[4] + t[5]))
            assert heads == list(range(D.group))
            chunks = sorted(t[6] for t in tasks.tolist() if t[0] == T_ATTN and t[1] == 0 and t[2] == b and t[3] == g)
            assert all(t[7] == chunks[0] and t[8] == len(chunks) for t in comb)
            assert chunks == list(range(chunks[0], chunks[0] + len(chunks)))


def test_full_bs1_phases_spread_over_all_ctas(mk):
    tasks, cs = mk.inspect_tasks(FULL, [8192], 152)
    per_cta = defaultdict(lambda: defaultdict(int))
    for c in range(152):
        for t in tasks[cs[c]:cs[c + 1]].tolist():
            if t[1] == 5:
                per_cta[t[0]][c] += 1
    for typ in (T_QKV, T_OPROJ, T_MOE, T_RED):
        assert len(per_cta[typ]) == 152, typ          # every CTA takes part in each big phase
        assert max(per_cta[typ].values()) == 1, typ   # and takes one tile of it
    # 513 pages x 4 groups in 14-page chunks: 148 chunks, at most one per CTA
    assert len(per_cta[T_ATTN]) == 148 and max(per_cta[T_ATTN].values()) == 1


def test_plan_create_rejects_unusable_temperatures(mk):
    # The temperature is checked before any CUDA call, so fake (aligned,
    # never dereferenced) device addresses are enough here.  Negative, NaN,
    # infinite and denormal-small temperatures (whose inverse overflows) are
    # MK_ERR_INVALID; the message names the rule.
    class Fake:
        def __init__(self, addr):
            self.addr = addr

        def data_ptr(self):
            return self.addr

    D = TINY
    L = D.n_layers
    addr = iter(range(1 << 20, 1 << 30, 1 << 12))
    weights = {k: Fake(next(addr)) for k in ("embed", "final_norm", "lm_head")}
    for k in ("attn_norm", "wqkv", "wo", "ffn_norm", "router", "w_gate_up", "w_down"):
        weights[k] = [Fake(next(addr)) for _ in range(L)]
    pools = [Fake(next(addr)) for _ in range(L)]

    class Pool(Fake):
        shape = (64,)

    kp = [Pool(p.addr) for p in pools]
    w, kv, keep = mk._weight_structs(D, weights, kp)
    dims = mk.dims_struct(D)
    lens = mk._int_array([20])
    pt = mk._int_array(list(range(4)))
    out = ctypes.c_void_p()
    for T in (-1.0, float("nan"), float("inf"), 1e-39):
        opts = mk.MkPlanOpts()
        opts.temperature = T
        rc = mk.lib().mk_plan_create(ctypes.byref(dims), ctypes.byref(w), ctypes.byref(kv), 1, lens, pt, 4,
                                     ctypes.byref(opts), ctypes.byref(out))
        assert rc == mk.MK_ERR_INVALID, T
        assert b"inverse" in mk.lib().mk_last_error(), T
        assert not out.value
    del keep
