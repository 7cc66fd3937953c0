"""Thin ctypes binding of libmk.so (include/mk.h): argument marshalling only.

Every step of the decode path runs inside the library's CUDA kernel; this
module never computes any of it.  It fails loudly when libmk.so is missing
(build it with ``persistent_moe_decode_02_gb300.build.build()``)."""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmk.so")

MK_OK, MK_ERR_INVALID, MK_ERR_CUDA, MK_ERR_DEP_TIMEOUT, MK_ERR_CAPACITY, MK_ERR_UNSUPPORTED = 0, -1, -2, -3, -4, -5
MK_DBG_HIDDEN, MK_DBG_EXPERT_IDS, MK_DBG_GATES, MK_DBG_ROUTER_LOGITS, MK_DBG_SEQ_LENS, MK_DBG_UNION = 1, 2, 3, 4, 5, 6
MK_DBG_TASKS, MK_DBG_TRACE, MK_DBG_STAGE_TRACE = 7, 8, 9
TRACE_SLOTS = ["fetch", "dep", "act", "stages", "done", "p_first", "p_last", "p_start", "s_first", "s_last",
               "mid1", "mid2"]

EXPORTS = [
    "mk_plan_create", "mk_decode_step", "mk_decode_steps", "mk_decode_step_host", "mk_plan_update", "mk_plan_sync",
    "mk_plan_read_debug", "mk_plan_info", "mk_plan_destroy", "mk_status_string", "mk_plan_inspect",
    "mk_last_error", "mk_decode_step_noalloc", "mk_plan_set_sampling", "mk_plan_set_top_p", "mk_sched_create", "mk_sched_submit", "mk_sched_next",
    "mk_sched_commit", "mk_sched_abandon", "mk_sched_result", "mk_sched_forget", "mk_sched_stats",
    "mk_sched_destroy", "mk_serve_step", "mk_sched_next_rows", "mk_sched_set_prefill", "mk_plan_update_rows",
    "mk_sched_peek_rows",
]


class MkModelDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim",
                                            "n_experts", "top_k", "expert_ffn", "vocab", "page_size")] + \
               [("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float)]


_PP = ctypes.POINTER(ctypes.c_void_p)


class MkWeights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("attn_norm", _PP), ("wqkv", _PP), ("wo", _PP), ("ffn_norm", _PP), ("router", _PP),
                ("w_gate_up", _PP), ("w_down", _PP)]


class MkKv(ctypes.Structure):
    _fields_ = [("kv_pool", _PP), ("num_pages", ctypes.c_int)]


class MkPlanOpts(ctypes.Structure):
    _fields_ = [("timeout_us", ctypes.c_int), ("num_ctas", ctypes.c_int), ("max_batch", ctypes.c_int),
                ("split_pages", ctypes.c_int), ("debug_drop_task", ctypes.c_int), ("trace", ctypes.c_int),
                ("temperature", ctypes.c_float), ("seed", ctypes.c_ulonglong), ("top_p", ctypes.c_float),
                ("chunk_first", ctypes.POINTER(ctypes.c_int)), ("tc_off", ctypes.c_int)]


class MkError(RuntimeError):
    def __init__(self, fn: str, code: int):
        detail = lib().mk_last_error().decode()
        super().__init__(f"{fn} failed: {code} ({status_string(code)})" + (f": {detail}" if detail else ""))
        self.code = code


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it first "
                              "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, p_int = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_int)
        L.mk_plan_create.argtypes = [ctypes.POINTER(MkModelDims), ctypes.POINTER(MkWeights), ctypes.POINTER(MkKv),
                                     i32, p_int, p_int, i32, ctypes.POINTER(MkPlanOpts), ctypes.POINTER(vp)]
        L.mk_decode_step.argtypes = [vp, vp, vp, vp, vp]
        L.mk_decode_steps.argtypes = [vp, vp, i32, vp, vp, vp]
        L.mk_decode_step_host.argtypes = [vp, p_int, ctypes.POINTER(ctypes.c_float), p_int, vp]
        L.mk_plan_update.argtypes = [vp, i32, p_int, p_int, i32, vp]
        L.mk_plan_sync.argtypes = [vp, vp]
        L.mk_plan_read_debug.argtypes = [vp, i32, vp, ctypes.c_size_t, vp]
        L.mk_plan_info.argtypes = [vp, p_int, i32]
        L.mk_plan_destroy.argtypes = [vp]
        L.mk_plan_destroy.restype = None
        L.mk_status_string.argtypes = [i32]
        L.mk_status_string.restype = ctypes.c_char_p
        L.mk_last_error.argtypes = []
        L.mk_last_error.restype = ctypes.c_char_p
        L.mk_plan_inspect.argtypes = [ctypes.POINTER(MkModelDims), i32, p_int, i32, i32, p_int, i32, p_int]
        L.mk_decode_step_noalloc.argtypes = [ctypes.POINTER(MkModelDims), ctypes.POINTER(MkWeights),
                                             ctypes.POINTER(MkKv), i32, p_int, p_int, i32, vp, vp, vp, vp, vp]
        i64, p_i64 = ctypes.c_longlong, ctypes.POINTER(ctypes.c_longlong)
        L.mk_plan_set_sampling.argtypes = [vp, ctypes.c_float, ctypes.c_ulonglong]
        L.mk_plan_set_top_p.argtypes = [vp, ctypes.c_float]
        L.mk_sched_create.argtypes = [i32, i32, i32, i32, ctypes.POINTER(vp)]
        L.mk_sched_submit.argtypes = [vp, i64, p_int, i32, i32, i32]
        L.mk_sched_next.argtypes = [vp, p_int, p_int, p_int, p_int, p_i64, p_int]
        L.mk_sched_next_rows.argtypes = [vp, p_int, p_int, p_int, p_int, p_i64, p_int, p_int]
        L.mk_sched_set_prefill.argtypes = [vp, i32]
        L.mk_sched_peek_rows.argtypes = [vp, p_int, p_int, p_int, p_int, p_i64, p_int]
        L.mk_plan_update_rows.argtypes = [vp, i32, p_int, p_int, i32, p_int, vp]
        L.mk_sched_commit.argtypes = [vp, p_int]
        L.mk_sched_abandon.argtypes = [vp]
        L.mk_sched_result.argtypes = [vp, i64, p_int, i32, p_int, p_int]
        L.mk_sched_forget.argtypes = [vp, i64]
        L.mk_sched_stats.argtypes = [vp, p_int, i32]
        L.mk_sched_destroy.argtypes = [vp]
        L.mk_sched_destroy.restype = None
        L.mk_serve_step.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(MkModelDims), ctypes.POINTER(MkWeights),
                                    ctypes.POINTER(MkKv), ctypes.POINTER(MkPlanOpts), vp]
        for f in ("mk_plan_create", "mk_decode_step", "mk_decode_steps", "mk_decode_step_host", "mk_plan_update", "mk_plan_sync",
                  "mk_plan_read_debug", "mk_plan_info", "mk_plan_inspect", "mk_decode_step_noalloc",
                  "mk_plan_set_sampling", "mk_plan_set_top_p", "mk_sched_create", "mk_sched_submit", "mk_sched_next", "mk_sched_commit", "mk_sched_abandon",
                  "mk_sched_result", "mk_sched_forget", "mk_sched_stats", "mk_serve_step", "mk_sched_next_rows",
                  "mk_sched_set_prefill", "mk_plan_update_rows", "mk_sched_peek_rows"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().mk_status_string(code).decode()


def dims_struct(D) -> MkModelDims:
    return MkModelDims(D.n_layers, D.hidden, D.n_q_heads, D.n_kv_heads, D.head_dim, D.n_experts, D.top_k,
                       D.expert_ffn, D.vocab, D.page_size, D.rms_eps, D.rope_theta)


def _int_array(vals: Sequence[int]):
    return (ctypes.c_int * len(vals))(*[int(v) for v in vals])


def _ptr_array(tensors):
    return (ctypes.c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def inspect_tasks(D, seq_lens: Sequence[int], num_ctas: int, split_pages: int = 0):
    """Host-only task list: returns (tasks [n, 12] int tensor, cta_start list)."""
    dims = dims_struct(D)
    sl = _int_array(seq_lens)
    n = lib().mk_plan_inspect(ctypes.byref(dims), len(seq_lens), sl, num_ctas, split_pages, None, 0, None)
    if n < 0:
        raise MkError("mk_plan_inspect", n)
    buf = (ctypes.c_int * (12 * n))()
    cs = (ctypes.c_int * (num_ctas + 1))()
    n2 = lib().mk_plan_inspect(ctypes.byref(dims), len(seq_lens), sl, num_ctas, split_pages, buf, n, cs)
    assert n2 == n
    return torch.tensor(list(buf), dtype=torch.int64).view(n, 12), list(cs)


def _weight_structs(D, weights: dict, kv_pools):
    """ctypes views of the weight and KV pointers (the arrays must outlive the call)."""
    arrays = {k: _ptr_array(weights[k]) for k in
              ("attn_norm", "wqkv", "wo", "ffn_norm", "router", "w_gate_up", "w_down")}
    kvp = _ptr_array(kv_pools)
    cast = lambda a: ctypes.cast(a, _PP)
    w = MkWeights(weights["embed"].data_ptr(), weights["final_norm"].data_ptr(), weights["lm_head"].data_ptr(),
                  *[cast(arrays[k]) for k in ("attn_norm", "wqkv", "wo", "ffn_norm", "router", "w_gate_up",
                                              "w_down")])
    kv = MkKv(cast(kvp), int(kv_pools[0].shape[0]))
    return w, kv, (arrays, kvp)


def decode_step_noalloc(D, weights: dict, kv_pools, seq_lens: Sequence[int], page_table, max_pages: int,
                        tokens: torch.Tensor, next_token: torch.Tensor, logits: Optional[torch.Tensor] = None,
                        status: Optional[torch.Tensor] = None, stream=None) -> int:
    """One step through mk_decode_step_noalloc (no plan, no allocation inside
    the library).  Returns the enqueue status; the device status goes to
    `status` (int32[4] on the device) when given."""
    w, kv, keep = _weight_structs(D, weights, kv_pools)
    dims = dims_struct(D)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr() if t is not None else 0)
    pt = [int(x) for x in page_table]
    rc = lib().mk_decode_step_noalloc(ctypes.byref(dims), ctypes.byref(w), ctypes.byref(kv), len(seq_lens),
                                      _int_array(seq_lens), _int_array(pt), max_pages, ptr(tokens), ptr(logits),
                                      ptr(next_token), ptr(status), _stream(stream))
    del keep
    return rc


class Plan:
    """Owns an mk_plan.  Weight/KV tensors are referenced, not copied.

    weights: dict with 'embed', 'final_norm', 'lm_head' tensors and per-layer
    lists 'attn_norm', 'wqkv', 'wo', 'ffn_norm', 'router', 'w_gate_up',
    'w_down' (bf16 CUDA tensors in the layout of include/mk.h).
    kv_pools: per-layer bf16 [num_pages, nkv, 2, head_dim, page_size] (per page
    and KV head the K block, then the V block, each stored transposed, slot
    fastest)."""

    def __init__(self, D, weights: dict, kv_pools, seq_lens: Sequence[int], page_table,
                 max_pages: int, timeout_us: int = 0, num_ctas: int = 0, max_batch: int = 0,
                 split_pages: int = 0, debug_drop_task: int = 0, trace: int = 0, tc_off: bool = False):
        self.D = D
        self._keep = (weights, kv_pools)
        self._arrays = {k: _ptr_array(weights[k]) for k in
                        ("attn_norm", "wqkv", "wo", "ffn_norm", "router", "w_gate_up", "w_down")}
        self._kvp = _ptr_array(kv_pools)
        cast = lambda a: ctypes.cast(a, _PP)
        self._w = MkWeights(weights["embed"].data_ptr(), weights["final_norm"].data_ptr(),
                            weights["lm_head"].data_ptr(), *[cast(self._arrays[k]) for k in
                                                             ("attn_norm", "wqkv", "wo", "ffn_norm", "router",
                                                              "w_gate_up", "w_down")])
        self._kv = MkKv(cast(self._kvp), int(kv_pools[0].shape[0]))
        self._dims = dims_struct(D)
        opts = MkPlanOpts(timeout_us, num_ctas, max_batch, split_pages, debug_drop_task, int(trace))
        opts.tc_off = int(bool(tc_off))
        self.batch = len(seq_lens)
        pt = [int(x) for x in page_table]
        h = ctypes.c_void_p()
        rc = lib().mk_plan_create(ctypes.byref(self._dims), ctypes.byref(self._w), ctypes.byref(self._kv),
                                  self.batch, _int_array(seq_lens), _int_array(pt), max_pages,
                                  ctypes.byref(opts), ctypes.byref(h))
        if rc != MK_OK:
            raise MkError("mk_plan_create", rc)
        self.h = h

    def step(self, tokens: torch.Tensor, next_token: torch.Tensor, logits: Optional[torch.Tensor] = None,
             stream=None) -> int:
        """Enqueue one decode step (device buffers).  Returns the status code."""
        return lib().mk_decode_step(self.h, ctypes.c_void_p(tokens.data_ptr()),
                                    ctypes.c_void_p(logits.data_ptr() if logits is not None else 0),
                                    ctypes.c_void_p(next_token.data_ptr()), _stream(stream))

    def steps(self, tokens: torch.Tensor, n_steps: int, next_tokens: torch.Tensor,
              logits: Optional[torch.Tensor] = None, stream=None) -> int:
        """Enqueue n_steps decode steps in one launch (device buffers):
        next_tokens int32 [n_steps, batch], logits float32 [n_steps, batch,
        vocab] or None.  Returns the status code."""
        return lib().mk_decode_steps(self.h, ctypes.c_void_p(tokens.data_ptr()), int(n_steps),
                                     ctypes.c_void_p(logits.data_ptr() if logits is not None else 0),
                                     ctypes.c_void_p(next_tokens.data_ptr()), _stream(stream))

    def step_host(self, tokens, next_token, logits=None, stream=None) -> int:
        """One step with host buffers (int32 / float32 CPU tensors, contiguous)."""
        tp = ctypes.cast(tokens.data_ptr(), ctypes.POINTER(ctypes.c_int))
        np_ = ctypes.cast(next_token.data_ptr(), ctypes.POINTER(ctypes.c_int))
        lp = ctypes.cast(logits.data_ptr(), ctypes.POINTER(ctypes.c_float)) if logits is not None else None
        return lib().mk_decode_step_host(self.h, tp, lp, np_, _stream(stream))

    def update_rows(self, seq_lens: Sequence[int], page_table, max_pages: int, chunk_first: Sequence[int],
                    stream=None) -> None:
        """Replace the batch with rows of which some are prefill chunks (include/mk.h)."""
        self.batch = len(seq_lens)
        pt = [int(x) for x in page_table]
        rc = lib().mk_plan_update_rows(self.h, self.batch, _int_array(seq_lens), _int_array(pt), max_pages,
                                       _int_array(chunk_first), _stream(stream))
        if rc != MK_OK:
            raise MkError("mk_plan_update_rows", rc)

    def update(self, seq_lens: Sequence[int], page_table, max_pages: int, stream=None) -> None:
        # int32 host arrays handed over by pointer (a numpy array or CPU tensor is not copied)
        sl = np.ascontiguousarray(np.asarray(seq_lens), dtype=np.int32)
        pt = np.ascontiguousarray(np.asarray(page_table), dtype=np.int32)
        p_int = ctypes.POINTER(ctypes.c_int)
        rc = lib().mk_plan_update(self.h, len(sl), sl.ctypes.data_as(p_int), pt.ctypes.data_as(p_int), max_pages,
                                  _stream(stream))
        if rc != MK_OK:
            raise MkError("mk_plan_update", rc)
        self.batch = len(seq_lens)

    def sync(self, stream=None) -> int:
        return lib().mk_plan_sync(self.h, _stream(stream))

    def set_sampling(self, temperature: float, seed: int = 0) -> None:
        """Temperature sampling for the following steps (0: greedy); see include/mk.h."""
        rc = lib().mk_plan_set_sampling(self.h, float(temperature), int(seed) & (2 ** 64 - 1))
        if rc != MK_OK:
            raise MkError("mk_plan_set_sampling", rc)

    def set_top_p(self, top_p: float) -> None:
        """Nucleus sampling (0 < top_p < 1) for the following sampled steps; 1: off."""
        rc = lib().mk_plan_set_top_p(self.h, float(top_p))
        if rc != MK_OK:
            raise MkError("mk_plan_set_top_p", rc)

    def read_debug(self, what: int, out: torch.Tensor, stream=None) -> torch.Tensor:
        rc = lib().mk_plan_read_debug(self.h, what, ctypes.c_void_p(out.data_ptr()),
                                      out.numel() * out.element_size(), _stream(stream))
        if rc != MK_OK:
            raise MkError("mk_plan_read_debug", rc)
        return out

    def timeline(self, stream=None):
        """(tasks int32 [n, 12], stamps int64 [n, 10]) of the last step (needs trace=True)."""
        n = self.info()["num_tasks"]
        tasks = torch.empty(n, 12, dtype=torch.int32)
        self.read_debug(MK_DBG_TASKS, tasks, stream)
        stamps = torch.empty(n, len(TRACE_SLOTS), dtype=torch.int64)
        self.read_debug(MK_DBG_TRACE, stamps, stream)
        self.sync(stream)
        return tasks, stamps

    def stage_timeline(self, stream=None) -> torch.Tensor:
        """int64 [num_ctas, 4096, 6] of the last step: per CTA and ring stage, the
        copy issue, landing and release stamps (ns, 0 = none), the task index, and
        the SM clock at landing and release (needs trace=2)."""
        out = torch.empty(self.info()["num_ctas"], 4096, 6, dtype=torch.int64)
        self.read_debug(MK_DBG_STAGE_TRACE, out, stream)
        self.sync(stream)
        return out

    def info(self) -> dict:
        buf = (ctypes.c_int * 12)()
        lib().mk_plan_info(self.h, buf, 12)
        keys = ["num_ctas", "num_tasks", "nstages", "stage_bytes", "smem_bytes", "batch", "attn_tasks",
                "gu_tasks", "lm_tiles", "replans", "tc_gate_up", "tc_proj"]
        return dict(zip(keys, list(buf)))

    def close(self):
        if getattr(self, "h", None):
            lib().mk_plan_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Scheduler:
    """Owns an mk_sched: the host-side request queue, batch and KV page
    allocator of continuous batching (include/mk.h describes the policy)."""

    def __init__(self, num_pages: int, page_size: int, max_batch: int, max_pages: int):
        h = ctypes.c_void_p()
        rc = lib().mk_sched_create(num_pages, page_size, max_batch, max_pages, ctypes.byref(h))
        if rc != MK_OK:
            raise MkError("mk_sched_create", rc)
        self.h, self.max_batch, self.max_pages = h, max_batch, max_pages

    def submit(self, rid: int, prompt: Sequence[int], max_new_tokens: int, eos_token: int = -1) -> None:
        rc = lib().mk_sched_submit(self.h, rid, _int_array(prompt), len(prompt), max_new_tokens, eos_token)
        if rc != MK_OK:
            raise MkError("mk_sched_submit", rc)

    def set_prefill(self, max_chunk: int) -> None:
        """Prompt tokens a request may feed per step as consecutive rows (1: one token per step)."""
        rc = lib().mk_sched_set_prefill(self.h, int(max_chunk))
        if rc != MK_OK:
            raise MkError("mk_sched_set_prefill", rc)

    def next(self):
        """The next batch's rows as a dict (seq_lens, page_table, tokens, rids,
        chunk_first, changed), or None when idle."""
        cap, mp = self.max_batch, self.max_pages
        b, ch = ctypes.c_int(), ctypes.c_int()
        sl, pt, tk = (ctypes.c_int * cap)(), (ctypes.c_int * (cap * mp))(), (ctypes.c_int * cap)()
        rids, cf = (ctypes.c_longlong * cap)(), (ctypes.c_int * cap)()
        rc = lib().mk_sched_next_rows(self.h, ctypes.byref(b), sl, pt, tk, rids, cf, ctypes.byref(ch))
        if rc != MK_OK:
            raise MkError("mk_sched_next_rows", rc)
        n = b.value
        if n == 0:
            return None
        return {"seq_lens": list(sl[:n]), "page_table": list(pt[:n * mp]), "tokens": list(tk[:n]),
                "rids": list(rids[:n]), "chunk_first": list(cf[:n]), "changed": bool(ch.value)}

    def peek(self):
        """The rows next() would return after the pending batch committed with no end token, or None."""
        cap, mp = self.max_batch, self.max_pages
        b = ctypes.c_int()
        sl, pt, tk = (ctypes.c_int * cap)(), (ctypes.c_int * (cap * mp))(), (ctypes.c_int * cap)()
        rids, cf = (ctypes.c_longlong * cap)(), (ctypes.c_int * cap)()
        rc = lib().mk_sched_peek_rows(self.h, ctypes.byref(b), sl, pt, tk, rids, cf)
        if rc != MK_OK:
            raise MkError("mk_sched_peek_rows", rc)
        n = b.value
        if n == 0:
            return None
        return {"seq_lens": list(sl[:n]), "page_table": list(pt[:n * mp]), "tokens": list(tk[:n]),
                "rids": list(rids[:n]), "chunk_first": list(cf[:n])}

    def commit(self, next_tokens: Sequence[int]) -> None:
        rc = lib().mk_sched_commit(self.h, _int_array(next_tokens))
        if rc != MK_OK:
            raise MkError("mk_sched_commit", rc)

    def abandon(self) -> None:
        rc = lib().mk_sched_abandon(self.h)
        if rc != MK_OK:
            raise MkError("mk_sched_abandon", rc)

    def result(self, rid: int):
        """(output tokens, done) of request rid."""
        n, d = ctypes.c_int(), ctypes.c_int()
        rc = lib().mk_sched_result(self.h, rid, None, 0, ctypes.byref(n), ctypes.byref(d))
        if rc != MK_OK:
            raise MkError("mk_sched_result", rc)
        buf = (ctypes.c_int * max(1, n.value))()
        rc = lib().mk_sched_result(self.h, rid, buf, n.value, ctypes.byref(n), ctypes.byref(d))
        if rc != MK_OK:
            raise MkError("mk_sched_result", rc)
        return list(buf[:n.value]), bool(d.value)

    def forget(self, rid: int) -> None:
        rc = lib().mk_sched_forget(self.h, rid)
        if rc != MK_OK:
            raise MkError("mk_sched_forget", rc)

    def stats(self) -> dict:
        buf = (ctypes.c_int * 5)()
        lib().mk_sched_stats(self.h, buf, 5)
        return dict(zip(["queued", "active", "retired", "free_pages", "steps"], list(buf)))

    def close(self):
        if getattr(self, "h", None):
            lib().mk_sched_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Server:
    """The serving loop: a Scheduler plus the plan it drives (created by the
    first mk_serve_step).  kv_pools: the KV pool the scheduler's pages index
    (every page of it is the scheduler's)."""

    def __init__(self, D, weights: dict, kv_pools, max_batch: int, max_pages: int, timeout_us: int = 0,
                 num_ctas: int = 0, split_pages: int = 0, temperature: float = 0.0, seed: int = 0,
                 prefill: int = 8):
        self.D = D
        self._keep = (weights, kv_pools)
        self._w, self._kv, self._arrays = _weight_structs(D, weights, kv_pools)
        self._dims = dims_struct(D)
        self._opts = MkPlanOpts(timeout_us, num_ctas, max_batch, split_pages, 0, 0, float(temperature),
                                int(seed) & (2 ** 64 - 1))
        self.sched = Scheduler(int(kv_pools[0].shape[0]), D.page_size, max_batch, max_pages)
        if prefill > 1:   # prompts enter the cache in chunks of up to `prefill` tokens per step
            self.sched.set_prefill(min(prefill, 8))
        self.plan = ctypes.c_void_p()

    def submit(self, rid: int, prompt: Sequence[int], max_new_tokens: int, eos_token: int = -1) -> None:
        self.sched.submit(rid, prompt, max_new_tokens, eos_token)

    def step(self, stream=None) -> int:
        """One serving step; returns the batch size that ran (0: idle)."""
        rc = lib().mk_serve_step(self.sched.h, ctypes.byref(self.plan), ctypes.byref(self._dims),
                                 ctypes.byref(self._w), ctypes.byref(self._kv), ctypes.byref(self._opts),
                                 _stream(stream))
        if rc < 0:
            raise MkError("mk_serve_step", rc)
        return rc

    def run(self, max_steps: int = 1 << 30, stream=None) -> int:
        """Step until nothing is queued or admitted (or max_steps); returns the steps run."""
        n = 0
        while n < max_steps and self.step(stream) > 0:
            n += 1
        return n

    def result(self, rid: int):
        return self.sched.result(rid)

    def close(self):
        if getattr(self, "plan", None) and self.plan.value:
            lib().mk_plan_destroy(self.plan)
            self.plan = ctypes.c_void_p()
        if getattr(self, "sched", None) is not None:
            self.sched.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
