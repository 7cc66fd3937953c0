"""Seeded synthetic inputs for the MoE decode step: model shapes, weights,
prior paged KV, first tokens, ragged lengths and page tables.

This module is the only code that both the CPU oracle and the GPU path use.
It holds none of the decode step's arithmetic: it only produces inputs.
Every value comes from a counter-based generator (``gen.h``) keyed by
(seed, stream name, element index), built once for the host (OpenMP) and
once for the device (CUDA) from the same source, so a tensor generated on
either side has the same bits.

Input recipe (the pages print no weights; they describe a 30B-total /
3.3B-active BF16 MoE model served from a paged KV cache):
  * weight matrices bf16 ~ N(0, 0.02); RMSNorm gains bf16(1 + N(0, 0.02));
  * prior K/V bf16 ~ N(0, 1), keyed by logical (request, layer, position),
    so physical page placement never changes a value;
  * first tokens uniform in [0, vocab);
  * page tables are seeded random permutations of the physical pages.
"N(0, s)" is realised as a 4-term Irwin-Hall sum scaled to standard
deviation s, which is exact integer arithmetic on any device.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_SRCS = [os.path.join(_HERE, "gen.cu"), os.path.join(_HERE, "gen.h")]

WEIGHT_SIGMA = 0.02
KV_SIGMA = 1.0
# Standard deviation of the sum of four uniform 16-bit integers.
_SD_IH4 = math.sqrt(4.0 * (65536.0 ** 2 - 1.0) / 12.0)


def build(force: bool = False) -> str:
    """Compile libsynth.so (host OpenMP + sm_103a device code) if stale."""
    newest = max(os.path.getmtime(s) for s in _SRCS)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = [
        "nvcc", "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
        "-Xcompiler", "-fPIC,-fopenmp,-ffp-contract=off", "-shared", _SRCS[0],
        "-o", tmp, "-lgomp",
    ]
    subprocess.run(cmd, check=True, cwd=_HERE)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, u64, u32, i32, dbl, vp = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                                       ctypes.c_int, ctypes.c_double, ctypes.c_void_p)
        lib.synth_fill_normal_bf16.argtypes = [vp, i64, u64, u32, i64, dbl, dbl, i32, vp]
        lib.synth_fill_uniform_int.argtypes = [vp, i64, u64, u32, i64, u32, i32, vp]
        lib.synth_fill_kv_paged.argtypes = [vp, vp, i64, i32, i32, i32, i64, u64, u32, dbl, i32, vp]
        for f in (lib.synth_fill_normal_bf16, lib.synth_fill_uniform_int, lib.synth_fill_kv_paged):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def stream_id(name: str) -> int:
    """32-bit FNV-1a hash of a stream name."""
    h = 0x811C9DC5
    for b in name.encode():
        h = ((h ^ b) * 0x01000193) & 0xFFFFFFFF
    return h


def _cuda_stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream) if t.is_cuda else None


def fill_normal_(out: torch.Tensor, seed: int, name: str, start: int = 0,
                 mean: float = 0.0, sigma: float = WEIGHT_SIGMA) -> torch.Tensor:
    """Fill a contiguous bf16 tensor with elements [start, start + numel) of a stream."""
    assert out.dtype == torch.bfloat16 and out.is_contiguous()
    rc = _L().synth_fill_normal_bf16(ctypes.c_void_p(out.data_ptr()), out.numel(), seed,
                                     stream_id(name), start, mean, sigma / _SD_IH4,
                                     int(out.is_cuda), _cuda_stream(out))
    if rc != 0:
        raise RuntimeError(f"synth_fill_normal_bf16 failed ({rc})")
    return out


def normal(shape, seed: int, name: str, start: int = 0, mean: float = 0.0,
           sigma: float = WEIGHT_SIGMA, device="cpu") -> torch.Tensor:
    return fill_normal_(torch.empty(shape, dtype=torch.bfloat16, device=device), seed, name,
                        start, mean, sigma)


def uniform_ints(n: int, hi: int, seed: int, name: str, start: int = 0) -> torch.Tensor:
    out = torch.empty(n, dtype=torch.int32)
    rc = _L().synth_fill_uniform_int(ctypes.c_void_p(out.data_ptr()), n, seed, stream_id(name),
                                     start, hi, 0, None)
    if rc != 0:
        raise RuntimeError("synth_fill_uniform_int failed")
    return out


def fill_kv_paged_(pool: torch.Tensor, page_table: torch.Tensor, n_tok: int, seed: int,
                   name: str) -> None:
    """Write the first n_tok logical K (or V) rows of one request/layer into a
    paged pool [num_pages, nkv, d, page_size] (each page stores its block
    transposed, one row per dimension) through its page table.  The pool may
    be a view whose (page, head) blocks lie pool.stride(1) elements apart (the
    K or V half of an interleaved pool); each block is contiguous."""
    assert pool.dtype == torch.bfloat16 and pool.dim() == 4
    _, nkv, d, ps = pool.shape
    assert pool.stride(3) == 1 and pool.stride(2) == ps and pool.stride(0) == nkv * pool.stride(1)
    assert page_table.dtype == torch.int32 and page_table.device == pool.device
    need = (n_tok + ps - 1) // ps
    assert page_table.numel() >= need
    rc = _L().synth_fill_kv_paged(ctypes.c_void_p(pool.data_ptr()),
                                  ctypes.c_void_p(page_table.data_ptr()), n_tok, nkv, ps, d,
                                  pool.stride(1), seed, stream_id(name), KV_SIGMA / _SD_IH4,
                                  int(pool.is_cuda), _cuda_stream(pool))
    if rc != 0:
        raise RuntimeError("synth_fill_kv_paged failed")


# --------------------------------------------------------------------------
# Model shapes and workloads
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Dims:
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_experts: int
    top_k: int
    expert_ffn: int
    vocab: int
    page_size: int = 16
    rms_eps: float = 1e-6
    rope_theta: float = 1e4

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


TINY = Dims(2, 256, 4, 2, 64, 8, 2, 512, 4096)
MID = Dims(8, 2048, 32, 4, 128, 64, 8, 768, 32000)
FULL = Dims(48, 2048, 32, 4, 128, 128, 8, 768, 151936)


@dataclass
class Workload:
    """One benchmark/parity configuration: shapes, batch and context lengths."""
    name: str
    dims: Dims
    ctx: List[int]                 # prior tokens cached per request at step 0
    steps: int
    seed: int = 0
    churn_leave: int = 0           # requests that finish after each step
    churn_join_ctx: int = 0        # context length of each joining request
    note: str = ""

    @property
    def batch(self) -> int:
        return len(self.ctx)


def log_uniform_lengths(n: int, lo: int, hi: int, seed: int, name: str) -> List[int]:
    """n integer lengths, log-uniform in [lo, hi], rounded down."""
    u = uniform_ints(n, 1 << 24, seed, name).double().numpy() / float(1 << 24)
    return [int(math.floor(lo * math.exp(x * math.log(hi / lo)))) for x in u]


def workload(name: str) -> Workload:
    if name == "tiny":
        return Workload(name, TINY, [128], 32,
                        note="2 layers, hidden 256, 4q/2kv x 64, 8 experts top-2, F 512, vocab 4096, ctx 128")
    if name == "mid":
        return Workload(name, MID, [4096], 16,
                        note="8 layers, hidden 2048, 32q/4kv x 128, 64 experts top-8, F 768, vocab 32000, ctx 4096")
    if name == "full_bs1_8k":
        return Workload(name, FULL, [8192], 64,
                        note="48 layers, hidden 2048, 32q/4kv x 128, 128 experts top-8, F 768, vocab 151936, batch 1, ctx 8192")
    if name == "full_b32_churn":
        return Workload(name, FULL, log_uniform_lengths(32, 512, 32768, 0, "ctx.b32"), 64,
                        churn_leave=2, churn_join_ctx=512,
                        note="full shape, batch 32, ctx log-uniform [512, 32768], 2 leave / 2 join at 512 per step")
    if name == "full_b1_256k":
        return Workload(name, FULL, [262144], 16, note="full shape, batch 1, ctx 262144")
    if name == "mid_b8":
        return Workload(name, MID, log_uniform_lengths(8, 512, 4096, 0, "ctx.mid_b8"), 4,
                        note="mid shape, batch 8, ctx log-uniform [512, 4096] (a few GB on the device: profiling case)")
    if name == "full_b8_long":
        return Workload(name, FULL, log_uniform_lengths(8, 8192, 262144, 0, "ctx.b8"), 16,
                        note="full shape, batch 8, ctx log-uniform [8192, 262144]")
    raise KeyError(name)


WORKLOADS = ["tiny", "mid", "mid_b8", "full_bs1_8k", "full_b32_churn", "full_b1_256k", "full_b8_long"]


def first_token(dims: Dims, seed: int, rid: int) -> int:
    """Seeded first token of logical request rid, uniform in [0, vocab)."""
    return int(uniform_ints(1, dims.vocab, seed, "tok", start=rid)[0])


def page_permutation(num_pages: int, seed: int, salt: int = 0) -> np.ndarray:
    """Seeded random permutation of physical page ids."""
    return np.random.Generator(np.random.PCG64([seed, salt])).permutation(num_pages).astype(np.int32)


# --------------------------------------------------------------------------
# Weight streams.  Every tensor is its own stream; element index = row-major
# offset in the logical tensor listed here.
# --------------------------------------------------------------------------

def wname(kind: str, layer: Optional[int] = None) -> str:
    return kind if layer is None else f"L{layer}.{kind}"


class SynthWeights:
    """Logical weights generated on demand on the host (bf16, CPU tensors).

    Logical tensors (row-major [out, in]):
      embed [V, H]; final_norm [H]; lm_head [V, H]
      per layer: attn_norm [H], wq [nq*d, H], wk [nkv*d, H], wv [nkv*d, H],
                 wo [H, nq*d], ffn_norm [H], router [E, H],
                 gate [E, F, H], up [E, F, H], down [E, H, F]
    """

    def __init__(self, dims: Dims, seed: int = 0, cache_limit_bytes: int = 8 << 30):
        self.dims, self.seed = dims, seed
        self._cache = {}
        self._cache_bytes = 0
        self._limit = cache_limit_bytes

    def _get(self, key, fn):
        t = self._cache.get(key)
        if t is None:
            t = fn()
            nb = t.numel() * 2
            if self._cache_bytes + nb <= self._limit:
                self._cache[key] = t
                self._cache_bytes += nb
        return t

    def _norm(self, name):
        return self._get(name, lambda: normal((self.dims.hidden,), self.seed, name, mean=1.0))

    def embed_rows(self, tokens: Sequence[int]) -> torch.Tensor:
        H = self.dims.hidden
        return torch.stack([normal((H,), self.seed, "embed", start=int(t) * H) for t in tokens])

    def final_norm(self):
        return self._norm("final_norm")

    def attn_norm(self, l):
        return self._norm(wname("attn_norm", l))

    def ffn_norm(self, l):
        return self._norm(wname("ffn_norm", l))

    def _mat(self, kind, l, rows, cols):
        n = wname(kind, l)
        return self._get(n, lambda: normal((rows, cols), self.seed, n))

    def wq(self, l):
        D = self.dims
        return self._mat("wq", l, D.n_q_heads * D.head_dim, D.hidden)

    def wk(self, l):
        D = self.dims
        return self._mat("wk", l, D.n_kv_heads * D.head_dim, D.hidden)

    def wv(self, l):
        D = self.dims
        return self._mat("wv", l, D.n_kv_heads * D.head_dim, D.hidden)

    def wo(self, l):
        D = self.dims
        return self._mat("wo", l, D.hidden, D.n_q_heads * D.head_dim)

    def router(self, l):
        D = self.dims
        return self._mat("router", l, D.n_experts, D.hidden)

    def expert(self, l, e):
        D = self.dims
        F, H = D.expert_ffn, D.hidden

        def gen():
            g = normal((F, H), self.seed, wname("gate", l), start=e * F * H)
            u = normal((F, H), self.seed, wname("up", l), start=e * F * H)
            dn = normal((H, F), self.seed, wname("down", l), start=e * H * F)
            return (g, u, dn)
        key = ("expert", l, e)
        t = self._cache.get(key)
        if t is None:
            t = gen()
            nb = sum(x.numel() for x in t) * 2
            if self._cache_bytes + nb <= self._limit:
                self._cache[key] = t
                self._cache_bytes += nb
        return t

    def lm_head(self):
        D = self.dims
        return self._mat("lm_head", None, D.vocab, D.hidden)


def kv_name(rid: int, layer: int, kind: str) -> str:
    return f"kv.R{rid}.L{layer}.{kind}"


def prior_kv(dims: Dims, seed: int, rid: int, layer: int, n_tok: int):
    """Logical prior K and V of one request/layer: bf16 [n_tok, nkv, d] each."""
    shape = (n_tok, dims.n_kv_heads, dims.head_dim)
    k = normal(shape, seed, kv_name(rid, layer, "K"), sigma=KV_SIGMA)
    v = normal(shape, seed, kv_name(rid, layer, "V"), sigma=KV_SIGMA)
    return k, v
