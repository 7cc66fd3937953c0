"""Decode-throughput benchmark of the persistent MoE decode megakernel.

Default workload: the full-scale shape (48 layers, hidden 2048, 32q/4kv x 128,
128 experts top-8, expert FFN 768, vocab 151936), batch 1, 8192 cached tokens,
bf16 random-init weights, paged bf16 KV cache.  One step = one decode step of
the whole model = one megakernel launch.  Inputs stay resident in HBM; every
step streams ~6.9 GB, far larger than the 129 MB L2, so no flush is needed.

Prints one JSON line (see the keys below).  `--impl reference` times the CPU
oracle instead (the reference arm): a bounded sample of the same step on the
host cores.  Under torchrun each rank runs an independent replica on its own
GPU (the path does not shard), timed between barriers, max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode tok/s (bs1, 8K ctx) and achieved HBM GB/s as % of speed-of-light"
KERNEL_SOURCES = ["persistent_moe_decode_02_gb300/csrc/megakernel.cuh",
                  "persistent_moe_decode_02_gb300/csrc/megakernel.cu",
                  "persistent_moe_decode_02_gb300/csrc/mk_internal.h",
                  "persistent_moe_decode_02_gb300/csrc/plan.cu"]


def kernel_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def max_over_ranks(x: float, world: int, device: str = "cuda") -> float:
    """The largest x over the ranks of the process group (x itself on one rank):
    the job's time is its slowest replica's."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t)


def job_tok_s(world: int, batch: int, steps: int, seconds: float) -> float:
    """Whole-job throughput: every replica decodes `batch` tokens per step."""
    return world * batch * steps / seconds


def ncu_traffic(workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 7:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self) -> dict:
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ---------------------------------------------------------------- reference arm / CPU baseline

def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the baseline line."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


class OracleSample:
    """One whole decode step of the CPU oracle: every transformer layer of
    request 0 plus the final norm, LM head and argmax, timed for real (no
    extrapolation).  For a batch above 1 the step's time is that of request 0
    times the batch (requests are independent; said in describe()).  The
    weights, prior K/V and embedding rows the step reads are generated and
    cached by prepare(), an untimed first pass of the same step, so the clock
    covers only the oracle's arithmetic."""

    def __init__(self, wl):
        import synth
        self.wl, self.D = wl, wl.dims
        self.W = synth.SynthWeights(self.D, wl.seed, cache_limit_bytes=48 << 30)
        self.store = {}
        self.tok = synth.first_token(self.D, wl.seed, 0)
        self.emb = None

    def _prior(self, rid, l, n):
        import synth
        if (rid, l, n) not in self.store:
            self.store[(rid, l, n)] = synth.prior_kv(self.D, self.wl.seed, rid, l, n)
        return self.store[(rid, l, n)]

    def _run(self) -> float:
        from oracle import decode as O
        D = self.D
        if self.emb is None:
            self.emb = self.W.embed_rows([self.tok])[0]
        req = O.OracleRequest(0, self.wl.ctx[0], self._prior, D.n_layers)
        t0 = time.perf_counter()
        x = O.widen(self.emb)
        for l in range(D.n_layers):
            x, _ = O.decode_layer(self.W, D, l, x, req, self.wl.ctx[0])
        O.lm_head(self.W, D, x)
        return (time.perf_counter() - t0) * self.wl.batch

    def prepare(self):
        self._run()          # generates and caches every input the step reads (not timed)
        return self

    def step_seconds(self) -> float:
        return self._run()

    def describe(self) -> str:
        D = self.D
        what = (f"one whole decode step ({D.n_layers} layers, final norm, LM head, argmax) of request 0, "
                f"timed; inputs generated and cached by an untimed first pass")
        if self.wl.batch > 1:
            what += f"; scaled by the batch of {self.wl.batch} (requests are independent)"
        return what


REFERENCE_BUDGET_S = 120.0   # timed oracle work of one --impl reference run


def reference_arm(args, wl):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    smp = OracleSample(wl).prepare()
    warm = min(args.warmup, 1)
    for _ in range(warm):
        smp.step_seconds()
    # every step is a whole oracle step: as many of the requested steps as fit
    # the time budget are run, and the line reports how many ran
    times = [smp.step_seconds()]
    n = min(args.steps, max(1, int(REFERENCE_BUDGET_S / max(times[0], 1e-6))))
    while len(times) < n:
        times.append(smp.step_seconds())
    step_s = statistics.mean(times)
    cores = torch.get_num_threads()
    v = wl.batch / step_s
    out = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s", "n_gpus": args.gpus,
           "steps": len(times), "steps_requested": args.steps, "warmup": warm + 1,
           "ms_per_step": step_s * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": config_of(wl),
           "cpu_baseline": {"value": v, "unit": "tok/s", "cores": cores, "cpu": cpu_model(), "kind": "oracle",
                            "sample": smp.describe() + f"; {len(times)} timed steps"},
           "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def config_of(wl) -> dict:
    D = wl.dims
    return {"workload": wl.name, "layers": D.n_layers, "hidden": D.hidden,
            "heads": f"{D.n_q_heads}q/{D.n_kv_heads}kv x {D.head_dim}",
            "experts": f"{D.n_experts} top-{D.top_k}, ffn {D.expert_ffn}", "vocab": D.vocab,
            "batch": wl.batch, "ctx": wl.ctx if wl.batch <= 8 else f"{min(wl.ctx)}..{max(wl.ctx)}",
            "weights": "bf16 random-init", "kv": "paged bf16, page 16, shuffled",
            "l2": "inputs larger than L2 (the step streams GBs; no flush needed)", "logits": False}


# ---------------------------------------------------------------- our arm

def our_arm(args, wl):
    import torch
    import torch.distributed as dist

    import synth
    from persistent_moe_decode_02_gb300 import mk
    from persistent_moe_decode_02_gb300.roofline import step_bytes
    from synth.device import DeviceModel, PagedKV, initial_tokens, kv_pages_needed

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()

    D = wl.dims
    model = DeviceModel(D, wl.seed)
    e2e_steps = max(3, args.steps // 4)
    total_steps = args.warmup + args.steps + e2e_steps + 2 + (args.steps + args.steps_per_launch
                                                               if args.steps_per_launch > 1 else 0)
    ps = D.page_size
    max_pages = max((c + total_steps + ps) // ps for c in wl.ctx) + 1
    kv = PagedKV(D, kv_pages_needed(D, wl.ctx, total_steps) + 4, max_pages, wl.seed)
    reqs = [kv.admit(rid, c, total_steps) for rid, c in enumerate(wl.ctx)]
    plan = mk.Plan(D, model.weights(), kv.kv, [r.length for r in reqs], kv.page_table(reqs), max_pages,
                   tc_off=args.tc_off)
    B = wl.batch
    tok = torch.tensor(initial_tokens(wl, list(range(B))), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    # warm-up (next token feeds back in place: d_tokens aliases d_next_token)
    for _ in range(args.warmup):
        rc = plan.step(tok, tok)
        assert rc == 0, mk.status_string(rc)
    st = plan.sync()
    assert st == 0, mk.status_string(st)
    ctx_at_start = [r.length + args.warmup for r in reqs]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ev[0].record(stream)
        for i in range(args.steps):
            plan.step(tok, tok)
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
    barrier()
    st = plan.sync()
    assert st == 0, mk.status_string(st)
    per_launch = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    elapsed_ms = max_over_ranks(ev[0].elapsed_time(ev[-1]), world)
    # distinct experts per layer over the whole batch (the experts a step must read)
    ids = torch.zeros(B, D.n_layers, D.top_k, dtype=torch.int32)
    plan.read_debug(mk.MK_DBG_EXPERT_IDS, ids)
    plan.sync()
    union = torch.tensor([len(set(ids[:, l, :].flatten().tolist())) for l in range(D.n_layers)])
    nbytes = 0
    for s in range(args.steps):
        nbytes += step_bytes(D, [c + s for c in ctx_at_start], union_per_layer=union.tolist())["total"]
    bytes_per_launch = nbytes / args.steps
    mean_launch_ms = statistics.mean(per_launch)
    achieved = bytes_per_launch / (mean_launch_ms * 1e-3) / 1e9
    peaks = measured_peaks()
    value = job_tok_s(world, B, args.steps, elapsed_ms * 1e-3)

    # end to end through the host-buffer entry point: H2D tokens, step, D2H next tokens, sync
    # (right after the headline loop, so both see the plan at the same age)
    h_tok = torch.tensor(tok.cpu().tolist(), dtype=torch.int32).pin_memory()
    h_next = torch.empty(B, dtype=torch.int32).pin_memory()
    barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        rc = plan.step_host(h_tok, h_next)
        assert rc == 0, mk.status_string(rc)
        h_tok.copy_(h_next)
    t1 = time.perf_counter()
    e2e_s = max_over_ranks(t1 - t0, world)
    e2e = {"value": job_tok_s(world, B, e2e_steps, e2e_s), "unit": "tok/s", "h2d_bytes_per_step": 4 * B,
           "d2h_bytes_per_step": 4 * B + 16, "steps": e2e_steps}

    tok.copy_(h_tok.cuda())

    # several steps per launch (tokens fed back on the device): the same
    # number of steps, timed the same way
    K = max(1, args.steps_per_launch)
    multi = None
    if K > 1:
        n_launch = max(1, args.steps // K)
        # two row buffers in turn: a launch reads the last row of the other
        rows = [torch.empty(K, B, dtype=torch.int32, device="cuda") for _ in range(2)]
        rows[1][-1].copy_(tok)
        rc = plan.steps(rows[1][-1], K, rows[0])   # warm-up launch
        assert rc == 0, mk.status_string(rc)
        evm = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        barrier()
        torch.cuda.synchronize()
        evm[0].record(stream)
        for i in range(n_launch):
            plan.steps(rows[i % 2][-1], K, rows[(i + 1) % 2])
        evm[1].record(stream)
        torch.cuda.synchronize()
        st = plan.sync()
        assert st == 0, mk.status_string(st)
        ms = max_over_ranks(evm[0].elapsed_time(evm[1]), world)
        multi = {"steps_per_launch": K, "launches": n_launch, "value": job_tok_s(world, B, n_launch * K, ms * 1e-3),
                 "unit": "tok/s", "ms_per_step": ms / (n_launch * K)}
        tok.copy_(rows[n_launch % 2][-1])

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        smp = OracleSample(wl).prepare()
        s = smp.step_seconds()
        cpu = {"value": B / s, "unit": "tok/s", "cores": torch.get_num_threads(), "cpu": cpu_model(),
               "kind": "oracle", "sample": smp.describe() + "; 1 timed step"}
    if rank == 0:
        info = plan.info()
        out = {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
               "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
               "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
               "config": config_of(wl),
               "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
               "weights_gb": round(model.nbytes() / 1e9, 2),
               "sol_pct_of_8tbs": 100.0 * achieved / 8000.0,
               "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": achieved / peaks["hbm_gbs"], "peak_source": peaks["source"],
                            "traffic": ncu_traffic(wl.name), "algorithmic_bytes_per_launch": bytes_per_launch,
                            "kernel": "mk_megakernel", "mean_launch_ms": mean_launch_ms},
               "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps, "multi_step": multi,
               "clocks": clk.summary(), "plan": info, "kernel_hash": kernel_hash()}
        print(json.dumps(out), flush=True)
    plan.close()
    if world > 1:
        dist.destroy_process_group()


def churn_arm(args, wl):
    """Continuous batching inside the timed loop (workloads with churn, e.g.
    batch 32 with 2 requests leaving and 2 joining at 512 tokens every step):
    each timed step is one decode step of the whole batch followed by the
    plan update for the next batch (the leaving requests' pages released, the
    joiners' rows added: host task-list rebuild and upload).  The joiners'
    pages and their synthetic prior K/V are written before the clock starts
    (input preparation, like every other workload's cache)."""
    import torch

    from persistent_moe_decode_02_gb300 import mk
    from persistent_moe_decode_02_gb300.roofline import step_bytes
    from synth.device import DeviceModel, PagedKV, initial_tokens, kv_pages_needed

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    D, B = wl.dims, wl.batch
    leave, jctx = wl.churn_leave, wl.churn_join_ctx
    e2e_steps = max(3, args.steps // 4)
    n_steps = args.warmup + args.steps + e2e_steps
    n_join = leave * n_steps
    ps = D.page_size
    max_pages = max((c + n_steps + ps) // ps for c in wl.ctx + [jctx]) + 1
    model = DeviceModel(D, wl.seed)
    kv = PagedKV(D, kv_pages_needed(D, wl.ctx, n_steps, n_join, jctx) + 4, max_pages, wl.seed)
    live = [kv.admit(rid, c, n_steps + 1) for rid, c in enumerate(wl.ctx)]
    joiners = [kv.admit(B + i, jctx, n_steps + 1) for i in range(n_join)]
    join_tok = torch.tensor(initial_tokens(wl, [r.rid for r in joiners]), dtype=torch.int32, device="cuda")
    plan = mk.Plan(D, model.weights(), kv.kv, [r.length for r in live], kv.page_table(live), max_pages,
                   max_batch=B, tc_off=args.tc_off)
    tok = torch.tensor(initial_tokens(wl, list(range(B))), dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    state = {"j": 0, "lens": []}

    def churn_step(tokens_in, tokens_out):
        rc = plan.step(tokens_in, tokens_out)
        assert rc == 0, mk.status_string(rc)
        state["lens"].append([r.length for r in live])
        for r in live:
            r.length += 1
        del live[:leave]
        j = state["j"]
        live.extend(joiners[j:j + leave])
        state["j"] = j + leave
        # next inputs: the staying requests' outputs, then the joiners' first tokens
        tokens_in[:B - leave].copy_(tokens_out[leave:])
        tokens_in[B - leave:].copy_(join_tok[j:j + leave])
        plan.update([r.length for r in live], kv.page_table(live), max_pages)

    for _ in range(args.warmup):
        churn_step(tok, nxt)
    assert plan.sync() == 0
    state["lens"].clear()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with ClockSampler(0) as clk:
        t0 = time.perf_counter()
        ev[0].record(stream)
        for _ in range(args.steps):
            churn_step(tok, nxt)
        ev[1].record(stream)
        torch.cuda.synchronize()
        wall_s = time.perf_counter() - t0
    st = plan.sync()
    assert st == 0, mk.status_string(st)
    elapsed_ms = ev[0].elapsed_time(ev[1])
    ids = torch.zeros(B, D.n_layers, D.top_k, dtype=torch.int32)
    plan.read_debug(mk.MK_DBG_EXPERT_IDS, ids)
    plan.sync()
    union = [len(set(ids[:, l, :].flatten().tolist())) for l in range(D.n_layers)]
    nbytes = sum(step_bytes(D, lens, union_per_layer=union)["total"] for lens in state["lens"]) / args.steps
    ms = elapsed_ms / args.steps
    achieved = nbytes / (ms * 1e-3) / 1e9
    peaks = measured_peaks()
    # end to end: the same churn loop through the host-buffer entry point
    h_tok = torch.tensor(tok.cpu().tolist(), dtype=torch.int32).pin_memory()
    h_next = torch.empty(B, dtype=torch.int32).pin_memory()
    t1 = time.perf_counter()
    for _ in range(e2e_steps):
        rc = plan.step_host(h_tok, h_next)
        assert rc == 0, mk.status_string(rc)
        for r in live:
            r.length += 1
        del live[:leave]
        j = state["j"]
        live.extend(joiners[j:j + leave])
        state["j"] = j + leave
        h_tok[:B - leave].copy_(h_next[leave:])
        h_tok[B - leave:].copy_(join_tok[j:j + leave].cpu())
        plan.update([r.length for r in live], kv.page_table(live), max_pages)
    e2e_s = time.perf_counter() - t1
    out = {"metric": METRIC, "value": B * args.steps / (elapsed_ms * 1e-3), "unit": "tok/s", "n_gpus": 1,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config_of(wl),
           "churn": {"leave_per_step": leave, "join_per_step": leave, "join_ctx": jctx,
                     "in_timed_loop": "decode step + plan update (host rebuild and upload) every step",
                     "wall_ms_per_step": 1e3 * wall_s / args.steps},
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": achieved / peaks["hbm_gbs"], "peak_source": peaks["source"], "traffic": None,
                        "algorithmic_bytes_per_launch": nbytes, "kernel": "mk_megakernel",
                        "note": "bytes per step from the steps' actual lengths and the last step's expert union; "
                                "the batch runs as 4 launches of 8 requests"},
           "cpu_baseline": None,
           "e2e": {"value": B * e2e_steps / e2e_s, "unit": "tok/s", "h2d_bytes_per_step": 4 * B,
                   "d2h_bytes_per_step": 4 * B + 16, "steps": e2e_steps},
           "gpu_launches": args.steps * ((B + 7) // 8), "clocks": clk.summary(), "kernel_hash": kernel_hash()}
    print(json.dumps(out), flush=True)
    plan.close()


PHASES = ["QKV", "ATTN", "OPROJ", "EXPERT", "REDUCE", "LM", "COMBINE"]


def summarize_timeline(tasks, stamps, step_ms) -> str:
    """Text summary of one traced step: per task kind the mean time spent
    waiting for the dependency, loading activations, consuming stages and
    finishing; the producer's lead; and the per-layer phase windows."""
    import statistics as st

    import torch
    S = stamps.double()
    t0 = S[S > 0].min()
    S = torch.where(S > 0, (S - t0) / 1000.0, torch.zeros_like(S))   # microseconds
    typ, lay = tasks[:, 0], tasks[:, 1]
    out = [f"traced step ms: {', '.join(f'{x:.3f}' for x in step_ms)}; span of last step {float(S.max()):.1f} us"]
    seg = [("wait", 0, 1), ("act", 1, 2), ("stages", 2, 3), ("tail", 3, 4), ("prod_lead", 5, 1),
           ("prod_issue", 5, 6), ("act>stage0", 2, 8), ("stage0>last", 8, 9), ("last>done", 9, 3)]
    out.append("kind      n      " + "  ".join(f"{n:>10s}" for n, _, _ in seg) + "   (us, mean per task)")
    for k, name in enumerate(PHASES):
        m = typ == k
        if int(m.sum()) == 0:
            continue
        vals = [float((S[m, b] - S[m, a]).mean()) for _, a, b in seg]
        out.append(f"{name:8s} {int(m.sum()):6d} " + "  ".join(f"{v:10.2f}" for v in vals))
        mm = m & (S[:, 10] > 0) & (S[:, 11] > 0)
        if S.shape[1] >= 12 and int(mm.sum()) > 0:
            out.append(f"{'':8s} activation steps: dep>mid1 {float((S[mm, 10] - S[mm, 1]).mean()):.2f}  "
                       f"mid1>mid2 {float((S[mm, 11] - S[mm, 10]).mean()):.2f}  "
                       f"mid2>act {float((S[mm, 2] - S[mm, 11]).mean()):.2f}")
    L = int(lay.max()) + 1
    red, lmk = PHASES.index("REDUCE"), PHASES.index("LM")
    ends = [float(S[(typ == red) & (lay == l), 4].max()) for l in range(L)]
    dl = [b - a for a, b in zip(ends, ends[1:])] or [ends[0]]
    out.append(f"per-layer time us: median {st.median(dl):.2f} min {min(dl):.2f} max {max(dl):.2f}")
    l = L // 2
    out.append(f"layer {l} phase windows (us): dependency met first..last | done last | producer first copy")
    for k in range(len(PHASES)):
        m = (typ == k) & (lay == l)
        if k == lmk:
            continue
        if int(m.sum()) == 0:
            continue
        out.append(f"  {PHASES[k]:8s} dep {float(S[m, 1].min()):9.1f}..{float(S[m, 1].max()):9.1f} | done "
                   f"{float(S[m, 4].max()):9.1f} | prod {float(S[m, 5].min()):9.1f}..{float(S[m, 5].max()):9.1f}")
    m = typ == lmk
    out.append(f"LM head: start {float(S[m, 1].min()):.1f} end {float(S[m, 4].max()):.1f}")
    return "\n".join(out)


def timeline_arm(args, wl):
    """Trace a few steps (globaltimer stamps per task) and print the summary."""
    import torch

    from persistent_moe_decode_02_gb300 import mk
    from synth.device import DeviceModel, PagedKV, initial_tokens, kv_pages_needed
    D = wl.dims
    model = DeviceModel(D, wl.seed)
    steps = args.steps
    ps = D.page_size
    max_pages = max((c + steps + 2 + ps) // ps for c in wl.ctx) + 1
    kv = PagedKV(D, kv_pages_needed(D, wl.ctx, steps + 2) + 4, max_pages, wl.seed)
    reqs = [kv.admit(i, c, steps + 2) for i, c in enumerate(wl.ctx)]
    plan = mk.Plan(D, model.weights(), kv.kv, [r.length for r in reqs], kv.page_table(reqs), max_pages,
                   trace=2 if args.stage_trace else 1)
    tok = torch.tensor(initial_tokens(wl, list(range(wl.batch))), dtype=torch.int32, device="cuda")
    times = []
    for _ in range(steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        rc = plan.step(tok, tok)
        e1.record()
        torch.cuda.synchronize()
        assert rc == 0 and plan.sync() == 0
        times.append(e0.elapsed_time(e1))
    tasks, stamps = plan.timeline()
    text = summarize_timeline(tasks, stamps, times)
    head = f"workload {wl.name}: {wl.dims}; batch {wl.batch}; plan {plan.info()}; kernel {kernel_hash()}"
    print(head + "\n" + text, flush=True)
    if args.timeline != "-":
        with open(args.timeline, "w") as f:
            f.write(head + "\n" + text + "\n")
        extra = {"stages": plan.stage_timeline()} if args.stage_trace else {}
        torch.save({"tasks": tasks, "stamps": stamps, "times": times, **extra}, args.timeline + ".pt")
    plan.close()


def serve_arm(args, wl):
    """The continuous-batching loop (mk_serve_step) on the workload's model:
    a seeded stream of requests (prompt and output lengths log-uniform), half
    queued at the start and the rest after a quarter of the expected steps,
    prompts fed through decode steps into an empty cache.  Prints one JSON
    line: tokens through the model per second of wall time, and per step the
    wall time and the stream time of the same calls (CUDA events around each
    mk_serve_step; the difference is host time the GPU does not overlap)."""
    import torch

    import synth
    from persistent_moe_decode_02_gb300 import mk
    from synth.device import DeviceModel
    D = wl.dims
    cap = args.serve_batch
    n_req = 4 * cap
    plen = synth.log_uniform_lengths(n_req, 16, 256, wl.seed, "serve prompt")
    olen = synth.log_uniform_lengths(n_req, 16, 128, wl.seed, "serve output")
    ps = D.page_size
    max_pages = (256 + 128 + ps - 1) // ps
    num_pages = cap * max_pages
    shape = (num_pages, D.n_kv_heads, 2, D.head_dim, ps)
    model = DeviceModel(D, wl.seed)
    kv = [torch.zeros(shape, dtype=torch.bfloat16, device="cuda") for _ in range(D.n_layers)]
    toks = synth.uniform_ints(int(sum(plen)), D.vocab, wl.seed, "serve tokens").tolist()
    prompts, o = [], 0
    for n in plen:
        prompts.append(toks[o:o + n])
        o += n
    srv = mk.Server(D, model.weights(), kv, max_batch=cap, max_pages=max_pages)
    half = n_req // 2
    for i in range(half):
        srv.submit(i, prompts[i], olen[i])
    expected = sum(p + m - 1 for p, m in zip(plen, olen)) // cap
    stream = torch.cuda.current_stream()
    steps, tokens, gpu_ms, wall, rest = 0, 0, 0.0, 0.0, False
    torch.cuda.synchronize()
    while True:
        if not rest and steps >= expected // 4:
            for i in range(half, n_req):
                srv.submit(i, prompts[i], olen[i])
            rest = True
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(stream)
        b = srv.step(stream)
        e1.record(stream)
        e1.synchronize()
        wall += time.perf_counter() - t0
        if b == 0:
            if rest:
                break
            for i in range(half, n_req):   # the first half finished early: queue the rest now
                srv.submit(i, prompts[i], olen[i])
            rest = True
            continue
        gpu_ms += e0.elapsed_time(e1)
        steps += 1
        tokens += b
    st = srv.sched.stats()
    assert st["retired"] == n_req and st["free_pages"] == num_pages, st
    gen = int(sum(olen))
    out = {"metric": "serving loop tokens/s (prompt and output tokens through the model, wall time)",
           "value": tokens / wall, "unit": "tok/s", "generated_tok_s": gen / wall, "requests": n_req,
           "max_batch": cap, "steps": steps, "ms_per_step_wall": 1e3 * wall / steps,
           "ms_per_step_stream": gpu_ms / steps, "mean_batch": tokens / steps,
           "config": {"workload": wl.name, "layers": D.n_layers, "prompt_tokens": "16-256 log-uniform",
                      "output_tokens": "16-128 log-uniform", "weights": "bf16 random-init", "data": "synthetic"}}
    print(json.dumps(out))
    srv.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="full_bs1_8k")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tc-off", action="store_true",
                    help="expert gate/up and projections of batches 3-8 on the CUDA cores instead of the tensor cores")
    ap.add_argument("--steps-per-launch", type=int, default=8,
                    help="also time this many decode steps per launch (tokens fed back on the device); 1: off")
    ap.add_argument("--timeline", default=None,
                    help="trace --steps steps per task and write a summary to this path ('-': print only)")
    ap.add_argument("--stage-trace", action="store_true",
                    help="with --timeline: also record every ring stage (saved beside the summary)")
    ap.add_argument("--serve", action="store_true",
                    help="time the continuous-batching loop (mk_serve_step) on the workload's model")
    ap.add_argument("--serve-batch", type=int, default=8)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    import synth
    wl = synth.workload(args.workload)
    if args.timeline:
        import __graft_entry__
        __graft_entry__.build()
        timeline_arm(args, wl)
    elif args.serve:
        import __graft_entry__
        __graft_entry__.build()
        serve_arm(args, wl)
    elif args.impl == "reference":
        reference_arm(args, wl)
    elif wl.churn_leave > 0:
        import __graft_entry__
        __graft_entry__.build()
        churn_arm(args, wl)
    else:
        import __graft_entry__
        __graft_entry__.build()
        our_arm(args, wl)


if __name__ == "__main__":
    main()
