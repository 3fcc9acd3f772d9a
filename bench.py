"""Benchmark of the exact greedy verify step on GB300.

One step = one spec_verify_step (k = 15, 16 rows) of the full synthetic target:
52 Q4_K blocks at hidden 6656 (QKV 6656->7680, O 6656->6656, gate|up
6656->2x17920, down 17920->6656), LM head 6656->131072, KV context 2048 bf16,
argmax, accept and KV rollback — followed by a metadata rollback to the same
context so every timed step sees the same depth.  Weights (13.75 GB) are far
larger than L2, so nothing is served from cache between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  --impl reference times the CPU oracle on a bounded
sample of the same step on the host cores (the oracle is the only reference
this method has).  With N > 1 (torchrun) each rank runs an independent replica
(the step has no exchange); the whole-job value sums them and timing is the
max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify steps/s and weight GB/s (% of GB300 HBM roofline) at k+1=16 rows"
CTX = 2048
K_DRAFT = 15
ROWS = K_DRAFT + 1


def full_cfg():
    from speculative_decoding_exact_gb300 import runtime, synth
    return runtime.ModelConfig(**synth.FULL)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def max_over_ranks(x, world, device):
    """The max of x over the ranks of the job (x itself at world 1): the job's
    time is its slowest rank's."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as tdist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_steps_per_s(ms_max, steps, world):
    """Whole-job verify steps/s: every rank runs `steps` steps of its own
    replica within the slowest rank's `ms_max` milliseconds."""
    return steps * world * 1000.0 / ms_max


def gemm_algorithmic_bytes(cfg):
    """Per step: weights N*K*0.5625 + fp32 inputs M*K*4 + fp32 outputs M*N*4 of every GEMM."""
    tot = 0
    launches = 0
    mats = [(N, K) for _, N, K in cfg.matrices()] * cfg.n_layers + [(cfg.vocab, cfg.hidden)]
    for N, K in mats:
        tot += N * (K // 256) * 144 + ROWS * K * 4 + ROWS * N * 4
        launches += 1
    return tot, launches


def kv_read_bytes(cfg, ctx):
    return cfg.n_layers * 2 * cfg.n_kv_heads * cfg.head_dim * 2 * (ctx + ROWS)


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class Clocks:
    """nvidia-smi sampling every 50 ms; only the samples whose timestamps fall
    inside the timed window [mark_start, mark_stop] are reported (the nearest
    ones if the window is shorter than the sampling period)."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
            return
        # wait (up to 10 s) for the first sample so that the window is covered
        for _ in range(200):
            if os.path.getsize(self.f.name) > 0:
                break
            time.sleep(0.05)

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    @staticmethod
    def _ts(x):
        import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(x.strip(), fmt).timestamp()
            except ValueError:
                continue
        return None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        samples = []
        for r in rows:
            r = [x.strip() for x in r]
            try:
                samples.append((self._ts(r[0]), float(r[2]), float(r[3]), r[6:10]))
            except (ValueError, IndexError):
                continue
        inside = [x for x in samples
                  if x[0] is not None and self.t0 is not None and self.t0 <= x[0] <= self.t1]
        if not inside and samples and self.t0 is not None:
            mid = 0.5 * (self.t0 + (self.t1 or self.t0))
            timed = [x for x in samples if x[0] is not None]
            inside = sorted(timed, key=lambda x: abs(x[0] - mid))[:2] if timed else samples[-2:]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for x in inside:
            for nm, v in zip(names, x[3]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(nm)
        sm = [x[1] for x in inside]
        mx = [x[2] for x in inside]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "window_s": (self.t1 - self.t0) if self.t0 and self.t1 else None,
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# CPU oracle sample (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------
class OracleSample:
    """A bounded sample of the same step through the oracle on one host core:
    1/COLF of the columns of each block GEMM of one layer (16 rows, full K),
    the layer's full attention at context 2048, 1/HEADF of the head columns.
    Extrapolated: step = 52 * (COLF * t_gemms + t_attn) + HEADF * t_head."""
    COLF, HEADF = 16, 128

    def __init__(self, cfg):
        import oracle
        from speculative_decoding_exact_gb300 import synth
        self.oracle, self.cfg = oracle, cfg
        H = cfg.hidden
        self.mats = []
        for j, (name, N, K) in enumerate(cfg.matrices()):
            n = N // self.COLF
            self.mats.append((synth.q4k_matrix(n, K, 0, 1000 * 0 + j), n, K))
        self.head = synth.q4k_matrix(cfg.vocab // self.HEADF, H, 0, 999999)
        self.x_h = synth.normal((ROWS, H), 0, 5)
        self.x_f = synth.normal((ROWS, cfg.ffn), 0, 6)
        ocfg = oracle.Config(hidden=H, n_layers=1, n_q_heads=cfg.n_q_heads, n_kv_heads=cfg.n_kv_heads,
                             head_dim=cfg.head_dim, ffn=cfg.ffn, vocab=cfg.vocab)
        self.kv = oracle.KV(ocfg, (CTX + ROWS) // 16 + 1, (CTX + ROWS) // 16 + 1)
        self.kv.extend(CTX + ROWS)
        nkv = cfg.n_kv_heads * cfg.head_dim
        kb = synth.bf16_bits(synth.normal((CTX + ROWS, nkv), 0, 7))
        vb = synth.bf16_bits(synth.normal((CTX + ROWS, nkv), 0, 8))
        for p in range(CTX + ROWS):
            pg, sl = self.kv.page_table[p // 16], p % 16
            self.kv.pool[pg, 0, 0, :, sl] = kb[p].reshape(cfg.n_kv_heads, cfg.head_dim)
            self.kv.pool[pg, 0, 1, :, sl] = vb[p].reshape(cfg.n_kv_heads, cfg.head_dim)
        self.q = synth.normal((ROWS, cfg.n_q_heads, cfg.head_dim), 0, 9)

    def run(self):
        o, t = self.oracle, time.perf_counter
        t0 = t()
        xn = o.rmsnorm(self.x_h, None, 1e-6)
        for W, n, K in self.mats:
            o.linear(W, n, K, xn if K == self.cfg.hidden else self.x_f)
        t1 = t()
        self.kv.attention(0, self.q, CTX)
        t2 = t()
        o.linear(self.head, self.cfg.vocab // self.HEADF, self.cfg.hidden, xn)
        t3 = t()
        step_s = self.cfg.n_layers * (self.COLF * (t1 - t0) + (t2 - t1)) + self.HEADF * (t3 - t2)
        return step_s, t3 - t0

    def describe(self):
        return (f"oracle on 1 host core: one layer's block GEMMs on 1/{self.COLF} of their columns "
                f"(16 rows, full K), that layer's attention at context {CTX}, 1/{self.HEADF} of the "
                f"LM-head columns; extrapolated x52 layers, x{self.COLF} columns, x{self.HEADF} head")


def host_cpu():
    """The host the oracle runs on: architecture, logical CPUs, and the CPU
    model from /proc/cpuinfo (x86: "model name"; Arm: implementer and part
    codes, e.g. 0x41 / 0xd4f for a Neoverse V2)."""
    import platform
    info = {"machine": platform.machine(), "nproc": os.cpu_count()}
    try:
        fields = {}
        for line in open("/proc/cpuinfo"):
            k, _, v = line.partition(":")
            fields.setdefault(k.strip(), v.strip())
        if "model name" in fields:
            info["model"] = fields["model name"]
        elif "CPU part" in fields:
            info["model"] = f"implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    except OSError:
        pass
    return info


def cpu_baseline(cfg, min_seconds=10.0):
    s = OracleSample(cfg)
    times, spent = [], 0.0
    while spent < min_seconds:
        step_s, wall = s.run()
        times.append(step_s)
        spent += wall
    return {"value": 1.0 / statistics.median(times), "unit": "verify steps/s", "cores": 1,
            "kind": "oracle", "sample": s.describe() + f"; {len(times)} samples", "host": host_cpu()}


def run_reference(args, rank, world):
    cfg = full_cfg()
    if rank != 0:
        return
    s = OracleSample(cfg)
    for _ in range(args.warmup):
        s.run()
    steps = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        steps.append(s.run()[0])
    wall = time.perf_counter() - t0
    v = 1.0 / statistics.mean(steps)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "verify steps/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 / v, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8xint4 dot, f32 combine", "data": "synthetic",
            "config": workload_config(cfg),
            "cpu_baseline": {"value": v, "unit": "verify steps/s", "cores": 1, "kind": "oracle",
                             "sample": s.describe(), "host": host_cpu()},
            "e2e": {"value": v, "unit": "verify steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "sample_wall_s": wall}
    print(json.dumps(line), flush=True)


def workload_config(cfg):
    return {"workload": f"full synthetic verify pass: 52 Q4_K blocks hidden 6656 + LM head 131072, "
                        f"k+1=16 rows, KV context {CTX} bf16",
            "layers": cfg.n_layers, "hidden": cfg.hidden, "ffn": cfg.ffn, "vocab": cfg.vocab,
            "q_heads": cfg.n_q_heads, "kv_heads": cfg.n_kv_heads, "rows": ROWS, "context": CTX,
            "weight_bytes": cfg.weight_bytes(),
            "l2": "inputs larger than L2 (13.75 GB of weights streamed per step)",
            "parallelism": "replicas"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def kernel_source_sha():
    h = hashlib.sha256()
    for f in ("gemm.cu", "common.cuh", "gemm_plan.h"):
        h.update(open(os.path.join(ROOT, "speculative_decoding_exact_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(cfg):
    """DRAM bytes (read + write) per GEMM launch of a step, averaged over the
    step's launches, from the committed per-shape ncu captures; None if the
    kernel changed since the capture or a shape of the step was not captured."""
    p = os.path.join(ROOT, "profiles", "gemm_q4k_ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    sha, shapes = None, {}
    for line in open(p):
        if line.startswith("kernel_source_sha:"):
            sha = line.split(":", 1)[1].strip()
        elif line.startswith("shape "):
            name, rest = line[len("shape "):].split(":", 1)
            f = rest.split()
            shapes[name.strip()] = int(f[0]) + int(f[1])
    if sha != kernel_source_sha():
        return None
    mats = [(N, K) for _, N, K in cfg.matrices()] * cfg.n_layers + [(cfg.vocab, cfg.hidden)]
    try:
        return sum(shapes[f"{N}x{K}"] for N, K in mats) / len(mats)
    except KeyError:
        return None


def setup_model(rank):
    """The full synthetic model on this rank's GPU: random Q4_K weights of the
    52-block architecture + head, a paged KV filled to CTX with random bf16,
    16 hidden rows and 15 draft tokens.  Returns a namespace of the pieces."""
    import types

    import torch

    from speculative_decoding_exact_gb300 import runtime, synth
    from speculative_decoding_exact_gb300 import build as b

    b.build()
    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    cfg = full_cfg()
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    max_ctx = CTX + 64
    ctx = runtime.Context(cfg, max_ctx=max_ctx, stream=stream)
    pages = max_ctx // 16
    t_setup = time.perf_counter()
    dw = runtime.DeviceWeights(cfg)
    for l in range(cfg.n_layers):
        for j, (name, N, K) in enumerate(cfg.matrices()):
            getattr(dw, name).append(runtime.upload_tiled(ctx, synth.q4k_matrix(N, K, rank, 1000 * l + j),
                                                          N, K))
    dw.w_head = runtime.upload_tiled(ctx, synth.q4k_matrix(cfg.vocab, cfg.hidden, rank, 999999),
                                     cfg.vocab, cfg.hidden)
    kv = runtime.DeviceKV(cfg, pages, pages)
    kv.reset(ctx)
    kv.extend(ctx, CTX)
    g = torch.Generator(device="cuda").manual_seed(1234 + rank)
    with torch.cuda.stream(stream):
        kv.pool.copy_(torch.randn(kv.pool.shape, generator=g, device="cuda").to(torch.bfloat16))
    hidden = torch.from_numpy(synth.normal((ROWS, cfg.hidden), rank, 5)).cuda()
    draft = torch.from_numpy(synth.tokens(K_DRAFT, cfg.vocab, rank, 6)).cuda()
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    return types.SimpleNamespace(cfg=cfg, ctx=ctx, stream=stream, dw=dw, kv=kv, hidden=hidden, draft=draft,
                                 res=res, ws=dw.struct(), ks=kv.struct(), local=local,
                                 setup_s=time.perf_counter() - t_setup)


def run_gpu(args, rank, world):
    import torch

    from speculative_decoding_exact_gb300 import abi, runtime, synth
    from speculative_decoding_exact_gb300 import build as b

    mdl = setup_model(rank)
    cfg, ctx, stream, local = mdl.cfg, mdl.ctx, mdl.stream, mdl.local
    hidden, draft, res, ws, ks = mdl.hidden, mdl.draft, mdl.res, mdl.ws, mdl.ks
    setup_s = mdl.setup_s

    def step():
        rc = abi.spec_verify_step(ctx.h, ws, ks, hidden.data_ptr(), draft.data_ptr(), K_DRAFT,
                                  res.data_ptr())
        if rc != 0:
            raise abi.SpecError("spec_verify_step", rc)
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, ks, CTX))

    clocks = Clocks(local)
    clocks.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    r = res.cpu().numpy()
    assert r[2] == 0, f"step status {r[2]}"
    launches = abi.spec_last_step_launches(ctx.h) + 1

    dist = world > 1
    if dist:
        import torch.distributed as tdist
    if dist:
        tdist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed")
    clocks.mark_start()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.mark_stop()
    torch.cuda.nvtx.range_pop()
    if dist:
        tdist.barrier()
    ms = e0.elapsed_time(e1)
    clk = clocks.stop()
    ms = max_over_ranks(ms, world, "cuda")
    ms_per_step = ms / args.steps
    steps_per_s = job_steps_per_s(ms, args.steps, world)

    # per-step distribution: a separate pass of the same steps with an event
    # after each one (kept out of the timed region above, whose consecutive
    # steps overlap through programmatic dependent launch)
    step_ms = step_time_stats(torch, stream, step, args.steps)

    # GEMM kernel timing: CUDA events around every GEMM launch of the same steps
    gemm_ms, gemm_launches = profile_gemms(ctx, abi, torch, stream, ws, ks, hidden, draft, res,
                                           args.steps)
    gbytes, glaunch = gemm_algorithmic_bytes(cfg)
    peak, peak_kind = measured_peaks()
    achieved = gbytes / (gemm_ms * 1e-3) / 1e9 if gemm_ms else None
    traffic = committed_traffic(cfg)

    # end to end through the host-buffer entry point
    hid_h = torch.from_numpy(synth.normal((ROWS, cfg.hidden), rank, 5)).pin_memory()
    dr_h = torch.from_numpy(synth.tokens(K_DRAFT, cfg.vocab, rank, 6)).pin_memory()
    res_h = abi.spec_result()
    for _ in range(2):
        abi.check("spec_verify_step_host", abi.spec_verify_step_host(ctx.h, ws, ks, hid_h.data_ptr(),
                                                                     dr_h.data_ptr(), K_DRAFT, res_h))
        abi.spec_kv_rollback(ctx.h, ks, CTX)
    torch.cuda.synchronize()
    if dist:
        tdist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        abi.check("spec_verify_step_host", abi.spec_verify_step_host(ctx.h, ws, ks, hid_h.data_ptr(),
                                                                     dr_h.data_ptr(), K_DRAFT, res_h))
        abi.spec_kv_rollback(ctx.h, ks, CTX)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, "cuda")
    e2e = job_steps_per_s(e2e_s * 1000.0, args.steps, world)

    if rank != 0:
        ctx.close()
        return
    wb = cfg.weight_bytes()
    line = {
        "metric": METRIC, "value": steps_per_s, "unit": "verify steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8xuint4 dot (exact integers on e4m3 tcgen05 MMAs), f32 combine, bf16 KV", "data": "synthetic",
        "config": workload_config(cfg),
        "weight_gbs": wb * steps_per_s / world / 1e9,
        "weight_frac_of_hbm": {"measured": wb * steps_per_s / world / 1e9 / peak, "peak_gbs": peak,
                               "spec_8tbs": wb * steps_per_s / world / 1e9 / 8000.0},
        "total_gbs": (wb + kv_read_bytes(cfg, CTX)) * steps_per_s / world / 1e9,
        "roofline": {"kernel": "gemm_q4k_kernel (all Q4_K GEMM launches of a step)",
                     "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": (achieved / peak) if achieved else None, "peak_kind": peak_kind,
                     "traffic": traffic, "launches_per_step": glaunch,
                     "avg_launch_us": gemm_ms * 1e3 / glaunch if gemm_ms else None,
                     "algorithmic_bytes_per_launch": gbytes / glaunch},
        "cpu_baseline": cpu_baseline(cfg) if world == 1 or rank == 0 else None,
        "e2e": {"value": e2e, "unit": "verify steps/s",
                "h2d_bytes_per_step": ROWS * cfg.hidden * 4 + K_DRAFT * 4,
                "d2h_bytes_per_step": 16},
        "gpu_launches": launches * args.steps,
        "clocks": clk,
        "step_ms": step_ms,
        "setup_s": setup_s,
        "accepted_len_last": int(r[0]),
    }
    print(json.dumps(line), flush=True)
    ctx.close()


def step_time_stats(torch, stream, step, steps):
    """Median and 95th percentile of single-step times: `steps` more steps,
    a CUDA event on the step's stream after each one."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(steps):
        step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    t = sorted(ev[i].elapsed_time(ev[i + 1]) for i in range(steps))
    p95 = t[min(len(t) - 1, int(math.ceil(0.95 * len(t))) - 1)]
    return {"median": statistics.median(t), "p95": p95, "min": t[0], "max": t[-1], "steps": steps,
            "pass": "separate, an event after every step"}


def profile_gemms(ctx, abi, torch, stream, ws, ks, hidden, draft, res, steps):
    """Same steps with CUDA events recorded around each GEMM launch on the ctx
    stream; returns (total GEMM ms per step, GEMM launches per step)."""
    abi.check("spec_profile_gemms", abi.spec_profile_gemms(ctx.h, 1))
    tot, n = 0.0, 0
    for _ in range(steps):
        abi.check("spec_verify_step", abi.spec_verify_step(ctx.h, ws, ks, hidden.data_ptr(),
                                                           draft.data_ptr(), K_DRAFT, res.data_ptr()))
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, ks, CTX))
        ms, n = abi.spec_profile_read(ctx.h)
        tot += ms
    abi.check("spec_profile_gemms", abi.spec_profile_gemms(ctx.h, 0))
    return tot / steps, n


def run_gemm_shape(args):
    """Time one Q4_K GEMM shape (16 rows, synthetic weights) through
    spec_gemm_q4k; a small device footprint, used as the ncu capture target."""
    import torch

    from speculative_decoding_exact_gb300 import abi, runtime, synth
    from speculative_decoding_exact_gb300 import build as b

    b.build()
    N, K = (int(v) for v in args.gemm_shape.lower().split("x"))
    ctx = runtime.Context(runtime.ModelConfig(**synth.FULL), max_ctx=2112)
    W = runtime.upload_tiled(ctx, synth.q4k_matrix(N, K, 7, N + K), N, K)
    x = torch.from_numpy(synth.normal((16, K), 7, 16)).cuda()
    y = torch.zeros((16, N), dtype=torch.float32, device="cuda")

    def call():
        abi.check("spec_gemm_q4k", abi.spec_gemm_q4k(ctx.h, W.data_ptr(), N, K, x.data_ptr(), 16,
                                                     y.data_ptr()))

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / args.steps
    wbytes = N * (K // 256) * 144
    print(json.dumps({"metric": "q4k gemm weight GB/s (16 rows, quantise + GEMM + piece sum)",
                      "value": wbytes / us / 1e3, "unit": "GB/s", "us_per_call": us,
                      "shape": {"N": N, "K": K, "rows": 16}, "weight_bytes": wbytes,
                      "l2": "weights resident from the previous call when smaller than L2"}))
    ctx.close()


def _time_steps(torch, stream, step, warmup, steps):
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_sampled(args):
    """The verify step with the sampled decision (Ch. 33 §33.2) on the full
    model at context --ctx: q = the draft's distributions (softmax of random
    logits, 15 x V, on the device), the MT19937 state on the device.  One JSON
    line with steps/s next to the greedy step's, timed the same way."""
    import torch

    from speculative_decoding_exact_gb300 import abi

    mdl = setup_model(0)
    cfg, ctx, stream = mdl.cfg, mdl.ctx, mdl.stream
    g = torch.Generator(device="cuda").manual_seed(77)
    q = torch.softmax(torch.randn((K_DRAFT, cfg.vocab), generator=g, device="cuda") * 3.0, dim=1).contiguous()
    st = np.zeros(abi.MT_WORDS, dtype=np.uint32)
    abi.check("spec_mt_seed", abi.spec_mt_seed(st.ctypes.data, 5489))
    mt = torch.from_numpy(st.view(np.int32).copy()).cuda()
    hist = torch.zeros((args.steps, 4), dtype=torch.int32, device="cuda")
    it = [0]

    def sampled():
        abi.check("spec_verify_step_sampled",
                  abi.spec_verify_step_sampled(ctx.h, mdl.ws, mdl.ks, mdl.hidden.data_ptr(), mdl.draft.data_ptr(),
                                               q.data_ptr(), K_DRAFT, mt.data_ptr(), mdl.res.data_ptr(), None))
        hist[it[0] % args.steps].copy_(mdl.res)
        it[0] += 1
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, mdl.ks, CTX))

    def greedy():
        abi.check("spec_verify_step", abi.spec_verify_step(ctx.h, mdl.ws, mdl.ks, mdl.hidden.data_ptr(),
                                                           mdl.draft.data_ptr(), K_DRAFT, mdl.res.data_ptr()))
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, mdl.ks, CTX))

    ms_s = _time_steps(torch, stream, sampled, args.warmup, args.steps)
    h = hist.cpu().numpy()
    assert np.all(h[:, 2] == 0), "sampled step status"
    ms_g = _time_steps(torch, stream, greedy, args.warmup, args.steps)
    print(json.dumps({"metric": "verify steps/s, sampled acceptance (Ch. 33 section 33.2)",
                      "value": 1000.0 / ms_s, "unit": "verify steps/s", "ms_per_step": ms_s,
                      "greedy_steps_per_s": 1000.0 / ms_g, "sampled_overhead_us": (ms_s - ms_g) * 1e3,
                      "mean_accepted": float(h[:, 0].mean()), "steps": args.steps, "warmup": args.warmup,
                      "config": dict(workload_config(cfg), draft_q="softmax(3 N(0,1)) per position",
                                     rng="MT19937 seed 5489 on the device")}), flush=True)
    ctx.close()


def run_accept_profile(args):
    """Verify steps at context --ctx with drafts planted so that the accepted
    length L follows a target mean (each position accepted with probability
    a, a solved from E[min(Geom, 15)] = mean), plus an all-accepted run; one
    JSON line per profile with steps/s and accepted tokens/s = steps/s x
    mean(L + 1), next to the draft front projection (Q4_K 33,280 -> 6,656)
    timed at M = round(mean L) + 1 and M = 16."""
    import torch

    from speculative_decoding_exact_gb300 import abi, runtime, synth

    mdl = setup_model(0)
    cfg, ctx, stream = mdl.cfg, mdl.ctx, mdl.stream
    V = cfg.vocab
    # the target argmax of every row (the same every step: fixed rows, rolled-back KV)
    am = torch.zeros(ROWS, dtype=torch.int32, device="cuda")
    taps = abi.spec_taps(None, am.data_ptr(), None)
    abi.check("spec_verify_step_ex", abi.spec_verify_step_ex(ctx.h, mdl.ws, mdl.ks, mdl.hidden.data_ptr(),
                                                             mdl.draft.data_ptr(), K_DRAFT, mdl.res.data_ptr(),
                                                             taps))
    abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, mdl.ks, CTX))
    torch.cuda.synchronize()
    idx = am.cpu().numpy()

    def alpha_for(mean):
        lo, hi = 0.0, 1.0
        for _ in range(60):
            a = 0.5 * (lo + hi)
            e = sum(a ** i for i in range(1, K_DRAFT + 1))
            lo, hi = (a, hi) if e < mean else (lo, a)
        return 0.5 * (lo + hi)

    fc_N, fc_K = cfg.hidden, 5 * cfg.hidden
    Wfc = runtime.upload_tiled(ctx, synth.q4k_matrix(fc_N, fc_K, 3, 4242), fc_N, fc_K)
    xfc = torch.from_numpy(synth.normal((16, fc_K), 3, 17)).cuda()
    yfc = torch.zeros((16, fc_N), dtype=torch.float32, device="cuda")

    def fc_us(M):
        def call():
            abi.check("spec_gemm_q4k", abi.spec_gemm_q4k(ctx.h, Wfc.data_ptr(), fc_N, fc_K, xfc.data_ptr(), M,
                                                         yfc.data_ptr()))
        return _time_steps(torch, stream, call, 3, 20) * 1e3

    rng = np.random.default_rng(5)
    for mean in (1.0, 4.0, 12.0, float(K_DRAFT)):
        a = alpha_for(mean) if mean < K_DRAFT else 1.0
        Ls = np.zeros(args.steps, dtype=np.int32)
        drafts = np.zeros((args.steps, K_DRAFT), dtype=np.int32)
        for t in range(args.steps):
            L = 0
            while L < K_DRAFT and rng.random() < a:
                L += 1
            Ls[t] = L
            d = rng.integers(0, V, K_DRAFT).astype(np.int32)
            d[:L] = idx[:L]
            if L < K_DRAFT:
                d[L] = (idx[L] + 1) % V
            drafts[t] = d
        dd = torch.from_numpy(drafts).cuda()
        hist = torch.zeros((args.steps, 4), dtype=torch.int32, device="cuda")
        it = [0]

        def step():
            t = it[0] % args.steps
            mdl.draft.copy_(dd[t])
            abi.check("spec_verify_step", abi.spec_verify_step(ctx.h, mdl.ws, mdl.ks, mdl.hidden.data_ptr(),
                                                               mdl.draft.data_ptr(), K_DRAFT, mdl.res.data_ptr()))
            hist[t].copy_(mdl.res)
            it[0] += 1
            abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, mdl.ks, CTX))

        it[0] = 0
        ms = _time_steps(torch, stream, step, 0, args.steps)
        h = hist.cpu().numpy()
        assert np.all(h[:, 2] == 0) and np.array_equal(h[:, 0], Ls), "planted accepted lengths"
        sps = 1000.0 / ms
        m_acc = float(h[:, 0].mean())
        print(json.dumps({"metric": "accepted tokens/s at k+1=16 rows (verify steps/s x mean(L+1))",
                          "value": sps * (m_acc + 1.0), "unit": "tokens/s", "steps_per_s": sps,
                          "target_mean_accepted": mean, "mean_accepted": m_acc, "steps": args.steps,
                          "fc_front_projection_us": {"M": int(round(m_acc)) + 1,
                                                     "us": fc_us(int(round(m_acc)) + 1), "M16_us": fc_us(16)},
                          "config": dict(workload_config(cfg), acceptance=f"per-position {a:.4f}")}),
              flush=True)
    ctx.close()


def run_sweep(args):
    """Projection sweep: Q4_K 6656->6656 and 6656->26624 at M in {1, 2, 4, 8,
    16} rows through spec_gemm_q4k (quantise + GEMM + ordered piece sum), a
    bandwidth test of the skinny dequant-GEMM.  The weights rotate over >= 2 GB
    of distinct device copies (82 of the small matrix, 21 of the large), so no
    call finds its weights in the 129 MB L2.  One JSON line per (shape, M):
    weight GB/s, us per call, fraction of the measured copy bandwidth."""
    import torch

    from speculative_decoding_exact_gb300 import abi, runtime, synth
    from speculative_decoding_exact_gb300 import build as b

    b.build()
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    ctx = runtime.Context(runtime.ModelConfig(**synth.FULL), max_ctx=2112, stream=stream)
    peak, peak_kind = measured_peaks()
    K = 6656
    for N in (6656, 26624):
        wbytes = N * (K // 256) * 144
        ncopies = max(2, -(-2 * 10**9 // wbytes))
        W0 = runtime.upload_tiled(ctx, synth.q4k_matrix(N, K, 7, N), N, K)
        copies = [W0] + [W0.clone() for _ in range(ncopies - 1)]
        x = torch.from_numpy(synth.normal((16, K), 7, 16)).cuda()
        y = torch.zeros((16, N), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        for M in (1, 2, 4, 8, 16):
            it = [0]

            def call():
                W = copies[it[0] % ncopies]
                it[0] += 1
                abi.check("spec_gemm_q4k", abi.spec_gemm_q4k(ctx.h, W.data_ptr(), N, K, x.data_ptr(), M,
                                                             y.data_ptr()))

            calls = max(args.steps, 2 * ncopies)
            ms = _time_steps(torch, stream, call, max(args.warmup, 3), calls)
            us = ms * 1e3
            alg = wbytes + M * K * 4 + M * N * 4
            gbs = wbytes / us / 1e3
            print(json.dumps({"metric": "Q4_K projection weight GB/s (quantise + GEMM + piece sum)",
                              "value": gbs, "unit": "GB/s", "us_per_call": us,
                              "algorithmic_gbs": alg / us / 1e3,
                              "roofline": {"bound": "hbm", "achieved": alg / us / 1e3, "peak": peak,
                                           "unit": "GB/s", "frac": alg / us / 1e3 / peak,
                                           "peak_kind": peak_kind},
                              "frac_of_8tbs": gbs / 8000.0,
                              "shape": {"N": N, "K": K, "rows": M}, "weight_bytes": wbytes,
                              "calls": calls, "warmup": max(args.warmup, 3),
                              "config": {"workload": f"projection sweep {K}->{N}, {M} rows",
                                         "l2": f"weights rotated over {ncopies} device copies "
                                               f"({ncopies * wbytes / 1e9:.2f} GB) so L2 serves no repeat"}}),
                  flush=True)
        del copies, W0
        torch.cuda.empty_cache()
    ctx.close()


def run_cudacore(args):
    """The tensor-core GEMM against the CUDA-core (dp4a) one on one Q4_K
    shape (--cudacore NxK), 16 rows, weights rotated over >= 2 GB of device
    copies; one JSON line with both weight GB/s."""
    import torch

    from speculative_decoding_exact_gb300 import abi, runtime, synth
    from speculative_decoding_exact_gb300 import build as b

    b.build()
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    ctx = runtime.Context(runtime.ModelConfig(**synth.FULL), max_ctx=2112, stream=stream)
    N, K = (int(v) for v in args.cudacore.lower().split("x"))
    wbytes = N * (K // 256) * 144
    ncopies = max(2, -(-2 * 10**9 // wbytes))
    W0 = runtime.upload_tiled(ctx, synth.q4k_matrix(N, K, 7, N), N, K)
    copies = [W0] + [W0.clone() for _ in range(ncopies - 1)]
    x = torch.from_numpy(synth.normal((16, K), 7, 16)).cuda()
    y = torch.zeros((16, N), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    out = {}
    for name, fn in (("tensor_core", abi.spec_gemm_q4k), ("cuda_core_dp4a", abi.spec_gemm_q4k_cudacore)):
        it = [0]

        def call():
            W = copies[it[0] % ncopies]
            it[0] += 1
            abi.check(name, fn(ctx.h, W.data_ptr(), N, K, x.data_ptr(), 16, y.data_ptr()))

        ms = _time_steps(torch, stream, call, max(args.warmup, 3), max(args.steps, 2 * ncopies))
        out[name] = {"us_per_call": ms * 1e3, "weight_gbs": wbytes / (ms * 1e-3) / 1e9}
    peak, peak_kind = measured_peaks()
    print(json.dumps({"metric": "Q4_K GEMM weight GB/s, tensor cores vs CUDA cores (16 rows)",
                      "value": out["tensor_core"]["weight_gbs"], "unit": "GB/s", **out,
                      "speedup_tensor_over_cuda_core": out["cuda_core_dp4a"]["us_per_call"] /
                      out["tensor_core"]["us_per_call"],
                      "peak": peak, "peak_kind": peak_kind, "shape": {"N": N, "K": K, "rows": 16},
                      "config": {"workload": f"one Q4_K projection {K}->{N}, 16 rows",
                                 "l2": f"weights rotated over {ncopies} device copies"}}), flush=True)
    ctx.close()


def run_head_accept(args):
    """LM head + accept: final RMSNorm, the Q4_K head 6656 -> 131072 with its
    fused per-row argmax over 16 rows (spec_lm_head_argmax), then the accept
    kernel with the KV rollback (spec_accept) on a paged bf16 KV of 52 layers x
    4 heads x 128 at n_past = 2055 (the block straddles a page).  Drafts are
    planted so that the accepted lengths are uniform in 0..15 over >= 64
    trials; the device result of every trial is checked against the planted
    length.  One trial = KV block reserve (spec_kv_extend by 16) + head/argmax
    + accept/rollback + rollback to n_past."""
    import torch

    from speculative_decoding_exact_gb300 import abi, runtime, synth
    from speculative_decoding_exact_gb300 import build as b

    b.build()
    cfg = full_cfg()
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    n_past, max_ctx = 2055, 2112
    ctx = runtime.Context(cfg, max_ctx=max_ctx, stream=stream)
    H, V = cfg.hidden, cfg.vocab
    Wh = runtime.upload_tiled(ctx, synth.q4k_matrix(V, H, 0, 999999), V, H)
    gamma = torch.ones(H, dtype=torch.float32, device="cuda")
    x = torch.from_numpy(synth.normal((ROWS, H), 0, 11)).cuda()
    pages = max_ctx // 16
    kv = runtime.DeviceKV(cfg, pages, pages)
    kv.reset(ctx)
    kv.extend(ctx, n_past)
    ks = kv.struct()
    idx = torch.zeros(ROWS, dtype=torch.int32, device="cuda")
    abi.check("spec_lm_head_argmax", abi.spec_lm_head_argmax(ctx.h, Wh.data_ptr(), gamma.data_ptr(), x.data_ptr(),
                                                             ROWS, idx.data_ptr(), None))
    torch.cuda.synchronize()
    target = idx.cpu().numpy()
    trials = max(64, args.steps)
    rng = np.random.default_rng(2055)
    Ls = rng.integers(0, K_DRAFT + 1, trials).astype(np.int32)
    drafts = torch.from_numpy(np.stack([synth.plant_draft(target, int(L), V, 0, 4000 + t)
                                        for t, L in enumerate(Ls)])).cuda()
    hist = torch.zeros((trials, 4), dtype=torch.int32, device="cuda")
    res = torch.zeros(4, dtype=torch.int32, device="cuda")
    it = [0]

    def trial():
        t = it[0] % trials
        it[0] += 1
        abi.check("spec_kv_extend", abi.spec_kv_extend(ctx.h, ks, ROWS))
        abi.check("spec_lm_head_argmax", abi.spec_lm_head_argmax(ctx.h, Wh.data_ptr(), gamma.data_ptr(),
                                                                 x.data_ptr(), ROWS, idx.data_ptr(), None))
        abi.check("spec_accept", abi.spec_accept(ctx.h, idx.data_ptr(), drafts[t].data_ptr(), K_DRAFT, ks,
                                                 res.data_ptr()))
        hist[t].copy_(res)
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, ks, n_past))

    it[0] = 0
    ms = _time_steps(torch, stream, trial, 0, trials)
    h = hist.cpu().numpy()
    assert np.all(h[:, 2] == 0) and np.array_equal(h[:, 0], Ls), "planted accepted lengths"
    assert np.array_equal(h[:, 3], n_past + Ls + 1), "rolled-back lengths"
    assert abi.spec_last_status(ctx.h) == 0
    peak, peak_kind = measured_peaks()
    wbytes = V * (H // 256) * 144
    print(json.dumps({"metric": "LM head + argmax + accept/rollback per second (16 rows, V = 131072)",
                      "value": 1000.0 / ms, "unit": "head+accept/s", "ms_per_trial": ms,
                      "head_weight_gbs": wbytes / (ms * 1e-3) / 1e9,
                      "head_frac_of_measured_hbm": wbytes / (ms * 1e-3) / 1e9 / peak, "peak_kind": peak_kind,
                      "trials": trials, "accepted_hist": np.bincount(Ls, minlength=K_DRAFT + 1).tolist(),
                      "config": {"workload": "Q4_K head 6656->131072 + argmax + accept + KV rollback, "
                                             "16 rows, n_past 2055, paged bf16 KV 52 x 4 x 128, page 16",
                                 "l2": "head weights (491 MB) larger than L2"}}), flush=True)
    ctx.close()


def run_ctx_sweep(args):
    """The 52-block verify pass with the KV context swept over 2,048 / 16,384 /
    32,768 and planted acceptance profiles of mean accepted length 1, 4 and 12
    (each position accepted with probability a, E[min(Geom, 15)] = mean),
    with the DFlash-style front projection (Q4_K 33,280 -> 6,656) timed at
    M = round(mean L) + 1 and M = 16.  One JSON line per (context, mean):
    steps/s and accepted tokens/s = steps/s x mean(L + 1)."""
    import torch

    from speculative_decoding_exact_gb300 import abi, runtime, synth

    mdl = setup_model(0)
    cfg, stream = mdl.cfg, mdl.stream
    V = cfg.vocab
    mdl.ctx.close()
    fc_N, fc_K = cfg.hidden, 5 * cfg.hidden
    for ctx_len in (2048, 16384, 32768):
        max_ctx = ctx_len + 64
        ctx = runtime.Context(cfg, max_ctx=max_ctx, stream=stream)
        pages = max_ctx // 16
        kv = runtime.DeviceKV(cfg, pages, pages)
        kv.reset(ctx)
        kv.extend(ctx, ctx_len)
        g = torch.Generator(device="cuda").manual_seed(1234 + ctx_len)
        with torch.cuda.stream(stream):
            for l in range(cfg.n_layers):
                kv.pool[:, l].copy_(torch.randn(kv.pool[:, l].shape, generator=g, device="cuda")
                                    .to(torch.bfloat16))
        ks = kv.struct()
        ws = mdl.dw.struct()
        if ctx_len == 2048:
            Wfc = runtime.upload_tiled(ctx, synth.q4k_matrix(fc_N, fc_K, 3, 4242), fc_N, fc_K)
            xfc = torch.from_numpy(synth.normal((16, fc_K), 3, 17)).cuda()
            yfc = torch.zeros((16, fc_N), dtype=torch.float32, device="cuda")
        am = torch.zeros(ROWS, dtype=torch.int32, device="cuda")
        abi.check("spec_verify_step_ex", abi.spec_verify_step_ex(ctx.h, ws, ks, mdl.hidden.data_ptr(),
                                                                 mdl.draft.data_ptr(), K_DRAFT, mdl.res.data_ptr(),
                                                                 abi.spec_taps(None, am.data_ptr(), None)))
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, ks, ctx_len))
        torch.cuda.synchronize()
        idx = am.cpu().numpy()

        def fc_us(M):
            def call():
                abi.check("spec_gemm_q4k", abi.spec_gemm_q4k(ctx.h, Wfc.data_ptr(), fc_N, fc_K, xfc.data_ptr(),
                                                             M, yfc.data_ptr()))
            return _time_steps(torch, stream, call, 3, 20) * 1e3

        rng = np.random.default_rng(ctx_len)
        for mean in (1.0, 4.0, 12.0):
            a = _alpha_for_mean(mean)
            Ls = np.zeros(args.steps, dtype=np.int32)
            drafts = np.zeros((args.steps, K_DRAFT), dtype=np.int32)
            for t in range(args.steps):
                L = 0
                while L < K_DRAFT and rng.random() < a:
                    L += 1
                Ls[t] = L
                d = rng.integers(0, V, K_DRAFT).astype(np.int32)
                d[:L] = idx[:L]
                if L < K_DRAFT:
                    d[L] = (idx[L] + 1) % V
                drafts[t] = d
            dd = torch.from_numpy(drafts).cuda()
            hist = torch.zeros((args.steps, 4), dtype=torch.int32, device="cuda")
            it = [0]

            def step():
                t = it[0] % args.steps
                it[0] += 1
                abi.check("spec_verify_step", abi.spec_verify_step(ctx.h, ws, ks, mdl.hidden.data_ptr(),
                                                                   dd[t].data_ptr(), K_DRAFT, mdl.res.data_ptr()))
                hist[t].copy_(mdl.res)
                abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, ks, ctx_len))

            for _ in range(max(args.warmup, 3)):
                step()
            it[0] = 0
            ms = _time_steps(torch, stream, step, 0, args.steps)
            h = hist.cpu().numpy()
            assert np.all(h[:, 2] == 0) and np.array_equal(h[:, 0], Ls), "planted accepted lengths"
            sps = 1000.0 / ms
            m_acc = float(h[:, 0].mean())
            wb = cfg.weight_bytes()
            print(json.dumps({"metric": "accepted tokens/s at k+1=16 rows (verify steps/s x mean(L+1))",
                              "value": sps * (m_acc + 1.0), "unit": "tokens/s", "steps_per_s": sps,
                              "ms_per_step": ms, "context": ctx_len, "target_mean_accepted": mean,
                              "mean_accepted": m_acc, "steps": args.steps,
                              "weight_gbs": wb * sps / 1e9,
                              "total_gbs": (wb + kv_read_bytes(cfg, ctx_len)) * sps / 1e9,
                              "fc_front_projection_us": {"M": int(round(m_acc)) + 1,
                                                         "us": fc_us(int(round(m_acc)) + 1), "M16_us": fc_us(16)},
                              "config": dict(workload_config(cfg), context=ctx_len,
                                             acceptance=f"per-position {a:.4f}")}), flush=True)
        del kv
        ctx.close()
        torch.cuda.empty_cache()


def run_overlap(args):
    """Split submit (Ch. 33 §33.2 / Figure 33.1) on the full model at context
    --ctx: the step captures the block outputs of layers 1, 13, 25, 37, 49
    (the draft's five hidden rows) and records an event after block 49; a
    second stream with its own spec_ctx waits on it and runs the draft's
    front projection (Q4_K 33,280 -> 6,656, 16 rows) while the step's last
    blocks and LM head run.  Reports, in ms: the step alone (recorded graph),
    the step with the split event (enqueued launch by launch), the projection
    alone, the two one after the other on one stream, and overlapped."""
    import torch

    from speculative_decoding_exact_gb300 import abi, runtime, synth

    mdl = setup_model(0)
    cfg, ctx, sa = mdl.cfg, mdl.ctx, mdl.stream
    H = cfg.hidden
    ids = np.array([1, 13, 25, 37, 49], dtype=np.int32)
    cap = torch.zeros((16, 5 * H), dtype=torch.float32, device="cuda")
    abi.check("spec_set_capture", abi.spec_set_capture(ctx.h, ids.ctypes.data, 5, cap.data_ptr()))
    sb = torch.cuda.Stream()
    ctx_b = runtime.Context(cfg, max_ctx=CTX + 64, stream=sb)
    fc_N, fc_K = H, 5 * H
    Wfc = runtime.upload_tiled(ctx_b, synth.q4k_matrix(fc_N, fc_K, 3, 4242), fc_N, fc_K)
    yfc = torch.zeros((16, fc_N), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()

    def step():
        abi.check("spec_verify_step", abi.spec_verify_step(ctx.h, mdl.ws, mdl.ks, mdl.hidden.data_ptr(),
                                                           mdl.draft.data_ptr(), K_DRAFT, mdl.res.data_ptr()))
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, mdl.ks, CTX))

    def fc(c):
        abi.check("spec_gemm_q4k", abi.spec_gemm_q4k(c.h, Wfc.data_ptr(), fc_N, fc_K, cap.data_ptr(), 16,
                                                     yfc.data_ptr()))

    ms_step = _time_steps(torch, sa, step, args.warmup, args.steps)
    ms_fc = _time_steps(torch, sb, lambda: fc(ctx_b), args.warmup, args.steps)

    def serial():
        step()
        # the projection on the step's stream: a spec_ctx of the same stream
        fc(ctx_serial)

    ctx_serial = runtime.Context(cfg, max_ctx=CTX + 64, stream=sa)
    ms_serial = _time_steps(torch, sa, serial, args.warmup, args.steps)
    ctx_serial.close()

    ev = torch.cuda.Event()
    ev.record(sa)
    torch.cuda.synchronize()
    abi.check("spec_set_split", abi.spec_set_split(ctx.h, 49, ev.cuda_event))
    ms_step_split = _time_steps(torch, sa, step, args.warmup, args.steps)
    done_b = torch.cuda.Event()

    def overlapped():
        step()
        sb.wait_event(ev)
        fc(ctx_b)
        done_b.record(sb)
        sa.wait_event(done_b)                        # the round ends when both are done

    ms_overlap = _time_steps(torch, sa, overlapped, args.warmup, args.steps)
    abi.check("spec_set_split", abi.spec_set_split(ctx.h, -1, None))
    abi.check("spec_set_capture", abi.spec_set_capture(ctx.h, None, 0, None))
    print(json.dumps({"metric": "verify step + draft front projection, split submit (ms per round)",
                      "value": ms_overlap, "unit": "ms", "higher_is_better": False,
                      "step_ms": ms_step, "step_with_split_event_ms": ms_step_split, "fc_ms": ms_fc,
                      "serial_ms": ms_serial, "overlapped_ms": ms_overlap,
                      "saved_vs_serial_ms": ms_serial - ms_overlap, "steps": args.steps, "warmup": args.warmup,
                      "config": dict(workload_config(cfg), capture_layers=ids.tolist(), split_after=49,
                                     fc="Q4_K 33280->6656, 16 rows, own spec_ctx on a second stream")}),
          flush=True)
    ctx_b.close()
    ctx.close()


def run_draft(args):
    """A DFlash-shaped draft forward (Ch. 8 §8.2) with random Q4_K weights,
    timed beside the verify step: the front projection fc 33,280 -> 6,656 over
    16 rows of five concatenated target hidden states, five blocks at hidden
    6,656 (52 query heads, FFN 17,920), attention over a context of 2,112 rows
    (the 64-row sink plus the 2,048-row window of Ch. 8 §8.3) and the 16-row
    block, then the target's own LM head and the per-row argmax (the draft
    borrows the target's head, Ch. 8 §8.2).  The draft's k and v project
    6,656 -> 1,024 (8 KV heads of 128, Ch. 8 §8.2); its query head count is
    not given and is taken as 48 (6 per KV head, an attention width of
    6,144).  q and k are QK-normed and rotated (RoPE, theta 1e6: the base is
    not given either).  Everything runs through the library's own kernels: spec_gemm_q4k
    for fc, then a 5-layer verify step for the blocks, head and argmax.
    Reports ms per draft forward, per verify step, and per cycle."""
    import torch

    from speculative_decoding_exact_gb300 import abi, runtime, synth

    mdl = setup_model(0)
    cfg, ctx, stream = mdl.cfg, mdl.ctx, mdl.stream
    H = cfg.hidden
    dcfg = runtime.ModelConfig(**dict(synth.FULL, n_layers=5, n_q_heads=48, n_kv_heads=8, rope_theta=1.0e6))
    dctx_len = 64 + 2048
    dmax = dctx_len + 64
    dctx = runtime.Context(dcfg, max_ctx=dmax, stream=stream)
    dw = runtime.DeviceWeights(dcfg)
    for l in range(dcfg.n_layers):
        for j, (name, N, K) in enumerate(dcfg.matrices()):
            getattr(dw, name).append(runtime.upload_tiled(dctx, synth.q4k_matrix(N, K, 9, 5000 + 10 * l + j), N, K))
    dw.w_head = mdl.dw.w_head                     # the target's LM head
    # QK-norm gains per layer (random around 1)
    dw.q_norm = [torch.from_numpy((1.0 + 0.1 * synth.normal((128,), 9, 5100 + l)).astype(np.float32)).cuda()
                 for l in range(dcfg.n_layers)]
    dw.k_norm = [torch.from_numpy((1.0 + 0.1 * synth.normal((128,), 9, 5200 + l)).astype(np.float32)).cuda()
                 for l in range(dcfg.n_layers)]
    fc_N, fc_K = H, 5 * H
    Wfc = runtime.upload_tiled(dctx, synth.q4k_matrix(fc_N, fc_K, 9, 5999), fc_N, fc_K)
    pages = dmax // 16
    dkv = runtime.DeviceKV(dcfg, pages, pages)
    dkv.reset(dctx)
    dkv.extend(dctx, dctx_len)
    g = torch.Generator(device="cuda").manual_seed(99)
    with torch.cuda.stream(stream):
        dkv.pool.copy_(torch.randn(dkv.pool.shape, generator=g, device="cuda").to(torch.bfloat16))
    cap = torch.from_numpy(synth.normal((16, fc_K), 9, 6000)).cuda()
    hid = torch.zeros((16, H), dtype=torch.float32, device="cuda")
    dtok = torch.from_numpy(synth.tokens(K_DRAFT, cfg.vocab, 9, 6001)).cuda()
    dres = torch.zeros(4, dtype=torch.int32, device="cuda")
    prop = torch.zeros(16, dtype=torch.int32, device="cuda")
    dws, dks = dw.struct(), dkv.struct()
    taps = abi.spec_taps(None, prop.data_ptr(), None)
    torch.cuda.synchronize()

    def draft():
        abi.check("spec_gemm_q4k", abi.spec_gemm_q4k(dctx.h, Wfc.data_ptr(), fc_N, fc_K, cap.data_ptr(), 16,
                                                     hid.data_ptr()))
        abi.check("spec_verify_step_ex", abi.spec_verify_step_ex(dctx.h, dws, dks, hid.data_ptr(), dtok.data_ptr(),
                                                                 K_DRAFT, dres.data_ptr(), taps))
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(dctx.h, dks, dctx_len))

    def verify():
        abi.check("spec_verify_step", abi.spec_verify_step(ctx.h, mdl.ws, mdl.ks, mdl.hidden.data_ptr(),
                                                           mdl.draft.data_ptr(), K_DRAFT, mdl.res.data_ptr()))
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, mdl.ks, CTX))

    def cycle():
        draft()
        verify()

    ms_d = _time_steps(torch, stream, draft, args.warmup, args.steps)
    assert int(dres[2].item()) == 0
    ms_v = _time_steps(torch, stream, verify, args.warmup, args.steps)
    ms_c = _time_steps(torch, stream, cycle, args.warmup, args.steps)
    dbytes = dcfg.weight_bytes() + fc_N * (fc_K // 256) * 144
    print(json.dumps({"metric": "DFlash-shaped draft forward (fc + 5 blocks + target LM head + argmax), ms",
                      "value": ms_d, "unit": "ms", "higher_is_better": False,
                      "draft_ms": ms_d, "verify_ms": ms_v, "cycle_ms": ms_c,
                      "draft_weight_bytes": dbytes, "draft_weight_gbs": dbytes / (ms_d * 1e-3) / 1e9,
                      "steps": args.steps, "warmup": args.warmup,
                      "config": {"workload": "draft: fc Q4_K 33280->6656, 5 blocks hidden 6656 (48 q / 8 kv heads: "
                                             "k/v 6656->1024, FFN 17920), context 64 sink + 2048 window, "
                                             "target LM head 131072, "
                                             "16 rows; verify: the full 52-block step at context "
                                             f"{CTX}", "draft_weights": "random Q4_K"}}), flush=True)
    dctx.close()
    ctx.close()


def run_swa(args):
    """Sliding-window layers (Ch. 8 §8.6 item 4) on the full model at context
    --ctx: every second block is a window layer of --swa positions (its K/V in
    a ring of W + 16 rows, attended by the same tensor-core kernel over the
    window's chunks), the others attend the whole paged context.  Timed beside
    the plain step at the same context, sharing the weights."""
    import torch

    from speculative_decoding_exact_gb300 import abi, runtime, synth

    mdl = setup_model(0)
    cfg, ctx, stream = mdl.cfg, mdl.ctx, mdl.stream

    def plain():
        abi.check("spec_verify_step", abi.spec_verify_step(ctx.h, mdl.ws, mdl.ks, mdl.hidden.data_ptr(),
                                                           mdl.draft.data_ptr(), K_DRAFT, mdl.res.data_ptr()))
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, mdl.ks, CTX))

    ms_plain = _time_steps(torch, stream, plain, args.warmup, args.steps)
    scfg = runtime.ModelConfig(**dict(synth.FULL, swa_window=args.swa, swa_period=2))
    sctx = runtime.Context(scfg, max_ctx=CTX + 64, stream=stream)
    pages = (CTX + 64) // 16
    skv = runtime.DeviceKV(scfg, pages, pages)
    skv.reset(sctx)
    skv.extend(sctx, CTX)
    g = torch.Generator(device="cuda").manual_seed(4321)
    with torch.cuda.stream(stream):
        for l in range(scfg.n_layers):
            if scfg.swa_index(l) < 0:
                skv.pool[:, l].copy_(torch.randn(skv.pool[:, l].shape, generator=g, device="cuda").to(torch.bfloat16))
        skv.swa_ring.copy_(torch.randn(skv.swa_ring.shape, generator=g, device="cuda").to(torch.bfloat16))
    torch.cuda.synchronize()
    sks = skv.struct()

    def windowed():
        abi.check("spec_verify_step", abi.spec_verify_step(sctx.h, mdl.ws, sks, mdl.hidden.data_ptr(),
                                                           mdl.draft.data_ptr(), K_DRAFT, mdl.res.data_ptr()))
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(sctx.h, sks, CTX))

    ms_swa = _time_steps(torch, stream, windowed, args.warmup, args.steps)
    r = mdl.res.cpu().numpy()
    assert r[2] == 0 and abi.spec_last_status(sctx.h) == 0, "sliding-window step status"
    print(json.dumps({"metric": "verify steps/s with sliding-window layers (every second block)",
                      "value": 1000.0 / ms_swa, "unit": "verify steps/s", "ms_per_step": ms_swa,
                      "plain_steps_per_s": 1000.0 / ms_plain, "window": args.swa, "context": CTX,
                      "window_layers": scfg.n_swa, "steps": args.steps, "warmup": args.warmup,
                      "config": dict(workload_config(cfg), swa_window=args.swa, swa_period=2)}), flush=True)
    sctx.close()
    ctx.close()


def _alpha_for_mean(mean):
    """Per-position acceptance a with E[min(Geom(a), 15)] = sum_{i=1..15} a^i = mean."""
    lo, hi = 0.0, 1.0
    for _ in range(60):
        a = 0.5 * (lo + hi)
        e = sum(a ** i for i in range(1, K_DRAFT + 1))
        lo, hi = (a, hi) if e < mean else (lo, a)
    return 0.5 * (lo + hi)


def run_tree(args):
    """Token-tree verify steps (Ch. 33 section 33.7) on the full model at
    context --ctx: a random tree of --tree nodes (node 0 = the carried
    frontier, parent[i] uniform in [0, i), random tokens, random rows), timed
    like the linear step, which is timed beside it."""
    import torch

    from speculative_decoding_exact_gb300 import abi, synth

    mdl = setup_model(0)
    cfg, ctx, stream = mdl.cfg, mdl.ctx, mdl.stream
    n = args.tree
    rng = np.random.default_rng(3)
    parent = torch.from_numpy(np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)],
                                       dtype=np.int32)).cuda()
    tokens = torch.from_numpy(rng.integers(0, cfg.vocab, n).astype(np.int32)).cuda()
    rows = torch.from_numpy(synth.normal((n, cfg.hidden), 0, 55)).cuda()
    path = torch.zeros(max(16, n), dtype=torch.int32, device="cuda")

    def tree():
        abi.check("spec_verify_tree", abi.spec_verify_tree(ctx.h, mdl.ws, mdl.ks, rows.data_ptr(), tokens.data_ptr(),
                                                           parent.data_ptr(), n, mdl.res.data_ptr(),
                                                           path.data_ptr(), None))
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, mdl.ks, CTX))

    def linear():
        abi.check("spec_verify_step", abi.spec_verify_step(ctx.h, mdl.ws, mdl.ks, mdl.hidden.data_ptr(),
                                                           mdl.draft.data_ptr(), K_DRAFT, mdl.res.data_ptr()))
        abi.check("spec_kv_rollback", abi.spec_kv_rollback(ctx.h, mdl.ks, CTX))

    ms_t = _time_steps(torch, stream, tree, args.warmup, args.steps)
    r = mdl.res.cpu().numpy()
    assert r[2] == 0, f"tree step status {r[2]}"
    ms_l = _time_steps(torch, stream, linear, args.warmup, args.steps)
    print(json.dumps({"metric": f"token-tree verify steps/s ({n} nodes, {(n + 15) // 16} pass(es) of <= 16 rows)",
                      "value": 1000.0 / ms_t,
                      "unit": "verify steps/s", "ms_per_step": ms_t, "linear_16_rows_steps_per_s": 1000.0 / ms_l,
                      "steps": args.steps, "warmup": args.warmup,
                      "config": dict(workload_config(cfg), tree="random parents, random tokens")}), flush=True)
    ctx.close()


def run_attention(args):
    """Time the verify attention alone: 16 rows, the full model's 52 query / 4 KV
    heads of 128, KV context --ctx (the block of 16 rows appended after it),
    through spec_attention on a one-layer paged KV pool.  The L2 is flushed
    with a 256 MB write before every call (one layer's KV at 2k is 4.2 MB), and
    each call is timed alone with CUDA events.  A small device footprint, used
    as the ncu capture target of the attention kernels."""
    import torch

    from speculative_decoding_exact_gb300 import abi, runtime, synth
    from speculative_decoding_exact_gb300 import build as b

    b.build()
    cfg = runtime.ModelConfig(**dict(synth.FULL, n_layers=1))
    max_ctx = CTX + 64
    ctx = runtime.Context(cfg, max_ctx=max_ctx)
    pages = max_ctx // cfg.page_size
    kv = runtime.DeviceKV(cfg, pages, pages)
    kv.reset(ctx)
    kv.extend(ctx, CTX + 16)
    g = torch.Generator(device="cuda").manual_seed(5)
    kv.pool.copy_(torch.randn(kv.pool.shape, generator=g, device="cuda").to(torch.bfloat16))
    q = torch.from_numpy(synth.normal((16, cfg.n_q_heads * cfg.head_dim), 5, 1)).cuda()
    out = torch.zeros((16, cfg.n_q_heads * cfg.head_dim), dtype=torch.float32, device="cuda")
    flush = torch.empty(256 * 2**20 // 4, dtype=torch.float32, device="cuda")
    kvs = kv.struct()

    def call():
        abi.check("spec_attention", abi.spec_attention(ctx.h, kvs, 0, q.data_ptr(), 16, out.data_ptr()))

    for _ in range(args.warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    total = 0.0
    for _ in range(args.steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1)
    us = total * 1000.0 / args.steps
    kv_bytes = (CTX + 16) * cfg.n_kv_heads * 2 * cfg.head_dim * 2
    print(json.dumps({"metric": "verify attention KV GB/s (16 rows, q tiles + partials + merge)",
                      "value": kv_bytes / us / 1e3, "unit": "GB/s", "us_per_call": us,
                      "config": {"ctx": CTX, "rows": 16, "n_q_heads": cfg.n_q_heads,
                                 "n_kv_heads": cfg.n_kv_heads, "head_dim": cfg.head_dim},
                      "kv_bytes": kv_bytes, "l2": "flushed (256 MB write) before every call"}))
    ctx.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--gemm-shape", default=None,
                    help="NxK: time one Q4_K GEMM shape instead of the verify step")
    ap.add_argument("--sampled", action="store_true",
                    help="time the verify step with the sampled decision (Ch. 33 section 33.2)")
    ap.add_argument("--accept-profile", action="store_true",
                    help="steps with planted drafts at mean accepted lengths 1, 4, 12, 15: accepted tokens/s")
    ap.add_argument("--tree", type=int, default=0,
                    help="time token-tree verify steps with a random tree of this many nodes (1..64; "
                         "more than 16 run in passes of 16 rows)")
    ap.add_argument("--attn", action="store_true",
                    help="time the verify attention alone at context --ctx instead of the verify step")
    ap.add_argument("--sweep", action="store_true",
                    help="projection sweep 6656->6656 and 6656->26624 at M = 1..16, weights rotated over 2 GB")
    ap.add_argument("--cudacore", default=None,
                    help="NxK: the tensor-core GEMM against the CUDA-core (dp4a) GEMM on one shape")
    ap.add_argument("--head-accept", action="store_true",
                    help="LM head 6656->131072 + argmax + accept/rollback at n_past 2055, L ~ U{0..15}")
    ap.add_argument("--ctx-sweep", action="store_true",
                    help="verify steps at context 2k/16k/32k x mean accepted length 1/4/12, with the fc timing")
    ap.add_argument("--draft", action="store_true",
                    help="time a DFlash-shaped draft forward (fc + 5 blocks + LM head) beside the verify step")
    ap.add_argument("--swa", type=int, default=0,
                    help="W: every second block a sliding-window layer of W positions, at context --ctx")
    ap.add_argument("--overlap", action="store_true",
                    help="split submit: the draft front projection on a second stream overlaps the step's suffix")
    ap.add_argument("--ctx", type=int, default=2048,
                    help="KV context of the verify step (the long-context sweep uses 16384, 32768)")
    args = ap.parse_args()
    global CTX
    if args.ctx % 16 or args.ctx < 16:
        ap.error("--ctx must be a positive multiple of 16")
    CTX = args.ctx
    if args.gemm_shape:
        run_gemm_shape(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.head_accept:
        run_head_accept(args)
        return
    if args.cudacore:
        run_cudacore(args)
        return
    if args.ctx_sweep:
        run_ctx_sweep(args)
        return
    if args.overlap:
        run_overlap(args)
        return
    if args.swa:
        run_swa(args)
        return
    if args.draft:
        run_draft(args)
        return
    if args.attn:
        run_attention(args)
        return
    if args.sampled:
        run_sampled(args)
        return
    if args.tree:
        run_tree(args)
        return
    if args.accept_profile:
        run_accept_profile(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as tdist
        if args.impl == "ours":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world)
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()
