#!/usr/bin/env python3
"""Benchmark of the decode-time skinny linears on GB300.

Workload (the headline): the bf16 skinny GEMM sweep, y = x . W^T with
M in {1,2,4,8,16,32,64,128} over (N,K) in {(4096,4096), (12288,4096), (4096,12288),
(32768,1024), (8192,4096)}; x ~ N(0,1), W ~ N(0,1/K), seeded per shape, bf16.
One step = one call of every one of those 40 shapes.

Metric: microseconds per call and achieved HBM GB/s on weight bytes (fraction of
the measured HBM peak) per (N,K,M); `value` is the whole step's weight bytes
divided by its device time (GB/s).  The other hot-path workloads (the bf16 GEMV
2048x1024 at M=1, fused gate/up, fp8 head + argmax, MoE W1/W2, mid-M rows, the A8W8
block-scaled linear with its activation quantisation, the batch-invariant numerics
mode at 1-8 rows, and chained gate/up -> down and W1 -> W2 pairs) are measured in the
same run and reported under "ops".

Timing: each shape's calls are captured in a CUDA graph of R back-to-back calls
that rotate over enough weight copies to exceed 3x the L2 size (so no call finds
its weights in L2; up to 16 copies their count is a power of two, so consecutive
graphs over the same copies continue the rotation); the graph is replayed once per
step between CUDA events on the capturing stream; per-call time = event time / R.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

SWEEP_NK = [(4096, 4096), (12288, 4096), (4096, 12288), (32768, 1024), (8192, 4096)]
SWEEP_M = [1, 2, 4, 8, 16, 32, 64, 128]
GATE_UP_M = [1, 2, 3, 4, 6, 8, 12, 16, 32, 64, 128]
HEAD_M = [1, 2, 3, 4, 8]
CHAIN_M = [1, 2, 4, 8, 16]
MID_M = [192, 256, 384, 512]
MID_NK = [(32768, 1024), (8192, 1024), (4096, 12288)]
MOE_M = [1, 2, 4, 8, 16]
A8_NK = [(32768, 1024), (8192, 4096)]
A8_M = [1, 2, 4, 8, 16, 32, 64]
INV_M = [1, 2, 4, 8]
MOE_E, MOE_I, MOE_K, MOE_TOPK = 128, 1536, 4096, 6
HEAD_N, HEAD_K = 248320, 4096
FALLBACK_HBM_GBS = 6800.0
WORKLOAD = ("bf16 skinny GEMM sweep M{1..128} x (N,K){(4096,4096),(12288,4096),(4096,12288),"
            "(32768,1024),(8192,4096)}")
METRIC = "µs/call and achieved HBM GB/s (% of GB300 peak) per (N,K,M) decode shape"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            for k in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
                if k in d:
                    return float(d[k]), "measured"
        except (OSError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU arm

def _max_over_ranks(x: float, device) -> float:
    """The largest x over all ranks of the process group (x itself without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_value(world: int, step_bytes: float, step_us: float) -> float:
    """Whole-job GB/s: every rank (an independent replica) streams step_bytes per step,
    and the job's step lasts as long as its slowest rank's."""
    return world * step_bytes / (step_us * 1e-6) / 1e9


def _graph_case(torch, calls, reps: int, stream):
    """Capture `reps` calls (a list of closures, used round-robin) into one CUDA graph."""
    for c in calls[:2]:
        c()                       # warm: attribute setup, occupancy cache
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(reps):
            calls[i % len(calls)]()
    torch.cuda.synchronize()
    return g


def _copies_for(nbytes: int, l2: int) -> int:
    """Weight copies for one shape: at least 3x L2 of them.  Up to 16 copies the count is
    rounded up to a power of two, so that a graph of 16 calls makes whole rotations and
    the next graph over the same copies (the next row count) starts on the copy used
    longest ago, not on one a few calls old that may still sit in L2."""
    n = max(2, -(-3 * l2 // max(1, nbytes)))
    if n <= 16:
        n = 1 << (n - 1).bit_length()
    return n


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import gemv_dg_bf16_gb300 as dg
    from synth import decode_inputs as S

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    dg.dg_init(local)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    peak, peak_src = _peaks()
    stream = torch.cuda.Stream(device=dev)
    R = args.reps

    table = None
    if args.table:
        # a shape table measured on this device and build (dg_sweep): every call
        # below dispatches through it; the headline shapes are timed both ways
        if args.sweep_table and rank == 0:
            dg.dg_sweep(_table_shapes(dg), args.table, reps=args.sweep_reps, resume=True)
        if world > 1:
            dist.barrier()
        with open(args.table) as f:
            table = json.load(f)
        dg.dg_table_load(args.table)

    cases = []        # (name, dict(meta), graph, weight_bytes_per_call)
    keep = []         # every tensor a captured graph reads or writes stays alive with it
    pattern = re.compile(args.cases) if args.cases else None

    def case_id(name, meta):
        return name + "/" + "/".join(f"{k}{v}" for k, v in meta.items() if k in ("M", "N", "K", "N_half"))

    def wanted(name, meta):
        return pattern is None or pattern.search(case_id(name, meta)) is not None

    kernels = []      # kernel launches of one call of each case

    def add(name, meta, calls, wbytes, launches_per_call=1):
        if not wanted(name, meta):
            return
        with torch.cuda.stream(stream):
            g = _graph_case(torch, calls, R, stream)
        cases.append((name, meta, g, wbytes))
        keep.append(calls)
        kernels.append(launches_per_call)

    # --- the headline sweep
    sweep_cases = []
    dcases = []       # shape-table arm: the sweep shapes' graphs with the compiled defaults
    only = None
    if args.only:
        only = tuple(int(v) for v in args.only.split(","))       # M,N,K
    for (N, K) in SWEEP_NK if only is None else [(only[1], only[2])]:
        if not any(wanted("gemv_bf16", {"M": M, "N": N, "K": K}) for M in SWEEP_M):
            continue
        W0 = S.linear_inputs(1, N, K, device=dev)[1]
        wb = N * K * 2
        Ws = [W0] + [W0.clone() for _ in range(_copies_for(wb, l2) - 1)]
        for M in SWEEP_M if only is None else [only[0]]:
            x = S.linear_inputs(M, N, K, device=dev)[0]
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = dg.workspace(dg.DG_OP_GEMV_BF16, M, N, K, device=dev)
            calls = [(lambda W=W, x=x, y=y, ws=ws: dg.dg_gemv_bf16(x, W, y, ws=ws, stream=stream)) for W in Ws]
            if wanted("gemv_bf16", {"M": M, "N": N, "K": K}):
                if table is not None:
                    # the same calls with the compiled defaults, captured before the
                    # table is loaded again (dispatch happens when a call is captured);
                    # timed in steps of their own, in the same shape order
                    dg.dg_table_clear()
                    with torch.cuda.stream(stream):
                        dcases.append(({"M": M, "N": N, "K": K}, _graph_case(torch, calls, R, stream), wb))
                    dg.dg_table_load(args.table)
                add("gemv_bf16", {"M": M, "N": N, "K": K}, calls, wb)
                sweep_cases.append(len(cases) - 1)
    def need(name, metas):
        return any(wanted(name, m) for m in metas)

    if not args.sweep_only and only is None:
        # --- GEMV 2048x1024 at M=1
        N, K = 2048, 1024
        x, W0 = S.linear_inputs(1, N, K, device=dev)
        wb = N * K * 2
        Ws = [W0] + [W0.clone() for _ in range(_copies_for(wb, l2) - 1)]
        y = torch.empty((1, N), dtype=torch.bfloat16, device=dev)
        ws = dg.workspace(dg.DG_OP_GEMV_BF16, 1, N, K, device=dev)
        add("gemv_bf16_2048x1024", {"M": 1, "N": N, "K": K},
            [(lambda W=W, x=x, y=y, ws=ws: dg.dg_gemv_bf16(x, W, y, ws=ws, stream=stream)) for W in Ws], wb)
        # --- gate/up
        Nh, K = 12288, 4096
        W0 = (S.gate_up_inputs(1, Nh, K, device=dev)[1]
              if need("gate_up_silu", [{"M": M, "N_half": Nh, "K": K} for M in GATE_UP_M]) else None)
        wb = 2 * Nh * K * 2
        Ws = [W0] + [W0.clone() for _ in range(_copies_for(wb, l2) - 1)] if W0 is not None else []
        for M in GATE_UP_M if Ws else []:
            x = S.gate_up_inputs(M, Nh, K, device=dev)[0]
            out = torch.empty((M, Nh), dtype=torch.bfloat16, device=dev)
            ws = dg.workspace(dg.DG_OP_GATE_UP_SILU, M, Nh, K, device=dev)
            add("gate_up_silu", {"M": M, "N_half": Nh, "K": K},
                [(lambda W=W, x=x, out=out, ws=ws: dg.dg_gate_up_silu(x, W, out, ws=ws, stream=stream)) for W in Ws], wb)
        # --- fp8 head
        head_on = need("head_fp8_argmax", [{"M": M, "N": HEAD_N, "K": HEAD_K} for M in HEAD_M])
        if head_on:
            x8, Wq, scale = S.head_inputs(8, HEAD_N, HEAD_K, device=dev)
        for M in HEAD_M if head_on else []:
            x = x8[:M].contiguous()
            logits = torch.empty((M, HEAD_N), dtype=torch.bfloat16, device=dev)
            am = torch.empty((M,), dtype=torch.int32, device=dev)
            ws = dg.workspace(dg.DG_OP_HEAD_FP8_ARGMAX, M, HEAD_N, HEAD_K, device=dev)
            add("head_fp8_argmax", {"M": M, "N": HEAD_N, "K": HEAD_K},
                [lambda x=x, logits=logits, am=am, ws=ws, Wq=Wq, scale=scale: dg.dg_head_fp8_argmax(
                    x, Wq, scale, logits, am, ws=ws, stream=stream)], HEAD_N * HEAD_K + 4)
        # --- MoE
        moe_on = need("moe_w1_silu", [{"M": M} for M in MOE_M]) or need("moe_w2", [{"M": M} for M in MOE_M])
        if moe_on:
            W1q, s1, W2q, s2 = S.moe_weights(MOE_E, MOE_I, MOE_K, MOE_K, device=dev)
        for M in MOE_M if moe_on else []:
            routs = [S.moe_inputs(M, MOE_K, MOE_TOPK, MOE_E, rep=r, device=dev) for r in range(8)]
            uniq = [len(set(r[1].cpu().flatten().tolist())) for r in routs]
            a = torch.empty((M, MOE_TOPK, MOE_I), dtype=torch.bfloat16, device=dev)
            yv = torch.empty((M, MOE_K), dtype=torch.bfloat16, device=dev)
            ws1 = dg.workspace(dg.DG_OP_MOE_W1, M, MOE_I, MOE_K, MOE_TOPK, device=dev)
            ws2 = dg.workspace(dg.DG_OP_MOE_W2, M, MOE_K, MOE_I, MOE_TOPK, device=dev)
            u_mean = sum(uniq) / len(uniq)
            b1 = u_mean * (2 * MOE_I * MOE_K + 2 * MOE_I * 4)
            b2 = u_mean * (MOE_K * MOE_I + MOE_K * 4)
            add("moe_w1_silu", {"M": M, "U_mean": u_mean},
                [(lambda r=r, a=a, ws1=ws1, W1q=W1q, s1=s1: dg.dg_moe_w1_silu(r[0], r[1], W1q, s1, a, ws=ws1, stream=stream))
                 for r in routs], b1)
            add("moe_w2", {"M": M, "U_mean": u_mean},
                [(lambda r=r, a=a, yv=yv, ws2=ws2, W2q=W2q, s2=s2: dg.dg_moe_w2(a, r[1], r[2], W2q, s2, yv, ws=ws2, stream=stream))
                 for r in routs], b2)

        # --- mid-M bf16 linear (129..512 token rows) on three shapes
        for (N, K) in MID_NK:
            if not need("gemv_mid_m", [{"M": M, "N": N, "K": K} for M in MID_M]):
                continue
            W0 = S.linear_inputs(1, N, K, device=dev)[1]
            wb = N * K * 2
            Wm = [W0] + [W0.clone() for _ in range(_copies_for(wb, l2) - 1)]
            for M in MID_M:
                x = S.linear_inputs(M, N, K, device=dev)[0]
                y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
                ws = dg.workspace(dg.DG_OP_GEMV_BF16, M, N, K, device=dev)
                add("gemv_mid_m", {"M": M, "N": N, "K": K, "tflops_per_call": round(2 * M * N * K / 1e12, 6)},
                    [(lambda W=W, x=x, y=y, ws=ws: dg.dg_gemv_bf16(x, W, y, ws=ws, stream=stream)) for W in Wm], wb,
                    launches_per_call=(M + 255) // 256)
            del Wm
        # --- A8W8 block-scaled linear with the activation quantisation fused in
        for (N, K) in A8_NK:
            if not need("gemv_a8w8", [{"M": M, "N": N, "K": K} for M in A8_M]):
                continue
            _, Wq0, sw = S.a8w8_inputs(1, N, K, device=dev)
            wb = N * K + sw.numel() * 4
            Wa = [Wq0] + [Wq0.clone() for _ in range(_copies_for(wb, l2) - 1)]
            for M in A8_M:
                x = S.normal_bf16((M, K), 1.0, S.seed_for("a8w8", "x", N, K, M), dev)
                y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
                ws = dg.workspace(dg.DG_OP_GEMV_A8W8, M, N, K, device=dev)
                sep = dg.dg_select(dg.DG_OP_GEMV_A8W8, M, N, K).params[1] == 1    # quantisation launch first
                add("gemv_a8w8", {"M": M, "N": N, "K": K, "quant": "separate launch" if sep else "fused"},
                    [(lambda W=W, x=x, y=y, ws=ws, sw=sw: dg.dg_gemv_a8w8_blockscale(x, W, sw, y, ws=ws, stream=stream))
                     for W in Wa], wb, launches_per_call=2 if sep else 1)
            del Wa
        # --- the bf16 sweep shapes at 1-8 rows in the batch-invariant numerics mode (the
        #     tcgen05 family where the fastest mode takes the CUDA cores or mma.sync)
        if need("gemv_bf16_invariant", [{"M": M, "N": N, "K": K} for (N, K) in SWEEP_NK for M in INV_M]):
            dg.dg_set_numerics(dg.DG_NUMERICS_BATCH_INVARIANT)
            try:
                for (N, K) in SWEEP_NK:
                    W0 = S.linear_inputs(1, N, K, device=dev)[1]
                    wb = N * K * 2
                    Wi = [W0] + [W0.clone() for _ in range(_copies_for(wb, l2) - 1)]
                    for M in INV_M:
                        x = S.linear_inputs(M, N, K, device=dev)[0]
                        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
                        ws = dg.workspace(dg.DG_OP_GEMV_BF16, M, N, K, device=dev)
                        add("gemv_bf16_invariant", {"M": M, "N": N, "K": K},
                            [(lambda W=W, x=x, y=y, ws=ws: dg.dg_gemv_bf16(x, W, y, ws=ws, stream=stream)) for W in Wi],
                            wb)
                    del Wi
            finally:
                dg.dg_set_numerics(dg.DG_NUMERICS_FASTEST)
        # --- chained pairs inside one graph (PDL lets the second kernel's prologue and
        #     first weight loads overlap the first one's tail): MLP gate/up -> down
        #     projection, and MoE W1 -> W2
        if need("chain_mlp", [{"M": M} for M in CHAIN_M]) and Ws:
            Nh, K = 12288, 4096
            Wd0 = S.linear_inputs(1, 4096, Nh, device=dev)[1]
            Wds = [Wd0, Wd0.clone()]
            for M in CHAIN_M:
                x = S.gate_up_inputs(M, Nh, K, device=dev)[0]
                h = torch.empty((M, Nh), dtype=torch.bfloat16, device=dev)
                yd = torch.empty((M, 4096), dtype=torch.bfloat16, device=dev)
                wsa = dg.workspace(dg.DG_OP_GATE_UP_SILU, M, Nh, K, device=dev)
                wsb = dg.workspace(dg.DG_OP_GEMV_BF16, M, 4096, Nh, device=dev)

                def pair(W, Wd, x=x, h=h, yd=yd, wsa=wsa, wsb=wsb):
                    dg.dg_gate_up_silu(x, W, h, ws=wsa, stream=stream)
                    dg.dg_gemv_bf16(h, Wd, yd, ws=wsb, stream=stream)
                add("chain_mlp", {"M": M},
                    [(lambda i=i, f=pair, wg=Ws, wd=Wds: f(wg[i % len(wg)], wd[i % 2]))
                     for i in range(max(len(Ws), 2))],
                    2 * Nh * K * 2 + 4096 * Nh * 2, launches_per_call=2)
        if moe_on and need("chain_moe", [{"M": M} for M in MOE_M]):
            for M in MOE_M:
                routs = [S.moe_inputs(M, MOE_K, MOE_TOPK, MOE_E, rep=r, device=dev) for r in range(8)]
                uniq = [len(set(r[1].cpu().flatten().tolist())) for r in routs]
                u_mean = sum(uniq) / len(uniq)
                a = torch.empty((M, MOE_TOPK, MOE_I), dtype=torch.bfloat16, device=dev)
                yv = torch.empty((M, MOE_K), dtype=torch.bfloat16, device=dev)
                ws1 = dg.workspace(dg.DG_OP_MOE_W1, M, MOE_I, MOE_K, MOE_TOPK, device=dev)
                ws2 = dg.workspace(dg.DG_OP_MOE_W2, M, MOE_K, MOE_I, MOE_TOPK, device=dev)

                def pair(r, a=a, yv=yv, ws1=ws1, ws2=ws2):
                    dg.dg_moe_w1_silu(r[0], r[1], W1q, s1, a, ws=ws1, stream=stream)
                    dg.dg_moe_w2(a, r[1], r[2], W2q, s2, yv, ws=ws2, stream=stream)
                add("chain_moe", {"M": M, "U_mean": u_mean}, [(lambda r=r, f=pair: f(r)) for r in routs],
                    u_mean * (3 * MOE_I * MOE_K + 2 * MOE_I * 4 + MOE_K * 4), launches_per_call=2)

    n_cases = len(cases)
    if n_cases == 0:
        raise SystemExit(f"no benchmark case matches --cases {args.cases!r} / --only {args.only!r}")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_cases)]
    times = [[] for _ in range(n_cases)]

    def one_step(record):
        for i, (_, _, g, _) in enumerate(cases):
            if record:
                ev[i][0].record(stream)
            g.replay()
            if record:
                ev[i][1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one_step(False)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = ClockSampler(local)
    clocks.start()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    step_ms = []
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            one_step(True)
            stream.synchronize()
            for i in range(n_cases):
                times[i].append(ev[i][0].elapsed_time(ev[i][1]) * 1e3 / R)   # µs per call
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if world > 1:
        dist.barrier()
    clk = clocks.stop()

    # ---- shape-table arm: the same sweep with the compiled defaults, timed the same way
    defaults = []
    if dcases:
        dev_ = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in dcases]
        dts = [[] for _ in dcases]
        with torch.cuda.stream(stream):
            for step in range(args.warmup + args.steps):
                for i, (_, g, _) in enumerate(dcases):
                    dev_[i][0].record(stream)
                    g.replay()
                    dev_[i][1].record(stream)
                stream.synchronize()
                if step >= args.warmup:
                    for i in range(len(dcases)):
                        dts[i].append(dev_[i][0].elapsed_time(dev_[i][1]) * 1e3 / R)
        defaults = [dict(**meta, us=round(statistics.median(t), 3), weight_bytes=int(wb))
                    for (meta, _, wb), t in zip(dcases, dts)]

    # ---- cold single calls (outside the timed region): L2 flushed before each call
    cold = None
    if not args.no_cold and sweep_cases:
        flush = torch.empty(max(2 * l2, 1 << 28), dtype=torch.uint8, device=dev)
        cev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        cold_us = {}
        with torch.cuda.stream(stream):
            for i in sweep_cases:
                call = keep[i][0]
                ts = []
                for _ in range(5):
                    flush.fill_(1)
                    cev[0].record(stream)
                    call()
                    cev[1].record(stream)
                    stream.synchronize()
                    ts.append(cev[0].elapsed_time(cev[1]) * 1e3)
                cold_us[i] = statistics.median(ts)
        del flush
        cb = sum(cases[i][3] for i in sweep_cases)
        ct = sum(cold_us.values())
        cold = {"value": round(cb / (ct * 1e-6) / 1e9, 1), "unit": "GB/s", "us_per_step": round(ct, 1),
                "method": "each sweep call alone, eager, after writing a 2xL2 buffer; CUDA events around "
                          "the call on its stream; median of 5",
                "us": {case_id(cases[i][0], cases[i][1]): round(cold_us[i], 3) for i in sweep_cases}}

    def summarize(i):
        name, meta, _, wb = cases[i]
        us = statistics.median(times[i])
        gbs = wb / (us * 1e-6) / 1e9
        return dict(op=name, **meta, us=round(us, 3), gbs=round(gbs, 1), frac=round(gbs / peak, 4),
                    weight_bytes=int(wb))

    sweep = [summarize(i) for i in sweep_cases]
    if not sweep:                       # profiling runs of other ops: report their totals
        sweep = [summarize(i) for i in range(n_cases)]
    step_us = sum(s["us"] for s in sweep)
    step_bytes = sum(s["weight_bytes"] for s in sweep)
    value_rank = step_bytes / (step_us * 1e-6) / 1e9
    step_us = _max_over_ranks(step_us, dev)
    value = _job_value(world, step_bytes, step_us)
    small = [s for s in sweep if s["M"] <= 16]
    # Which kernel family the dispatch sends each sweep shape to; the roofline is
    # reported for the family that takes the most time.
    fam_names = {dg.DG_VAR_CC_WARP: "cc_dense_kernel", dg.DG_VAR_CC_BULK: "cc_bulk_kernel",
                 dg.DG_VAR_TC: "tc_dense_kernel", dg.DG_VAR_MMA: "mw_dense_kernel"}
    by_kernel = {}
    for s_ in sweep:
        v = dg.dg_select(dg.DG_OP_GEMV_BF16, s_["M"], s_["N"], s_["K"]).variant if s_["op"] == "gemv_bf16" else -1
        k = by_kernel.setdefault(fam_names.get(v, "other"), {"us": 0.0, "bytes": 0, "launches_per_step": 0})
        k["us"] += s_["us"]
        k["bytes"] += s_["weight_bytes"]
        k["launches_per_step"] += 1
    for k in by_kernel.values():
        k["achieved"] = round(k["bytes"] / (k["us"] * 1e-6) / 1e9, 1)
        k["frac"] = round(k["achieved"] / peak, 4)
        k["us"] = round(k["us"], 3)
    dominant = max(by_kernel, key=lambda n: by_kernel[n]["us"]) if by_kernel else None
    ops = {}
    for i in range(n_cases):
        if i in sweep_cases:
            continue
        s = summarize(i)
        ops.setdefault(s["op"], []).append(s)
    for c in ops.get("gemv_mid_m", []):
        c["tflops"] = round(c["tflops_per_call"] / (c["us"] * 1e-6), 1)
    sweep_us = {(s_["M"], s_["N"], s_["K"]): s_["us"] for s_ in sweep if "N" in s_}
    for c in ops.get("gemv_bf16_invariant", []):
        c["fastest_mode_us"] = sweep_us.get((c["M"], c["N"], c["K"]))
    # chained pairs: the same two calls measured on their own, for the PDL overlap
    sweep_by = {(s_["M"], s_["N"], s_["K"]): s_["us"] for s_ in sweep if "N" in s_}
    for c in ops.get("chain_mlp", []):
        gu = next((o["us"] for o in ops.get("gate_up_silu", []) if o["M"] == c["M"]), None)
        dn = sweep_by.get((c["M"], 4096, 12288))
        if gu is not None and dn is not None:
            c["parts_us"] = round(gu + dn, 3)
    for c in ops.get("chain_moe", []):
        w1 = next((o["us"] for o in ops.get("moe_w1_silu", []) if o["M"] == c["M"]), None)
        w2 = next((o["us"] for o in ops.get("moe_w2", []) if o["M"] == c["M"]), None)
        if w1 is not None and w2 is not None:
            c["parts_us"] = round(w1 + w2, 3)

    # ---- e2e through the public API with host buffers (x in, y out, pinned)
    e2e = _e2e(torch, dg, S, dev, stream, args, l2) if only is None and not args.cases else None

    launches = args.steps * R * sum(kernels)
    res = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_us / 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,1/K) weights; no dataset)",
        "config": {"workload": WORKLOAD, "calls_per_step": len(sweep),
                   "l2_defeat": f"weights rotate over >= 3x L2 ({l2 // 2**20} MiB) of copies inside "
                                f"CUDA graphs of {R} calls",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "build_id": dg.dg_build_id()},
        "roofline": {"bound": "hbm",
                     "achieved": by_kernel[dominant]["achieved"] if dominant else round(value_rank, 1),
                     "peak": peak, "unit": "GB/s",
                     "frac": by_kernel[dominant]["frac"] if dominant else round(value_rank / peak, 4),
                     **_traffic(dg, dominant),
                     "peak_source": peak_src, "kernel": dominant,
                     "achieved_definition": "weight bytes of the kernel's sweep launches / their summed "
                                            "CUDA-event time",
                     "by_kernel": by_kernel,
                     "sweep_frac": round(value_rank / peak, 4),
                     "frac_m_le_16": (round(sum(s["weight_bytes"] for s in small) /
                                            (sum(s["us"] for s in small) * 1e-6) / 1e9 / peak, 4)
                                      if small else None)},
        "clocks": clk,
        "e2e": e2e,
        "cold": cold,
        "gpu_launches": launches,
        "shapes": sweep,
        "ops": ops,
        "timed_wall_s": round(wall, 3),
    }
    if table is not None:
        res["table"] = _table_report(table, args.table, dg, defaults, sweep, peak)
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res))


def _table_shapes(dg):
    """Every decode shape this benchmark times, as dg_sweep requests."""
    sh = [(dg.DG_OP_GEMV_BF16, M, N, K, 0, 0) for (N, K) in SWEEP_NK for M in SWEEP_M]
    sh.append((dg.DG_OP_GEMV_BF16, 1, 2048, 1024, 0, 0))
    sh += [(dg.DG_OP_GATE_UP_SILU, M, 12288, 4096, 0, 0) for M in GATE_UP_M]
    sh += [(dg.DG_OP_HEAD_FP8_ARGMAX, M, HEAD_N, HEAD_K, 0, 0) for M in HEAD_M]
    sh += [(dg.DG_OP_MOE_W1, M, MOE_I, MOE_K, MOE_TOPK, MOE_E) for M in MOE_M]
    sh += [(dg.DG_OP_MOE_W2, M, MOE_K, MOE_I, MOE_TOPK, MOE_E) for M in MOE_M]
    return sh


def _table_report(table, path, dg, defaults, sweep, peak):
    """The headline sweep with the loaded table against the compiled defaults (timed
    in steps of their own, the same way), plus the table's identity and the entries
    that differ."""
    by = {(d["M"], d["N"], d["K"]): d for d in defaults}
    rows, b_def, t_def = [], 0, 0.0
    for s_ in sweep:
        d = by.get((s_["M"], s_["N"], s_["K"]))
        if d is None:
            continue
        b_def += d["weight_bytes"]
        t_def += d["us"]
        rows.append({"M": s_["M"], "N": s_["N"], "K": s_["K"], "us_table": s_["us"], "us_default": d["us"]})
    changed = [e for e in table.get("entries", []) if e.get("pick") != e.get("default")]
    v_def = b_def / (t_def * 1e-6) / 1e9 if t_def > 0 else None
    return {"path": os.path.basename(path), "identity": table.get("identity"),
            "entries": dg.dg_table_entries(), "entries_not_default": len(changed),
            "defaults_value": round(v_def, 1) if v_def else None,
            "defaults_frac": round(v_def / peak, 4) if v_def else None,
            "changed": [{k: e.get(k) for k in ("op", "M", "N", "K", "pick", "pick_us", "default_us")}
                        for e in changed],
            "shapes": rows}


def _e2e(torch, dg, S, dev, stream, args, l2):
    """Whole sweep step through the Python API with host buffers: every call's x
    comes in from pinned host memory in one copy, every y goes back out in one."""
    weights = {(N, K): S.linear_inputs(1, N, K, device=dev)[1] for (N, K) in SWEEP_NK}
    shapes = [(M, N, K) for M in SWEEP_M for (N, K) in SWEEP_NK]
    xs_host = [S.linear_inputs(M, N, K)[0] for (M, N, K) in shapes]
    x_off, y_off = [0], [0]
    for (M, N, K) in shapes:
        x_off.append(x_off[-1] + M * K + (-(M * K)) % 8)      # 16-byte aligned slices
        y_off.append(y_off[-1] + M * N + (-(M * N)) % 8)
    xh = torch.empty(x_off[-1], dtype=torch.bfloat16).pin_memory()
    for x, (M, N, K), o in zip(xs_host, shapes, x_off):
        xh[o:o + M * K].copy_(x.reshape(-1))
    yh = torch.empty(y_off[-1], dtype=torch.bfloat16).pin_memory()
    xd = torch.empty_like(xh, device=dev)
    yd = torch.empty_like(yh, device=dev)
    # Every call of the step reads its own copy of the weights (the step's 40 copies
    # together are many times L2), so no call finds its weights in L2.
    items = []
    wbytes = 0
    for i, (M, N, K) in enumerate(shapes):
        items.append((xd[x_off[i]:x_off[i] + M * K].view(M, K), weights[(N, K)].clone(),
                      yd[y_off[i]:y_off[i] + M * N].view(M, N), dg.workspace(dg.DG_OP_GEMV_BF16, M, N, K, device=dev)))
        wbytes += N * K * 2
    h2d = sum(M * K * 2 for (M, N, K) in shapes)
    d2h = sum(M * N * 2 for (M, N, K) in shapes)

    def issue():
        xd.copy_(xh, non_blocking=True)
        for x, W, y, ws in items:
            dg.dg_gemv_bf16(x, W, y, ws=ws, stream=stream)
        yh.copy_(yd, non_blocking=True)

    def eager_step():
        with torch.cuda.stream(stream):
            issue()
        torch.cuda.synchronize()

    # The same step captured once as a CUDA graph (the library's calls are capturable):
    # every replay still copies x in from pinned host memory and y back out.
    with torch.cuda.stream(stream):
        issue()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        issue()

    def graph_step():
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()

    def timed(step):
        for _ in range(3):
            step()
        n = max(3, min(args.steps, 50))
        t0 = time.perf_counter()
        for _ in range(n):
            step()
        return (time.perf_counter() - t0) / n

    dt_graph = timed(graph_step)
    dt_eager = timed(eager_step)
    # the result really came back: spot-check one call against the device output
    assert torch.equal(yh[y_off[0]:y_off[1]].view(torch.int16), yd[y_off[0]:y_off[1]].cpu().view(torch.int16))
    return {"value": round(wbytes / dt_graph / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(dt_graph * 1e3, 3),
            "eager_value": round(wbytes / dt_eager / 1e9, 1), "eager_ms_per_step": round(dt_eager * 1e3, 3),
            "note": "wall clock per step on the host, synchronised every step; weights stay resident "
                    "(model parameters), one copy per call so that none is re-read from L2; each step "
                    "copies all 40 calls' x in from pinned host memory (one copy) and their y back out "
                    "(one copy).  value: the step replayed from one CUDA graph; eager_value: the same "
                    "calls issued one by one from Python"}


def _traffic(dg, kernel):
    """DRAM bytes per launch of `kernel` from its committed ncu summary
    (profiles/traffic_<kernel>.txt), only if that capture was taken on this build."""
    out = {"traffic": None}
    if not kernel:
        return out
    p = os.path.join(ROOT, "profiles", f"traffic_{kernel}.txt")
    try:
        kv = {}
        with open(p) as f:
            for ln in f:
                if ":" in ln and not ln.startswith("#"):
                    k, v = ln.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("build_id") != dg.dg_build_id():
            return out
        return {"traffic": float(kv["dram_bytes_per_launch"]), "traffic_shape": kv.get("shape"),
                "traffic_algorithmic_bytes": float(kv["algorithmic_bytes_per_launch"])}
    except (OSError, KeyError, ValueError):
        return out


# ----------------------------------------------------------------------------- CPU baseline

def _oracle_sweep_sample(budget_s: float, rows_frac: int = 8):
    """Time the fp64 oracle on the sweep shapes, every `rows_frac`-th weight row,
    in whole passes over all 40 shapes until about `budget_s` of work is done."""
    import numpy as np
    import torch

    from oracle import oracle as O
    from synth import decode_inputs as S

    O.lib()
    mats = []
    for (N, K) in SWEEP_NK:
        rows = np.arange(0, N, rows_frac, dtype=np.int64)
        g = torch.Generator().manual_seed(N * 7 + K)
        Wsub = (torch.randn((len(rows), K), generator=g) * K ** -0.5).to(torch.bfloat16)
        xs = [S.linear_inputs(M, 8, K, tag="cpu")[0].view(torch.int16).numpy().view(np.uint16) for M in SWEEP_M]
        mats.append((Wsub.view(torch.int16).numpy().view(np.uint16), xs))
    total_b = 0.0
    total_t = 0.0
    passes = 0
    while True:
        for Wb, xs in mats:
            for xb in xs:
                t0 = time.perf_counter()
                O.linear_bf16(xb, Wb)
                total_t += time.perf_counter() - t0
                total_b += Wb.size * 2
        passes += 1
        if total_t >= budget_s or passes >= 1000:
            break
    return total_b, total_t, f"{passes} pass(es) over every {rows_frac}th weight row of all 40 sweep shapes"


def _cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (x86 'model name', or Arm implementer/part)."""
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model", "CPU part"):
        m = re.search(rf"^{key}\s*:\s*(.+)$", info, re.M)
        if m:
            return (key + " " if key == "CPU part" else "") + m.group(1).strip()
    return "unknown"


def cpu_baseline(budget_s: float):
    b, t, sample = _oracle_sweep_sample(budget_s)
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return {"value": round(b / t / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "cpu_model": _cpu_model(), "nproc": os.cpu_count(),
            "sample": sample + f"; {t:.1f} s of fp64 oracle work (OpenMP over outputs, {cores} threads), "
                               "GB/s of weight bytes covered"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return
    budget = max(0.5, args.cpu_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        _oracle_sweep_sample(budget, rows_frac=64)
    b_tot = t_tot = 0.0
    sample = ""
    for _ in range(args.steps):
        b, t, sample = _oracle_sweep_sample(budget, rows_frac=64)
        b_tot += b
        t_tot += t
    value = b_tot / t_tot / 1e9
    cores = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
           "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(t_tot / max(1, args.steps) * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": WORKLOAD},
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                            "cpu_model": _cpu_model(), "nproc": os.cpu_count(),
                            "sample": sample},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--reps", type=int, default=16, help="calls per captured graph")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sweep-only", action="store_true", help="only the headline sweep (no other ops)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cold", action="store_true", help="skip the cold single-call timings")
    ap.add_argument("--only", default="", help="profiling: one sweep shape 'M,N,K' (no other ops, no e2e)")
    ap.add_argument("--cases", default="", help="profiling: regex over case ids such as 'moe_w2/M16' or "
                    "'head_fp8_argmax/M8/N248320/K4096' (only matching cases are built and timed)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--table", default="", help="dispatch through this shape table (dg_sweep JSON); the "
                    "headline shapes are also timed with the compiled defaults")
    ap.add_argument("--sweep-table", action="store_true", help="measure the table first (dg_sweep over "
                    "every shape this benchmark times; resumes a partial table of this build)")
    ap.add_argument("--sweep-reps", type=int, default=20)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
