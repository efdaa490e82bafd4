"""Benchmark of the block-causal attention hot path on one B300 (or N replicas).

A step is one pass of the whole hot path over one batch of the Minecraft 1.6B dynamics
layer shapes (B=1, T=256, S=290, 30 Q / 3 KV heads, head_dim 64, window 192, agent 289):
space attention forward, time attention forward, and (when enabled) both backward passes.
Metric: algorithmic TFLOP/s (allowed query-key pairs only; a backward counts 2.5 forward).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --workload minecraft_decode     # the rollout decode step (GB/s)
    python bench.py --workload tokenizer_enc --varlen   # space attention, dropped MAE patches

--impl reference times the fp64 CPU oracle (the only reference this project has) on a
bounded sample of the same workload.  Under torchrun each rank runs an independent replica
(the operator has no cross-GPU exchange); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_causal_video_attention_b300 import synth  # noqa: E402

METRIC = "space/time attention TFLOP/s (fwd, fwd+bwd) and % of B300 bf16 roofline"
UNIT = "TFLOP/s"


def pairs_space(w):
    n = w.S * w.S - (w.S - 1 if w.agent >= 0 else 0)
    return n * w.B * w.T * w.Hq


def pairs_time(w):
    n = sum(min(t + 1, w.window) for t in range(w.T))
    return n * w.B * w.S * w.Hq


def flops(w):
    """Algorithmic FLOPs per op: 4*D per allowed (query, key) pair and head; bwd = 2.5x."""
    f = {"space_fwd": 4.0 * w.D * pairs_space(w), "time_fwd": 4.0 * w.D * pairs_time(w)}
    f["space_bwd"] = 2.5 * f["space_fwd"]
    f["time_bwd"] = 2.5 * f["time_fwd"]
    return f


def fwd_bytes(w):
    rows = w.B * w.T * w.S
    return rows * (2 * w.Hq * w.D * 2 + 2 * w.Hkv * w.D * 2 + 4 * w.Hq)


def bwd_bytes(w):
    rows = w.B * w.T * w.S
    # read Q, K, V, O, dO, LSE; write dQ, dK, dV
    return rows * (3 * w.Hq * w.D * 2 + 2 * w.Hkv * w.D * 2 + 4 * w.Hq + w.Hq * w.D * 2
                   + 2 * w.Hkv * w.D * 2)


# DRAM bytes (read + write) per call of an operator, summed over its kernels, from one ncu
# capture of `python bench.py --op <op> --steps 1 --warmup 1 --no-cpu-baseline` with
# --metrics dram__bytes_read.sum,dram__bytes_write.sum (summary in profiles/).  They hold only
# for the kernel sources they were measured on: any change to those sources voids them.
MEASURED_TRAFFIC = {
    "csrc_sha256": "5621d56d5edc540aca42aa831a0c4027c0d688e687a7903a7590dae10fdbfd00",
    "minecraft_fwd_bwd": {
        # forward with the O residual; backward: K/V ranges, dQ (with Delta from O + O_lo), dK/dV
        "space_fwd": 919082189,
        "time_fwd": 915951053,
        "space_bwd": 2311614208,
        "time_bwd": 2317548902,
    },
    # decode: 4-rollout capture (176.42 MB read, 2.57 MB written, mean of 5 calls) scaled by
    # the units (x4); taken on sources whose decode kernel (od_decode.cuh and the helpers it
    # uses) is the same as these
    "minecraft_decode": {"decode": 715973837},
}


def csrc_digest():
    d = os.path.join(ROOT, "block_causal_video_attention_b300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(d)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(f.encode())
            with open(os.path.join(d, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()


def measured_traffic(workload, op):
    if csrc_digest() != MEASURED_TRAFFIC["csrc_sha256"]:
        return None
    return MEASURED_TRAFFIC.get(workload, {}).get(op)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6400.0, 1800.0, 1400.0, "fallback"


class Clocks:
    """Samples nvidia-smi SM clocks and throttle reasons while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu):
        self.gpu = gpu
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.time()
            while not self.rows and time.time() - t0 < 5.0:   # wait for the first sample
                time.sleep(0.02)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for n, val in zip(names, r[5:9]):
                    if val.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                pass
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x, device=None):
    """Largest value of `x` over all ranks (the slowest replica sets the job's time)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flop_per_step_per_rank, world, steps, ms):
    """Whole-job throughput: every rank runs its own replica of the step (weak scaling)."""
    return world * flop_per_step_per_rank * steps / (ms * 1e-3) / 1e12


# ----------------------------------------------------------------------------- CPU oracle
_INPUTS = {}


def oracle_sample(w, nunits, with_bwd):
    """Time the fp64 oracle on `nunits` whole units of each op; returns (flop, seconds,
    threads, description).  The workload's inputs are generated once per process."""
    import oracle
    oracle.build()
    if w.name not in _INPUTS:
        _INPUTS[w.name] = synth.make_inputs(w, with_dout=True)
    q, k, v, dout = _INPUTS[w.name]
    G = w.G
    rng = np.random.default_rng(1234)
    f = flops(w)
    tot_flop, tot_s = 0.0, 0.0
    units_space = w.B * w.T * w.Hkv
    units_time = w.B * w.S * w.Hkv
    per_unit = {"space_fwd": f["space_fwd"] / units_space, "time_fwd": f["time_fwd"] / units_time,
                "space_bwd": f["space_bwd"] / units_space, "time_bwd": f["time_bwd"] / units_time}
    # gather sub-problems: nunits space units stacked as B, same for time
    sb = [(int(rng.integers(w.B)), int(rng.integers(w.T)), int(rng.integers(w.Hkv))) for _ in range(nunits)]
    tb = [(int(rng.integers(w.B)), int(rng.integers(w.S)), int(rng.integers(w.Hkv))) for _ in range(nunits)]
    X = oracle.from_bf16
    sq = np.concatenate([X(q[b:b+1, t:t+1, :, h*G:(h+1)*G]) for b, t, h in sb])
    sk = np.concatenate([X(k[b:b+1, t:t+1, :, h:h+1]) for b, t, h in sb])
    sv = np.concatenate([X(v[b:b+1, t:t+1, :, h:h+1]) for b, t, h in sb])
    sd = np.concatenate([X(dout[b:b+1, t:t+1, :, h*G:(h+1)*G]) for b, t, h in sb])
    tq = np.concatenate([X(q[b:b+1, :, s:s+1, h*G:(h+1)*G]) for b, s, h in tb])
    tk = np.concatenate([X(k[b:b+1, :, s:s+1, h:h+1]) for b, s, h in tb])
    tv = np.concatenate([X(v[b:b+1, :, s:s+1, h:h+1]) for b, s, h in tb])
    td = np.concatenate([X(dout[b:b+1, :, s:s+1, h*G:(h+1)*G]) for b, s, h in tb])
    nth = oracle.num_threads(0)
    t0 = time.perf_counter()
    if with_bwd:
        oracle.space_bwd(sq, sk, sv, sd, w.agent, w.scale)
        oracle.time_bwd(tq, tk, tv, td, w.window, w.scale)
        tot_flop = nunits * (per_unit["space_fwd"] + per_unit["space_bwd"] + per_unit["time_fwd"]
                             + per_unit["time_bwd"])
    else:
        oracle.space_fwd(sq, sk, sv, w.agent, w.scale)
        oracle.time_fwd(tq, tk, tv, w.window, w.scale)
        tot_flop = nunits * (per_unit["space_fwd"] + per_unit["time_fwd"])
    tot_s = time.perf_counter() - t0
    desc = "%d space units (b,t,kv head) + %d time units (b,s,kv head) of %s, %s" % (
        nunits, nunits, w.name, "fwd+bwd" if with_bwd else "fwd")
    return tot_flop, tot_s, nth, desc


def oracle_full(w, with_bwd, chunk=48):
    """Time the fp64 oracle on every unit of the workload (all B*T*Hkv space units and all
    B*S*Hkv time units, `chunk` units per oracle call to bound host memory); returns
    (flop, seconds, threads, description) like oracle_sample."""
    import oracle
    oracle.build()
    if w.name not in _INPUTS:
        _INPUTS[w.name] = synth.make_inputs(w, with_dout=True)
    q, k, v, dout = _INPUTS[w.name]
    G = w.G
    X = oracle.from_bf16
    f = flops(w)
    units_space = [(b, t, h) for b in range(w.B) for t in range(w.T) for h in range(w.Hkv)]
    units_time = [(b, s_, h) for b in range(w.B) for s_ in range(w.S) for h in range(w.Hkv)]
    nth = oracle.num_threads(0)
    tot_s = 0.0
    for kind, units in (("space", units_space), ("time", units_time)):
        for c0 in range(0, len(units), chunk):
            part = units[c0:c0 + chunk]
            if kind == "space":
                sl = [(slice(b, b + 1), slice(t, t + 1), slice(None)) for b, t, h in part]
            else:
                sl = [(slice(b, b + 1), slice(None), slice(s_, s_ + 1)) for b, s_, h in part]
            hs = [h for _, _, h in part]
            cq = np.concatenate([X(q[a + (slice(h * G, (h + 1) * G),)]) for a, h in zip(sl, hs)])
            ck = np.concatenate([X(k[a + (slice(h, h + 1),)]) for a, h in zip(sl, hs)])
            cv = np.concatenate([X(v[a + (slice(h, h + 1),)]) for a, h in zip(sl, hs)])
            cd = np.concatenate([X(dout[a + (slice(h * G, (h + 1) * G),)]) for a, h in zip(sl, hs)])
            extra = w.agent if kind == "space" else w.window
            t0 = time.perf_counter()
            if with_bwd:
                getattr(oracle, kind + "_bwd")(cq, ck, cv, cd, extra, w.scale)
            else:
                getattr(oracle, kind + "_fwd")(cq, ck, cv, extra, w.scale)
            tot_s += time.perf_counter() - t0
    ops = ["space_fwd", "time_fwd"] + (["space_bwd", "time_bwd"] if with_bwd else [])
    tot_flop = sum(f[o] for o in ops)
    desc = "the whole %s workload: %d space units + %d time units, %s" % (
        w.name, len(units_space), len(units_time), "fwd+bwd" if with_bwd else "fwd")
    return tot_flop, tot_s, nth, desc


def varlen_config(w, lengths):
    """The `config` object of a variable-length line; both arms print the same one."""
    return {"workload": w.name + "_varlen", "B": w.B, "T": w.T, "S_max": w.S,
            "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.D,
            "tokens_per_block": {"mean": float(lengths.mean()),
                                 "min": int(lengths.min()), "max": int(lengths.max())},
            "ops": ["space_fwd", "space_bwd"], "l2": "inputs larger than L2",
            "parallelism": "single GPU"}


def fwd_bwd_config(args, w, with_bwd, world, ops):
    """The `config` object of a fwd/bwd line; both arms print the same one."""
    return {"workload": w.name, "B": w.B, "T": w.T, "S": w.S, "Hq": w.Hq,
            "Hkv": w.Hkv, "head_dim": w.D, "window": w.window, "agent": w.agent,
            "ops": ops, "delta": ("recomputed from P and dP" if (not with_bwd or args.no_residual)
                                  else "from O + O_lo (forward writes the residual)"),
            "qkv": "packed [B,T,S,Hq+2Hkv,D]" if args.packed else "separate",
            "l2": "inputs larger than L2 (Q alone %.0f MB)" % (w.B * w.T * w.S * w.Hq * w.D * 2 / 1e6),
            "parallelism": "replicas" if world > 1 else "single GPU"}


def run_reference(args, w, with_bwd):
    rank, world, _ = dist_info()
    if rank != 0:
        return
    nunits = args.ref_units
    vals = []
    for _ in range(args.warmup if args.warmup < 1 else 1):
        oracle_sample(w, max(1, nunits // 8), with_bwd)
    for _ in range(args.steps):
        if args.oracle_full:
            fl, s, nth, desc = oracle_full(w, with_bwd)
        else:
            fl, s, nth, desc = oracle_sample(w, nunits, with_bwd)
        vals.append((fl, s))
    fl = sum(v[0] for v in vals)
    s = sum(v[1] for v in vals)
    value = fl / s / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": fwd_bwd_config(args, w, with_bwd, world,
                                     ["space_fwd", "time_fwd"] + (["space_bwd", "time_bwd"] if with_bwd else [])),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nth, "kind": "oracle",
                             "sample": desc + " per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU path
def run_ours(args, w, with_bwd):
    import torch
    import torch.distributed as dist
    from block_causal_video_attention_b300 import api

    rank, world, local = dist_info()
    torch.cuda.set_device(local)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)

    q, k, v, dout = synth.make_inputs(w, with_dout=True)
    to = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    hq, hk, hv, hd = (to(a).pin_memory() for a in (q, k, v, dout))
    dq, dk, dv, dd = (t.to(dev) for t in (hq, hk, hv, hd))
    stream = torch.cuda.current_stream()
    o_s = torch.empty_like(dq)
    o_t = torch.empty_like(dq)
    l_s = torch.empty(dq.shape[:4], dtype=torch.float32, device=dev)
    l_t = torch.empty_like(l_s)
    ops = ["space_fwd", "time_fwd"]
    if with_bwd:
        ops += ["space_bwd", "time_bwd"]
    if args.op:
        if args.op not in ops:
            raise SystemExit("--op %s is not part of workload %s" % (args.op, w.name))
        ops = [args.op]
    run = set(ops)
    packed = bool(args.packed)
    if packed:
        # one fused-projection tensor [B,T,S,Hq+2Hkv,D] instead of three
        dqkv_in = torch.cat([dq, dk, dv], dim=3).contiguous()
    if with_bwd:
        g = [torch.empty_like(x) for x in (dq, dk, dv, dq, dk, dv)]
        if packed:
            g_packed = [torch.empty_like(dqkv_in), torch.empty_like(dqkv_in)]
        ws_s = torch.empty(max(api.bwd_workspace_bytes(0, w.B, w.T, w.S, w.Hq, w.Hkv), 16),
                           dtype=torch.uint8, device=dev)
        ws_t = torch.empty(max(api.bwd_workspace_bytes(1, w.B, w.T, w.S, w.Hq, w.Hkv), 16),
                           dtype=torch.uint8, device=dev)

    ev = {op: [] for op in ops}
    # the forward also writes O's rounding residual so that the backward reads Delta from
    # memory (unless --no-residual: then the backward recomputes it from P and dP)
    lo_s = lo_t = None
    if with_bwd and not args.no_residual:
        lo_s, lo_t = torch.empty_like(dq), torch.empty_like(dq)

    def step(record, Q=dq, K=dk, V=dv, DO=dd, QKV=None):
        if packed:
            return step_packed(record, dqkv_in if QKV is None else QKV, DO)

        def timed(op, fn):
            if record:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                ev[op].append((a, b))
            else:
                fn()
        if "space_fwd" in run:
            timed("space_fwd", lambda: api.space_attn_fwd(Q, K, V, w.agent, w.scale, o_s, l_s, stream,
                                                          o_lo=lo_s))
        if "time_fwd" in run:
            timed("time_fwd", lambda: api.time_attn_fwd(Q, K, V, w.window, w.scale, o_t, l_t, stream,
                                                        o_lo=lo_t))
        if "space_bwd" in run:
            timed("space_bwd", lambda: api.space_attn_bwd(Q, K, V, o_s, l_s, DO, w.agent, w.scale,
                                                          workspace=ws_s, out=g[:3], stream=stream,
                                                          o_lo=lo_s))
        if "time_bwd" in run:
            timed("time_bwd", lambda: api.time_attn_bwd(Q, K, V, o_t, l_t, DO, w.window, w.scale,
                                                        workspace=ws_t, out=g[3:], stream=stream,
                                                        o_lo=lo_t))

    def step_packed(record, QKV, DO):
        def timed(op, fn):
            if record:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                ev[op].append((a, b))
            else:
                fn()
        if "space_fwd" in run:
            timed("space_fwd", lambda: api.space_attn_fwd_packed(QKV, w.Hq, w.agent, w.scale, o_s, l_s,
                                                                 stream, o_lo=lo_s))
        if "time_fwd" in run:
            timed("time_fwd", lambda: api.time_attn_fwd_packed(QKV, w.Hq, w.window, w.scale, o_t, l_t,
                                                               stream, o_lo=lo_t))
        if "space_bwd" in run:
            timed("space_bwd", lambda: api.space_attn_bwd_packed(
                QKV, w.Hq, o_s, l_s, DO, w.agent, w.scale, workspace=ws_s, out=g_packed[0], stream=stream,
                o_lo=lo_s))
        if "time_bwd" in run:
            timed("time_bwd", lambda: api.time_attn_bwd_packed(
                QKV, w.Hq, o_t, l_t, DO, w.window, w.scale, workspace=ws_t, out=g_packed[1], stream=stream,
                o_lo=lo_t))

    if args.op and args.op.endswith("_bwd"):
        # the backward reads the forward's O and LSE: produce them once, outside the timing
        if args.op == "space_bwd":
            api.space_attn_fwd(dq, dk, dv, w.agent, w.scale, o_s, l_s, stream, o_lo=lo_s)
        else:
            api.time_attn_fwd(dq, dk, dv, w.window, w.scale, o_t, l_t, stream, o_lo=lo_t)
    clk = Clocks(local).__enter__()
    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize()
    if api.get_device_status() != 0:
        raise RuntimeError("device timeout during warm-up")
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(args.steps):
        step(True)
    end.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end), dev)
    if api.get_device_status() != 0:
        raise RuntimeError("device timeout during the timed region")
    f = flops(w)
    step_flop = sum(f[o] for o in ops)
    value = job_tflops(step_flop, world, args.steps, ms)
    per_op = {}
    for op in ops:
        t_ms = float(np.mean([a.elapsed_time(b) for a, b in ev[op]]))
        per_op[op] = {"ms": t_ms, "tflops": f[op] / (t_ms * 1e-3) / 1e12}

    # end to end: pinned host inputs -> device, the step, results back to pinned host memory
    outs = [o_s, l_s, o_t, l_t] + ((g_packed if packed else g) if with_bwd else [])
    hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    if packed:
        hqkv = dqkv_in.cpu().pin_memory()
        hin = [hqkv] + ([hd] if with_bwd else [])
        din = [torch.empty_like(dqkv_in), torch.empty_like(dd)]
    else:
        hin = [hq, hk, hv] + ([hd] if with_bwd else [])
        din = [torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv), torch.empty_like(dd)]
    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = sum(t.numel() * t.element_size() for t in hout)

    def e2e_step():
        for h, d in zip(hin, din):
            d.copy_(h, non_blocking=True)
        if packed:
            step(False, DO=din[1], QKV=din[0])
        else:
            step(False, din[0], din[1], din[2], din[3])
        for d, h in zip(outs, hout):
            h.copy_(d, non_blocking=True)
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    clk.__exit__()
    e2e_ms = max_over_ranks(a.elapsed_time(b), dev)
    e2e = job_tflops(step_flop, world, args.steps, e2e_ms)

    hbm, tc, tc_sus, src = load_peaks()
    # dominant kernel: the op with the largest share of device time
    dom = max(ops, key=lambda o: per_op[o]["ms"])
    fwd_b, bwd_b = fwd_bytes(w), bwd_bytes(w)
    op_bytes = {"space_fwd": fwd_b, "time_fwd": fwd_b, "space_bwd": bwd_b, "time_bwd": bwd_b}
    for op in ops:
        t_s = per_op[op]["ms"] * 1e-3
        bound = "tensor" if f[op] / (tc * 1e12) >= op_bytes[op] / (hbm * 1e9) else "hbm"
        per_op[op]["bound"] = bound
        per_op[op]["gbs"] = op_bytes[op] / t_s / 1e9
        per_op[op]["frac"] = (per_op[op]["tflops"] / tc) if bound == "tensor" else (per_op[op]["gbs"] / hbm)
    d = per_op[dom]
    if d["bound"] == "tensor":
        roof = {"bound": "tensor", "achieved": d["tflops"], "peak": tc, "unit": "TFLOP/s",
                "frac": d["tflops"] / tc, "traffic": measured_traffic(w.name, dom), "kernel": dom,
                "peak_source": "%s bf16 burst" % src}
    else:
        roof = {"bound": "hbm", "achieved": d["gbs"], "peak": hbm, "unit": "GB/s",
                "frac": d["gbs"] / hbm, "traffic": measured_traffic(w.name, dom), "kernel": dom,
                "peak_source": "%s HBM copy" % src}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.op:
        if args.oracle_full:
            fl, s, nth, desc = oracle_full(w, with_bwd)
        else:
            fl, s, nth, desc = oracle_sample(w, args.ref_units, with_bwd)
        cpu = {"value": fl / s / 1e12, "unit": UNIT, "cores": nth, "kind": "oracle", "sample": desc}

    launches_per_step = {"space_fwd": 1, "time_fwd": 1, "space_bwd": api.BWD_LAUNCHES,
                         "time_bwd": api.BWD_LAUNCHES}
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic",
                "config": fwd_bwd_config(args, w, with_bwd, world, ops),
                "per_op": per_op, "roofline": roof, "cpu_baseline": cpu,
                "e2e": {"value": e2e, "unit": UNIT, "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h},
                "gpu_launches": args.steps * sum(launches_per_step[o] for o in ops),
                "clocks": clk.summary()}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- varlen space
VARLEN_METRIC = ("variable-length space attention TFLOP/s (fwd+bwd, tokenizer encoder with "
                 "dropped MAE patches) and % of B300 bf16 roofline")


def varlen_space_flops(w, L):
    """Algorithmic FLOPs of one varlen space fwd and bwd: 4*D per allowed pair per head."""
    L = np.asarray(L, dtype=np.float64)
    pairs = L * L
    if w.agent >= 0:
        pairs = pairs - np.where(w.agent < L, L - 1, 0)
    fwd = 4.0 * w.D * w.Hq * float(pairs.sum())
    return fwd, 2.5 * fwd


def run_varlen(args, w):
    """Space attention forward + backward over timestep blocks of seeded MAE lengths (the
    padded [B,T,S,H,D] layout), timed next to the same calls with every block full."""
    import torch
    from block_causal_video_attention_b300 import api

    rank, world, local = dist_info()
    lengths = synth.mae_block_lengths(w.B, w.T, w.seed + 100)
    fl_f, fl_b = varlen_space_flops(w, lengths)
    if args.impl == "reference":
        if rank != 0:
            return
        import oracle
        oracle.build()
        q, k, v, dout = synth.make_inputs(w, with_dout=True)
        X = oracle.from_bf16
        vals = []
        for i in range(args.steps):
            b, t = i % w.B, (i // w.B) % w.T   # one whole block per step
            sl = (slice(b, b + 1), slice(t, t + 1))
            t0 = time.perf_counter()
            oracle.space_bwd_varlen(X(q[sl]), X(k[sl]), X(v[sl]), X(dout[sl]),
                                    lengths[b:b + 1, t:t + 1], w.agent, w.scale)
            s = time.perf_counter() - t0
            f, bb = varlen_space_flops(w, lengths[b:b + 1, t:t + 1])
            vals.append((f + bb, s))
        value = sum(v_[0] for v_ in vals) / sum(v_[1] for v_ in vals) / 1e12
        line = {"impl": "reference", "metric": VARLEN_METRIC, "value": value, "unit": UNIT,
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * sum(v_[1] for v_ in vals) / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic", "config": varlen_config(w, lengths),
                "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(0),
                                 "kind": "oracle", "sample": "one whole timestep block per step"},
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q, k, v, dout = synth.make_inputs(w, with_dout=True)
    to = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    hq, hk, hv, hd = (to(a).pin_memory() for a in (q, k, v, dout))
    dq, dk, dv, dd = (t.to(dev) for t in (hq, hk, hv, hd))
    hL = torch.from_numpy(lengths.reshape(-1).copy()).pin_memory()
    dL = hL.to(dev)
    full = torch.full_like(dL, w.S)
    stream = torch.cuda.current_stream()
    o = torch.zeros_like(dq)
    lse = torch.zeros(dq.shape[:4], dtype=torch.float32, device=dev)
    lo = torch.zeros_like(dq)
    g = [torch.zeros_like(x) for x in (dq, dk, dv)]
    ws = torch.empty(max(api.bwd_workspace_bytes(0, w.B, w.T, w.S, w.Hq, w.Hkv), 16),
                     dtype=torch.uint8, device=dev)

    def step(Lt, ev=None, Q=dq, K=dk, V=dv, DO=dd):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)] if ev is not None else None
        if e:
            e[0].record(stream)
        api.space_attn_fwd_varlen(Q, K, V, Lt, w.agent, w.scale, o, lse, stream, o_lo=lo)
        if e:
            e[1].record(stream)
        api.space_attn_bwd_varlen(Q, K, V, o, lse, DO, Lt, w.agent, w.scale, workspace=ws, out=g,
                                  stream=stream, o_lo=lo)
        if e:
            e[2].record(stream)
            ev.append(e)

    def timed(Lt):
        for _ in range(args.warmup):
            step(Lt)
        torch.cuda.synchronize()
        if api.get_device_status() != 0:
            raise RuntimeError("device timeout")
        ev = []
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            step(Lt, ev)
        b.record(stream)
        torch.cuda.synchronize()
        if api.get_device_status() != 0:
            raise RuntimeError("device timeout")
        fwd = float(np.mean([x[0].elapsed_time(x[1]) for x in ev]))
        bwd = float(np.mean([x[1].elapsed_time(x[2]) for x in ev]))
        return a.elapsed_time(b) / args.steps, fwd, bwd

    clk = Clocks(local).__enter__()
    ms, fwd_ms, bwd_ms = timed(dL)
    dense_ms, dense_fwd, dense_bwd = timed(full)
    # end to end: Q, K, V, dO and the lengths in from pinned host memory, O, LSE and the
    # gradients back
    hin = [hq, hk, hv, hd, hL]
    din = [torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv), torch.empty_like(dd),
           torch.empty_like(dL)]
    outs = [o, lse] + g
    hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = sum(t.numel() * t.element_size() for t in hout)

    def e2e_step():
        for h_, d_ in zip(hin, din):
            d_.copy_(h_, non_blocking=True)
        step(din[4], None, din[0], din[1], din[2], din[3])
        for d_, h_ in zip(outs, hout):
            h_.copy_(d_, non_blocking=True)
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    clk.__exit__()
    e2e_ms = a.elapsed_time(b) / args.steps
    value = (fl_f + fl_b) / (ms * 1e-3) / 1e12
    _, tc, _, src = load_peaks()
    bwd_tf = fl_b / (bwd_ms * 1e-3) / 1e12
    roof = {"bound": "tensor", "achieved": bwd_tf, "peak": tc, "unit": "TFLOP/s",
            "frac": bwd_tf / tc, "traffic": None, "kernel": "space_bwd (varlen)",
            "peak_source": "%s bf16 burst" % src}
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        oracle.build()
        X = oracle.from_bf16
        t0 = time.perf_counter()
        sl = (slice(0, 1), slice(0, 1))
        oracle.space_bwd_varlen(X(q[sl]), X(k[sl]), X(v[sl]), X(dout[sl]), lengths[:1, :1],
                                w.agent, w.scale)
        s_ = time.perf_counter() - t0
        f_, b_ = varlen_space_flops(w, lengths[:1, :1])
        cpu = {"value": (f_ + b_) / s_ / 1e12, "unit": UNIT, "cores": oracle.num_threads(0),
               "kind": "oracle", "sample": "timestep block (0, 0), %d tokens, fwd+bwd" %
               int(lengths[0, 0])}
    line = {"metric": VARLEN_METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": varlen_config(w, lengths),
            "per_op": {"space_fwd": {"ms": fwd_ms, "tflops": fl_f / (fwd_ms * 1e-3) / 1e12},
                       "space_bwd": {"ms": bwd_ms, "tflops": bwd_tf}},
            "dense": {"ms_per_step": dense_ms, "fwd_ms": dense_fwd, "bwd_ms": dense_bwd,
                      "note": "same calls with every block holding all %d slots" % w.S},
            "roofline": roof, "cpu_baseline": cpu,
            "e2e": {"value": (fl_f + fl_b) / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": 4 * args.steps, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- decode step
DECODE_METRIC = "rollout decode step (time attention over a ring-buffer KV cache) GB/s and % of B300 HBM roofline"


def decode_bytes(w):
    """Algorithmic HBM bytes of one decode step with a full window: the window's K and V rows
    once, the new frame's q / k_new / v_new, the two cache rows written, O and LSE."""
    n_valid = min(w.T, w.window)
    kv_row = w.D * 2
    return (w.B * w.S * w.Hkv * (2 * n_valid * kv_row + 4 * kv_row)
            + w.B * w.S * w.Hq * (2 * w.D * 2 + 4))


def decode_flops(w):
    return 4.0 * w.D * w.B * w.S * w.Hq * min(w.T, w.window)


def decode_oracle_sample(w, rollouts, inputs=None):
    """Time the oracle's decode step on `rollouts` whole rollouts (all S x Hkv units each);
    returns (algorithmic bytes of that sample, seconds, threads, description)."""
    import oracle
    oracle.build()
    q, kn, vn, kc, vc = inputs if inputs is not None else synth.make_decode_inputs(w)
    X = oracle.from_bf16
    sl = slice(0, rollouts)
    args = [X(a[sl]) for a in (q, kn, vn, kc, vc)]
    t0 = time.perf_counter()
    oracle.time_decode(*args, w.T - 1, w.scale)
    s = time.perf_counter() - t0
    return decode_bytes(w) * rollouts / w.B, s, 1, (
        "%d of %d rollouts of %s (all %d positions x %d KV heads each), one decode step" % (
            rollouts, w.B, w.name, w.S, w.Hkv))


def decode_config(w, world):
    """The `config` object of a decode line; both arms print the same one (the step decodes
    frame w.T - 1: every step reads a full window)."""
    return {"workload": w.name, "rollouts": w.B, "S": w.S, "Hq": w.Hq, "Hkv": w.Hkv,
            "head_dim": w.D, "window": w.window, "frame_index": w.T - 1,
            "l2": "inputs larger than L2 (KV cache %.0f MB)" %
            (2 * w.B * w.window * w.S * w.Hkv * w.D * 2 / 1e6),
            "parallelism": "replicas" if world > 1 else "single GPU"}


def run_decode(args, w):
    import torch
    import torch.distributed as dist
    from block_causal_video_attention_b300 import api

    rank, world, local = dist_info()
    if args.impl == "reference":
        if rank != 0:
            return
        inputs = synth.make_decode_inputs(w)
        vals = [decode_oracle_sample(w, 1, inputs) for _ in range(args.steps)]
        b = sum(v[0] for v in vals)
        s = sum(v[1] for v in vals)
        value = b / s / 1e9
        line = {"impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": "GB/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * s / args.steps, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": decode_config(w, world),
                "cpu_baseline": {"value": value, "unit": "GB/s", "cores": vals[0][2],
                                 "kind": "oracle", "sample": vals[0][3] + " per step"},
                "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    torch.cuda.set_device(local)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    to = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    inputs = synth.make_decode_inputs(w)
    q, kn, vn, kc, vc = inputs
    hq, hkn, hvn = (to(a).pin_memory() for a in (q, kn, vn))
    dq, dkn, dvn = (t.to(dev) for t in (hq, hkn, hvn))
    # the cache is device-resident state of the rollout (frames t-191 .. t-1 and a stale slot)
    dkc, dvc = to(kc).to(dev), to(vc).to(dev)
    stream = torch.cuda.current_stream()
    o = torch.empty_like(dq)
    lse = torch.empty(dq.shape[:3], dtype=torch.float32, device=dev)
    t0 = w.T - 1  # steady state: every step reads a full window (decode_config says so)

    def step(i, Q=dq, KN=dkn, VN=dvn):
        api.time_attn_decode(Q, KN, VN, dkc, dvc, t0 + i, w.scale, o, lse, stream)

    clk = Clocks(local).__enter__()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if api.get_device_status() != 0:
        raise RuntimeError("device timeout during warm-up")
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        evs[i][0].record(stream)
        step(args.warmup + i)
        evs[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end), dev)
    if api.get_device_status() != 0:
        raise RuntimeError("device timeout during the timed region")
    kern_ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    nbytes = decode_bytes(w)
    value = world * nbytes * args.steps / (ms * 1e-3) / 1e9

    # end to end: the new frame's q, k_new, v_new from pinned host memory, O and LSE back
    hin = [hq, hkn, hvn]
    din = [torch.empty_like(dq), torch.empty_like(dkn), torch.empty_like(dvn)]
    hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse)]
    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = sum(t.numel() * t.element_size() for t in hout)

    def e2e_step(i):
        for h, d in zip(hin, din):
            d.copy_(h, non_blocking=True)
        step(i, din[0], din[1], din[2])
        for d, h in zip((o, lse), hout):
            h.copy_(d, non_blocking=True)
    base = args.warmup + args.steps
    for i in range(2):
        e2e_step(base + i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(args.steps):
        e2e_step(base + 2 + i)
    b.record(stream)
    torch.cuda.synchronize()
    clk.__exit__()
    e2e_ms = max_over_ranks(a.elapsed_time(b), dev)
    e2e = world * nbytes * args.steps / (e2e_ms * 1e-3) / 1e9

    hbm, _, _, src = load_peaks()
    achieved = nbytes / (kern_ms * 1e-3) / 1e9
    traffic = None
    if csrc_digest() == MEASURED_TRAFFIC["csrc_sha256"]:
        traffic = MEASURED_TRAFFIC.get(w.name, {}).get("decode")
    roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "traffic": traffic, "kernel": "od_decode_kernel",
            "peak_source": "%s HBM copy" % src}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        b_, s_, nth, desc = decode_oracle_sample(w, w.B, inputs)
        cpu = {"value": b_ / s_ / 1e9, "unit": "GB/s", "cores": nth, "kind": "oracle",
               "sample": desc}
    if rank == 0:
        line = {"metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic",
                "config": decode_config(w, world),
                "tflops": decode_flops(w) / (kern_ms * 1e-3) / 1e12,
                "roofline": roof, "cpu_baseline": cpu,
                "e2e": {"value": e2e, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h},
                "gpu_launches": args.steps, "clocks": clk.summary()}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None)
    ap.add_argument("--fwd-only", action="store_true")
    ap.add_argument("--ref-units", type=int, default=6)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-full", action="store_true",
                    help="time the oracle on the whole workload instead of a bounded sample "
                         "(about a minute of host time for minecraft_fwd_bwd)")
    ap.add_argument("--varlen", action="store_true",
                    help="variable-length space attention (fwd+bwd) over seeded MAE block "
                         "lengths, e.g. with --workload tokenizer_enc")
    ap.add_argument("--no-residual", action="store_true",
                    help="the forward does not write O's residual; the backward recomputes Delta")
    ap.add_argument("--packed", action="store_true",
                    help="read Q, K, V from one packed [B,T,S,Hq+2Hkv,D] tensor (fused QKV "
                         "projection layout) and write packed dQKV")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (rollouts for the decode workload), e.g. "
                         "for a smaller profiling case")
    ap.add_argument("--op", default=None, choices=["space_fwd", "time_fwd", "space_bwd", "time_bwd"],
                    help="time one operator only (for profiling); the line then covers that op")
    args = ap.parse_args()
    name = args.workload or ("minecraft_fwd" if args.fwd_only else "minecraft_fwd_bwd")
    w = synth.WORKLOADS[name]
    if args.batch:
        w = dataclasses.replace(w, B=args.batch, name="%s_b%d" % (w.name, args.batch))
    if name.endswith("_decode"):
        run_decode(args, w)
        return
    if args.varlen:
        run_varlen(args, w)
        return
    with_bwd = w.backward and not args.fwd_only
    if args.impl == "reference":
        run_reference(args, w, with_bwd)
    else:
        run_ours(args, w, with_bwd)


if __name__ == "__main__":
    main()
