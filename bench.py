#!/usr/bin/env python3
"""Benchmark of the fused GEMM-epilogue transformer block (fwd + bwd).

Workload (one step): the non-attention block at 70B-ish width -- tokens 8192
(4 sequences of 2048), hidden 8192, 64 query / 8 KV heads of 128, SwiGLU
intermediate 28672, bf16 weights ~N(0, 1/fan_in) -- forward and backward
through libcoda.so: gamma folds, row RMS, QKV GEMM with QK-RMSNorm + RoPE
epilogue, O-proj GEMM with residual + partial-RMS epilogue, gate/up GEMM with
row-scale + SwiGLU epilogue, down-proj GEMM with residual epilogue, and the
backward GEMMs with dSwiGLU, RMSNorm-backward and weight-gradient epilogues.
The attention core is out of scope; its output and input gradients are seeded
inputs.

Prints one JSON line.  value = algorithmic TFLOP/s of the whole step (sum of
2*M*N*K over its GEMMs, 42.06 TFLOP per step) with every input resident in
HBM; e2e = the same with the step's activations copied host->device and the
block output and input gradient copied back inside the timed region.

--impl reference times the fp64 CPU oracle on a bounded token sample of the
same workload instead (the reference arm: there is no runnable upstream).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused GEMM-epilogue TFLOP/s & % bf16 peak; block fwd+bwd ms vs unfused"
WORKLOAD = ("non-attention transformer block fwd+bwd: tokens 8192 (4x2048), hidden 8192, 64 q / 8 kv heads x 128, "
            "SwiGLU intermediate 28672; QKV+QK-RMSNorm+RoPE, O-proj+residual+partial RMS, gate/up+SwiGLU, "
            "down+residual epilogues and their backward")
DOMINANT = "gateup"   # the step's largest single GEMM-epilogue launch (row-scale + SwiGLU epilogue)
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "gateup_swiglu_gemm_block8192.md")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="coda", choices=["coda", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-unfused", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-ce", action="store_true",
                   help="skip the side measurements (linear + cross-entropy, FP8 gate/up, MLP, RMSNorm-linear)")
    p.add_argument("--legs", default="ce,fp8,nvfp4,mlp,rms",
                   help="side measurements to run (comma list of ce, fp8, nvfp4, mlp, rms)")
    p.add_argument("--serial", action="store_true", help="run the step's calls on one stream")
    p.add_argument("--fold-weights", action="store_true",
                   help="fold the RMSNorm gains into the weights each step instead of applying them in the "
                        "producing epilogues")
    p.add_argument("--cpu-tokens", type=int, default=64, help="token sample of the CPU oracle timing")
    p.add_argument("--tokens", type=int, default=8192,
                   help="tokens per step (8192 is the benchmark workload; smaller values only for profiling)")
    return p.parse_args()


# ----------------------------------------------------------------------------- one GPU only
def world_size(args):
    """The benchmark runs on one GPU.  The default GEMM shares B tiles between
    the CTAs of a cluster with TMA multicast, and this library is built for a
    single device; a multi-process launch is refused instead of running
    replicas."""
    return max(int(os.environ.get("WORLD_SIZE", 1)), args.gpus)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = os.path.join("/tmp", f"coda_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit()),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- peaks / profile
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return d["bf16_tflops"], d["bf16_tflops_sustained"], d["hbm_gbs"], "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


# The sources the dominant kernel (gate/up GEMM + SwiGLU epilogue) and its
# host-side launch are built from; a change to any of them invalidates the
# committed DRAM-traffic figure.
DOMINANT_SOURCES = ["coda_api.cu", "coda_epilogues.cuh", "coda_gemm.cuh", "coda_gemm_swiglu.cu", "coda_internal.h",
                    "coda_launch.cuh", "coda_ptx.cuh", "coda_status.h"]


def source_digest():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gemm_epilogue_transformer_bf16_gb300", "csrc")
    for f in DOMINANT_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None if the kernel sources changed since it was taken."""
    try:
        txt = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    d = re.search(r"source_digest:\s*([0-9a-f]+)", txt)
    if not m or not d or d.group(1) != source_digest():
        return None
    return float(m.group(1))


# ----------------------------------------------------------------------------- unfused comparison
def unfused_step_fn(w, t, s):
    """The same block fwd+bwd as eager torch.matmul (cuBLAS) plus unfused
    element-wise ops, differentiated by autograd.  Comparison only."""
    import torch
    import torch.nn.functional as F

    params = {k: w[k].detach().clone().requires_grad_(True)
              for k in ("Wqkv", "Wo", "Wg", "Wu", "Wd", "gamma_attn", "gamma_mlp", "gamma_q", "gamma_k")}
    T, d = s.tokens, s.head_dim
    ang = t["pos"].double()[:, None] * (s.theta ** (-2.0 * torch.arange(d // 2, device=t["pos"].device,
                                                                         dtype=torch.float64) / d))[None, :]
    cos, sin = ang.cos().float(), ang.sin().float()

    def rope(v):
        a, b = v[..., 0::2], v[..., 1::2]
        c, sn = cos[:, None, :], sin[:, None, :]
        return torch.stack((a * c - b * sn, a * sn + b * c), dim=-1).flatten(-2)

    def rms(x, g):
        xf = x.float()
        return (xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + s.eps) * g).to(torch.bfloat16)

    def step():
        p = params
        x0 = t["x0"].detach().requires_grad_(True)
        A = t["A"].detach().requires_grad_(True)
        a0 = rms(x0, p["gamma_attn"])
        qkv = a0 @ p["Wqkv"].t()
        q = qkv[:, : s.n_q * d].view(T, s.n_q, d)
        k = qkv[:, s.n_q * d: (s.n_q + s.n_kv) * d].view(T, s.n_kv, d)
        v = qkv[:, (s.n_q + s.n_kv) * d:]
        Q = rope(rms(q, p["gamma_q"]).float()).to(torch.bfloat16)
        K = rope(rms(k, p["gamma_k"]).float()).to(torch.bfloat16)
        x1 = x0 + A @ p["Wo"].t()
        a1 = rms(x1, p["gamma_mlp"])
        H = F.silu(a1 @ p["Wg"].t()) * (a1 @ p["Wu"].t())
        x2 = x1 + H @ p["Wd"].t()
        torch.autograd.backward([x2, Q, K, v], [t["dx2"], t["dQ"].view(T, s.n_q, d), t["dK"].view(T, s.n_kv, d),
                                                t["dV"]])
        for q_ in params.values():
            q_.grad = None
    return step


# ----------------------------------------------------------------------------- CPU oracle timing
def oracle_inputs(host, tokens):
    """fp64 copies of the workload's weights and of its first `tokens` tokens."""
    import numpy as np
    sl = slice(0, tokens)
    p = {}
    for k, v in host.items():
        if k in ("x0", "A", "dx2", "dQ", "dK", "dV", "pos"):
            p[k] = v[sl].double().numpy() if k != "pos" else v[sl].numpy().astype(np.int64)
        else:
            p[k] = v.double().numpy()
    return p


def oracle_sample_timing(tokens, p):
    """Time the fp64 oracle (as it stands) on the sample prepared by
    oracle_inputs: block_fwd + block_bwd.  Returns (TFLOP/s, seconds, flops)."""
    from oracle import coda_oracle as O
    import synth
    s = synth.FULL["block"]
    cfg = dict(n_q=s.n_q, n_kv=s.n_kv, head_dim=s.head_dim, theta=s.theta, eps=s.eps)
    t0 = time.perf_counter()
    O.block_fwd(p, **cfg)
    O.block_bwd(p, **cfg)
    dt = time.perf_counter() - t0
    flops = O.block_flops(tokens, s.hidden, s.qkv_out, s.n_q * s.head_dim, s.inter)
    return flops / dt / 1e12, dt, flops


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    if int(os.environ.get("RANK", 0)) != 0:
        return 0
    import torch
    import synth
    s = synth.FULL["block"]
    host = synth.make_block(s, seed=0)
    torch.set_num_threads(cores())
    p = oracle_inputs(host, args.cpu_tokens)
    vals, secs = [], []
    for i in range(args.warmup + args.steps):
        v, dt, flops = oracle_sample_timing(args.cpu_tokens, p)
        if i >= args.warmup:
            vals.append(v)
            secs.append(dt)
    val = statistics.median(vals)
    sample = f"block fwd+bwd on the first {args.cpu_tokens} of 8192 tokens (full weights), fp64 NumPy"
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.median(secs) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "tokens": s.tokens, "hidden": s.hidden, "inter": s.inter,
                       "oracle_tokens_per_step": args.cpu_tokens},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores(), "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- main arm
def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if world_size(args) > 1:
        print("bench.py runs on one GPU only: the library is single-device and its cluster GEMMs share tiles by "
              "TMA multicast; launch it without --gpus > 1 / WORLD_SIZE > 1", file=sys.stderr)
        return 2
    import numpy as np
    import torch
    import synth
    import gemm_epilogue_transformer_bf16_gb300 as coda
    from gemm_epilogue_transformer_bf16_gb300.block import Block

    assert torch.cuda.is_available(), "bench.py needs a CUDA device"
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    coda.load()
    import dataclasses
    s = dataclasses.replace(synth.FULL["block"], tokens=args.tokens)
    host = synth.make_block(s, seed=0)
    t = {k: v.to(dev) for k, v in host.items()}
    blk = Block(s, t, device=dev, concurrent=not args.serial, fold_weights=args.fold_weights)
    flops_step = sum(blk.gemm_flops().values())
    launches_step = sum(blk.launches().values())
    stream = torch.cuda.current_stream(dev)
    args_step = (t["x0"], t["A"], t["pos"], t["dx2"], t["dQ"], t["dK"], t["dV"])

    # ---------------------------------------------------------------- device-resident timing
    names = list(blk.launches())
    for _ in range(args.warmup):
        blk.step(*args_step)
    torch.cuda.synchronize(dev)
    st = coda.get_status(blk.ws)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {coda.status_string(st)}")
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(args.steps)]
    gpu_id = None
    try:
        gpu_id = str(torch.cuda.get_device_properties(dev).uuid)
        gpu_id = gpu_id if gpu_id.startswith("GPU-") else "GPU-" + gpu_id
    except Exception:
        gpu_id = None
    clocks = ClockSampler(gpu_id)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        ev = marks[i]
        ev[0].record(stream)
        j = [1]

        def mark(name, ev=ev, j=j):
            ev[j[0]].record(stream)
            j[0] += 1
        blk.step(*args_step, mark=mark)
    stop.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms_total = start.elapsed_time(stop)
    ms_step = ms_total / args.steps
    value = flops_step * args.steps / (ms_total / 1e3) / 1e12
    stage_ms = {n: statistics.median(marks[i][k].elapsed_time(marks[i][k + 1]) for i in range(args.steps))
                for k, n in enumerate(names)}
    gf = blk.gemm_flops()
    burst, sustained, hbm, peak_src = measured_peaks()
    stages = {n: {"ms": round(stage_ms[n], 4), "launches": blk.launches()[n],
                  "tflops": round(gf[n] / (stage_ms[n] / 1e3) / 1e12, 1) if gf[n] else None} for n in names}
    ach = gf[DOMINANT] / (stage_ms[DOMINANT] / 1e3) / 1e12
    roofline = {"bound": "tensor", "achieved": round(ach, 1), "peak": sustained, "unit": "TFLOP/s",
                "frac": round(ach / sustained, 4), "traffic": profiled_traffic(),
                "kernel": "coda_gemm_kernel<256, EpiSwiglu> (gate/up GEMM, 8192x57344x8192)",
                "peak_kind": f"bf16 sustained ({peak_src})"}
    torch.cuda.synchronize(dev)
    if coda.get_status(blk.ws) != 0:
        raise RuntimeError("device status error in timed region")

    # ---------------------------------------------------------------- end to end through host buffers
    # Every step copies its inputs (x0, A, positions, dx2, dQ, dK, dV) from
    # pinned host memory and reads its results (x2, dx0) back, inside the timed
    # region.  The copies are pipelined the way a training loop prefetches: the
    # next step's inputs go host->device on their own stream into a second
    # buffer set while the current step computes, and results come back on a
    # third stream.  Events order every reuse: an input buffer is refilled only
    # after the step that read it has finished, a step starts only when its
    # inputs have landed, and x2 / dx0 are overwritten only after the previous
    # step's copy-out.
    e2e = None
    if not args.no_e2e:
        in_keys = ("x0", "A", "pos", "dx2", "dQ", "dK", "dV")
        hin = {k: host[k].pin_memory() for k in in_keys}
        hx2 = torch.empty_like(host["x0"]).pin_memory()
        hdx0 = torch.empty_like(host["x0"]).pin_memory()
        dbuf = [{k: torch.empty_like(t[k]) for k in in_keys} for _ in range(2)]
        h2d = sum(v.numel() * v.element_size() for v in hin.values())
        d2h = hx2.numel() * hx2.element_size() + hdx0.numel() * hdx0.element_size()
        h2d_s = torch.cuda.Stream(device=dev)
        d2h_s = torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        ev_used = [torch.cuda.Event(), torch.cuda.Event()]
        ev_x2, ev_x2_out, ev_dx0_out = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()

        def copy_in(bi, after=None):
            with torch.cuda.stream(h2d_s):
                if after is not None:
                    h2d_s.wait_event(after)
                for k in in_keys:
                    dbuf[bi][k].copy_(hin[k], non_blocking=True)
                ev_in[bi].record(h2d_s)

        def e2e_run(nsteps, start_ev=None):
            if start_ev is not None:
                h2d_s.wait_event(start_ev)
            copy_in(0)
            for i in range(nsteps):
                bi = i % 2
                if i + 1 < nsteps:
                    copy_in(1 - bi, ev_used[1 - bi] if i >= 1 else None)
                stream.wait_event(ev_in[bi])
                if i >= 1:
                    stream.wait_event(ev_x2_out)
                d = dbuf[bi]
                f = blk.forward(d["x0"], d["A"], d["pos"])
                ev_x2.record(stream)
                with torch.cuda.stream(d2h_s):
                    d2h_s.wait_event(ev_x2)
                    hx2.copy_(f["x2"], non_blocking=True)
                    ev_x2_out.record(d2h_s)
                if i >= 1:
                    stream.wait_event(ev_dx0_out)
                g = blk.backward(d["x0"], d["A"], d["pos"], d["dx2"], d["dQ"], d["dK"], d["dV"])
                ev_used[bi].record(stream)
                with torch.cuda.stream(d2h_s):
                    d2h_s.wait_event(ev_used[bi])
                    hdx0.copy_(g["dx0"], non_blocking=True)
                    ev_dx0_out.record(d2h_s)
            stream.wait_stream(h2d_s)
            stream.wait_stream(d2h_s)

        e2e_run(max(2, args.warmup // 2))
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_run(args.steps, a)
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms_e2e = a.elapsed_time(b)
        if not (torch.equal(hx2, blk.x2.cpu()) and torch.equal(hdx0, blk.grads_qkv["dX"].cpu())):
            raise RuntimeError("e2e results read back do not match the device buffers")
        e2e = {"value": round(flops_step * args.steps / (ms_e2e / 1e3) / 1e12, 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e / args.steps, 3),
               "copies": "pinned host buffers; next step's inputs prefetched on a copy stream, results read back "
                         "on another"}

    # ---------------------------------------------------------------- unfused torch comparison
    unfused_ms = None
    if not args.no_unfused:
        del blk
        torch.cuda.empty_cache()
        step = unfused_step_fn(t, t, s)
        for _ in range(2):
            step()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        n_unf = max(3, args.steps // 3)
        a.record(stream)
        for _ in range(n_unf):
            step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        unfused_ms = a.elapsed_time(b) / n_unf

    # ---------------------------------------------------------------- linear + CE (rows a8, a12)
    # Not part of the block step: the 8192 x 2048 x 128256 linear + cross-entropy
    # workload, forward and backward, timed the same way and reported beside it.
    other = {}
    legs = set(args.legs.split(","))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]

    def time_calls(fn, n=5, warm=2):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize(dev)
        ev[0].record(stream)
        for _ in range(n):
            fn()
        ev[1].record(stream)
        torch.cuda.synchronize(dev)
        return ev[0].elapsed_time(ev[1]) / n

    def unfused_leg(entry, fn, ours_ms, n=3):
        """Time the same workload as eager torch (cuBLAS matmuls, unfused
        element-wise ops, autograd backward) and add it to the leg's entry."""
        if args.no_unfused:
            return
        ms = time_calls(fn, n=n, warm=1)
        entry["unfused_ms"] = round(ms, 3)
        entry["speedup_vs_unfused"] = round(ms / ours_ms, 3)

    if not args.no_ce and "ce" in legs:
        from gemm_epilogue_transformer_bf16_gb300.block import LinearCE
        cs_ = synth.FULL["linear_ce"]
        hc = synth.make_ce(cs_, seed=0)
        dc = {k: v.to(dev) for k, v in hc.items()}
        ce = LinearCE(cs_.tokens, cs_.vocab, cs_.hidden, device=dev)
        for _ in range(2):
            ce.step(dc["X"], dc["W"], dc["labels"])
        torch.cuda.synchronize(dev)
        n_ce = 3
        fw, bw = [], []
        for _ in range(n_ce):
            ev[0].record(stream)
            coda.linear_cross_entropy(dc["X"], dc["W"], dc["labels"], out=ce.out, ws=ce.ws)
            ev[1].record(stream)
            coda.linear_cross_entropy_bwd(dc["X"], dc["W"], dc["labels"], ce.out["lse"], ce.out["n_valid"], 1.0,
                                          out=ce.grads, ws=ce.ws)
            ev[2].record(stream)
            torch.cuda.synchronize(dev)
            fw.append(ev[0].elapsed_time(ev[1]))
            bw.append(ev[1].elapsed_time(ev[2]))
        if coda.get_status(ce.ws) != 0:
            raise RuntimeError("device status error in the linear-CE measurement")
        # 2*M*N*K: the logits GEMM forward; the backward recomputes them, then dX and dW
        f_fwd = 2 * cs_.tokens * cs_.hidden * cs_.vocab
        f_all = 4 * f_fwd
        mf, mb = statistics.median(fw), statistics.median(bw)
        other["linear_cross_entropy"] = {
            "workload": "tokens 8192, hidden 2048, vocab 128256, 5% ignored labels; fwd (online LSE epilogue + "
                        "combine) and bwd (softmax-minus-onehot epilogue, dX, dW)",
            "fwd_ms": round(mf, 3), "bwd_ms": round(mb, 3),
            "fwd_tflops": round(f_fwd / (mf / 1e3) / 1e12, 1),
            "fwd_bwd_tflops": round(f_all / ((mf + mb) / 1e3) / 1e12, 1)}
        del ce
        Xr = dc["X"].detach().requires_grad_(True)
        Wr = dc["W"].detach().requires_grad_(True)
        lab_long = dc["labels"].long()

        def ce_unfused():
            # bf16 logits from cuBLAS (2.1 GB, they fit), fp32 cross-entropy, autograd backward
            z = Xr @ Wr.t()
            torch.nn.functional.cross_entropy(z.float(), lab_long, ignore_index=cs_.ignore_index).backward()
            Xr.grad = None
            Wr.grad = None
        unfused_leg(other["linear_cross_entropy"], ce_unfused, mf + mb)
        del dc, Xr, Wr

    if not args.no_ce and ("fp8" in legs or "nvfp4" in legs):
        T_, H_, I_ = s.tokens, s.hidden, s.inter
        r_ = coda.rms_rstd(t["x0"], s.eps)
        Hq = torch.empty(T_, I_, dtype=torch.bfloat16, device=dev)
        gq8, uq8 = torch.empty_like(Hq), torch.empty_like(Hq)
        ws8 = coda.workspace(256, dev)
    if not args.no_ce and "fp8" in legs:
        # FP8 (e4m3) gate/up + SwiGLU at the block's shape (NEXT row: the same
        # mainloop with kind::f8f6f4), beside the bf16 launch timed above.
        xq, sx = coda.quantize_fp8_rows(t["x0"])
        gq, sg = coda.quantize_fp8_rows(t["Wg"])
        uq, su = coda.quantize_fp8_rows(t["Wu"])
        f8 = []
        for i in range(5):
            ev[0].record(stream)
            coda.linear_swiglu_fp8(xq, sx, gq, sg, uq, su, rstd=r_, H=Hq, g=gq8, u=uq8, ws=ws8)
            ev[1].record(stream)
            torch.cuda.synchronize(dev)
            if i >= 2:
                f8.append(ev[0].elapsed_time(ev[1]))
        if coda.get_status(ws8) != 0:
            raise RuntimeError("device status error in the FP8 measurement")
        m8 = statistics.median(f8)
        fp8_peak = 2 * burst
        other["fp8_gateup_swiglu"] = {
            "workload": f"e4m3 gate/up GEMM with row-scale + SwiGLU epilogue, {T_} x 2x{I_} x {H_}, per-row scales",
            "ms": round(m8, 3), "tflops": round(gf[DOMINANT] / (m8 / 1e3) / 1e12, 1),
            "peak": round(fp8_peak, 1), "peak_kind": f"fp8 = 2 x bf16 burst ({peak_src}, nominal ratio)",
            "frac": round(gf[DOMINANT] / (m8 / 1e3) / 1e12 / fp8_peak, 4)}
        del xq, gq, uq
    if not args.no_ce and "nvfp4" in legs:
        # NVFP4 (e2m1 + e4m3 block scales) gate/up + SwiGLU at the same shape:
        # the block-scaled kind::mxf4nvf4 mainloop, single CTAs.
        fq = []
        xq4, sfx4, sx4 = coda.quantize_nvfp4_rows(t["x0"])
        gq4, sfg4, sg4 = coda.quantize_nvfp4_rows(t["Wg"])
        uq4, sfu4, su4 = coda.quantize_nvfp4_rows(t["Wu"])
        for i in range(5):
            ev[0].record(stream)
            coda.quantize_nvfp4_rows(t["x0"])
            ev[1].record(stream)
            coda.linear_swiglu_nvfp4(xq4, sfx4, sx4, gq4, sfg4, sg4, uq4, sfu4, su4, rstd=r_, H=Hq, g=gq8, u=uq8,
                                     ws=ws8)
            ev[2].record(stream)
            torch.cuda.synchronize(dev)
            if i >= 2:
                fq.append((ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])))
        if coda.get_status(ws8) != 0:
            raise RuntimeError("device status error in the NVFP4 measurement")
        mq4 = statistics.median(q for q, _ in fq)
        m4 = statistics.median(g for _, g in fq)
        fp4_peak = 6 * burst
        other["nvfp4_gateup_swiglu"] = {
            "workload": f"NVFP4 gate/up GEMM (e2m1, e4m3 scale per 16, fp32 row scale) with row-scale + SwiGLU "
                        f"epilogue, {T_} x 2x{I_} x {H_}, single-CTA tiles",
            "ms": round(m4, 3), "tflops": round(gf[DOMINANT] / (m4 / 1e3) / 1e12, 1),
            "peak": round(fp4_peak, 1), "peak_kind": f"fp4 = 6 x bf16 burst ({peak_src}, nominal ratio)",
            "frac": round(gf[DOMINANT] / (m4 / 1e3) / 1e12 / fp4_peak, 4),
            "quantize_x_ms": round(mq4, 3)}
        del xq4, gq4, uq4, sfx4, sfg4, sfu4
    if not args.no_ce and ("fp8" in legs or "nvfp4" in legs):
        del Hq, gq8, uq8

    # Two more workloads (also parity workloads), forward + backward, timed the
    # same way: the SwiGLU MLP at hidden 4096 and the RMSNorm-reparameterised
    # projection + residual at 4096 x 2048 (gain folded into W: the standalone
    # operator's form).  FLOPs 2*M*N*K per GEMM.
    if not args.no_ce and "mlp" in legs:
        s3 = synth.FULL["mlp"]
        d3 = {k: v.to(dev) for k, v in synth.make_mlp(s3, seed=0).items()}
        ws3 = coda.workspace(max(coda.load().coda_linear_swiglu_bwd_workspace_size(s3.tokens, s3.inter, s3.hidden),
                                 coda.load().coda_linear_residual_workspace_size(s3.tokens, s3.hidden, s3.inter)), dev)
        o3 = {}
        side3 = torch.cuda.Stream(device=dev)

        def mlp_step():
            H3, g3, u3 = coda.linear_swiglu(d3["X"], d3["Wg"], d3["Wu"], ws=ws3)
            coda.linear_residual(H3, d3["Wd"], d3["R"], ws=ws3)
            o3["g"] = coda.linear_swiglu_bwd(d3["dY"], d3["X"], d3["Wg"], d3["Wu"], d3["Wd"], g3, u3, H3, ws=ws3,
                                             side_stream=side3)
        m3 = time_calls(mlp_step)
        f3 = 2 * s3.tokens * s3.hidden * s3.inter * 3 * 3       # fwd 3 GEMMs, bwd 6
        other["mlp_swiglu"] = {
            "workload": f"SwiGLU MLP fwd+bwd, tokens {s3.tokens}, hidden {s3.hidden}, intermediate {s3.inter}",
            "ms": round(m3, 3), "tflops": round(f3 / (m3 / 1e3) / 1e12, 1),
            "frac_of_sustained": round(f3 / (m3 / 1e3) / 1e12 / sustained, 4)}
        del o3, ws3
        p3 = {k: d3[k].detach().requires_grad_(True) for k in ("X", "Wg", "Wu", "Wd")}

        def mlp_unfused():
            p = p3
            H = torch.nn.functional.silu(p["X"] @ p["Wg"].t()) * (p["X"] @ p["Wu"].t())
            (d3["R"] + H @ p["Wd"].t()).backward(d3["dY"])
            for v in p.values():
                v.grad = None
        unfused_leg(other["mlp_swiglu"], mlp_unfused, m3)
        del d3, p3
    if not args.no_ce and "rms" in legs:
        s2 = synth.FULL["rmsnorm_linear"]
        d2 = {k: v.to(dev) for k, v in synth.make_rms_linear(s2, seed=0).items()}
        # outputs and workspaces allocated once, as a training loop holds them;
        # dW on a second stream beside c -> dX
        M2, N2, K2 = s2.tokens, s2.out, s2.hidden
        lib = coda.load()
        Wf2 = torch.empty_like(d2["W"])
        Y2 = torch.empty(M2, N2, dtype=torch.bfloat16, device=dev)
        r2 = torch.empty(M2, dtype=torch.float32, device=dev)
        ws2a = coda.workspace(lib.coda_rmsnorm_linear_workspace_size(M2, N2, K2), dev)
        ws2b = coda.workspace(lib.coda_rmsnorm_linear_bwd_workspace_size(M2, N2, K2), dev)
        g2 = {"dX": torch.empty_like(d2["X"]), "dW": torch.empty_like(d2["W"]),
              "dgamma": torch.empty(K2, dtype=torch.float32, device=dev)}
        side2 = torch.cuda.Stream(device=dev)

        def rms_step():
            coda.fold_gamma(d2["W"], d2["gamma"], out=Wf2)
            coda.rmsnorm_linear(d2["X"], Wf2, d2["R"], eps=s2.eps, rstd_out=r2, Y=Y2, ws=ws2a)
            coda.rmsnorm_linear_bwd(d2["G"], d2["X"], d2["W"], d2["gamma"], r2, Y2, d2["R"], ws=ws2b, out=g2,
                                    side_stream=side2)
        m2 = time_calls(rms_step, n=20, warm=3)
        # the same calls captured once into a CUDA graph (on a capture stream
        # that has run them once outside the capture) and replayed
        cap2 = torch.cuda.Stream(device=dev)
        cap2.wait_stream(stream)
        with torch.cuda.stream(cap2):
            rms_step()
        stream.wait_stream(cap2)
        graph2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph2, stream=cap2):
            rms_step()
        mg2 = time_calls(graph2.replay, n=20, warm=3)
        if coda.get_status(ws2a) != 0 or coda.get_status(ws2b) != 0:
            raise RuntimeError("device status error in the RMSNorm-linear measurement")
        f2 = 2 * s2.tokens * s2.hidden * s2.out * 3               # fwd 1 GEMM, bwd 2
        other["rmsnorm_linear"] = {
            "workload": f"RMSNorm-reparameterised projection + residual fwd+bwd, tokens {s2.tokens}, "
                        f"hidden {s2.hidden}, out {s2.out} (gain fold, row RMS, prepass and combines included)",
            "ms": round(m2, 3), "tflops": round(f2 / (m2 / 1e3) / 1e12, 1),
            "frac_of_sustained": round(f2 / (m2 / 1e3) / 1e12 / sustained, 4),
            "graph_ms": round(mg2, 3), "graph_tflops": round(f2 / (mg2 / 1e3) / 1e12, 1)}
        del graph2
        p2 = {"X": d2["X"].detach().requires_grad_(True), "W": d2["W"].detach().requires_grad_(True),
              "gamma": d2["gamma"].detach().requires_grad_(True)}

        def rms_unfused():
            p = p2
            xf = p["X"].float()
            xn = (xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + s2.eps) * p["gamma"]).to(torch.bfloat16)
            (d2["R"] + xn @ p["W"].t()).backward(d2["G"])
            for v in p.values():
                v.grad = None
        unfused_leg(other["rmsnorm_linear"], rms_unfused, m2, n=20)
        del d2, p2

    # ---------------------------------------------------------------- CPU oracle baseline
    cpu = None
    if not args.no_cpu_baseline and args.tokens == synth.FULL["block"].tokens:
        torch.set_num_threads(cores())
        v, dt, fl = oracle_sample_timing(args.cpu_tokens, oracle_inputs(host, args.cpu_tokens))
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores(), "kind": "oracle",
               "sample": f"fp64 NumPy block_fwd+block_bwd on the first {args.cpu_tokens} of 8192 tokens "
                         f"(full weights): {fl / 1e12:.3f} TFLOP in {dt:.1f} s"}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens": s.tokens, "hidden": s.hidden, "n_q": s.n_q,
                   "n_kv": s.n_kv, "head_dim": s.head_dim, "inter": s.inter, "tflop_per_step":
                   round(flops_step / 1e12, 3), "l2": "inputs (1.7 GB of weights + activations) exceed the "
                   "129 MB L2; no flush", "parallelism": "single GPU",
                   "rmsnorm_gain": "folded into the weights each step" if args.fold_weights
                   else "applied by the producing epilogue (u = x ⊙ gamma)"},
        "pct_bf16_peak": {"burst": round(value / burst, 4), "sustained": round(value / sustained, 4),
                          "source": peak_src},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_step * args.steps,
        "clocks": clk,
        "unfused_ms_per_step": round(unfused_ms, 3) if unfused_ms else None,
        "speedup_vs_unfused": round(unfused_ms / ms_step, 3) if unfused_ms else None,
        "stages": stages,
        "other_workloads": other or None,
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
