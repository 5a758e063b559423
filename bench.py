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
N_LEG = 50            # timed calls per leg (median reported)
W_LEG = 10            # untimed calls before them
FLUSH_BYTES = 256 << 20   # buffer written between timed calls of a leg (L2 flush)
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
    p.add_argument("--legs", default="swiglu,rms,mlp,ce,fp8,fp8block,nvfp4",
                   help="other workloads to time after the block step (comma list of swiglu, rms, mlp, ce, fp8, "
                        "fp8block, nvfp4; none for none)")
    p.add_argument("--no-block", action="store_true", help="skip the block step (profiling of the other legs)")
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


def oracle_workload_timings(tokens, block_sample):
    """The fp64 oracle (as it stands) on every workload, on the host cores:
    linear + SwiGLU (256 x 512 -> 1024) and the RMSNorm-linear fwd+bwd
    (4096 x 2048 -> 2048) in full; the SwiGLU MLP, linear + cross-entropy and
    the block on their first `tokens` tokens with full weights, the seconds
    scaled to the full token count by FLOPs and labelled "extrapolated"."""
    from oracle import coda_oracle as O
    import synth

    def f64(d):
        return {k: (v.double().numpy() if v.dtype != torch_int32() else v.numpy()) for k, v in d.items()}

    out = {}

    def entry(name, secs, flops, how):
        out[name] = {"seconds": round(secs, 3), "tflops": round(flops / secs / 1e12, 4), "how": how}

    s1 = synth.FULL["swiglu"]
    p = f64(synth.make_swiglu(s1, seed=0))
    t0 = time.perf_counter()
    O.swiglu_fwd(p["X"], p["Wg"], p["Wu"])
    entry("swiglu", time.perf_counter() - t0, 2 * s1.tokens * s1.hidden * s1.inter * 2, "full")
    s2 = synth.FULL["rmsnorm_linear"]
    p = f64(synth.make_rms_linear(s2, seed=0))
    t0 = time.perf_counter()
    O.rmsnorm_linear_fwd(p["X"], p["gamma"], p["W"], s2.eps, p["R"])
    O.rmsnorm_linear_bwd(p["X"], p["gamma"], p["W"], s2.eps, p["G"])
    entry("rmsnorm_linear", time.perf_counter() - t0, 2 * s2.tokens * s2.hidden * s2.out * 3, "full")
    s3 = synth.FULL["mlp"]
    p = f64(synth.make_mlp(s3, seed=0))
    sl = slice(0, tokens)
    t0 = time.perf_counter()
    O.mlp_fwd(p["X"][sl], p["Wg"], p["Wu"], p["Wd"], p["R"][sl])
    O.mlp_bwd(p["X"][sl], p["Wg"], p["Wu"], p["Wd"], p["dY"][sl])
    dt = time.perf_counter() - t0
    full = O.mlp_flops(s3.tokens, s3.hidden, s3.inter)
    entry("mlp_swiglu", dt * full / O.mlp_flops(tokens, s3.hidden, s3.inter), full,
          f"extrapolated by FLOPs from the first {tokens} tokens ({dt:.2f} s)")
    s4 = synth.FULL["linear_ce"]
    p = f64(synth.make_ce(s4, seed=0))
    t0 = time.perf_counter()
    O.linear_cross_entropy_fwd(p["X"][sl], p["W"], p["labels"][sl])
    O.linear_cross_entropy_bwd(p["X"][sl], p["W"], p["labels"][sl])
    dt = time.perf_counter() - t0
    full = O.ce_flops(s4.tokens, s4.hidden, s4.vocab)
    entry("linear_cross_entropy", dt * full / O.ce_flops(tokens, s4.hidden, s4.vocab), full,
          f"extrapolated by FLOPs from the first {tokens} tokens ({dt:.2f} s)")
    _, bdt, bfl = block_sample
    s5 = synth.FULL["block"]
    full = O.block_flops(s5.tokens, s5.hidden, s5.qkv_out, s5.n_q * s5.head_dim, s5.inter)
    entry("block", bdt * full / bfl, full, f"extrapolated by FLOPs from the first {tokens} tokens ({bdt:.2f} s)")
    return out


def torch_int32():
    import torch
    return torch.int32


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
    stream = torch.cuda.current_stream(dev)
    burst, sustained, hbm, peak_src = measured_peaks()
    def block_leg():
        """The block step: device-resident timing (the headline), end to end
        through pinned host buffers, and the eager-torch comparison."""
        blk = Block(s, t, device=dev, concurrent=not args.serial, fold_weights=args.fold_weights)
        flops_step = sum(blk.gemm_flops().values())
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
        # the library's own launch counter (coda_launch_count): every kernel
        # it issues inside the timed region, split launches' second slices
        # included; per stage from the first timed step
        counts = [[0] * (len(names) + 1) for _ in range(args.steps)]
        n_launch0 = coda.launch_count()
        start.record(stream)
        for i in range(args.steps):
            ev = marks[i]
            ev[0].record(stream)
            counts[i][0] = coda.launch_count()
            j = [1]

            def mark(name, ev=ev, j=j, cnt=counts[i]):
                ev[j[0]].record(stream)
                cnt[j[0]] = coda.launch_count()
                j[0] += 1
            blk.step(*args_step, mark=mark)
        stop.record(stream)
        launches_timed = coda.launch_count() - n_launch0
        torch.cuda.synchronize(dev)
        clk = clocks.stop()
        ms_total = start.elapsed_time(stop)
        ms_step = ms_total / args.steps
        value = flops_step * args.steps / (ms_total / 1e3) / 1e12
        median_step = statistics.median(marks[i][0].elapsed_time(marks[i][-1]) for i in range(args.steps))
        stage_ms = {n: statistics.median(marks[i][k].elapsed_time(marks[i][k + 1]) for i in range(args.steps))
                    for k, n in enumerate(names)}
        gf = blk.gemm_flops()
        stages = {n: {"ms": round(stage_ms[n], 4), "launches": counts[0][k + 1] - counts[0][k],
                      "tflops": round(gf[n] / (stage_ms[n] / 1e3) / 1e12, 1) if gf[n] else None}
                  for k, n in enumerate(names)}
        ach = gf[DOMINANT] / (stage_ms[DOMINANT] / 1e3) / 1e12
        # the step lasts about 25 ms and the timed region about a second, so
        # the kernel is held to the burst peak (the sustained figure is a
        # seconds-long loop under the power cap)
        roofline = {"bound": "tensor", "achieved": round(ach, 1), "peak": burst, "unit": "TFLOP/s",
                    "frac": round(ach / burst, 4), "traffic": profiled_traffic(),
                    "kernel": "coda_gemm_kernel<256, EpiSwiglu> (gate/up GEMM, 8192x57344x8192)",
                    "peak_kind": f"bf16 burst ({peak_src})"}
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
            clocks_e2e = ClockSampler(gpu_id)   # the clocks of this loop too: it runs after the other
            clocks_e2e.start()
            time.sleep(0.3)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            e2e_run(args.steps, a)
            b.record(stream)
            torch.cuda.synchronize(dev)
            clk_e2e = clocks_e2e.stop()
            ms_e2e = a.elapsed_time(b)
            if not (torch.equal(hx2, blk.x2.cpu()) and torch.equal(hdx0, blk.grads_qkv["dX"].cpu())):
                raise RuntimeError("e2e results read back do not match the device buffers")
            e2e = {"value": round(flops_step * args.steps / (ms_e2e / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e / args.steps, 3),
                   "copies": "pinned host buffers; next step's inputs prefetched on a copy stream, results read back "
                             "on another", "clocks": clk_e2e}

        # ---------------------------------------------------------------- unfused torch comparison
        unfused_ms = None
        if not args.no_unfused:
            del blk
            torch.cuda.empty_cache()
            step = unfused_step_fn(t, t, s)
            for _ in range(3):
                step()
            torch.cuda.synchronize(dev)
            n_unf = max(N_LEG, args.steps)
            ue = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_unf)]
            for e in ue:
                e[0].record(stream)
                step()
                e[1].record(stream)
            torch.cuda.synchronize(dev)
            unfused_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ue)
        return dict(value=value, ms_step=ms_step, median_step=median_step, flops_step=flops_step,
                    launches_timed=launches_timed, roofline=roofline, e2e=e2e, clk=clk, unfused_ms=unfused_ms,
                    stages=stages)

    blk_res = None if args.no_block else block_leg()

    # ---------------------------------------------------------------- the other workloads
    # One leg per other workload, each timed the same way: 10 untimed
    # calls, then N_LEG calls, each between two CUDA events on the launching
    # stream with a 256 MB buffer written before it (an L2 flush, outside
    # the events); the median is reported.  Rates are 2*M*N*K per GEMM
    # against the measured bf16 burst peak (each call is timed alone).  The
    # eager-torch comparison of a leg runs the same workload as cuBLAS
    # matmuls plus unfused element-wise ops with an autograd backward, timed
    # the same way.
    other = {}
    legs = set(args.legs.split(","))
    flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def median_ms(fn, n=N_LEG, warm=W_LEG, parts=1):
        """Median over n calls of fn's device time (parts > 1: fn(mark) marks
        part boundaries, and the medians of every part are returned)."""
        for _ in range(warm):
            fn(lambda: None) if parts > 1 else fn()
        torch.cuda.synchronize(dev)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(parts + 1)] for _ in range(n)]
        for k in range(n):
            flush_buf.zero_()
            e = evs[k]
            e[0].record(stream)
            if parts > 1:
                pos = [1]

                def mark(e=e, pos=pos):
                    e[pos[0]].record(stream)
                    pos[0] += 1
                fn(mark)
            else:
                fn()
            e[parts].record(stream)
        torch.cuda.synchronize(dev)
        med = [statistics.median(e[p].elapsed_time(e[p + 1]) for e in evs) for p in range(parts)]
        return med if parts > 1 else med[0]

    def rate(flops, ms):
        return round(flops / (ms / 1e3) / 1e12, 1)

    def unfused_leg(entry, fn, ours_ms):
        if args.no_unfused:
            return
        ms = median_ms(fn)
        entry["unfused_ms"] = round(ms, 4)
        entry["speedup_vs_unfused"] = round(ms / ours_ms, 3)

    if "swiglu" in legs:
        # linear + SwiGLU forward, 256 x 512 -> 1024 (launch-latency bound)
        s1 = synth.FULL["swiglu"]
        d1 = {k: v.to(dev) for k, v in synth.make_swiglu(s1, seed=0).items()}
        ws1 = coda.workspace(256, dev)
        H1 = torch.empty(s1.tokens, s1.inter, dtype=torch.bfloat16, device=dev)
        m1 = median_ms(lambda: coda.linear_swiglu(d1["X"], d1["Wg"], d1["Wu"], H=H1, g=None, u=None, ws=ws1,
                                                  save=False))
        f1 = 2 * s1.tokens * s1.hidden * s1.inter * 2
        other["swiglu"] = {"workload": f"linear + SwiGLU forward, {s1.tokens} x {s1.hidden} -> {s1.inter} "
                                       f"(launch-latency bound)",
                           "ms": round(m1, 4), "tflops": rate(f1, m1), "frac_of_burst": round(rate(f1, m1) / burst, 4)}

        def swiglu_unfused():
            torch.nn.functional.silu(d1["X"] @ d1["Wg"].t()) * (d1["X"] @ d1["Wu"].t())
        unfused_leg(other["swiglu"], swiglu_unfused, m1)
        del d1

    if "rms" in legs:
        # RMSNorm-reparameterised projection + residual, 4096 x 2048 -> 2048,
        # forward and backward (gain fold, row RMS, prepass and combines
        # included); outputs and workspaces held across calls as a training
        # loop holds them; the gain fold beside the row RMS and dW beside
        # c -> dX on second streams
        s2 = synth.FULL["rmsnorm_linear"]
        d2 = {k: v.to(dev) for k, v in synth.make_rms_linear(s2, seed=0).items()}
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
        side2f = torch.cuda.Stream(device=dev)
        ev_prev, ev_fold = torch.cuda.Event(), torch.cuda.Event()

        def rms_step():
            # the gain fold runs on a second stream beside the row RMS (each
            # reads only inputs, and the fold waits for the previous step's
            # reads of W'); the projection waits for both
            cur = torch.cuda.current_stream()
            ev_prev.record(cur)
            side2f.wait_event(ev_prev)
            with torch.cuda.stream(side2f):
                coda.fold_gamma(d2["W"], d2["gamma"], out=Wf2)
                ev_fold.record(side2f)
            coda.rms_rstd(d2["X"], s2.eps, out=r2)
            cur.wait_event(ev_fold)
            coda.rmsnorm_linear(d2["X"], Wf2, d2["R"], rstd_in=r2, Y=Y2, ws=ws2a)
            coda.rmsnorm_linear_bwd(d2["G"], d2["X"], d2["W"], d2["gamma"], r2, Y2, d2["R"], ws=ws2b, out=g2,
                                    side_stream=side2)
        m2 = median_ms(rms_step)
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
        mg2 = median_ms(graph2.replay)
        if coda.get_status(ws2a) != 0 or coda.get_status(ws2b) != 0:
            raise RuntimeError("device status error in the RMSNorm-linear measurement")
        f2 = 2 * s2.tokens * s2.hidden * s2.out * 3               # fwd 1 GEMM, bwd 2
        other["rmsnorm_linear"] = {
            "workload": f"RMSNorm-reparameterised projection + residual fwd+bwd, tokens {s2.tokens}, "
                        f"hidden {s2.hidden}, out {s2.out} (gain fold, row RMS, prepass and combines included)",
            "ms": round(m2, 4), "tflops": rate(f2, m2), "frac_of_burst": round(rate(f2, m2) / burst, 4),
            "graph_ms": round(mg2, 4), "graph_tflops": rate(f2, mg2),
            "graph_frac_of_burst": round(rate(f2, mg2) / burst, 4)}
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
        unfused_leg(other["rmsnorm_linear"], rms_unfused, m2)
        del d2, p2

    if "mlp" in legs:
        # SwiGLU MLP fwd+bwd at hidden 4096 (weight gradients on a side stream)
        s3 = synth.FULL["mlp"]
        d3 = {k: v.to(dev) for k, v in synth.make_mlp(s3, seed=0).items()}
        ws3 = coda.workspace(max(coda.load().coda_linear_swiglu_bwd_workspace_size(s3.tokens, s3.inter, s3.hidden),
                                 coda.load().coda_linear_residual_workspace_size(s3.tokens, s3.hidden, s3.inter)), dev)
        side3 = torch.cuda.Stream(device=dev)
        o3 = {"H": torch.empty(s3.tokens, s3.inter, dtype=torch.bfloat16, device=dev)}
        o3["g"], o3["u"] = torch.empty_like(o3["H"]), torch.empty_like(o3["H"])
        o3["Y"] = torch.empty_like(d3["R"])
        o3["grads"] = {"dX": torch.empty_like(d3["X"]), "dWg": torch.empty_like(d3["Wg"]),
                       "dWu": torch.empty_like(d3["Wu"]), "dWd": torch.empty_like(d3["Wd"])}

        def mlp_step():
            coda.linear_swiglu(d3["X"], d3["Wg"], d3["Wu"], H=o3["H"], g=o3["g"], u=o3["u"], ws=ws3)
            coda.linear_residual(o3["H"], d3["Wd"], d3["R"], Y=o3["Y"], ws=ws3)
            coda.linear_swiglu_bwd(d3["dY"], d3["X"], d3["Wg"], d3["Wu"], d3["Wd"], o3["g"], o3["u"], o3["H"],
                                   ws=ws3, out=o3["grads"], side_stream=side3)
        m3 = median_ms(mlp_step)
        f3 = 2 * s3.tokens * s3.hidden * s3.inter * 3 * 3       # fwd 3 GEMMs, bwd 6
        other["mlp_swiglu"] = {
            "workload": f"SwiGLU MLP fwd+bwd, tokens {s3.tokens}, hidden {s3.hidden}, intermediate {s3.inter}",
            "ms": round(m3, 4), "tflops": rate(f3, m3), "frac_of_burst": round(rate(f3, m3) / burst, 4)}
        p3 = {k: d3[k].detach().requires_grad_(True) for k in ("X", "Wg", "Wu", "Wd")}

        def mlp_unfused():
            p = p3
            H = torch.nn.functional.silu(p["X"] @ p["Wg"].t()) * (p["X"] @ p["Wu"].t())
            (d3["R"] + H @ p["Wd"].t()).backward(d3["dY"])
            for v in p.values():
                v.grad = None
        unfused_leg(other["mlp_swiglu"], mlp_unfused, m3)
        del d3, p3, o3, ws3

    if "ce" in legs:
        # linear + cross-entropy, 8192 x 2048, vocabulary 128256: forward
        # (online LSE epilogue + combine) and backward (vocabulary slices)
        from gemm_epilogue_transformer_bf16_gb300.block import LinearCE
        cs_ = synth.FULL["linear_ce"]
        dc = {k: v.to(dev) for k, v in synth.make_ce(cs_, seed=0).items()}
        ce = LinearCE(cs_.tokens, cs_.vocab, cs_.hidden, device=dev)

        def ce_step(mark):
            coda.linear_cross_entropy(dc["X"], dc["W"], dc["labels"], out=ce.out, ws=ce.ws)
            mark()
            coda.linear_cross_entropy_bwd(dc["X"], dc["W"], dc["labels"], ce.out["lse"], ce.out["n_valid"], 1.0,
                                          out=ce.grads, ws=ce.ws)
        mf, mb = median_ms(ce_step, parts=2)
        if coda.get_status(ce.ws) != 0:
            raise RuntimeError("device status error in the linear-CE measurement")
        f_fwd = 2 * cs_.tokens * cs_.hidden * cs_.vocab
        f_all = 4 * f_fwd        # the backward recomputes the logits, then dX and dW
        other["linear_cross_entropy"] = {
            "workload": "tokens 8192, hidden 2048, vocab 128256, 5% ignored labels; fwd (online LSE epilogue + "
                        "combine) and bwd (softmax-minus-onehot epilogue, dX, dW, by vocabulary slices of 16384)",
            "fwd_ms": round(mf, 4), "bwd_ms": round(mb, 4), "ms": round(mf + mb, 4),
            "fwd_tflops": rate(f_fwd, mf), "bwd_tflops": rate(3 * f_fwd, mb), "tflops": rate(f_all, mf + mb),
            "frac_of_burst": round(rate(f_all, mf + mb) / burst, 4),
            "bwd_workspace_bytes": coda.load().coda_linear_cross_entropy_bwd_workspace_size(cs_.tokens, cs_.vocab,
                                                                                           cs_.hidden)}
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

    if "fp8" in legs or "nvfp4" in legs or "fp8block" in legs:
        T_, H_, I_ = s.tokens, s.hidden, s.inter
        x0_ = {k: t[k] for k in ("x0", "Wg", "Wu")}
        r_ = coda.rms_rstd(x0_["x0"], s.eps)
        Hq = torch.empty(T_, I_, dtype=torch.bfloat16, device=dev)
        gq8, uq8 = torch.empty_like(Hq), torch.empty_like(Hq)
        ws8 = coda.workspace(256, dev)
        f_gu = 2 * T_ * H_ * 2 * I_
    if "fp8" in legs:
        # e4m3 gate/up + SwiGLU at the block's shape (the same mainloop with
        # kind::f8f6f4), beside the bf16 launch timed in the block step
        xq, sx = coda.quantize_fp8_rows(x0_["x0"])
        gq, sg = coda.quantize_fp8_rows(x0_["Wg"])
        uq, su = coda.quantize_fp8_rows(x0_["Wu"])
        m8 = median_ms(lambda: coda.linear_swiglu_fp8(xq, sx, gq, sg, uq, su, rstd=r_, H=Hq, g=gq8, u=uq8, ws=ws8))
        if coda.get_status(ws8) != 0:
            raise RuntimeError("device status error in the FP8 measurement")
        fp8_peak = 2 * burst
        other["fp8_gateup_swiglu"] = {
            "workload": f"e4m3 gate/up GEMM with row-scale + SwiGLU epilogue, {T_} x 2x{I_} x {H_}, per-row scales",
            "ms": round(m8, 4), "tflops": rate(f_gu, m8),
            "peak": round(fp8_peak, 1), "peak_kind": f"fp8 = 2 x bf16 burst ({peak_src}, nominal ratio)",
            "frac": round(rate(f_gu, m8) / fp8_peak, 4)}
        # the other epilogues on the FP8 mainloop at the block's shapes: the
        # QKV projection with QK-norm + RoPE (8192 x 10240 x 8192), and the
        # MLP backward's input-gradient chain -- dH GEMM with the dSwiGLU
        # epilogue (8192 x 28672 x 8192), G' quantised per row, the dX GEMM
        # with the RMSNorm-backward epilogue (8192 x 8192 x 57344); weights'
        # transposed operands from the column quantiser (timed separately)
        n_qkv = s.qkv_out
        wqkv_q, swqkv = coda.quantize_fp8_rows(t["Wqkv"])
        qk_out = {"Q": torch.empty(T_, s.n_q * s.head_dim, dtype=torch.bfloat16, device=dev),
                  "K": torch.empty(T_, s.n_kv * s.head_dim, dtype=torch.bfloat16, device=dev),
                  "V": torch.empty(T_, s.n_kv * s.head_dim, dtype=torch.bfloat16, device=dev),
                  "qk_save": torch.empty(T_, (s.n_q + s.n_kv) * s.head_dim, dtype=torch.bfloat16, device=dev)}
        cs8 = coda.rope_table(s.theta, s.head_dim, s.seq_len, device=dev)
        gam = t["gamma_q"], t["gamma_k"]
        mq = median_ms(lambda: coda.linear_qknorm_rope_fp8(xq, sx, wqkv_q, swqkv, gam[0], gam[1], t["pos"], cs8,
                                                           s.n_q, s.n_kv, rstd=r_, eps=s.eps, out=qk_out, ws=ws8))
        mqb = median_ms(lambda: coda.linear_qknorm_rope(t["x0"], t["Wqkv"], gam[0], gam[1], t["pos"], cs8, s.n_q,
                                                        s.n_kv, rstd=r_, eps=s.eps, out=qk_out, ws=ws8))
        f_qkv = 2 * T_ * H_ * n_qkv
        other["fp8_qknorm_rope"] = {
            "workload": f"e4m3 QKV GEMM with QK-RMSNorm + RoPE epilogue, {T_} x {n_qkv} x {H_}",
            "ms": round(mq, 4), "tflops": rate(f_qkv, mq), "frac": round(rate(f_qkv, mq) / fp8_peak, 4),
            "bf16_ms": round(mqb, 4), "speedup_vs_bf16": round(mqb / mq, 3)}
        del wqkv_q, qk_out
        mwd = median_ms(lambda: coda.quantize_fp8_cols(t["Wd"]))
        wdt_q, swdt = coda.quantize_fp8_cols(t["Wd"])
        mwgu = median_ms(lambda: coda.quantize_fp8_cols(t["Wg"], t["Wu"]))
        wgut_q, swgut = coda.quantize_fp8_cols(t["Wg"], t["Wu"])
        dyq, sdy = coda.quantize_fp8_rows(t["dx2"])
        Gp8 = torch.empty(T_, 2 * I_, dtype=torch.bfloat16, device=dev)
        gq_, sgq_ = torch.empty(T_, 2 * I_, dtype=torch.uint8, device=dev), torch.empty(T_, dtype=torch.float32,
                                                                                       device=dev)
        coef8 = torch.empty(T_, dtype=torch.float32, device=dev)
        dx8 = {"dX": torch.empty(T_, H_, dtype=torch.bfloat16, device=dev),
               "dgamma": torch.empty(H_, dtype=torch.float32, device=dev)}
        ws_ds = coda.workspace(coda.load().coda_linear_dswiglu_fp8_workspace_size(T_, I_, H_), dev)
        ws_dx = coda.workspace(coda.load().coda_rmsnorm_linear_dx_fp8_workspace_size(T_, 2 * I_, H_), dev)

        def fp8_dgrad(mark):
            coda.linear_dswiglu_fp8(dyq, sdy, wdt_q, swdt, gq8, uq8, rstd=r_,
                                    out={"Gp": Gp8, "row": coef8, "H": None}, ws=ws_ds)
            mark()
            coda.quantize_fp8_rows(Gp8, Xq=gq_, scale=sgq_)
            mark()
            coda.rmsnorm_linear_dx_fp8(gq_, sgq_, wgut_q, swgut, t["x0"], t["gamma_mlp"], coef8,
                                       dX_resid=t["dx2"], out=dx8, ws=ws_dx)
        md = median_ms(fp8_dgrad, parts=3)
        if coda.get_status(ws_ds) != 0 or coda.get_status(ws_dx) != 0:
            raise RuntimeError("device status error in the FP8 backward measurement")
        f_dh, f_dx = 2 * T_ * H_ * I_, 2 * T_ * 2 * I_ * H_
        other["fp8_mlp_dgrad"] = {
            "workload": f"e4m3 MLP input-gradient chain: dH GEMM + dSwiGLU epilogue {T_} x {I_} x {H_}, G' row "
                        f"quantisation, dX GEMM + RMSNorm-backward epilogue {T_} x {H_} x {2 * I_}",
            "ms": round(sum(md), 4), "dswiglu_ms": round(md[0], 4), "quantize_g_ms": round(md[1], 4),
            "rms_dx_ms": round(md[2], 4), "dswiglu_tflops": rate(f_dh, md[0]), "rms_dx_tflops": rate(f_dx, md[2]),
            "gemm_frac": round(rate(f_dh + f_dx, md[0] + md[2]) / fp8_peak, 4),
            "weight_quant_ms": {"Wd^T": round(mwd, 4), "[Wg;Wu]^T": round(mwgu, 4)}}
        del wdt_q, wgut_q, dyq, Gp8, gq_, ws_ds, ws_dx, dx8
        del xq, gq, uq
    if "fp8block" in legs:
        # the whole block step with the FP8 GEMMs (BlockFP8): forward
        # projections and the MLP / O-projection input gradients on e4m3
        # operands, weights quantised every step inside the step
        from gemm_epilogue_transformer_bf16_gb300.block import BlockFP8
        args8 = (t["x0"], t["A"], t["pos"], t["dx2"], t["dQ"], t["dK"], t["dV"])
        n8 = max(10, min(args.steps, 30))
        res8 = {}
        for fw in (True, False):
            b8 = BlockFP8(s, t, device=dev, fp8_wgrad=fw)

            def fp8_step(mark, b8=b8):
                b8.step(*args8, mark=lambda name: mark())
            res8[fw] = median_ms(fp8_step, n=n8, warm=3, parts=3)
            if coda.get_status(b8.ws) != 0 or coda.get_status(b8.ws2) != 0:
                raise RuntimeError("device status error in the FP8 block measurement")
            f_blk = sum(b8.gemm_flops().values())
            del b8
        mq8, mf8, mb8 = res8[True]
        m8 = mq8 + mf8 + mb8
        m8b = sum(res8[False])
        other["fp8_block"] = {
            "workload": "the block step (tokens 8192, hidden 8192) with every GEMM on e4m3 operands: forward "
                        "projections, input gradients, weight gradients (operands quantised per column over the "
                        "tokens) and both GEMMs of the QKV backward; weights quantised inside the step",
            "ms": round(m8, 4), "tflops": rate(f_blk, m8), "quantize_weights_ms": round(mq8, 4),
            "fwd_ms": round(mf8, 4), "bwd_ms": round(mb8, 4),
            "bf16_wgrad_and_qkv_bwd_ms": round(m8b, 4),
            "bf16_block_ms": round(blk_res["median_step"], 4) if blk_res else None,
            "speedup_vs_bf16_block": round(blk_res["median_step"] / m8, 3) if blk_res else None}
    if "nvfp4" in legs:
        # NVFP4 (e2m1 + e4m3 block scales) gate/up + SwiGLU at the same shape:
        # the block-scaled kind::mxf4nvf4 mainloop, single CTAs
        xq4, sfx4, sx4 = coda.quantize_nvfp4_rows(x0_["x0"])
        gq4, sfg4, sg4 = coda.quantize_nvfp4_rows(x0_["Wg"])
        uq4, sfu4, su4 = coda.quantize_nvfp4_rows(x0_["Wu"])
        mq4 = median_ms(lambda: coda.quantize_nvfp4_rows(x0_["x0"]))
        m4 = median_ms(lambda: coda.linear_swiglu_nvfp4(xq4, sfx4, sx4, gq4, sfg4, sg4, uq4, sfu4, su4, rstd=r_,
                                                        H=Hq, g=gq8, u=uq8, ws=ws8))
        if coda.get_status(ws8) != 0:
            raise RuntimeError("device status error in the NVFP4 measurement")
        fp4_peak = 6 * burst
        other["nvfp4_gateup_swiglu"] = {
            "workload": f"NVFP4 gate/up GEMM (e2m1, e4m3 scale per 16, fp32 row scale) with row-scale + SwiGLU "
                        f"epilogue, {T_} x 2x{I_} x {H_}, single-CTA tiles",
            "ms": round(m4, 4), "tflops": rate(f_gu, m4),
            "peak": round(fp4_peak, 1), "peak_kind": f"fp4 = 6 x bf16 burst ({peak_src}, nominal ratio)",
            "frac": round(rate(f_gu, m4) / fp4_peak, 4), "quantize_x_ms": round(mq4, 4)}
        del xq4, gq4, uq4, sfx4, sfg4, sfu4
    if "fp8" in legs or "nvfp4" in legs or "fp8block" in legs:
        del Hq, gq8, uq8, x0_

    # ---------------------------------------------------------------- CPU oracle baseline
    cpu = None
    if not args.no_cpu_baseline and args.tokens == synth.FULL["block"].tokens:
        torch.set_num_threads(cores())
        v, dt, fl = oracle_sample_timing(args.cpu_tokens, oracle_inputs(host, args.cpu_tokens))
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores(), "kind": "oracle",
               "sample": f"fp64 NumPy block_fwd+block_bwd on the first {args.cpu_tokens} of 8192 tokens "
                         f"(full weights): {fl / 1e12:.3f} TFLOP in {dt:.1f} s",
               "per_workload": oracle_workload_timings(args.cpu_tokens, (v, dt, fl))}

    r = blk_res or {}
    value, ms_step = r.get("value"), r.get("ms_step")
    line = {
        "metric": METRIC, "value": round(value, 2) if value else None, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3) if ms_step else None,
        "median_ms_per_step": round(r["median_step"], 3) if r else None, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens": s.tokens, "hidden": s.hidden, "n_q": s.n_q,
                   "n_kv": s.n_kv, "head_dim": s.head_dim, "inter": s.inter,
                   "tflop_per_step": round(r["flops_step"] / 1e12, 3) if r else None,
                   "l2": "block step: inputs (1.7 GB of weights + activations) exceed the 129 MB L2, no flush; "
                         f"other workloads: {FLUSH_BYTES >> 20} MB written between timed calls",
                   "parallelism": "single GPU",
                   "rmsnorm_gain": "folded into the weights each step" if args.fold_weights
                   else "applied by the producing epilogue (u = x ⊙ gamma)"},
        "pct_bf16_peak": {"burst": round(value / burst, 4), "sustained": round(value / sustained, 4),
                          "source": peak_src} if value else None,
        "roofline": r.get("roofline"),
        "cpu_baseline": cpu,
        "e2e": r.get("e2e"),
        "gpu_launches": r["launches_timed"] if r else None,
        "clocks": r.get("clk"),
        "unfused_ms_per_step": round(r["unfused_ms"], 3) if r.get("unfused_ms") else None,
        "speedup_vs_unfused": round(r["unfused_ms"] / r["median_step"], 3) if r.get("unfused_ms") else None,
        "stages": r.get("stages"),
        "other_workloads": other or None,
    }
    print(json.dumps(line), flush=True)
    return 0

if __name__ == "__main__":
    sys.exit(main())
