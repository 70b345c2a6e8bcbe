#!/usr/bin/env python
"""Benchmark of the exact tiled attention hot path on GB300.

One STEP is one pass of the whole path over one batch of synthetic input:
  bf16 forward (causal)  ->  backward: preprocess, main kernel, dQ conversion
  ->  E4M3 quantisation of Q, K, V  ->  FP8 forward (non-causal)
all through the C ABI of libfa_gb300.so.  Default workload: B=2, H=16,
N=4096, d=128 (the long-head shape; the accuracy/throughput targets are stated
for N >= 4096, d = 128).  The metric is algorithmic TFLOPS:
  F = 4 B H N^2 d per forward, 2.5 F per backward, halved when causal;
  the FP8 forward counts its F (non-causal).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  --impl reference times the fp64 CPU oracle
(as it stands) on the host cores instead.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOPS on 1 GB300 and % of dense BF16/FP8 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal dense tensor-core ratios (FP8 runs at twice the BF16 rate).
FP8_OVER_BF16 = 2.0
L2_FLUSH_BYTES = 512 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long_head")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=0, help="0 = min(steps, 100)")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {k: float(pk[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def dist_setup(want_gpus):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def flops_fwd(w, causal):
    return 4.0 * w.B * w.H * w.N * w.N * w.d * (0.5 if causal else 1.0)


# --------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clk", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- kernel source id
def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_tiled_attention_10_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel):
    """DRAM bytes per launch recorded from an ncu capture of the current
    kernel sources (profiles/dram_traffic.json), else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            rec = json.load(f)
        if rec.get("source_hash") != kernel_source_hash():
            return None
        return rec["kernels"][kernel]["bytes_per_launch_full_workload"]
    except Exception:
        return None


# ---------------------------------------------------------------- CPU oracle
def oracle_sample(w, causal, heads, R, nthreads):
    """Time the fp64 oracle (materialised forward + backward) on the first R
    positions of `heads` heads of the workload.  With a causal mask that prefix
    is a self-contained causal problem; without one it is the top-left R x R
    block.  Returns (seconds, algorithmic flops)."""
    import oracle
    from exact_tiled_attention_10_gb300.inputs import qkv
    q, k, v, do = qkv(1, heads, R, w.d, w.seed + 17)
    t0 = time.perf_counter()
    oracle.bwd(q, k, v, do, w.scale, causal=causal, nthreads=nthreads)
    dt = time.perf_counter() - t0
    f = 4.0 * heads * R * R * w.d * (0.5 if causal else 1.0) * 3.5
    return dt, f


def cpu_baseline(w, causal, budget_s=20.0):
    import oracle
    cores = oracle.default_threads()
    heads = max(1, min(cores, w.B * w.H))
    # calibrate on a small prefix, then size R so the sample takes ~budget_s
    R0 = 512
    t0, _ = oracle_sample(w, causal, heads, R0, heads)
    R = int(R0 * math.sqrt(max(budget_s, 1e-3) / max(t0, 1e-6)))
    R = max(R0, min(w.N, (R // 64) * 64))
    dt, f = oracle_sample(w, causal, heads, R, heads)
    return {"value": f / dt / 1e12, "unit": "TFLOPS", "cores": heads, "kind": "oracle",
            "sample": "fp64 oracle forward+backward (materialised S, P) on %d heads x the first "
                      "%d of %d positions (%s), one thread per head, %.1f s" % (
                          heads, R, w.N, "causal" if causal else "non-causal", dt)}


def run_reference(args, w, causal):
    """The reference arm: the fp64 oracle as it stands, on the host cores."""
    import oracle
    cores = oracle.default_threads()
    heads = max(1, min(cores, w.B * w.H))
    total_budget = 150.0
    per_step = total_budget / max(1, args.steps + args.warmup)
    R0 = 128
    tc, _ = oracle_sample(w, causal, heads, R0, heads)
    R = int(R0 * math.sqrt(max(per_step, 1e-3) / max(tc, 1e-6)))
    R = max(64, min(w.N, (R // 64) * 64))
    for _ in range(args.warmup):
        oracle_sample(w, causal, heads, R, heads)
    tot_t, tot_f = 0.0, 0.0
    for _ in range(args.steps):
        dt, f = oracle_sample(w, causal, heads, R, heads)
        tot_t += dt
        tot_f += f
    value = tot_f / tot_t / 1e12
    sample = ("fp64 oracle forward+backward on %d heads x the first %d of %d positions per step "
              "(%s), one thread per head" % (heads, R, w.N, "causal" if causal else "non-causal"))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * tot_t / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": causal},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": heads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU step
class Step:
    """All buffers of one step, preallocated; run() enqueues the step's launches
    on the current stream with an event before and after every phase."""

    PHASES = ["fwd", "bwd_pre", "bwd_main", "bwd_dq", "quant_fp8", "fwd_fp8"]

    def __init__(self, w, causal, device, seed_offset=0):
        import torch
        import exact_tiled_attention_10_gb300 as fa
        from exact_tiled_attention_10_gb300.inputs import qkv
        self.fa, self.torch, self.w, self.causal = fa, torch, w, causal
        self.lib = fa.load_library()
        self.dev = device
        B, H, N, d = w.B, w.H, w.N, w.d
        self.q, self.k, self.v, self.do = qkv(B, H, N, d, w.seed + seed_offset, device=device)
        t = lambda *s, dt=torch.bfloat16: torch.empty(*s, dtype=dt, device=device)
        self.o, self.dq, self.dk, self.dv = (t(B, H, N, d) for _ in range(4))
        self.lse = t(B, H, N, dt=torch.float32)
        self.ws_bytes = fa.bwd_workspace_size(torch.bfloat16, B, H, N, d)
        self.ws = t(self.ws_bytes, dt=torch.uint8)
        nb = self.lib.fa_fp8_num_blocks(N)
        self.x8 = [t(B, H, N, d, dt=torch.uint8) for _ in range(3)]
        self.sc = [t(B, H, nb, dt=torch.float32) for _ in range(3)]
        self.o8 = t(B, H, N, d)
        self.lse8 = t(B, H, N, dt=torch.float32)
        self.flush = t(L2_FLUSH_BYTES, dt=torch.uint8)
        # split-key plans (automatic): the causal bf16 forward is never split;
        # the non-causal FP8 forward may be (its merge kernel is part of the call)
        self.split_bf16 = self.lib.fa_fwd_split_count(B, H, N, d, int(causal), 0, 0)
        self.split_fp8 = self.lib.fa_fwd_split_count(B, H, N, d, 0, 0, 0)
        self.sws_bytes = max(self.lib.fa_fwd_split_workspace_size(B, H, N, d, int(causal), 0, 0),
                             self.lib.fa_fwd_split_workspace_size(B, H, N, d, 0, 0, 0))
        self.sws = t(max(self.sws_bytes, 256), dt=torch.uint8)
        self.scale = 1.0 / math.sqrt(d)
        F = flops_fwd(w, causal)
        self.flops = {"fwd": F, "bwd_pre": 0.0, "bwd_main": 2.5 * F, "bwd_dq": 0.0,
                      "quant_fp8": 0.0, "fwd_fp8": flops_fwd(w, False)}
        n = B * H * N * d
        Np = (N + 127) // 128 * 128
        self.bytes = {"fwd": 4 * n * 2 + B * H * N * 4,
                      "bwd_pre": 2 * n * 2 + B * H * N * 4 + 2 * B * H * Np * 4 + B * H * Np * d * 4,
                      "bwd_main": 4 * n * 2 + 2 * B * H * Np * 4 + 2 * n * 2 + 2 * B * H * Np * d * 4,
                      "bwd_dq": B * H * Np * d * 4 + n * 2,
                      "quant_fp8": 3 * (n * 2 + n + B * H * nb * 4),
                      "fwd_fp8": 3 * n + n * 2 + B * H * N * 4}
        self.launches_per_step = 6 + int(self.split_bf16 > 1) + int(self.split_fp8 > 1)

    def _ck(self, st):
        if st != 0:
            raise RuntimeError(self.lib.fa_last_error().decode())

    def run(self, events=None):
        lib, w, s = self.lib, self.w, self.torch.cuda.current_stream(self.dev).cuda_stream
        B, H, N, d = w.B, w.H, w.N, w.d
        p = lambda x: x.data_ptr()
        rec = (lambda i: events[i].record()) if events is not None else (lambda i: None)
        rec(0)
        self._ck(lib.fa_fwd_split(p(self.q), p(self.k), p(self.v), p(self.o), p(self.lse), B, H, N, d,
                                  self.scale, int(self.causal), None, 0, p(self.sws), self.sws_bytes, s))
        rec(1)
        self._ck(lib.fa_bwd_preprocess(p(self.o), p(self.lse), p(self.do), B, H, N, d, p(self.ws),
                                       self.ws_bytes, s))
        rec(2)
        self._ck(lib.fa_bwd_main(p(self.q), p(self.k), p(self.v), p(self.do), p(self.dk), p(self.dv),
                                 B, H, N, d, self.scale, int(self.causal), None, p(self.ws),
                                 self.ws_bytes, s))
        rec(3)
        self._ck(lib.fa_bwd_dq(p(self.dq), B, H, N, d, self.scale, p(self.ws), self.ws_bytes, s))
        rec(4)
        self._ck(lib.fa_quantize_fp8_qkv(p(self.q), p(self.k), p(self.v), p(self.x8[0]), p(self.x8[1]),
                                         p(self.x8[2]), p(self.sc[0]), p(self.sc[1]), p(self.sc[2]), B, H, H, N, d,
                                         s))
        rec(5)
        self._ck(lib.fa_fwd_fp8_split(p(self.x8[0]), p(self.x8[1]), p(self.x8[2]), p(self.sc[0]),
                                      p(self.sc[1]), p(self.sc[2]), p(self.o8), p(self.lse8), B, H, N, d,
                                      self.scale, 0, None, 0, p(self.sws), self.sws_bytes, s))
        rec(6)

    def flush_l2(self):
        self.flush.zero_()


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, x, device):
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def e2e_pipelined(step_a, step_b, steps):
    """End to end through the C ABI with pinned host buffers: every step copies
    its inputs (Q, K, V, dO) in from the host, runs the whole step and copies
    its results (O, LSE, dQ, dK, dV, FP8 O) back.  The copies of step k+1 (in)
    and k-1 (out) run on their own streams while step k computes, on two sets
    of device buffers; events keep a buffer from being overwritten while it is
    still read or written.  Returns the milliseconds of `steps` steps, from
    the first copy in to the last copy out."""
    import torch
    dev = step_a.dev
    steps_ = (step_a, step_b)
    ins = lambda st: (st.q, st.k, st.v, st.do)
    outs = lambda st: (st.o, st.lse, st.dq, st.dk, st.dv, st.o8)
    hin = [[t.cpu().pin_memory() for t in ins(st)] for st in steps_]
    hout = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs(st)] for st in steps_]
    s_in, s_c, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()

    def run(n, timed):
        done_c = [None, None]   # compute of the last step on buffer b
        done_o = [None, None]   # copy out of the last step on buffer b
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        s_in.record_event(t0)
        for k in range(n):
            b = k % 2
            st = steps_[b]
            with torch.cuda.stream(s_in):
                if done_c[b] is not None:
                    s_in.wait_event(done_c[b])
                for dd, hh in zip(ins(st), hin[b]):
                    dd.copy_(hh, non_blocking=True)
                e_in = ev()
                s_in.record_event(e_in)
            with torch.cuda.stream(s_c):
                s_c.wait_event(e_in)
                if done_o[b] is not None:
                    s_c.wait_event(done_o[b])
                st.run()
                done_c[b] = ev()
                s_c.record_event(done_c[b])
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_c[b])
                for hh, dd in zip(hout[b], outs(st)):
                    hh.copy_(dd, non_blocking=True)
                done_o[b] = ev()
                s_out.record_event(done_o[b])
        for e in done_o:
            if e is not None:
                s_in.wait_event(e)
        s_in.record_event(t1)
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1)

    run(3, False)  # warm-up
    return run(steps, True)


def main():
    args = parse_args()
    ws, rank, local = dist_setup(args.gpus)
    from exact_tiled_attention_10_gb300.inputs import WORKLOADS
    w = WORKLOADS[args.workload]
    causal = True

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, w, causal)
        return

    import torch
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from exact_tiled_attention_10_gb300 import build as fa_build
    if rank == 0 or ws == 1:
        fa_build.build()
    barrier(ws)
    import exact_tiled_attention_10_gb300 as fa
    fa.load_library()

    step = Step(w, causal, device, seed_offset=1000 * rank)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(args.steps)]
    for _ in range(max(args.warmup, 3)):
        step.run()
        step.flush_l2()
    torch.cuda.synchronize()
    fa.check_device_status(device)

    clocks = ClockSampler(local)
    barrier(ws)
    torch.cuda.synchronize()
    clocks.start()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        step.run(ev[i])
        step.flush_l2()  # outside the step's events: L2 holds nothing of the next step
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(ws)
    clk = clocks.stop()
    fa.check_device_status(device)

    phase_ms = {ph: [] for ph in Step.PHASES}
    step_ms = []
    for e in ev:
        step_ms.append(e[0].elapsed_time(e[6]))
        for j, ph in enumerate(Step.PHASES):
            phase_ms[ph].append(e[j].elapsed_time(e[j + 1]))
    total_ms = max_over_ranks(ws, sum(step_ms), device)
    flops_step = sum(step.flops.values())
    value = ws * flops_step * args.steps / (total_ms / 1e3) / 1e12

    peaks, peak_src = load_peaks()
    bf16_peak = peaks["bf16_tflops_sustained"]
    passes = {}
    for ph in Step.PHASES:
        ms = statistics.mean(phase_ms[ph])
        ent = {"ms": round(ms, 4)}
        if step.flops[ph]:
            tf = step.flops[ph] / (ms / 1e3) / 1e12
            pk = bf16_peak * (FP8_OVER_BF16 if ph == "fwd_fp8" else 1.0)
            ent.update({"tflops": round(tf, 1), "frac_of_peak": round(tf / pk, 4),
                        "peak_tflops": pk})
        ent["gbs"] = round(step.bytes[ph] / (ms / 1e3) / 1e9, 1)
        if not step.flops[ph]:
            ent["frac_of_hbm"] = round(ent["gbs"] / peaks["hbm_gbs"], 4)
        passes[ph] = ent
    dom = max(("fwd", "bwd_main", "fwd_fp8"), key=lambda ph: statistics.mean(phase_ms[ph]))
    dom_ms = statistics.mean(phase_ms[dom])
    dom_peak = bf16_peak * (FP8_OVER_BF16 if dom == "fwd_fp8" else 1.0)
    achieved = step.flops[dom] / (dom_ms / 1e3) / 1e12
    roofline = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1),
                "peak": dom_peak, "unit": "TFLOP/s", "frac": round(achieved / dom_peak, 4),
                "traffic": recorded_traffic(dom),
                "peak_source": "%s (%s)" % (peak_src, "dense bf16 sustained" +
                                            (" x2 for e4m3" if dom == "fwd_fp8" else ""))}

    # ---- end to end through the public API with pinned host buffers
    e2e_steps = args.e2e_steps or min(args.steps, 100)
    e2e_ms = e2e_pipelined(step, Step(w, causal, device, seed_offset=1000 * rank), e2e_steps)
    hin_bytes = sum(t.numel() * t.element_size() for t in (step.q, step.k, step.v, step.do))
    hout_bytes = sum(t.numel() * t.element_size() for t in (step.o, step.lse, step.dq, step.dk, step.dv, step.o8))
    h2d, d2h = hin_bytes, hout_bytes
    e2e_ms = max_over_ranks(ws, e2e_ms, device)
    e2e_value = ws * flops_step * e2e_steps / (e2e_ms / 1e3) / 1e12

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        try:
            cpu = cpu_baseline(w, causal)
        except Exception as ex:  # reported, not fatal
            cpu = {"value": None, "unit": "TFLOPS", "cores": 0, "kind": "oracle",
                   "sample": "failed: %s" % ex}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOPS", "n_gpus": ws,
            "steps": args.steps, "warmup": max(args.warmup, 3),
            "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16+e4m3", "data": "synthetic",
            "config": {"workload": "%s: B=%d H=%d N=%d d=%d; bf16 causal fwd + bwd, then E4M3 "
                                   "quantise Q/K/V + FP8 non-causal fwd" % (w.name, w.B, w.H, w.N, w.d),
                       "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": causal,
                       "l2": "flushed between steps (512 MiB write outside the timed events)",
                       "parallelism": "replicas" if ws > 1 else "single GPU"},
            "passes": passes,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 2), "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "how": "C ABI with pinned host buffers; every step copies Q, K, V, dO in and O, LSE, "
                           "dQ, dK, dV, FP8 O out; copies of neighbouring steps overlap compute (two "
                           "device buffer sets, three streams); inputs of %.0f MB per step, "
                           "L2 129 MB" % (h2d / 1e6)},
            "gpu_launches": step.launches_per_step * args.steps,
            "clocks": clk,
            "wall_s": round(wall, 3),
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
