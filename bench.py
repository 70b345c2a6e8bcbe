#!/usr/bin/env python
"""Benchmark of the exact tiled attention hot path on GB300.

One STEP is one pass of the whole path over one batch of synthetic input:
  bf16 forward (causal)  ->  backward: preprocess, main kernel, dQ conversion
  ->  E4M3 quantisation of Q, K, V  ->  FP8 forward (non-causal)
all through the C ABI of libfa_gb300.so.  L2 is flushed before the step and
again between its bf16 and FP8 parts, outside the timed events, so that each
part starts cold, with no dirty lines of the other part's outputs to write
back (the bf16 backward leaves ~100 MB of dK, dV and dQ in L2, which cost the
HBM-bound quantiser ~15% when it ran right behind it).  Default workload: B=2, H=16,
N=4096, d=128 (the long-head shape; the accuracy/throughput targets are stated
for N >= 4096, d = 128).  The metric is algorithmic TFLOPS:
  F = 4 B H N^2 d per forward, 2.5 F per backward, halved when causal.

The headline `value` is the bf16 rate: (F_fwd + F_bwd) over the time of the
bf16 forward plus the whole backward call (preprocess + main + dQ
conversion), summed over the timed steps.  The FP8 rows (quantiser + FP8
forward) run inside the same steps and are reported on their own (`fp8`),
against the FP8 peak; no figure mixes bf16 and E4M3 FLOPs.  Fractions use the
measured BURST dense bf16 peak (FP8: twice that): each kernel runs for well
under a second at a time.  `configs` holds the same figures for the other
workload shapes (mid, ragged with its effective FLOPs, long_seq).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  --impl reference times the fp64 CPU oracle
(as it stands) on the host cores instead.
"""
from __future__ import annotations

import argparse
import ctypes
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
    ap.add_argument("--no-configs", action="store_true", help="skip the other workload shapes")
    ap.add_argument("--config-reps", type=int, default=20)
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
    BF16 = ("fwd", "bwd_pre", "bwd_main", "bwd_dq")

    def __init__(self, w, causal, device, seed_offset=0, fp8=True):
        import torch
        import exact_tiled_attention_10_gb300 as fa
        from exact_tiled_attention_10_gb300.inputs import kv_lens_ragged, qkv
        self.fa, self.torch, self.w, self.causal, self.with_fp8 = fa, torch, w, causal, fp8
        self.lib = fa.load_library()
        self.dev = device
        B, H, N, d = w.B, w.H, w.N, w.d
        self.q, self.k, self.v, self.do = qkv(B, H, N, d, w.seed + seed_offset, device=device)
        self.kv = kv_lens_ragged(B, N, w.seed, device=device) if w.ragged else None
        t = lambda *s, dt=torch.bfloat16: torch.empty(*s, dtype=dt, device=device)
        self.o, self.dq, self.dk, self.dv = (t(B, H, N, d) for _ in range(4))
        self.lse = t(B, H, N, dt=torch.float32)
        self.ws_bytes = fa.bwd_workspace_size(torch.bfloat16, B, H, N, d)
        self.ws = t(self.ws_bytes, dt=torch.uint8)
        nb = self.lib.fa_fp8_num_blocks(N)
        if fp8:
            self.x8 = [t(B, H, N, d, dt=torch.uint8) for _ in range(3)]
            self.sc = [t(B, H, nb, dt=torch.float32) for _ in range(3)]
            self.o8 = t(B, H, N, d)
            self.lse8 = t(B, H, N, dt=torch.float32)
        self.flush = t(L2_FLUSH_BYTES, dt=torch.uint8)
        self.flush_rd = torch.ones(L2_FLUSH_BYTES // 2, dtype=torch.uint8, device=device)
        # split-key plans (automatic): the causal bf16 forward is never split;
        # the non-causal FP8 forward may be (its merge kernel is part of the call)
        has_kv = self.kv is not None
        self.split_bf16 = fa.split_count(B, H, N, d, causal, has_kv, 0)
        self.split_fp8 = fa.split_count(B, H, N, d, False, False, 0)
        self.sws_bytes = max(fa.split_workspace_size(B, H, N, d, causal, has_kv, 0),
                             fa.split_workspace_size(B, H, N, d, False, False, 0))
        self.sws = t(max(self.sws_bytes, 256), dt=torch.uint8)
        self.scale = 1.0 / math.sqrt(d)
        # the two forwards as fa_attn_fwd parameter blocks (automatic key split)
        self.p_fwd = fa.attn_params(batch=B, heads=H, seqlen_q=N, head_dim=d, scale=self.scale, causal=int(causal),
                                    kv_lens=self.kv, num_splits=0, q=self.q, k=self.k, v=self.v, o=self.o,
                                    lse=self.lse, workspace=self.sws, workspace_bytes=self.sws_bytes)
        if fp8:
            self.p_fp8 = fa.attn_params(dtype=fa.FA_E4M3, batch=B, heads=H, seqlen_q=N, head_dim=d, scale=self.scale,
                                        num_splits=0, q=self.x8[0], k=self.x8[1], v=self.x8[2], q_scale=self.sc[0],
                                        k_scale=self.sc[1], v_scale=self.sc[2], o=self.o8, lse=self.lse8,
                                        workspace=self.sws, workspace_bytes=self.sws_bytes)
        F = flops_fwd(w, causal)
        self.flops = {"fwd": F, "bwd_pre": 0.0, "bwd_main": 2.5 * F, "bwd_dq": 0.0,
                      "quant_fp8": 0.0, "fwd_fp8": flops_fwd(w, False)}
        # the ragged workload: the FLOPs of the visible (query, key) pairs only
        self.flops_eff = None
        if self.kv is not None:
            Feff = 4.0 * H * d * N * float(self.kv.sum().item()) * (0.5 if causal else 1.0)
            self.flops_eff = {"fwd": Feff, "bwd": 2.5 * Feff}
        n = B * H * N * d
        Np = (N + 127) // 128 * 128
        self.bytes = {"fwd": 4 * n * 2 + B * H * N * 4,
                      "bwd_pre": 2 * n * 2 + B * H * N * 4 + 2 * B * H * Np * 4 + B * H * Np * d * 4,
                      "bwd_main": 4 * n * 2 + 2 * B * H * Np * 4 + 2 * n * 2 + 2 * B * H * Np * d * 4,
                      "bwd_dq": B * H * Np * d * 4 + n * 2,
                      "quant_fp8": 3 * (n * 2 + n + B * H * nb * 4),
                      "fwd_fp8": 3 * n + n * 2 + B * H * N * 4}
        self.launches_bf16 = 4 + int(self.split_bf16 > 1)
        self.launches_fp8 = 2 + int(self.split_fp8 > 1)
        self.launches_per_step = self.launches_bf16 + (self.launches_fp8 if fp8 else 0)

    def _ck(self, st):
        if st != 0:
            raise RuntimeError(self.lib.fa_last_error().decode())

    def phases(self):
        return list(self.PHASES) if self.with_fp8 else list(self.BF16)

    def events(self):
        """A start and an end event for each phase of phases()."""
        return [self.torch.cuda.Event(enable_timing=True) for _ in range(2 * len(self.phases()))]

    def run(self, events=None):
        """One step; events[2i] / events[2i + 1] bracket phase i of phases()."""
        lib, w, s = self.lib, self.w, self.torch.cuda.current_stream(self.dev).cuda_stream
        B, H, N, d = w.B, w.H, w.N, w.d
        p = lambda x: x.data_ptr()
        kv = None if self.kv is None else p(self.kv)
        ev = iter(events) if events is not None else None
        rec = (lambda: next(ev).record()) if ev is not None else (lambda: None)
        rec()
        self._ck(lib.fa_attn_fwd(ctypes.byref(self.p_fwd), s))
        rec(), rec()
        self._ck(lib.fa_bwd_preprocess(p(self.o), p(self.lse), p(self.do), B, H, N, d, p(self.ws),
                                       self.ws_bytes, s))
        rec(), rec()
        self._ck(lib.fa_bwd_main(p(self.q), p(self.k), p(self.v), p(self.do), p(self.dk), p(self.dv),
                                 B, H, N, d, self.scale, int(self.causal), kv, p(self.ws),
                                 self.ws_bytes, s))
        rec(), rec()
        self._ck(lib.fa_bwd_dq(p(self.dq), B, H, N, d, self.scale, p(self.ws), self.ws_bytes, s))
        rec()
        if not self.with_fp8:
            return
        self.flush_l2()  # between the parts, outside every phase's events
        rec()
        self._ck(lib.fa_quantize_fp8_qkv(p(self.q), p(self.k), p(self.v), p(self.x8[0]), p(self.x8[1]),
                                         p(self.x8[2]), p(self.sc[0]), p(self.sc[1]), p(self.sc[2]), B, H, H,
                                         N, d, s))
        rec(), rec()
        self._ck(lib.fa_attn_fwd(ctypes.byref(self.p_fp8), s))
        rec()

    def flush_l2(self):
        """Writes a buffer four times the size of L2, then reads one twice its
        size: L2 ends holding none of the step's data and no dirty lines."""
        self.flush.zero_()
        self._sink = self.flush_rd.max()


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
    its inputs (Q, K, V, dO) in from the host, runs the bf16 forward and
    backward (the headline's work) and copies its results (O, LSE, dQ, dK, dV)
    back.  The copies of step k+1 (in)
    and k-1 (out) run on their own streams while step k computes, on two sets
    of device buffers; events keep a buffer from being overwritten while it is
    still read or written.  Returns the milliseconds of `steps` steps, from
    the first copy in to the last copy out."""
    import torch
    dev = step_a.dev
    steps_ = (step_a, step_b)
    ins = lambda st: (st.q, st.k, st.v, st.do)
    outs = lambda st: (st.o, st.lse, st.dq, st.dk, st.dv)
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


def summarise(step, phase_ms, peaks):
    """Per-pass figures of one workload from per-step phase times (ms lists):
    TFLOPS and fraction of the burst peak for the contractions, GB/s and
    fraction of the copy bandwidth for the HBM-bound kernels, and the two
    passes as the C ABI calls them: the bf16 forward (fa_fwd) and the whole
    backward call (fa_bwd = preprocess + main + dQ conversion)."""
    bf16_peak = peaks["bf16_tflops"]
    passes = {}
    for ph, ms_list in phase_ms.items():
        if not ms_list:
            continue
        ms = statistics.mean(ms_list)
        ent = {"ms": round(ms, 4)}
        if step.flops[ph]:
            tf = step.flops[ph] / (ms / 1e3) / 1e12
            pk = bf16_peak * (FP8_OVER_BF16 if ph == "fwd_fp8" else 1.0)
            ent.update({"tflops": round(tf, 1), "frac_of_peak": round(tf / pk, 4), "peak_tflops": pk})
        ent["gbs"] = round(step.bytes[ph] / (ms / 1e3) / 1e9, 1)
        if not step.flops[ph]:
            ent["frac_of_hbm"] = round(ent["gbs"] / peaks["hbm_gbs"], 4)
        passes[ph] = ent
    fwd_ms = passes["fwd"]["ms"]
    bwd_ms = sum(statistics.mean(phase_ms[ph]) for ph in ("bwd_pre", "bwd_main", "bwd_dq"))
    # key-padded workloads: the rates and fractions count the visible (query,
    # key) pairs only (the work the method has to do); the nominal B*N*N rate
    # is kept beside them
    Ff, Fb = step.flops["fwd"], step.flops["bwd_main"]
    if step.flops_eff is not None:
        Ff, Fb = step.flops_eff["fwd"], step.flops_eff["bwd"]
    out = {"fwd_tflops": round(Ff / (fwd_ms / 1e3) / 1e12, 1),
           "fwd_frac_burst": round(Ff / (fwd_ms / 1e3) / 1e12 / bf16_peak, 4),
           "bwd_call_ms": round(bwd_ms, 4),
           "bwd_call_tflops": round(Fb / (bwd_ms / 1e3) / 1e12, 1),
           "bwd_call_frac_burst": round(Fb / (bwd_ms / 1e3) / 1e12 / bf16_peak, 4)}
    if step.flops_eff is not None:
        out["flops"] = "visible pairs only (sum of kv_len in place of B*N)"
        out["fwd_tflops_nominal"] = round(step.flops["fwd"] / (fwd_ms / 1e3) / 1e12, 1)
        out["bwd_call_tflops_nominal"] = round(step.flops["bwd_main"] / (bwd_ms / 1e3) / 1e12, 1)
    if "fwd_fp8" in passes:
        out["fp8_fwd_tflops"] = passes["fwd_fp8"]["tflops"]
        out["fp8_fwd_frac_burst"] = passes["fwd_fp8"]["frac_of_peak"]
        out["quant_fp8_gbs"] = passes["quant_fp8"]["gbs"]
    return passes, out


def time_steps(step, steps, warmup):
    """Runs `warmup` then `steps` steps (L2 flushed between steps, outside the
    events) and returns {phase: [ms per step]}."""
    import torch
    phases = step.phases()
    ev = [step.events() for _ in range(steps)]
    for _ in range(max(warmup, 3)):
        step.run()
        step.flush_l2()
    torch.cuda.synchronize()
    for i in range(steps):
        step.run(ev[i])
        step.flush_l2()
    torch.cuda.synchronize()
    out = {ph: [] for ph in phases}
    for e in ev:
        for j, ph in enumerate(phases):
            out[ph].append(e[2 * j].elapsed_time(e[2 * j + 1]))
    return out


def time_fp8_backward(step, peaks, reps):
    """The FP8 backward (chapter 18 §18.6.2) of the step's FP8 forward (same
    codes, scales, O and LSE; non-causal), timed on its own: every kernel of
    the call (dO quantiser, preprocess, K transpose, main kernel, dQ
    conversion) between two events, L2 flushed between calls."""
    import torch
    fa, w = step.fa, step.w
    B, H, N, d = w.B, w.H, w.N, w.d
    f32 = lambda: torch.empty((B, H, N, d), dtype=torch.float32, device=step.dev)
    dq, dk, dv = f32(), f32(), f32()
    prm = fa.attn_params(dtype=fa.FA_E4M3, batch=B, heads=H, seqlen_q=N, head_dim=d, scale=step.scale,
                         q=step.x8[0], k=step.x8[1], v=step.x8[2], q_scale=step.sc[0], k_scale=step.sc[1],
                         v_scale=step.sc[2], o=step.o8, lse=step.lse8, dout=step.do, dq=dq, dk=dk, dv=dv)
    nbytes = int(step.lib.fa_attn_bwd_workspace_size(ctypes.byref(prm)))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=step.dev)
    prm.workspace, prm.workspace_bytes = ws.data_ptr(), nbytes
    s = torch.cuda.current_stream(step.dev).cuda_stream
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for i in range(reps + 3):
        if i >= 3:
            ev[i - 3][0].record()
        step._ck(step.lib.fa_attn_bwd(ctypes.byref(prm), s))
        if i >= 3:
            ev[i - 3][1].record()
        step.flush_l2()
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    F = 2.5 * flops_fwd(w, False)
    tf = F / (ms / 1e3) / 1e12
    pk = peaks["bf16_tflops"] * FP8_OVER_BF16
    return {"ms": round(ms, 4), "tflops": round(tf, 1), "frac_of_fp8_peak": round(tf / pk, 4), "reps": reps,
            "workload": "non-causal backward of the FP8 forward, float32 gradients, whole fa_attn_bwd call"}


def other_configs(device, peaks, reps):
    """The other workload shapes, each timed on its own (bf16 forward and
    whole backward call; FP8 where the workload has one)."""
    from exact_tiled_attention_10_gb300.inputs import WORKLOADS
    res = {}
    for name, causal, fp8 in (("mid", True, False), ("mid", False, False), ("ragged", False, False),
                              ("long_seq", True, False), ("long_seq", False, True)):
        w = WORKLOADS[name]
        st = Step(w, causal, device, fp8=fp8)
        ph = time_steps(st, reps, 3)
        passes, summ = summarise(st, ph, peaks)
        key = "%s_%s" % (name, "causal" if causal else "noncausal")
        summ.update({"B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": causal, "reps": reps})
        if w.ragged:
            summ["kv_lens_sum"] = int(st.kv.sum().item())
        if fp8:  # the FP8 figures are the point of this line (the pages' FP8 workload is non-causal)
            summ["passes"] = {k: passes[k] for k in ("quant_fp8", "fwd_fp8")}
        res[key] = summ
        del st
    return res


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
    ev = [step.events() for _ in range(args.steps)]
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

    phases = step.phases()
    phase_ms = {ph: [] for ph in phases}
    step_ms, bf16_ms = [], []
    for e in ev:
        t = [e[2 * j].elapsed_time(e[2 * j + 1]) for j in range(len(phases))]
        step_ms.append(sum(t))
        bf16_ms.append(sum(x for ph, x in zip(phases, t) if ph in Step.BF16))
        for ph, x in zip(phases, t):
            phase_ms[ph].append(x)
    total_ms = max_over_ranks(ws, sum(step_ms), device)
    bf16_total_ms = max_over_ranks(ws, sum(bf16_ms), device)
    flops_bf16 = step.flops["fwd"] + step.flops["bwd_main"]
    value = ws * flops_bf16 * args.steps / (bf16_total_ms / 1e3) / 1e12

    peaks, peak_src = load_peaks()
    passes, summ = summarise(step, phase_ms, peaks)
    dom = max(("fwd", "bwd_main", "fwd_fp8"), key=lambda ph: statistics.mean(phase_ms[ph]))
    roofline = {"bound": "tensor", "kernel": dom, "achieved": passes[dom]["tflops"],
                "peak": passes[dom]["peak_tflops"], "unit": "TFLOP/s", "frac": passes[dom]["frac_of_peak"],
                "traffic": recorded_traffic(dom),
                "peak_source": "%s (%s)" % (peak_src, "dense bf16 burst" +
                                            (" x2 for e4m3" if dom == "fwd_fp8" else "")),
                "peak_sustained": peaks["bf16_tflops_sustained"] * (FP8_OVER_BF16 if dom == "fwd_fp8" else 1.0)}
    fp8 = {"tflops": summ["fp8_fwd_tflops"], "frac_of_fp8_peak": summ["fp8_fwd_frac_burst"],
           "fp8_peak_tflops": peaks["bf16_tflops"] * FP8_OVER_BF16,
           "ms": passes["fwd_fp8"]["ms"], "quant_ms": passes["quant_fp8"]["ms"],
           "quant_gbs": passes["quant_fp8"]["gbs"], "quant_frac_of_hbm": passes["quant_fp8"]["frac_of_hbm"],
           "workload": "non-causal forward on E4M3 codes with per-64-row block scales (quantiser timed apart)"}

    fp8["bwd"] = time_fp8_backward(step, peaks, args.config_reps)

    # ---- end to end through the public API with pinned host buffers
    e2e_steps = args.e2e_steps or min(args.steps, 100)
    e2e_ms = e2e_pipelined(Step(w, causal, device, seed_offset=1000 * rank, fp8=False),
                           Step(w, causal, device, seed_offset=1000 * rank + 1, fp8=False), e2e_steps)
    hin_bytes = sum(t.numel() * t.element_size() for t in (step.q, step.k, step.v, step.do))
    hout_bytes = sum(t.numel() * t.element_size() for t in (step.o, step.lse, step.dq, step.dk, step.dv))
    h2d, d2h = hin_bytes, hout_bytes
    e2e_ms = max_over_ranks(ws, e2e_ms, device)
    e2e_value = ws * flops_bf16 * e2e_steps / (e2e_ms / 1e3) / 1e12

    configs = None
    if not args.no_configs:
        configs = other_configs(device, peaks, args.config_reps)

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
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "%s: B=%d H=%d N=%d d=%d; bf16 causal fwd + bwd, then E4M3 quantise Q/K/V "
                                   "+ FP8 non-causal fwd" % (w.name, w.B, w.H, w.N, w.d),
                       "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": causal,
                       "value_basis": "bf16 (F_fwd + F_bwd) / time of the bf16 forward and the whole backward "
                                      "call (%.4f ms per step); ms_per_step also holds the FP8 rows" % (
                                          bf16_total_ms / args.steps),
                       "l2": "flushed before each step and between its bf16 and FP8 parts, outside the timed "
                             "events (512 MiB written, then 256 MiB read: L2 left cold and clean)",
                       "parallelism": "replicas" if ws > 1 else "single GPU"},
            "targets": {"fwd_frac_burst": summ["fwd_frac_burst"], "fwd_target": 0.60,
                        "bwd_call_frac_burst": summ["bwd_call_frac_burst"], "bwd_target": 0.45,
                        "peak_tflops": peaks["bf16_tflops"], "peak": "%s dense bf16 burst" % peak_src},
            "passes": passes,
            "bf16": summ,
            "fp8": fp8,
            "roofline": roofline,
            "configs": configs,
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 2), "unit": "TFLOPS", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "how": "C ABI with pinned host buffers; every step copies Q, K, V, dO in and O, LSE, "
                           "dQ, dK, dV out around the bf16 forward + backward; copies of neighbouring steps "
                           "overlap compute (two device buffer sets, three streams); inputs of %.0f MB per "
                           "step, L2 129 MB" % (h2d / 1e6)},
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
