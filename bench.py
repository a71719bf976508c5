"""Benchmark of the fused GEMM + row-reduce/broadcast path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--quick]

One step = one call of the fused kernel over one batch of the workload
(default: GEMM + bias + GELU(tanh) + LayerNorm, X[16384,4096] . W[4096,4096],
the largest single-GPU workload of the metric's list, tensor-bound).  Inputs are resident in HBM when the timed
region starts; between steps the input/output buffer set rotates so the
footprint of consecutive steps exceeds L2 three times over.  The K timed
steps are replayed from CUDA graphs and timed with CUDA events on the
launching stream, bracketed by a barrier and synchronize on both sides; the
max over ranks is reported.  Under torchrun every rank runs its own batch on
its own GPU (weak scaling; no collective on the data path).

The JSON line also carries: roofline (dominant kernel vs the measured HBM
or tensor peak), e2e (the same metric through the public C-ABI call with
host buffers, H2D/D2H copies inside the timed region), the CPU oracle timed
on a bounded sample (cpu_baseline), SM clocks sampled during the timed
region, and each page workload's fused-kernel numbers: in full
(per_workload_detail) and, last on the line, compact (per_workload: per
launch microseconds and roofline fraction).

``--impl reference`` times the fp64 CPU oracle instead (the reference arm).
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from memory_fusion_gb300 import dist as mdist  # noqa: E402
from memory_fusion_gb300 import inputs  # noqa: E402

HEADLINE = "gelu_ln_16384x4096x4096"
METRIC = "fused GEMM+row-reduce TFLOP/s and HBM GB/s at 1 GB300; % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    return mdist.env()


def kind_of(w):
    """Kernel kind of a GEMM workload for the plan query (RMSNorm runs in the
    LayerNorm kernels, the causal softmax plans like the plain one)."""
    if w.kind in ("softmax", "softmax_causal"):
        return 2
    return 1 if w.act == "gelu_tanh" else 0


def fused_call(cf, w, X, W, bias, gamma, beta, Y, ws, wsb, stream=None, R=None, tuning=None):
    """The public fused call of workload w (tuning: optional cf_tuning)."""
    if w.kind == "softmax":
        return cf.cf_gemm_fused_rowsoftmax(X, W, None, Y, w.M, w.N, w.K, w.scale, ws, wsb, stream, tuning)
    if w.kind == "softmax_causal":
        return cf.cf_gemm_fused_rowsoftmax_causal(X, W, None, Y, w.M, w.N, w.K, w.scale, w.mask_offset, ws, wsb,
                                                  stream, tuning)
    act = cf.CF_ACT_GELU_TANH if w.act == "gelu_tanh" else cf.CF_ACT_NONE
    if w.resid_std is not None:
        norm = cf.CF_NORM_RMS if w.kind == "rmsnorm" else cf.CF_NORM_LAYER
        return cf.cf_gemm_fused_residual_norm(X, W, bias, R, gamma, beta, Y, w.M, w.N, w.K, w.alpha, w.eps, act,
                                              norm, ws, wsb, stream, tuning)
    fn = cf.cf_gemm_fused_rmsnorm if w.kind == "rmsnorm" else cf.cf_gemm_fused_rownorm
    return fn(X, W, bias, gamma, beta, Y, w.M, w.N, w.K, w.alpha, w.eps, act, ws, wsb, stream, tuning)


def unfused_call(cf, w, X, W, bias, gamma, beta, Y, ws, wsb, stream=None, R=None):
    if w.kind == "softmax":
        return cf.cf_unfused_gemm_rowsoftmax(X, W, None, Y, w.M, w.N, w.K, w.scale, ws, wsb, stream)
    act = cf.CF_ACT_GELU_TANH if w.act == "gelu_tanh" else cf.CF_ACT_NONE
    if w.resid_std is not None:
        norm = cf.CF_NORM_RMS if w.kind == "rmsnorm" else cf.CF_NORM_LAYER
        return cf.cf_unfused_gemm_residual_norm(X, W, bias, R, gamma, beta, Y, w.M, w.N, w.K, w.alpha, w.eps, act,
                                                norm, ws, wsb, stream)
    fn = cf.cf_unfused_gemm_rmsnorm if w.kind == "rmsnorm" else cf.cf_unfused_gemm_rownorm
    return fn(X, W, bias, gamma, beta, Y, w.M, w.N, w.K, w.alpha, w.eps, act, ws, wsb, stream)


def oracle_rows(oracle, w, d, rows):
    if w.kind == "b2b":
        return oracle.b2b_gemm(d["X"], d["W1"], d["W2"], op=w.op, alpha=w.alpha, b1=d["b1"], rows=rows,
                               gamma1=d.get("gamma1"), beta1=d.get("beta1"), eps=1e-5)
    if w.kind == "softmax":
        return oracle.gemm_rowsoftmax(d["X"], d["W"], scale=w.scale, rows=rows)
    if w.kind == "softmax_causal":
        return oracle.gemm_rowsoftmax_causal(d["X"], d["W"], scale=w.scale, offset=w.mask_offset, rows=rows)
    if w.resid_std is not None:
        return oracle.gemm_bias_residual_norm(d["X"], d["W"], d["bias"], d["R"], d["gamma"], d["beta"],
                                              alpha=w.alpha, eps=w.eps, act=w.act,
                                              norm="rms" if w.kind == "rmsnorm" else "layer", rows=rows)
    fn = oracle.gemm_bias_rmsnorm if w.kind == "rmsnorm" else oracle.gemm_bias_rownorm
    return fn(d["X"], d["W"], d["bias"], d["gamma"], d["beta"], alpha=w.alpha, eps=w.eps, act=w.act, rows=rows)


def row_vectors(w):
    """The fp32 [N] inputs of a workload's epilogue that are present."""
    if w.kind in ("softmax", "softmax_causal"):
        return ()
    return tuple(k for k, sd in (("bias", w.bias_std), ("gamma", w.gamma_std), ("beta", w.beta_std))
                 if sd is not None)


def roofline_time_s(w, peaks):
    t_flop = w.flops / (peaks["bf16_tflops"] * 1e12)
    t_byte = w.unavoidable_bytes / (peaks["hbm_gbs"] * 1e9)
    return max(t_flop, t_byte), ("tensor" if t_flop >= t_byte else "hbm")


KERNEL_TU = {"gemm_fused_kernel": "gemm_fused.cu", "stitch_": "stitch.cu", "b2b_kernel": "b2b.cu",
             "b2b_stream_kernel": "b2b_stream.cu", "addln_": "stitch_norm.cu", "bn_": "stitch_norm.cu"}


def _code_only(text):
    """Source text without comments and with whitespace runs collapsed (a
    comment edit does not change the code)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel):
    """Hash of the device code behind `kernel`: the translation unit that holds
    it, every shared device header (.cuh) and the internal header of shared
    constants and launch-argument structs (cf_internal.h), comments and layout
    ignored.  A kernel's DRAM traffic can only change when one of them does."""
    csrc = os.path.join(ROOT, "memory_fusion_gb300", "csrc")
    tu = next((f for k, f in KERNEL_TU.items() if kernel.startswith(k)), None)
    files = sorted(f for f in os.listdir(csrc) if f.endswith(".cuh") or f == tu or f == "cf_internal.h")
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def _traffic_entry(workload, kernel):
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(workload, {}).get(kernel)
        if e and e.get("source_hash") == kernel_source_hash(kernel):
            return e
    except Exception:
        pass
    return None


def profiled_traffic(workload, kernel):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    e = _traffic_entry(workload, kernel)
    return float(e["dram_bytes_per_launch"]) if e else None


def profiled_traffic_kind(workload, kernel):
    """How that figure was taken: one cold launch, or steady state (no cache
    flush between launches, so a launch also writes back the previous one's
    output that the L2 still held)."""
    e = _traffic_entry(workload, kernel)
    return e.get("kind") if e else None


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self, window=None):
        """Median SM clock and the throttle reasons seen; with `window` = (t0, t1)
        (time.time() around the timed region) only the samples inside it count,
        unless none fell inside (a region shorter than the 50 ms sampling
        period), which the result says."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        samples = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                samples.append((ts, float(parts[1]), float(parts[2]),
                                {nm for nm, v in zip(names, parts[5:9]) if v.lower() == "active"}))
            except ValueError:
                continue
        inside = [x for x in samples if window and window[0] - 0.02 <= x[0] <= window[1] + 0.02]
        use = inside if inside else samples
        reasons = set().union(*[x[3] for x in use]) if use else set()
        res = {"sm_mhz": statistics.median([x[1] for x in use]) if use else None,
               "sm_max_mhz": max(x[2] for x in use) if use else None,
               "reasons": sorted(reasons), "samples": len(use)}
        if window and not inside:
            res["note"] = "no sample inside the timed region (shorter than the sampling period); all samples"
        return res


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
class FusedRunner:
    """Device buffers of one workload, rotating over `nsets` sets, and one
    launcher per set that calls the C ABI on the current stream."""

    def __init__(self, torch, cf, w, nsets, seed_offset=0, device="cuda"):
        self.torch, self.cf, self.w = torch, cf, w
        d = (inputs.workload_inputs(w.name) if seed_offset == 0 else
             _seeded_inputs(w, seed_offset))
        self.host = d
        bf = torch.bfloat16
        X = torch.from_numpy(d["X"]).to(device, bf)
        W = torch.from_numpy(d["W"]).to(device, bf)
        self.sets = []
        for i in range(nsets):
            s = {"X": X if i == 0 else X.clone(), "W": W if i == 0 else W.clone(),
                 "Y": torch.empty((w.M, w.N), dtype=bf, device=device)}
            for k in ("bias", "gamma", "beta"):
                s[k] = torch.from_numpy(d[k]).to(device) if k in row_vectors(w) else None
            s["R"] = torch.from_numpy(d["R"]).to(device, bf) if d.get("R") is not None else None
            self.sets.append(s)
        self.ws_bytes = cf.cf_gemm_fused_workspace_size(w.M, w.N, w.K)
        self.ws = cf.new_workspace(self.ws_bytes, device)

    def launch(self, i, stream=None):
        cf, w = self.cf, self.w
        s = self.sets[i % len(self.sets)]
        st = fused_call(cf, w, s["X"], s["W"], s["bias"], s["gamma"], s["beta"], s["Y"], self.ws, self.ws_bytes,
                        stream, R=s["R"])
        cf.check(st, "fused launch")


def _seeded_inputs(w, rank):
    seed = mdist.seed_for(w.seed, rank)
    if w.kind in ("rownorm", "rmsnorm"):
        return inputs.gemm_inputs(w.M, w.N, w.K, seed, x_std=w.x_std, w_std=w.w_std,
                                  bias_std=w.bias_std, gamma_std=w.gamma_std, beta_std=w.beta_std,
                                  resid_std=w.resid_std)
    return inputs.gemm_inputs(w.M, w.N, w.K, seed, x_std=w.x_std, w_std=w.w_std,
                              bias_std=None, gamma_std=None, beta_std=None)


def bytes_per_set(w):
    return 2 * w.M * w.K + 2 * w.K * w.N + 2 * w.M * w.N


def capture_graph(torch, runner, start, count):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(count):
                runner.launch(start + i)
    torch.cuda.current_stream().wait_stream(s)
    return g


def time_steps(torch, runner, steps, warmup, barrier, sampler=None, graph_len=500):
    """Warm up, then time exactly `steps` launches replayed from CUDA graphs.
    Returns (seconds, launches)."""
    for i in range(warmup):
        runner.launch(i)
    torch.cuda.synchronize()
    R = max(1, min(steps, graph_len))
    reps, rem = divmod(steps, R)
    g = capture_graph(torch, runner, 0, R)
    g_rem = capture_graph(torch, runner, R, rem) if rem else None
    g.replay()  # upload + one untimed pass
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.3)
    w0 = time.time()
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    if g_rem is not None:
        g_rem.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    barrier()
    clocks = sampler.stop((w0, w1)) if sampler else None
    return e0.elapsed_time(e1) / 1e3, reps * R + rem, clocks


def time_e2e(torch, cf, w, steps, device, depth=3):
    """The public call with host buffers: every step copies its inputs X and W
    (and the row vectors, R) from pinned host memory, makes the fused call and
    copies Y back into pinned host memory.  Steps are pipelined over `depth`
    buffer sets on three streams (copy-in, compute, copy-out), so the copies
    of one step overlap the compute of its neighbours; events order each
    set's reuse.  Returns (seconds per step, H2D bytes, D2H bytes)."""
    d = inputs.workload_inputs(w.name)
    bf = torch.bfloat16
    names = ["X", "W"] + list(row_vectors(w)) + (["R"] if d.get("R") is not None else [])
    host = {}
    for k in names:
        t = torch.from_numpy(d[k])
        host[k] = (t.to(bf) if k in ("X", "W", "R") else t).pin_memory()
    sets = []
    for _ in range(depth):
        dev = {k: torch.empty_like(host[k], device=device) for k in names}
        dev["Y"] = torch.empty((w.M, w.N), dtype=bf, device=device)
        dev["hY"] = torch.empty((w.M, w.N), dtype=bf).pin_memory()
        sets.append(dev)
    wsb = cf.cf_gemm_fused_workspace_size(w.M, w.N, w.K)
    ws = cf.new_workspace(wsb, device)
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(depth)]
    ev_cmp = [torch.cuda.Event() for _ in range(depth)]
    ev_out = [torch.cuda.Event() for _ in range(depth)]
    used = [False] * depth

    def step(i):
        b = i % depth
        dv = sets[b]
        if used[b]:
            s_in.wait_event(ev_cmp[b])    # the previous use of this set's inputs is consumed
        with torch.cuda.stream(s_in):
            for k in names:
                dv[k].copy_(host[k], non_blocking=True)
            ev_in[b].record(s_in)
        s_cmp.wait_event(ev_in[b])
        if used[b]:
            s_cmp.wait_event(ev_out[b])   # the previous use of this set's Y has been read out
        cf.check(fused_call(cf, w, dv["X"], dv["W"], dv.get("bias"), dv.get("gamma"), dv.get("beta"), dv["Y"], ws,
                            wsb, s_cmp.cuda_stream, R=dv.get("R")))
        ev_cmp[b].record(s_cmp)
        s_out.wait_event(ev_cmp[b])
        with torch.cuda.stream(s_out):
            dv["hY"].copy_(dv["Y"], non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    for i in range(2 * depth):
        step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    s_cmp.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(steps):
        step(i)
    s_in.wait_stream(s_out)
    s_in.wait_stream(s_cmp)
    e1.record(s_in)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3 / steps
    h2d = sum(host[k].numel() * host[k].element_size() for k in names)
    d2h = w.M * w.N * 2
    return t, h2d, d2h


class B2bRunner:
    """Device buffers of a back-to-back GEMM workload over `nsets` rotating
    sets, launched through the public C ABI."""

    def __init__(self, torch, cf, w, nsets, seed_offset=0, device="cuda"):
        self.torch, self.cf, self.w = torch, cf, w
        d = inputs.workload_inputs(w.name) if seed_offset == 0 else inputs.b2b_inputs(
            w.M, w.K, w.N1, w.N2, mdist.seed_for(w.seed, seed_offset), x_std=w.x_std, w1_std=w.w1_std,
            w2_std=w.w2_std, b1_std=w.b1_std, ln=w.op == "layernorm")
        self.host = d
        bf = torch.bfloat16
        X = torch.from_numpy(d["X"]).to(device, bf)
        W1 = torch.from_numpy(d["W1"]).to(device, bf)
        W2 = torch.from_numpy(d["W2"]).to(device, bf)
        b1 = torch.from_numpy(d["b1"]).to(device) if d["b1"] is not None else None
        self.g1 = torch.from_numpy(d["gamma1"]).to(device) if d.get("gamma1") is not None else None
        self.be1 = torch.from_numpy(d["beta1"]).to(device) if d.get("beta1") is not None else None
        self.sets = [{"X": X if i == 0 else X.clone(), "W1": W1 if i == 0 else W1.clone(),
                      "W2": W2 if i == 0 else W2.clone(), "b1": b1,
                      "O": torch.empty((w.M, w.N2), dtype=bf, device=device)} for i in range(nsets)]
        self.op = {"softmax": cf.CF_B2B_SOFTMAX, "gelu_tanh": cf.CF_B2B_GELU_TANH,
                   "layernorm": cf.CF_B2B_LAYERNORM}[w.op]
        self.ws_bytes = cf.cf_b2b_workspace_size()
        self.ws = cf.new_workspace(self.ws_bytes, device)

    def launch(self, i, stream=None):
        w, s = self.w, self.sets[i % len(self.sets)]
        if w.op == "layernorm":
            st = self.cf.cf_b2b_gemm_layernorm(s["X"], s["W1"], s["b1"], self.g1, self.be1, s["W2"], s["O"], w.M,
                                               w.K, w.N1, w.N2, w.alpha, 1e-5, self.ws, self.ws_bytes, stream)
        else:
            st = self.cf.cf_b2b_gemm(s["X"], s["W1"], s["b1"], s["W2"], s["O"], w.M, w.K, w.N1, w.N2, w.alpha,
                                     self.op, self.ws, self.ws_bytes, stream)
        self.cf.check(st, "b2b launch")


def b2b_bytes_per_set(w):
    return w.unavoidable_bytes


def b2b_kernel_name(w, plan):
    """The kernel the plan launches: the stream kernel (n_slice 128: one CTA per
    row block) or the cluster kernel (n_slice 256)."""
    op = {"softmax": "SOFTMAX", "gelu_tanh": "GELU", "layernorm": "LN"}[w.op]
    return f"b2b_stream_kernel<{op}>" if plan.n_slice == 128 else f"b2b_kernel<{op}>"


def torch_b2b_time(torch, runner, reps):
    """The same chain as a user writes it without fusion: cuBLAS GEMM to a bf16
    P, F in torch (fp32 math, bf16 S stored), cuBLAS GEMM of S with W2.  Library
    kernels, not this package's: the context for what keeping S on chip saves."""
    w = runner.w

    class U:
        def launch(self, i, stream=None):
            s = runner.sets[i % len(runner.sets)]
            P = torch.matmul(s["X"], s["W1"]).float() * w.alpha
            if s["b1"] is not None:
                P = P + s["b1"]
            if w.op == "softmax":
                S = torch.softmax(P, dim=1)
            elif w.op == "gelu_tanh":
                S = torch.nn.functional.gelu(P, approximate="tanh")
            else:
                S = torch.nn.functional.layer_norm(P, (w.N1,), runner.g1, runner.be1, 1e-5)
            torch.matmul(S.to(torch.bfloat16), s["W2"], out=s["O"])

    t, n, _ = time_steps(torch, U(), reps, 3, lambda: None, graph_len=reps)
    return t / n


def b2b_numbers(torch, cf, w, peaks, device, l2):
    nsets = max(1, min(32, math.ceil(3 * l2 / b2b_bytes_per_set(w))))
    r = B2bRunner(torch, cf, w, nsets, device=device)
    reps = max(nsets, 200)
    t, n, _ = time_steps(torch, r, reps, 3, lambda: None, graph_len=reps)
    t1 = t / n
    troof, bound = roofline_time_s(w, peaks)
    _, plan = cf.cf_query_b2b_plan(w.M, w.K, w.N1, w.N2, r.op)
    tu = torch_b2b_time(torch, r, reps)
    out = {"us": round(t1 * 1e6, 2), "tflops": round(w.flops / t1 / 1e12, 1),
           "gbs": round(w.unavoidable_bytes / t1 / 1e9, 1), "bound": bound, "roofline_frac": round(troof / t1, 3),
           "buffer_sets": nsets, "unfused_torch_us": round(tu * 1e6, 2), "fused_speedup_vs_torch": round(tu / t1, 2),
           "plan": plan.as_dict()}
    del r
    torch.cuda.empty_cache()
    return out


def per_workload(torch, cf, peaks, device, names):
    """Each page workload's fused kernel, timed alone (graph of launches,
    rotating buffers where one set is smaller than 3x L2)."""
    out = {}
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    for name in names:
        w = inputs.WORKLOADS[name]
        if isinstance(w, inputs.StitchWorkload):
            out[name] = stitch_numbers(torch, cf, w, peaks, device, l2)
            continue
        if isinstance(w, inputs.B2bWorkload):
            out[name] = b2b_numbers(torch, cf, w, peaks, device, l2)
            continue
        if isinstance(w, inputs.StitchNormWorkload):
            out[name] = stitch_norm_numbers(torch, cf, w, peaks, device, l2)
            continue
        if isinstance(w, inputs.StitchPowWorkload):
            out[name] = stitch_pow_numbers(torch, cf, w, peaks, device, l2)
            continue
        nsets = max(1, min(32, math.ceil(3 * l2 / bytes_per_set(w))))
        r = FusedRunner(torch, cf, w, nsets, device=device)
        reps = max(nsets, 20 if w.flops > 1e11 else 400)
        t, n, _ = time_steps(torch, r, reps, 3, lambda: None, graph_len=reps)
        t1 = t / n
        troof, bound = roofline_time_s(w, peaks)
        _, plan, _ = cf.cf_query_gemm_fused_plan(w.M, w.N, w.K, kind_of(w))
        # the unfused composition exists for the unmasked epilogues only
        tu = unfused_time(torch, cf, r, reps) if w.kind != "softmax_causal" else None
        out[name] = {"us": round(t1 * 1e6, 2), "tflops": round(w.flops / t1 / 1e12, 1),
                     "gbs": round(w.unavoidable_bytes / t1 / 1e9, 1), "bound": bound,
                     "roofline_frac": round(troof / t1, 3), "buffer_sets": nsets,
                     "unfused_us": round(tu * 1e6, 2) if tu else None,
                     "fused_speedup": round(tu / t1, 2) if tu else None,
                     "plan": plan.as_dict()}
        del r
        torch.cuda.empty_cache()
    return out


# the compact per-workload summary lists the page workloads first (the
# other single-GPU configs of the metric, then the stitched shapes), then the
# next-in-line epilogues
SUMMARY_ORDER = ["wide_ln_8192x16384x2048", "softmax_4096x2048x128", "stitch_750000x32", "stitch_64x30000",
                 "ln_tiny_128x512x256", "gelu_ln_16384x4096x4096"]


def compact_summary(detail):
    """{workload: [microseconds per launch, roofline fraction]} in SUMMARY_ORDER,
    then the rest in table order."""
    names = [n for n in SUMMARY_ORDER if n in detail] + [n for n in detail if n not in SUMMARY_ORDER]
    return {n: [detail[n]["us"], detail[n]["roofline_frac"]] for n in names}


def unfused_time(torch, cf, runner, reps):
    """The same workload through the unfused two-kernel composition (GEMM to an
    fp32 intermediate, then the row kernel), same buffer rotation."""
    w = runner.w
    wsb = cf.cf_unfused_workspace_size(w.M, w.N, w.K)
    ws = torch.empty(wsb, dtype=torch.uint8, device=runner.sets[0]["X"].device)

    class U:
        def launch(self, i, stream=None):
            s = runner.sets[i % len(runner.sets)]
            st = unfused_call(cf, w, s["X"], s["W"], s["bias"], s["gamma"], s["beta"], s["Y"], ws, wsb, stream,
                              R=s["R"])
            cf.check(st, "unfused launch")

    t, n, _ = time_steps(torch, U(), reps, 3, lambda: None, graph_len=reps)
    del ws
    return t / n


def stitch_pow_numbers(torch, cf, w, peaks, device, l2):
    """The stitched power -> broadcast -> add -> softmax subgraph, timed alone."""
    d = inputs.workload_inputs(w.name)
    nsets = max(1, min(32, math.ceil(3 * l2 / w.unavoidable_bytes)))
    A = [torch.from_numpy(d["A"]).to(device) for _ in range(nsets)]
    wv = torch.from_numpy(d["w"]).to(device)
    O = [torch.empty_like(A[0]) for _ in range(nsets)]
    wsb = cf.cf_stitch_workspace_size(w.rows, w.cols)
    ws = cf.new_workspace(wsb, device)

    class R:
        def launch(self, i, stream=None):
            cf.check(cf.cf_stitch_powadd_softmax(A[i % nsets], wv, w.p, O[i % nsets], w.rows, w.cols, ws, wsb,
                                                 stream))

    reps = max(nsets, 200)
    t, n, _ = time_steps(torch, R(), reps, 3, lambda: None, graph_len=reps)
    t1 = t / n
    gbs = w.unavoidable_bytes / t1 / 1e9
    return {"us": round(t1 * 1e6, 2), "gbs": round(gbs, 1), "bound": "hbm",
            "roofline_frac": round(gbs / peaks["hbm_gbs"], 3), "buffer_sets": nsets}


def stitch_numbers(torch, cf, w, peaks, device, l2):
    d = inputs.workload_inputs(w.name)
    nsets = max(1, min(32, math.ceil(3 * l2 / w.unavoidable_bytes)))
    A = [torch.from_numpy(d["A"]).to(device) for _ in range(nsets)]
    b = torch.from_numpy(d["row_bias"]).to(device)
    O = [torch.empty_like(A[0]) for _ in range(nsets)]
    wsb = cf.cf_stitch_workspace_size(w.rows, w.cols)
    ws = cf.new_workspace(wsb, device)

    class R:
        def launch(self, i, stream=None):
            cf.check(cf.cf_stitch_rowreduce_broadcast(A[i % nsets], b, O[i % nsets], w.rows, w.cols,
                                                      ws, wsb, stream))

    reps = max(nsets, 200)
    t, n, _ = time_steps(torch, R(), reps, 3, lambda: None, graph_len=reps)
    t1 = t / n
    gbs = w.unavoidable_bytes / t1 / 1e9
    return {"us": round(t1 * 1e6, 2), "gbs": round(gbs, 1), "bound": "hbm",
            "roofline_frac": round(gbs / peaks["hbm_gbs"], 3), "buffer_sets": nsets}


class StitchNormRunner:
    """Device buffers of a stitched normalisation workload over `nsets`
    rotating sets, launched through the public C ABI."""

    def __init__(self, torch, cf, w, nsets, seed_offset=0, device="cuda"):
        self.torch, self.cf, self.w = torch, cf, w
        seed = w.seed if seed_offset == 0 else mdist.seed_for(w.seed, seed_offset)
        d = inputs.stitch_norm_inputs(w.rows, w.cols, seed, with_R=w.kind == "add_layernorm")
        self.host = d
        A = torch.from_numpy(d["A"]).to(device)
        R = torch.from_numpy(d["R"]).to(device) if d["R"] is not None else None
        self.g = torch.from_numpy(d["gamma"]).to(device)
        self.b = torch.from_numpy(d["beta"]).to(device)
        self.sets = [{"A": A if i == 0 else A.clone(), "R": (R if i == 0 else R.clone()) if R is not None else None,
                      "out": torch.empty_like(A)} for i in range(nsets)]
        self.mean = torch.empty(w.cols, device=device)
        self.var = torch.empty(w.cols, device=device)
        if w.kind == "add_layernorm":
            self.ws_bytes = cf.cf_stitch_workspace_size(w.rows, w.cols)
        else:
            self.ws_bytes = cf.cf_stitch_batchnorm_workspace_size(w.rows, w.cols)
        self.ws = cf.new_workspace(self.ws_bytes, device)

    def launch(self, i, stream=None):
        w, s, cf = self.w, self.sets[i % len(self.sets)], self.cf
        if w.kind == "add_layernorm":
            st = cf.cf_stitch_add_layernorm(s["A"], s["R"], self.g, self.b, s["out"], w.rows, w.cols, w.eps, self.ws,
                                            self.ws_bytes, stream)
        else:
            st = cf.cf_stitch_batchnorm(s["A"], self.g, self.b, s["out"], self.mean, self.var, w.rows, w.cols, w.eps,
                                        self.ws, self.ws_bytes, stream)
        cf.check(st, "stitched normalisation launch")


def stitch_norm_kernel_name(cf, w):
    if w.kind == "add_layernorm":
        return "addln_packed_kernel" if (w.cols + 3) // 4 <= 32 else "addln_split_kernel"
    _, mapping, _ = cf.cf_query_stitch_batchnorm_plan(w.rows, w.cols)
    if mapping == 3:
        return "bn_regional_kernel"
    # 128-bit rows stream through shared memory (the planner's rule)
    return "bn_global_tma_kernel" if w.cols % 4 == 0 else "bn_global_kernel"


def stitch_norm_numbers(torch, cf, w, peaks, device, l2):
    nsets = max(1, min(32, math.ceil(3 * l2 / w.unavoidable_bytes)))
    r = StitchNormRunner(torch, cf, w, nsets, device=device)
    reps = max(nsets, 200)
    t, n, _ = time_steps(torch, r, reps, 3, lambda: None, graph_len=reps)
    t1 = t / n
    gbs = w.unavoidable_bytes / t1 / 1e9
    out = {"us": round(t1 * 1e6, 2), "gbs": round(gbs, 1), "bound": "hbm",
           "roofline_frac": round(gbs / peaks["hbm_gbs"], 3), "buffer_sets": nsets,
           "kernel": stitch_norm_kernel_name(cf, w)}
    del r
    torch.cuda.empty_cache()
    return out


def pdl_chain_numbers(torch, cf, device, reps=200):
    """Three dependent fused calls on one stream -- GEMM+LayerNorm (1024x512x256),
    GEMM+softmax on its output (1024x256x512), B2B GEMM on that (K 256, N1 512,
    N2 128) -- replayed from CUDA graphs with programmatic dependent launch
    off and on: what overlapping each kernel's set-up with its predecessor's
    tail saves at a kernel boundary that is not fused."""
    M, K, N1, N2, NB1, NB2 = 1024, 256, 512, 256, 512, 128
    rng = np.random.Generator(np.random.PCG64(43))
    bf = torch.bfloat16

    def mat(r, c, sd):
        return torch.from_numpy(inputs.round_to_bf16(rng.standard_normal((r, c)).astype(np.float32) * sd)).to(
            device, bf)

    X, W1, W2, W3, W4 = mat(M, K, 1.0), mat(K, N1, K ** -0.5), mat(N1, N2, N1 ** -0.5), mat(N2, NB1, 4.0), \
        mat(NB1, NB2, NB1 ** -0.5)
    ones = torch.ones(N1, device=device)
    zeros = torch.zeros(N1, device=device)
    Y1 = torch.empty((M, N1), dtype=bf, device=device)
    Y2 = torch.empty((M, N2), dtype=bf, device=device)
    O = torch.empty((M, NB2), dtype=bf, device=device)
    ws = [cf.new_workspace(n, device) for n in (cf.cf_gemm_fused_workspace_size(M, N1, K),
                                                 cf.cf_gemm_fused_workspace_size(M, N2, N1),
                                                 cf.cf_b2b_workspace_size())]
    out = {}
    for label, tun in (("pdl_off_us", cf.tuning(disable_pdl=1)), ("pdl_on_us", cf.tuning())):
        class R:
            def launch(self, i, stream=None, t=tun):
                cf.check(cf.cf_gemm_fused_rownorm(X, W1, zeros, ones, zeros, Y1, M, N1, K, 1.0, 1e-5, cf.CF_ACT_NONE,
                                                  ws[0], ws[0].numel(), stream, t))
                cf.check(cf.cf_gemm_fused_rowsoftmax(Y1, W2, None, Y2, M, N2, N1, N1 ** -0.5, ws[1], ws[1].numel(),
                                                     stream, t))
                cf.check(cf.cf_b2b_gemm(Y2, W3, None, W4, O, M, N2, NB1, NB2, 1.0, cf.CF_B2B_GELU_TANH, ws[2],
                                        ws[2].numel(), stream, t))

        t, n, _ = time_steps(torch, R(), reps, 3, lambda: None, graph_len=reps)
        out[label] = round(t / n * 1e6, 2)
    out["saved_us_per_boundary"] = round((out["pdl_off_us"] - out["pdl_on_us"]) / 3, 2)
    out["chain"] = "GEMM+LN 1024x512x256 -> GEMM+softmax 1024x256x512 -> B2B GELU 1024x256x512x128, per chain"
    return out


def cpu_oracle_sample(w, budget_s=10.0, max_rows=None):
    """The fp64 oracle as it stands, on whole-row samples of the workload,
    repeated until ~budget_s of CPU time; returns (flops/s, seconds, rows)."""
    import oracle
    d = inputs.workload_inputs(w.name)
    rows_per = min(w.M, max_rows or w.M)
    rng = np.random.Generator(np.random.PCG64(0))
    done_rows, t_total = 0, 0.0
    while t_total < budget_s:
        rows = np.sort(rng.choice(w.M, size=rows_per, replace=False))
        t0 = time.perf_counter()
        oracle_rows(oracle, w, d, rows)
        t_total += time.perf_counter() - t0
        done_rows += rows_per
    return flops_per_row(w) * done_rows / t_total, t_total, done_rows


def flops_per_row(w):
    return w.flops / w.M


def workload_config(w):
    if isinstance(w, inputs.B2bWorkload):
        return {"workload": w.name, "op": w.op, "M": w.M, "K": w.K, "N1": w.N1, "N2": w.N2}
    return {"workload": w.name, "M": w.M, "N": w.N, "K": w.K}


def blas_threads():
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return len(os.sched_getaffinity(0))


def run_ours(args):
    import torch
    from memory_fusion_gb300 import cf

    ws_, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    ranks = mdist.Ranks("nccl", device)
    barrier = ranks.barrier
    peaks, peak_src = load_peaks()
    w = inputs.WORKLOADS[args.workload]
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    nsets = max(1, min(64, math.ceil(3 * l2 / bytes_per_set(w))))
    runner = FusedRunner(torch, cf, w, nsets, seed_offset=rank, device=device)
    props = torch.cuda.get_device_properties(device)
    gpu_id = str(getattr(props, "uuid", local))
    if gpu_id and not gpu_id.startswith("GPU-") and len(gpu_id) > 8:
        gpu_id = "GPU-" + gpu_id
    sampler = ClockSampler(gpu_id if gpu_id.startswith("GPU-") else str(local))
    t, n, clocks = time_steps(torch, runner, args.steps, args.warmup, barrier, sampler)
    t = ranks.max(t)  # the slowest rank sets the job time
    t1 = t / n
    value = mdist.job_throughput(w.flops * n, ws_, t) / 1e12
    troof, bound = roofline_time_s(w, peaks)
    kernel = {2: "gemm_fused_kernel<SOFTMAX>", 1: "gemm_fused_kernel<GELU_LN>", 0: "gemm_fused_kernel<LN>"}[kind_of(w)]
    if w.kind == "softmax_causal":
        kernel = "gemm_fused_kernel<SOFTMAX_MASK>"
    if w.kind == "rmsnorm":
        kernel += " (RMSNorm)"
    if w.resid_std is not None:
        kernel += " (residual)"
    if bound == "hbm":
        achieved = w.unavoidable_bytes / t1 / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4)}
    else:
        achieved = w.flops / t1 / 1e12
        pk = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": pk, "unit": "TFLOP/s",
                "frac": round(achieved / pk, 4),
                # the same against the power-capped (seconds-long loop) cuBLAS figure
                "peak_sustained": peaks["bf16_tflops_sustained"],
                "frac_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4)}
    traffic = profiled_traffic(w.name, kernel)
    roof["traffic"] = traffic
    roof["traffic_kind"] = profiled_traffic_kind(w.name, kernel)
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback"
    roof["kernel"] = kernel
    roof["algorithmic_bytes_per_launch"] = w.unavoidable_bytes
    roof["flops_per_launch"] = w.flops

    _, plan, active = cf.cf_query_gemm_fused_plan(w.M, w.N, w.K, kind_of(w))
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": ws_, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t1 * 1e3, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "dtype_detail": "bf16 operands, fp32 accumulate (TMEM) and fp32 epilogue, bf16 output",
        "data": "synthetic (seeded, shaped like the page workload)",
        "config": {"workload": w.name, "description": w.description, "M": w.M, "N": w.N, "K": w.K,
                   "batch_per_gpu": 1, "parallelism": f"replicas x{ws_} (rows independent)",
                   "l2": f"{nsets} rotating input/output sets (>= 3x L2 of {l2 >> 20} MiB)",
                   "plan": plan.as_dict()},
        "hbm_gbs": round(mdist.job_throughput(w.unavoidable_bytes * n, ws_, t) / 1e9, 1),
        "roofline_frac": round(troof / t1, 4),
        "roofline": roof,
        "gpu_launches": n,
        "clocks": clocks,
    }
    if rank == 0:
        te, h2d, d2h = time_e2e(torch, cf, w, max(10, min(args.steps, 200)), device)
        line["e2e"] = {"value": round(w.flops * ws_ / te / 1e12, 3), "unit": "TFLOP/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": round(te * 1e3, 4)}
        detail = None
        if not args.quick:
            names = [k for k in inputs.WORKLOADS]
            detail = per_workload(torch, cf, peaks, device, names)
            line["per_workload_detail"] = detail
            line["pdl_chain"] = pdl_chain_numbers(torch, cf, device)
        if not args.no_cpu:
            v, secs, rows = cpu_oracle_sample(w, budget_s=args.cpu_budget, max_rows=512)
            line["cpu_baseline"] = {"value": round(v / 1e12, 6), "unit": "TFLOP/s", "cores": blas_threads(),
                                    "kind": "oracle",
                                    "sample": f"{rows} whole rows of {w.name} (fp64 numpy oracle, "
                                              f"{secs:.1f} s; BLAS threads = cores, elementwise single-thread)"}
        if detail is not None:
            # last on the line, so that a record keeping only the line's tail keeps it
            line["per_workload"] = compact_summary(detail)
        print(json.dumps(line), flush=True)
    ranks.close()


def run_stitch(args):
    """A stitched workload as the timed workload (GB/s; used to profile the
    stitched kernels from a plain command line)."""
    import torch
    from memory_fusion_gb300 import cf

    ws_, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    ranks = mdist.Ranks("nccl", device)
    peaks, peak_src = load_peaks()
    w = inputs.WORKLOADS[args.workload]
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    nsets = max(1, min(32, math.ceil(3 * l2 / w.unavoidable_bytes)))
    if isinstance(w, inputs.StitchNormWorkload):
        runner = StitchNormRunner(torch, cf, w, nsets, seed_offset=rank, device=device)
        kernel = stitch_norm_kernel_name(cf, w)
        metric = f"stitched {w.kind} HBM GB/s"
    elif isinstance(w, inputs.StitchPowWorkload):
        d = inputs.powadd_inputs(w.rows, w.cols, mdist.seed_for(w.seed, rank))
        A = [torch.from_numpy(d["A"]).to(device) for _ in range(nsets)]
        wv = torch.from_numpy(d["w"]).to(device)
        O = [torch.empty_like(A[0]) for _ in range(nsets)]
        wsb = cf.cf_stitch_workspace_size(w.rows, w.cols)
        ws = cf.new_workspace(wsb, device)

        class RP:
            def launch(self, i, stream=None):
                cf.check(cf.cf_stitch_powadd_softmax(A[i % nsets], wv, w.p, O[i % nsets], w.rows, w.cols, ws, wsb,
                                                     stream))

        runner = RP()
        kernel = "stitch_packed_kernel" if (w.cols + 3) // 4 <= 32 else "stitch_split_kernel"
        metric = "stitched power->broadcast->softmax HBM GB/s"
    else:
        d = inputs.stitch_inputs(w.rows, w.cols, mdist.seed_for(w.seed, rank))
        A = [torch.from_numpy(d["A"]).to(device) for _ in range(nsets)]
        b = torch.from_numpy(d["row_bias"]).to(device)
        O = [torch.empty_like(A[0]) for _ in range(nsets)]
        wsb = cf.cf_stitch_workspace_size(w.rows, w.cols)
        ws = cf.new_workspace(wsb, device)

        class R:
            def launch(self, i, stream=None):
                cf.check(cf.cf_stitch_rowreduce_broadcast(A[i % nsets], b, O[i % nsets], w.rows, w.cols, ws, wsb,
                                                          stream))

        runner = R()
        # the planner's rule: rows of at most 32 float4 groups go packed, wider ones split
        kernel = "stitch_packed_kernel" if (w.cols + 3) // 4 <= 32 else "stitch_split_kernel"
        metric = "stitched reduce->broadcast HBM GB/s"

    props = torch.cuda.get_device_properties(device)
    gpu_id = str(getattr(props, "uuid", local))
    if gpu_id and not gpu_id.startswith("GPU-") and len(gpu_id) > 8:
        gpu_id = "GPU-" + gpu_id
    sampler = ClockSampler(gpu_id if gpu_id.startswith("GPU-") else str(local))
    t, n, clocks = time_steps(torch, runner, args.steps, args.warmup, ranks.barrier, sampler)
    t = ranks.max(t)
    gbs = mdist.job_throughput(w.unavoidable_bytes * n, ws_, t) / 1e9
    if rank == 0:
        print(json.dumps({"metric": metric, "value": round(gbs, 1), "unit": "GB/s",
                          "n_gpus": ws_, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": round(t / n * 1e3, 6), "higher_is_better": True, "scaling": "weak",
                          "dtype": "f32", "data": "synthetic (seeded, shaped like the page workload)",
                          "config": {"workload": w.name, "rows": w.rows, "cols": w.cols,
                                     "l2": f"{nsets} rotating input/output sets (>= 3x L2 of {l2 >> 20} MiB)"},
                          "roofline": {"bound": "hbm", "achieved": round(gbs / ws_, 1), "peak": peaks["hbm_gbs"],
                                       "unit": "GB/s", "frac": round(gbs / ws_ / peaks["hbm_gbs"], 4),
                                       "traffic": profiled_traffic(w.name, kernel),
                                       "traffic_kind": profiled_traffic_kind(w.name, kernel), "kernel": kernel,
                                       "algorithmic_bytes_per_launch": w.unavoidable_bytes,
                                       "peak_source": f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured"
                                       else "fallback"},
                          "gpu_launches": n, "clocks": clocks}), flush=True)
    ranks.close()


def run_b2b(args):
    """A back-to-back GEMM workload as the timed workload (TFLOP/s; used to
    profile the B2B kernel from a plain command line)."""
    import torch
    from memory_fusion_gb300 import cf

    ws_, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    ranks = mdist.Ranks("nccl", device)
    peaks, peak_src = load_peaks()
    w = inputs.WORKLOADS[args.workload]
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    nsets = max(1, min(32, math.ceil(3 * l2 / b2b_bytes_per_set(w))))
    r = B2bRunner(torch, cf, w, nsets, seed_offset=rank, device=device)
    props = torch.cuda.get_device_properties(device)
    gpu_id = str(getattr(props, "uuid", local))
    if gpu_id and not gpu_id.startswith("GPU-") and len(gpu_id) > 8:
        gpu_id = "GPU-" + gpu_id
    sampler = ClockSampler(gpu_id if gpu_id.startswith("GPU-") else str(local))
    t, n, clocks = time_steps(torch, r, args.steps, args.warmup, ranks.barrier, sampler)
    t = ranks.max(t)
    t1 = t / n
    tf = mdist.job_throughput(w.flops * n, ws_, t) / 1e12
    _, plan = cf.cf_query_b2b_plan(w.M, w.K, w.N1, w.N2, r.op)
    kernel = b2b_kernel_name(w, plan)
    # LayerNorm on the stream kernel: the fold kernel (gamma1^T W2, beta1^T W2)
    # launches before it every call; the step time covers both
    per_step = 2 if (w.op == "layernorm" and plan.n_slice == 128) else 1
    if rank == 0:
        print(json.dumps({"metric": "back-to-back GEMM TFLOP/s", "value": round(tf, 3), "unit": "TFLOP/s",
                          "n_gpus": ws_, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": round(t1 * 1e3, 6), "higher_is_better": True, "scaling": "weak",
                          "dtype": "bf16", "data": "synthetic (seeded)",
                          "config": dict(workload_config(w), plan=plan.as_dict(),
                                         l2=f"{nsets} rotating input/output sets (>= 3x L2 of {l2 >> 20} MiB)"),
                          "roofline": {"bound": "tensor", "achieved": round(tf / ws_, 1),
                                       "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                       "frac": round(tf / ws_ / peaks["bf16_tflops"], 4),
                                       "traffic": profiled_traffic(w.name, kernel),
                                       "traffic_kind": profiled_traffic_kind(w.name, kernel), "kernel": kernel,
                                       "algorithmic_bytes_per_launch": w.unavoidable_bytes,
                                       "flops_per_launch": w.flops,
                                       "launches_per_step": per_step,
                                       "peak_source": f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured"
                                       else "fallback"},
                          "gpu_launches": n * per_step, "clocks": clocks}), flush=True)
    ranks.close()


# ---------------------------------------------------------------------------
# reference arm: the fp64 CPU oracle
# ---------------------------------------------------------------------------
def _ref_sample_size(step_of, n_max, calls, budget_s):
    """Rows per step for the reference arm: the largest sample (at most n_max
    rows, at least one) whose `calls` oracle calls fit in budget_s, found by
    timing the oracle on this host at growing sample sizes."""
    target = budget_s / max(1, calls)
    step_of(1)  # first touch of the inputs and the BLAS threads
    n, best = 1, 1
    while True:
        t0 = time.perf_counter()
        step_of(n)
        t = time.perf_counter() - t0
        if t > target:
            return best
        best = n
        if n >= n_max:
            return n
        # grow at least twofold, faster while far below the target
        n = min(n_max, max(2 * n, int(n * 0.5 * target / max(t, 1e-6))))


def run_reference_stitched(args, w):
    """The oracle on a stitched workload: GB/s over the bytes of the rows it
    processed.  Each step is a random sample of whole rows, sized so that the
    warm-up and the K timed steps take about --ref-budget seconds (BatchNorm:
    the column statistics of the sampled rows, i.e. BatchNorm of a smaller
    batch drawn from the matrix)."""
    import oracle
    d = inputs.workload_inputs(w.name)
    rng = np.random.Generator(np.random.PCG64(1))
    per_row = w.unavoidable_bytes / w.rows
    bn = isinstance(w, inputs.StitchNormWorkload) and w.kind == "batchnorm"

    def step_of(n):
        # a contiguous block of rows at a random offset (drawing n distinct row
        # indices out of 750000 would cost more than the oracle's own step)
        r0 = int(rng.integers(0, w.rows - n + 1))
        rows = np.arange(r0, r0 + n)
        if bn:
            oracle.stitch_batchnorm(d["A"][r0:r0 + n], d["gamma"], d["beta"], w.eps)
        elif isinstance(w, inputs.StitchNormWorkload):
            oracle.stitch_add_layernorm(d["A"], d["R"], d["gamma"], d["beta"], w.eps, rows=rows)
        elif isinstance(w, inputs.StitchPowWorkload):
            oracle.stitch_powadd_softmax(d["A"], d["w"], w.p, rows=rows)
        else:
            oracle.stitch_rowreduce_broadcast(d["A"], d["row_bias"], rows=rows)

    n_max = w.rows if bn else min(w.rows, max(1, int(2e6 // w.cols)))
    n_rows = _ref_sample_size(step_of, n_max, args.steps + args.warmup, args.ref_budget)
    sample = (f"{n_rows} whole rows of {w.name} per step, a block at a random offset "
              f"({'BatchNorm over the sampled rows; ' if bn else ''}"
              f"fp64 numpy oracle; sized for about {args.ref_budget:.0f} s over warm-up and timed steps)")
    for _ in range(args.warmup):
        step_of(n_rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step_of(n_rows)
    t = time.perf_counter() - t0
    v = per_row * n_rows * args.steps / t / 1e9
    metric = (f"stitched {w.kind} HBM GB/s" if isinstance(w, inputs.StitchNormWorkload)
              else "stitched power->broadcast->softmax HBM GB/s" if isinstance(w, inputs.StitchPowWorkload)
              else "stitched reduce->broadcast HBM GB/s")
    print(json.dumps({
        "impl": "reference", "metric": metric, "value": round(v, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "rows": w.rows, "cols": w.cols},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_reference(args):
    ws_, rank, _ = dist_env()
    if rank != 0:
        return
    w = inputs.WORKLOADS[args.workload]
    if isinstance(w, (inputs.StitchWorkload, inputs.StitchNormWorkload, inputs.StitchPowWorkload)):
        run_reference_stitched(args, w)
        return
    import oracle
    # bf16 / fp32 inputs widened to float64 once, before any timing: the same
    # values the oracle would widen them to on every call
    d = {k: (v.astype(np.float64) if isinstance(v, np.ndarray) else v)
         for k, v in inputs.workload_inputs(w.name).items()}
    rng = np.random.Generator(np.random.PCG64(1))

    def step_of(n):
        oracle_rows(oracle, w, d, np.sort(rng.choice(w.M, size=n, replace=False)))

    rows_per_step = _ref_sample_size(step_of, 128, args.steps + args.warmup, args.ref_budget)
    for _ in range(args.warmup):
        step_of(rows_per_step)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step_of(rows_per_step)
    t = time.perf_counter() - t0
    flops = flops_per_row(w) * rows_per_step * args.steps
    v = flops / t / 1e12
    sample = (f"{rows_per_step} random whole rows of {w.name} per step (fp64 numpy oracle; sized for about "
              f"{args.ref_budget:.0f} s over warm-up and timed steps)")
    metric = "back-to-back GEMM TFLOP/s" if isinstance(w, inputs.B2bWorkload) else METRIC
    print(json.dumps({
        "impl": "reference", "metric": metric, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": ws_,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w),
        "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # defaults: ours, 100000 launches (about half a minute on the headline
    # workload); the reference arm (the fp64 CPU oracle), 20 steps
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="skip the per-workload table")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--ref-budget", type=float, default=90.0,
                    help="reference arm: seconds of oracle time over warm-up and timed steps")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 20 if args.impl == "reference" else 100000
    if args.warmup is None:
        args.warmup = 5 if args.impl == "reference" else 200
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    stitched = isinstance(inputs.WORKLOADS[args.workload],
                          (inputs.StitchWorkload, inputs.StitchNormWorkload, inputs.StitchPowWorkload))
    if args.impl == "reference":
        run_reference(args)
    elif stitched:
        run_stitch(args)
    elif isinstance(inputs.WORKLOADS[args.workload], inputs.B2bWorkload):
        run_b2b(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
