#!/usr/bin/env python3
"""Benchmark of the xHC per-sublayer residual-stream update on B300.

One step = the whole per-sublayer hot path on one batch: the fused forward in
training mode (in-place state update, dense read x_in, saved logits and the
saved active rows) followed by the fused backward (dL/dX', no gradient through
x_in), on the bf16 workload B=4, S=4096, N=16, C=2048, k=4 with seeded
synthetic inputs (X, out ~ N(0,1); conv weights and W ~ N(0, 0.02)).

Prints one JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
(on host cores) on a bounded sample of the same workload instead.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from residual_stream_expansion_xhc_b300 import inputs as xin  # noqa: E402

METRIC = "tokens/s per xHC sublayer (fwd, fwd+bwd) and achieved HBM GB/s vs peak"

# Algorithmic bytes per token of each kernel, in C-units (one row of C
# elements of the state dtype) plus fixed per-token fp32 side data.
#   forward, fused:   16 (read X) + 1 (read out) + 4 (write active rows)
#                     + 1 (write x_in) + 4 (write saved active rows) = 26
#   backward, token:  4 (dX' active) + 4 (old active rows) + 1 (out) = 9
#   backward, stream: 16 (X) + 16 (dX') + 1 (out) + 16 (dX) + 1 (dout) = 50
ALG_C = {  # algorithmic bytes per token in C-units (one row of C state elements)
    "coeffs_tc": 16, "fwd_update": 26, "bwd_col": 14, "bwd_stream_tc": 48, "flash_tc": 22,
    "restore_active": 8,  # read the k saved rows, write them back into the state
    "coeffs_simt": 17, "update_simt": 26,
    "bwd_token_simt": 9, "bwd_dx_simt": 48, "bwd_dw_simt": 16, "bwd_tfa_simt": 6,
}
ALG_SIDE = {  # fp32 bytes per token
    "coeffs_tc": 196, "coeffs_simt": 196, "flash_tc": 192 + 196,
    "coeffs_tc_router": 196 + 196,  # the logits and the router's inputs
}
# The fused stack step (flash_tc) of sublayer l: 16 (read X) + 1 (read out) +
# 4 (write the active rows in place) + 1 (write x_in) = 22 C, plus sublayer
# l's coefficient block read (192 B) and sublayer l+1's logits and block
# written (196 B).  The closing update of a stack writes no saved rows: 22 C.


def pass_c_units(N: int, k: int, mode: str) -> int:
    """Algorithmic bytes per token of one pass, in C-units (the minimum a pass
    must move; N streams, k active):
      forward, inference: N (read X) + 1 (read out) + k (write the active rows)
                          + 1 (write x_in)                      = 22 at N=16, k=4
      forward, training:  adds the k saved active rows          = 26
      backward:           2k + 1 (per-token quantities: dX' and the old rows
                          of the active streams, out) + 3N + 2 (stream pass:
                          X, dX', dX, out, dout)                = 59"""
    fwd = N + 1 + k + 1
    if mode == "fwd_inference":
        return fwd
    if mode == "fwd_training":
        return fwd + k
    if mode == "bwd":
        return (2 * k + 1) + (3 * N + 2)
    raise ValueError(mode)


def kernel_c_units(name: str, N: int, k: int, saved_active: bool = True) -> int:
    """Algorithmic bytes per token of one launch of a kernel, in C-units: what
    its own job must read and write at least."""
    table = {
        "coeffs_tc": N,                                   # read X
        "coeffs_tc_router": N,                            # read X (the router rows ride along)
        "fwd_update": N + 1 + k + 1 + (k if saved_active else 0),
        "flash_tc": N + 1 + k + 1,                        # dense read + sparse write of sublayer l
        "bwd_col": 3 * k + 2,                             # read dX'[a], old rows, out; write mix, dout
        "bwd_stream_tc": 3 * N,                           # read X, dX'; write dX
        "restore_active": 2 * k,                          # read the saved rows, write them into the state
    }
    if name in table:
        return table[name]
    return ALG_C.get(name, 0)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- oracle timing

def oracle_sample(wl, tensors, ntok: int):
    """The first ``ntok`` tokens of sequence 0 of the workload (exact for those
    tokens: nothing before a sequence start enters the update)."""
    X = xin.to_f64(wl, tensors.X[:1, :ntok])
    out = xin.to_f64(wl, tensors.out[:1, :ntok])
    dXp = xin.to_f64(wl, tensors.dXp[:1, :ntok])
    conv = None if tensors.conv is None else tuple(np.asarray(w, np.float64) for w in tensors.conv)
    if wl.router_fixed >= 0:
        W_r = np.asarray(tensors.extra["W_r"], np.float64)
        return X, out, conv, np.asarray(tensors.W, np.float64), (W_r, list(tensors.idx[: wl.router_fixed])), dXp
    return X, out, conv, np.asarray(tensors.W, np.float64), tensors.idx, dXp


def stack_sample(wl, layers, ntok: int):
    """The first ``ntok`` tokens of sequence 0 through every sublayer of a stack."""
    X = xin.to_f64(wl, layers[0].X[:1, :ntok])
    outs = [xin.to_f64(wl, t.out[:1, :ntok]) for t in layers]
    convs = [None if t.conv is None else tuple(np.asarray(w, np.float64) for w in t.conv) for t in layers]
    return X, outs, convs, [np.asarray(t.W, np.float64) for t in layers], [list(t.idx) for t in layers]


def time_oracle_stack(sample, wl):
    from oracle import xhc_oracle as xo
    X, outs, convs, Ws, idxs = sample
    t0 = time.perf_counter()
    xo.forward_stack(X, outs, convs, Ws, idxs, iters=wl.iters, eps=wl.eps, gs=wl.gram_schmidt, store="bf16")
    return time.perf_counter() - t0


def time_oracle(sample, wl):
    from oracle import xhc_oracle as xo
    X, out, conv, W, idx, dXp = sample
    t0 = time.perf_counter()
    if wl.router_fixed >= 0:
        W_r, fixed = idx
        xo.forward_routed(X, out, conv, W, W_r, fixed, wl.k, iters=wl.iters, eps=wl.eps)
        xo.backward_routed(X, out, conv, W, W_r, fixed, wl.k, dXp, None, iters=wl.iters, eps=wl.eps)
    else:
        xo.forward(X, out, conv, W, idx, iters=wl.iters, eps=wl.eps, gs=wl.gram_schmidt)
        xo.backward(X, out, conv, W, idx, dXp, None, iters=wl.iters, eps=wl.eps, gs=wl.gram_schmidt)
    return time.perf_counter() - t0


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads", 1) for d in threadpool_info()]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline_stack(wl, layers, ntok=256):
    sample = stack_sample(wl, layers, ntok)
    dt = time_oracle_stack(sample, wl)
    return {"value": ntok * wl.layers / dt, "unit": "sublayer-tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"fp64 numpy oracle, the {wl.layers}-sublayer stack forward of the first {ntok} tokens of "
                      f"sequence 0 ({dt:.1f} s)"}


def cpu_baseline(wl, tensors, ntok=1024, ntok1=1024):
    """The oracle on all host cores (its BLAS calls threaded), and beside it
    the same oracle on one thread (BLAS limited to one thread)."""
    sample = oracle_sample(wl, tensors, ntok)
    dt = time_oracle(sample, wl)
    res = {"value": ntok / dt, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
           "sample": f"fp64 numpy oracle, forward+backward of the first {ntok} tokens of sequence 0 "
                     f"({dt:.1f} s)", "host_cpus": os.cpu_count()}
    # one thread: a child process whose BLAS pools are started with one
    # thread (the thread counts are read when the BLAS library loads)
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-once", str(ntok1),
                            "--workload", wl.name], env=env, capture_output=True, text=True, timeout=600)
        dt1 = float(json.loads(r.stdout.strip().splitlines()[-1])["seconds"])
    except (subprocess.SubprocessError, ValueError, IndexError, KeyError, OSError):
        return res
    res["single_thread"] = {"value": ntok1 / dt1, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                            "sample": f"fp64 numpy oracle on one thread (1 of {os.cpu_count()} host CPUs), "
                                      f"forward+backward of one sequence of {ntok1} tokens drawn with the "
                                      f"workload's widths and distributions ({dt1:.1f} s)"}
    return res


def oracle_once(wl, ntok):
    """Child-process leg of the one-thread oracle timing: draw the workload,
    time the oracle on the first ``ntok`` tokens, print the seconds."""
    tensors = xin.make(xin.scaled(wl, B=1, S=max(ntok, 1)), grads=True)
    dt = time_oracle(oracle_sample(wl, tensors, ntok), wl)
    print(json.dumps({"seconds": dt, "tokens": ntok, "blas_threads": blas_threads()}), flush=True)


def run_reference(args, wl):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    ntok = args.ref_tokens
    if wl.layers > 1:
        layers = [xin.make(wl, l, state=(l == 0)) for l in range(wl.layers)]
        sample = stack_sample(wl, layers, ntok)
        for _ in range(args.warmup):
            time_oracle_stack(sample, wl)
        t = sum(time_oracle_stack(sample, wl) for _ in range(args.steps))
        value = ntok * wl.layers * args.steps / t
        desc = f"fp64 numpy oracle, the {wl.layers}-sublayer stack forward of the first {ntok} tokens of sequence 0"
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "sublayer-tokens/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": wl_desc(wl), "sample_tokens_per_step": ntok},
                "cpu_baseline": {"value": value, "unit": "sublayer-tokens/s", "cores": blas_threads(),
                                 "kind": "oracle", "sample": desc + " per step"},
                "e2e": {"value": value, "unit": "sublayer-tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    tensors = xin.make(wl, grads=True)
    sample = oracle_sample(wl, tensors, ntok)
    for _ in range(args.warmup):
        time_oracle(sample, wl)
    t = sum(time_oracle(sample, wl) for _ in range(args.steps))
    value = ntok * args.steps / t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl_desc(wl), "sample_tokens_per_step": ntok},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": f"fp64 numpy oracle, forward+backward of the first {ntok} tokens of "
                                       f"sequence 0 per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def wl_desc(wl):
    head = f"{wl.name}: B={wl.B} S={wl.S} N={wl.N} C={wl.C} k={wl.k} {wl.dtype}; "
    if wl.layers > 1:
        return head + (f"stack of {wl.layers} sublayers, forward in place (inference: x_in of every sublayer, no "
                       f"saved rows), each update fused with the next sublayer's coefficient projection")
    if wl.router_fixed >= 0:
        return head + (f"router: {wl.router_fixed} fixed + {wl.k - wl.router_fixed} routed slots per token; forward "
                       f"(in place, x_in, saved logits, saved active rows, router record) + backward (the saved rows "
                       f"written back first; dX', no dx_in)")
    gs = "; Gram-Schmidt of the TFA components" if wl.gram_schmidt else ""
    if not wl.backward:
        return head + f"forward (inference: in place, x_in written, no saved logits or rows){gs}"
    return head + (f"forward (training mode: in place, x_in, saved logits, saved active rows) + backward (dX', "
                   f"no dx_in){gs}")


# ----------------------------------------------------------------------------- GPU arm

class Step:
    """Device buffers of one sublayer and the fused forward + backward calls."""

    def __init__(self, wl, tensors, dev):
        import torch
        from residual_stream_expansion_xhc_b300 import api
        self.api, self.wl, self.torch = api, wl, torch
        dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32

        def act(a):
            if wl.dtype == "f32":
                return torch.from_numpy(a).to(dev)
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

        self.sh = api.make_shape(wl.B, wl.S, wl.N, wl.C, wl.k, dt, wl.iters, wl.eps, wl.gram_schmidt)
        self.X = act(tensors.X)
        self.out = act(tensors.out)
        self.dXp = act(tensors.dXp)
        self.conv = None if tensors.conv is None else tuple(torch.from_numpy(w).to(dev) for w in tensors.conv)
        self.W = torch.from_numpy(tensors.W).to(dev)
        self.idx = [int(i) for i in tensors.idx]
        B, S, N, C, k, P = wl.B, wl.S, wl.N, wl.C, wl.k, wl.P
        self.x_in = torch.empty(B, S, C, dtype=dt, device=dev)
        self.saved = torch.empty(B, S, P + 1, dtype=torch.float32, device=dev)
        self.act = torch.empty(B, S, k, C, dtype=dt, device=dev)
        self.dX = torch.empty_like(self.X)
        self.dout = torch.empty_like(self.out)
        self.dconv = None if self.conv is None else tuple(torch.empty_like(w) for w in self.conv)
        self.dW = torch.empty_like(self.W)
        self.ws = api.workspace(api.xhc_bwd_workspace_bytes(self.sh), dev)
        self.fws = api.workspace(api.xhc_fwd_workspace_need(self.sh, True), dev)

    def fwd(self):
        self.api.xhc_sublayer_fwd(self.sh, self.X, self.X, self.out, self.conv, self.W, self.idx, x_in=self.x_in,
                                  saved=self.saved, saved_active=self.act, workspace=self.fws)

    def bwd(self):
        self.api.xhc_sublayer_bwd(self.sh, self.X, self.act, self.out, self.conv, self.W, self.idx, self.saved,
                                  self.dXp, None, self.dX, self.dout, self.dconv, self.dW, self.ws)

    def __call__(self):
        self.fwd()
        self.bwd()


class RoutedStep(Step):
    """The router's forward, in place with the old active rows saved, and its
    backward, which writes those rows back (the state before the update) before
    it reads the state."""

    def __init__(self, wl, tensors, dev):
        super().__init__(wl, tensors, dev)
        torch = self.torch
        B, S, N, k = wl.B, wl.S, wl.N, wl.k
        self.W_r = torch.from_numpy(tensors.extra["W_r"]).to(dev)
        self.fixed = self.idx[: wl.router_fixed]
        self.tok_idx = torch.empty(B, S, k, dtype=torch.int32, device=dev)
        self.rrec = torch.empty(B, S, 2 * N + 2, dtype=torch.float32, device=dev)
        self.dW_r = torch.empty_like(self.W_r)
        self.fws = self.api.workspace(self.api.xhc_fwd_routed_workspace_bytes(self.sh), dev)
        self.ws = self.api.workspace(self.api.xhc_bwd_routed_workspace_bytes(self.sh), dev)

    def fwd(self):
        self.api.xhc_sublayer_fwd_routed(self.sh, self.X, self.X, self.out, self.conv, self.W, self.W_r, self.fixed,
                                         self.tok_idx, self.rrec, self.fws, x_in=self.x_in, saved=self.saved,
                                         saved_active=self.act)

    def bwd(self):
        self.api.xhc_sublayer_bwd_routed(self.sh, self.X, self.out, self.conv, self.W, self.W_r, self.fixed,
                                         self.saved, self.tok_idx, self.rrec, self.dXp, None, self.dX, self.dout,
                                         self.dconv, self.dW, self.dW_r, self.ws, saved_active=self.act)


class StackStep:
    """Device buffers of a stack of sublayers and the fused stack forward."""

    def __init__(self, wl, layers, dev):
        import torch
        from residual_stream_expansion_xhc_b300 import api
        self.api, self.wl, self.torch = api, wl, torch

        def act(a):
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

        self.sh = api.make_shape(wl.B, wl.S, wl.N, wl.C, wl.k, torch.bfloat16, wl.iters, wl.eps, wl.gram_schmidt)
        self.X = act(layers[0].X)
        self.outs = [act(t.out) for t in layers]
        self.convs = None if layers[0].conv is None else [tuple(torch.from_numpy(w).to(dev) for w in t.conv)
                                                          for t in layers]
        self.Ws = [torch.from_numpy(t.W).to(dev) for t in layers]
        self.idxs = [[int(i) for i in t.idx] for t in layers]
        self.x_ins = [torch.empty(wl.B, wl.S, wl.C, dtype=torch.bfloat16, device=dev) for _ in layers]
        self.ws = api.workspace(api.xhc_stack_fwd_workspace_bytes(self.sh), dev)

    def fwd(self):
        self.api.xhc_stack_fwd(self.sh, self.X, self.outs, self.convs, self.Ws, self.idxs, self.ws, x_ins=self.x_ins)

    def __call__(self):
        self.fwd()


class InfStep:
    """The inference forward of one sublayer: in place, x_in written, no saved
    logits and no saved rows (the logits go to the workspace)."""

    def __init__(self, wl, tensors, dev):
        import torch
        from residual_stream_expansion_xhc_b300 import api
        self.api, self.wl, self.torch = api, wl, torch

        def act(a):
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

        self.sh = api.make_shape(wl.B, wl.S, wl.N, wl.C, wl.k, torch.bfloat16, wl.iters, wl.eps, wl.gram_schmidt)
        self.X = act(tensors.X)
        self.out = act(tensors.out)
        self.conv = None if tensors.conv is None else tuple(torch.from_numpy(w).to(dev) for w in tensors.conv)
        self.W = torch.from_numpy(tensors.W).to(dev)
        self.idx = [int(i) for i in tensors.idx]
        self.x_in = torch.empty(wl.B, wl.S, wl.C, dtype=torch.bfloat16, device=dev)
        self.fws = api.workspace(api.xhc_fwd_workspace_need(self.sh, False), dev)

    def __call__(self):
        self.api.xhc_sublayer_fwd(self.sh, self.X, self.X, self.out, self.conv, self.W, self.idx, x_in=self.x_in,
                                  saved=None, saved_active=None, workspace=self.fws)


def measure_leg(step, wl, steps, warmup, alg_c_per_unit, units_per_step, unit, peak, saved_active=True):
    """Time one workload leg: ``steps`` steps after ``warmup`` (CUDA events on
    the launching stream), then the same steps again with the library's
    per-kernel events for the kernel table.  Bytes: ``alg_c_per_unit`` C-units
    (the pass model) per unit of work; moved = what the launched kernels must
    move by their own jobs (kernel_c_units) per step."""
    import torch
    from residual_stream_expansion_xhc_b300 import api
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    ms = timed(step, steps) / steps
    api.xhc_timing_collect()
    api.xhc_timing_enable(True)
    timed(step, steps)
    api.xhc_timing_enable(False)
    torch.cuda.synchronize()
    kern = api.xhc_timing_collect()
    cunit = wl.C * wl.esize
    alg = alg_c_per_unit * cunit * units_per_step
    moved_c = sum((c / steps) * kernel_c_units(n, wl.N, wl.k, saved_active) for n, (c, _) in kern.items())
    moved = moved_c * cunit * wl.tokens
    total = sum(t for _, t in kern.values())
    dname, (dcount, dtotal) = max(kern.items(), key=lambda kv: kv[1][1])
    d_ms = dtotal / dcount
    d_alg = (kernel_c_units(dname, wl.N, wl.k, saved_active) * cunit + ALG_SIDE.get(dname, 0)) * wl.tokens
    return {
        "workload": wl_desc(wl), "ms_per_step": ms, "value": units_per_step / (ms * 1e-3), "unit": unit,
        "alg_C_per_unit": alg_c_per_unit, "alg_bytes_per_step": alg,
        "alg_GBps": alg / (ms * 1e-3) / 1e9, "alg_frac": alg / (ms * 1e-3) / 1e9 / peak,
        "moved_C_per_token": moved_c, "moved_GBps": moved / (ms * 1e-3) / 1e9,
        "moved_frac": moved / (ms * 1e-3) / 1e9 / peak,
        "dominant": {"kernel": dname, "avg_ms": d_ms, "alg_bytes_per_launch": d_alg,
                     "GBps": d_alg / (d_ms * 1e-3) / 1e9, "frac": d_alg / (d_ms * 1e-3) / 1e9 / peak},
        "kernels": {n: {"launches_per_step": c / steps, "avg_ms": t / c, "share": t / total}
                    for n, (c, t) in kern.items()},
    }


def extra_legs(args, dev, peak):
    """The other bf16 workloads of the benchmark suite, one line each, on the
    same GPU after the main leg: the inference forward (B4 S4096 C2048), the
    eight-sublayer stack (B2 S8192 C4096, fused stack forward) and the
    mHC-shaped forward + backward (N = k = 4, no TFA)."""
    import torch
    out = {}
    steps = max(3, args.steps)
    wl = xin.WORKLOADS["fwd_bf16"]
    st = InfStep(wl, xin.make(wl), dev)
    out["fwd_inference"] = measure_leg(st, wl, steps, args.warmup, pass_c_units(wl.N, wl.k, "fwd_inference"),
                                       wl.tokens, "tokens/s", peak, saved_active=False)
    del st
    torch.cuda.empty_cache()
    wl = xin.WORKLOADS["mhc_bf16"]
    st = Step(wl, xin.make(wl, grads=True), dev)
    out["mhc"] = measure_leg(st, wl, steps, args.warmup,
                             pass_c_units(wl.N, wl.k, "fwd_training") + pass_c_units(wl.N, wl.k, "bwd"),
                             wl.tokens, "tokens/s", peak)
    out["mhc"]["forward_ms"] = timed(st.fwd, steps) / steps
    out["mhc"]["backward_ms"] = timed(st.bwd, steps) / steps
    del st
    torch.cuda.empty_cache()
    wl = xin.WORKLOADS["stack8_bf16"]
    layers = [xin.make(wl, l, state=(l == 0)) for l in range(wl.layers)]
    st = StackStep(wl, layers, dev)
    del layers
    out["stack8"] = measure_leg(st, wl, max(3, steps // 4), args.warmup, pass_c_units(wl.N, wl.k, "fwd_inference"),
                                wl.tokens * wl.layers, "sublayer-tokens/s", peak, saved_active=False)
    out["stack8"]["moved_C_per_sublayer"] = out["stack8"].pop("moved_C_per_token") / wl.layers
    del st
    torch.cuda.empty_cache()
    return out


def stack_e2e_run(step, layers, steps):
    """Host buffers through the public API: every step copies the state and
    every sublayer's `out` from pinned host memory, runs the stack and reads
    the final state and every sublayer's x_in back (one stream, in order)."""
    torch = step.torch
    hX = torch.from_numpy(layers[0].X.view(np.int16)).pin_memory()
    houts = [torch.from_numpy(t.out.view(np.int16)).pin_memory() for t in layers]
    rX = torch.empty_like(hX).pin_memory()
    rxin = [torch.empty(o.shape, dtype=torch.int16).pin_memory() for o in houts]

    def one():
        step.X.view(torch.int16).copy_(hX, non_blocking=True)
        for d, h in zip(step.outs, houts):
            d.view(torch.int16).copy_(h, non_blocking=True)
        step()
        rX.copy_(step.X.view(torch.int16), non_blocking=True)
        for h, d in zip(rxin, step.x_ins):
            h.copy_(d.view(torch.int16), non_blocking=True)

    one()
    ms = timed(one, steps)
    h2d = hX.numel() * 2 + sum(h.numel() * 2 for h in houts)
    d2h = rX.numel() * 2 + sum(h.numel() * 2 for h in rxin)
    return {"value": step.wl.tokens * step.wl.layers * steps / (ms * 1e-3), "unit": "sublayer-tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": ms / steps}


def timed(fn, steps):
    import torch
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(s)
    for _ in range(steps):
        fn()
    e1.record(s)
    e1.synchronize()
    return e0.elapsed_time(e1)


def copy_peak(dev):
    import torch
    from residual_stream_expansion_xhc_b300 import api
    n = 1 << 30
    a = torch.empty(n, dtype=torch.uint8, device=dev)
    a.fill_(1)
    b = torch.empty_like(a)
    api.xhc_copy(a, b)
    ms = timed(lambda: api.xhc_copy(a, b), 10)
    del a, b
    torch.cuda.empty_cache()                 # the 2 GB go back to the device
    return 2 * n * 10 / (ms * 1e-3) / 1e9


def e2e_run(step, tensors, steps):
    """Host buffers through the public API: every step copies its inputs
    (X, out, dX') from pinned host memory to the device, runs the forward +
    backward, and reads its results (X', dX, dout, dW, conv-weight gradients)
    back to pinned host memory.

    Steps are pipelined the way a training loop would: two sets of device
    buffers, host-to-device copies on one stream, the update on another and
    device-to-host reads on a third, so that step i + 1's inputs travel while
    step i's results come back (the link is full duplex).  The timed region
    starts before the first step's copies and ends after the last step's
    reads have landed."""
    torch = step.torch
    wl = step.wl
    dev = step.X.device

    def pinned(a):
        t = torch.from_numpy(a if wl.dtype == "f32" else a.view(np.int16))
        return t.pin_memory()

    hX, hout, hdXp = pinned(tensors.X), pinned(tensors.out), pinned(tensors.dXp)
    as_raw = (lambda t: t) if wl.dtype == "f32" else (lambda t: t.view(torch.int16))
    sets = [step, type(step)(wl, tensors, dev)]
    res = []
    for _ in sets:
        rdc = None if step.dconv is None else [torch.empty(w.shape, dtype=torch.float32).pin_memory()
                                               for w in step.dconv]
        res.append(dict(X=torch.empty_like(hX).pin_memory(), dX=torch.empty_like(hdXp).pin_memory(),
                        dout=torch.empty_like(hout).pin_memory(),
                        dW=torch.empty(step.W.shape, dtype=torch.float32).pin_memory(), dconv=rdc))
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    done_out = [None, None]                       # D2H of the last step that used each set

    def one(i):
        st, r = sets[i % 2], res[i % 2]
        ev_free = done_out[i % 2]
        with torch.cuda.stream(s_in):
            if ev_free is not None:
                s_in.wait_event(ev_free)
            as_raw(st.X).copy_(hX, non_blocking=True)
            as_raw(st.out).copy_(hout, non_blocking=True)
            as_raw(st.dXp).copy_(hdXp, non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev_in)
            st()
            ev_c = torch.cuda.Event()
            ev_c.record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_c)
            r["X"].copy_(as_raw(st.X), non_blocking=True)
            r["dX"].copy_(as_raw(st.dX), non_blocking=True)
            r["dout"].copy_(as_raw(st.dout), non_blocking=True)
            r["dW"].copy_(st.dW, non_blocking=True)
            if r["dconv"] is not None:
                for h, d in zip(r["dconv"], st.dconv):
                    h.copy_(d, non_blocking=True)
            ev_o = torch.cuda.Event()
            ev_o.record(s_out)
            done_out[i % 2] = ev_o

    one(0)
    one(1)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(steps):
        one(i)
    s_in.wait_stream(s_out)
    e1.record(s_in)
    e1.synchronize()
    ms = e0.elapsed_time(e1)
    h2d = sum(t.numel() * t.element_size() for t in (hX, hout, hdXp))
    r = res[0]
    d2h = sum(r[k].numel() * r[k].element_size() for k in ("X", "dX", "dout", "dW")) + (
        0 if r["dconv"] is None else sum(t.numel() * 4 for t in r["dconv"]))
    return {"value": wl.tokens * steps / (ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": ms / steps,
            "pipeline": "two buffer sets; H2D, compute and D2H on three streams"}


def run_gpu(args, wl):
    import torch
    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from residual_stream_expansion_xhc_b300 import api

    if wl.layers > 1:
        return run_gpu_stack(args, wl, world, rank, local, dev)
    tensors = xin.make(wl, grads=True)
    step = RoutedStep(wl, tensors, dev) if wl.router_fixed >= 0 else Step(wl, tensors, dev)
    same_run_copy = copy_peak(dev)
    esz = wl.esize
    cunit = wl.C * esz

    for _ in range(args.warmup):
        step()
    # forward alone and backward alone (for the per-pass numbers)
    torch.cuda.synchronize()
    fwd_ms = timed(step.fwd, args.steps) / args.steps
    bwd_ms = timed(step.bwd, args.steps) / args.steps

    api.xhc_timing_collect()
    torch.cuda.synchronize()
    barrier(world)
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    api.xhc_timing_enable(True)
    ms = timed(step, args.steps)
    api.xhc_timing_enable(False)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    kern = api.xhc_timing_collect()
    ms = max_over_ranks(ms, world)
    ms_step = ms / args.steps
    tokens = wl.tokens * world
    value = tokens * args.steps / (ms * 1e-3)

    peak, peak_kind = load_peaks()
    dom = max(kern.items(), key=lambda kv: kv[1][1])
    dname, (dcount, dtotal) = dom
    per_launch_ms = dtotal / dcount
    alg = (kernel_c_units(dname, wl.N, wl.k) * cunit + ALG_SIDE.get(dname, 0)) * wl.tokens
    achieved = alg / (per_launch_ms * 1e-3) / 1e9
    traffic = load_traffic(dname, wl.tokens)
    e2e = None
    if not args.no_e2e:
        e2e = e2e_run(step, tensors, args.e2e_steps)
        e2e["value"] *= world
    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(wl, tensors, args.cpu_tokens)
    extras = None
    if not args.no_extra and wl.name == "fwdbwd_bf16":
        del step, tensors
        torch.cuda.empty_cache()
        sampler2 = ClockSampler(local) if rank == 0 else None
        if sampler2:
            sampler2.start()
            time.sleep(0.3)
        extras = extra_legs(args, dev, peak)
        clocks2 = sampler2.stop() if sampler2 else None
        for v in extras.values():
            v["clocks"] = clocks2
    if rank != 0:
        return
    fwd_alg = pass_c_units(wl.N, wl.k, "fwd_training") * cunit * wl.tokens
    bwd_alg = pass_c_units(wl.N, wl.k, "bwd") * cunit * wl.tokens
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl_desc(wl), "tokens_per_step_per_gpu": wl.tokens,
                   "l2": "inputs larger than L2 (state X is %.2f GB per GPU)" % (wl.tokens * wl.N * cunit / 1e9),
                   "parallelism": f"replicas x{world} (independent batches, no collective)"},
        "roofline": {"kernel": dname, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})",
                     "alg_bytes_per_launch": alg, "launch_ms": per_launch_ms},
        "step": {"alg_C_per_token": (fwd_alg + bwd_alg) / (cunit * wl.tokens),
                 "alg_GBps": (fwd_alg + bwd_alg) / (ms_step * 1e-3) / 1e9,
                 "alg_frac": (fwd_alg + bwd_alg) / (ms_step * 1e-3) / 1e9 / peak},
        "fwd": {"tokens_per_s": wl.tokens / (fwd_ms * 1e-3), "ms": fwd_ms,
                "alg_GBps": fwd_alg / (fwd_ms * 1e-3) / 1e9, "alg_bytes": fwd_alg,
                "alg_frac": fwd_alg / (fwd_ms * 1e-3) / 1e9 / peak},
        "bwd": {"tokens_per_s": wl.tokens / (bwd_ms * 1e-3), "ms": bwd_ms,
                "alg_GBps": bwd_alg / (bwd_ms * 1e-3) / 1e9, "alg_bytes": bwd_alg,
                "alg_frac": bwd_alg / (bwd_ms * 1e-3) / 1e9 / peak},
        "kernels": {k: {"launches": c, "avg_ms": t / c, "share": t / sum(v[1] for v in kern.values())}
                    for k, (c, t) in kern.items()},
        "gpu_launches": int(sum(c for c, _ in kern.values())),
        "same_run_copy_GBps": same_run_copy,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if extras:
        line.update(extras)
    print(json.dumps(line), flush=True)


def run_gpu_stack(args, wl, world, rank, local, dev):
    """The fused stack forward: a step is the whole stack of wl.layers
    sublayers over one batch; the metric counts tokens x sublayers."""
    import torch
    from residual_stream_expansion_xhc_b300 import api
    layers = [xin.make(wl, l, state=(l == 0)) for l in range(wl.layers)]
    step = StackStep(wl, layers, dev)
    same_run_copy = copy_peak(dev)
    cunit = wl.C * wl.esize
    for _ in range(args.warmup):
        step()
    api.xhc_timing_collect()
    torch.cuda.synchronize()
    barrier(world)
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    api.xhc_timing_enable(True)
    ms = timed(step, args.steps)
    api.xhc_timing_enable(False)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    kern = api.xhc_timing_collect()
    ms = max_over_ranks(ms, world)
    units = wl.tokens * wl.layers * world
    value = units * args.steps / (ms * 1e-3)
    peak, peak_kind = load_peaks()
    dname, (dcount, dtotal) = max(kern.items(), key=lambda kv: kv[1][1])
    per_launch_ms = dtotal / dcount
    c_units = kernel_c_units(dname, wl.N, wl.k, saved_active=False)
    alg = (c_units * cunit + ALG_SIDE.get(dname, 0)) * wl.tokens
    achieved = alg / (per_launch_ms * 1e-3) / 1e9
    e2e = None
    if not args.no_e2e:
        e2e = stack_e2e_run(step, layers, max(1, args.e2e_steps // 2))
        e2e["value"] *= world
    cpu = cpu_baseline_stack(wl, layers, min(args.cpu_tokens, 512)) if rank == 0 and not args.no_cpu else None
    if rank != 0:
        return
    # bytes per sublayer of the stack as the fused schedule moves them
    stack_alg = ((wl.layers - 1) * 22 + 22 + 16) * cunit * wl.tokens
    line = {
        "metric": METRIC, "value": value, "unit": "sublayer-tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl_desc(wl), "tokens_per_step_per_gpu": wl.tokens, "sublayers": wl.layers,
                   "l2": "inputs larger than L2 (state X is %.2f GB per GPU)" % (wl.tokens * wl.N * cunit / 1e9),
                   "parallelism": f"replicas x{world} (independent batches, no collective)"},
        "roofline": {"kernel": dname, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": load_traffic(dname, wl.tokens),
                     "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})",
                     "alg_bytes_per_launch": alg, "launch_ms": per_launch_ms},
        "stack": {"C_units_per_sublayer": stack_alg / (cunit * wl.tokens * wl.layers),
                  "alg_GBps": stack_alg / (ms / args.steps * 1e-3) / 1e9, "alg_bytes": stack_alg},
        "kernels": {k: {"launches": c, "avg_ms": t / c, "share": t / sum(v[1] for v in kern.values())}
                    for k, (c, t) in kern.items()},
        "gpu_launches": int(sum(c for c, _ in kern.values())),
        "same_run_copy_GBps": same_run_copy,
        "clocks": clocks,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def load_traffic(kernel: str, tokens: int):
    """DRAM bytes (read + write) per launch of a kernel, from the committed ncu
    summary ``profiles/dram_traffic.txt`` (lines: kernel, measured bytes per
    launch, tokens of the captured launch), scaled to ``tokens``; None when the
    kernel has no entry there."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel:
                return float(parts[1]) * tokens / float(parts[2])
    return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["xhc", "reference"], default="xhc")
    ap.add_argument("--workload", default="fwdbwd_bf16", choices=sorted(xin.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the inference-forward, stack and mHC-shape lines of the default run")
    ap.add_argument("--cpu-tokens", type=int, default=8192)
    ap.add_argument("--ref-tokens", type=int, default=256)
    ap.add_argument("--oracle-once", type=int, default=0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    wl = xin.WORKLOADS[args.workload]
    if args.oracle_once:
        oracle_once(wl, args.oracle_once)
        return
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_gpu(args, wl)


if __name__ == "__main__":
    main()
