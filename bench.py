#!/usr/bin/env python
"""Benchmark of the speculative-decoding verify/sample step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one verify call (every kernel of the path) over one batch of
synthetic input.  Default workload: B=1, gamma=5, V=32000 bfloat16 logits,
T=0.7 (the single-sequence verify); --workload picks another entry of
workloads.WORKLOADS.  Inputs are resident in HBM before timing; each step uses
its own input set and the sets together exceed twice the 129 MB L2, so no
step starts with its inputs in L2.  The timed region replays a CUDA graph of
calls (one call per input set) on one stream, bracketed by CUDA events and a
synchronize; ms_per_step = elapsed / steps.

Printed as one JSON line (rank 0).  Under torchrun each rank runs an
independent replica on its own GPU (the path has no exchange step), the time
is the max over ranks and value = all ranks' positions / that time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "verify positions/sec (B*(gamma+1)) and achieved HBM GB/s as % of GB300 peak"
UNIT = "positions/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--workload", default=workloads.HEADLINE, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle time budget for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size B (smaller cases for ncu captures)")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the short summary runs of the other workloads (N=1 only)")
    return ap.parse_args()


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend=backend)
    return rank, ws, local


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """The largest value of x over all ranks (x itself on one rank)."""
    if ws <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _elt_bytes(w):
    return {"f32": 4, "bf16": 2, "f16": 2}[w.dtype]


def _q_elt_bytes(w) -> int:
    """Bytes per q element the step reads: float32 q, the draft's logits in
    w's dtype, or none (greedy, deterministic drafts)."""
    if w.mode != "sample" or w.deterministic:
        return 0
    return _elt_bytes(w) if w.qlogits else 4


def _workspace(sv, w, B, G, V, dev):
    if w.qlogits:
        return sv.alloc_qlogits_workspace(B, G, V, w.top_k, dev)
    return sv.alloc_workspace(B, G, V, w.top_k if w.mode == "sample" else 0, dev)


def algorithmic_bytes(w, n_accepted: np.ndarray, kept_per_row: int = 0, gamma_b=None):
    """Bytes the method must move for one step, split by kernel.

    streaming kernel: every logit once, plus the gathers of l(d_i) and q(d_i);
    final-draw kernel (untruncated sampling): one row of logits per sequence,
    plus the q row of a rejected sequence.  q as the draft's logits: every
    draft row once more (to form q) and q elements counted at the logits'
    size; the float32 q the library may form from them is the
    implementation's own traffic.  With top-k the final draw reads
    only the kept candidates' q values (inside the streaming kernel).
    Deterministic drafts (q one-hot, passed as None) read no q bytes.  A
    ragged round (gamma_b given) needs only rows 0..gamma_b of each sequence."""
    s = _elt_bytes(w)
    B, G, V = len(n_accepted), w.gamma, w.V
    qb = _q_elt_bytes(w)
    gsum = int(np.sum(gamma_b)) if gamma_b is not None else B * G
    if w.mode == "greedy":
        return {"stream": (gsum + B) * V * s, "final": 0}
    stream = (gsum + B) * V * s + gsum * (qb + s)
    if w.qlogits:
        stream += gsum * V * s           # the draft rows, read once to form their q
    if w.top_k > 0 or w.top_p < 1.0:
        return {"stream": stream + B * kept_per_row * qb, "final": 0}
    gb = np.asarray(gamma_b) if gamma_b is not None else np.full(B, G)
    rejected = int((n_accepted < gb).sum())
    final = rejected * V * (qb + s) + (B - rejected) * V * s
    return {"stream": stream, "final": final}


class Clocks:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"sv_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def _kernel_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_46_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def _traffic(workload: str, kernel: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum)
    from the committed ncu summary profiles/dram_traffic.txt, whose lines read
    `<workload> <kernel> <kernel source hash> <bytes per launch> ...`; None if
    absent or if the kernel source changed since the capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 4 and not line.startswith("#") and parts[0] == workload and parts[1] == kernel:
                    return float(parts[3]) if parts[2] == _kernel_hash() else None
    except OSError:
        pass
    return None


def _input_sets(w, n_sets: int, device):
    """n_sets independent input batches, generated as one batch of
    n_sets * B sequences and sliced (each slice is contiguous)."""
    big = workloads.make_inputs(w, seed=w.seed + 1000 * int(os.environ.get("RANK", "0")), device=device,
                                B=n_sets * w.B)
    sets = []
    for i in range(n_sets):
        sl = slice(i * w.B, (i + 1) * w.B)
        # stop_tokens is one list for the batch, everything else per sequence
        sets.append({k: (v[sl] if v is not None and k != "stop_tokens" else v) for k, v in big.items()})
    return sets


def _packed(named, dev):
    """One pinned host buffer and one device buffer holding every tensor of
    `named` (None entries stay None) at 256-byte aligned offsets, the host
    one filled with the tensors' values; returns (host buffer, device buffer,
    {name: device view})."""
    offs, o = {}, 0
    for k, v in named.items():
        if v is not None:
            offs[k] = o
            o += (v.numel() * v.element_size() + 255) // 256 * 256
    host = torch.empty(max(o, 256), dtype=torch.uint8, pin_memory=True)
    devb = torch.empty(max(o, 256), dtype=torch.uint8, device=dev)
    views = {}
    for k, v in named.items():
        if v is None:
            views[k] = None
            continue
        n = v.numel() * v.element_size()
        host[offs[k]:offs[k] + n].view(v.dtype).view(v.shape).copy_(v)
        views[k] = devb[offs[k]:offs[k] + n].view(v.dtype).view(v.shape)
    return host, devb, views


def _call(sv, w, inp, out, ws, stream):
    if w.qlogits:
        return sv.verify_sample_qlogits(inp["logits"], inp["q_logits"], inp["draft"], inp["uniforms"],
                                        w.temperature, w.top_k, w.top_p, workspace=ws, stream=stream, outputs=out)
    if w.mode == "greedy":
        return sv.verify_greedy(inp["logits"], inp["draft"], workspace=ws, stream=stream,
                                outputs=(out[0], out[1], out[3]))
    r = sv.verify_sample(inp["logits"], inp["q"], inp["draft"], inp["uniforms"], w.temperature, w.top_k,
                         w.top_p, workspace=ws, stream=stream, outputs=out, gamma_b=inp.get("gamma_b"))
    if w.ragged:
        # end the round at stop tokens / token budgets (one more kernel)
        sv.truncate_emitted(r[0], r[1], inp["stop_tokens"], inp["max_new"], stream=stream)
    return r


def run_gb300(args, rank, ws_n, local):
    import speculative_decoding_verification_46_gb300 as sv

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sv.load_library()
    w = workloads.WORKLOADS[args.workload]
    if args.batch is not None:
        w = w.with_(B=args.batch, name=f"{w.name}@B={args.batch}")
    B, G, V = w.B, w.gamma, w.V
    positions = B * (G + 1)

    per_set = B * (G + 1) * V * _elt_bytes(w) + B * G * V * _q_elt_bytes(w)
    n_sets = max(2, min(1024, math.ceil(2 * L2_BYTES / per_set) + 1))
    sets = _input_sets(w, n_sets, dev)
    outs = [(torch.empty(B, G + 1, dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev),
             torch.empty(B, G, dtype=torch.float32, device=dev) if w.mode == "sample" and G > 0 else None,
             torch.empty(B, dtype=torch.int32, device=dev)) for _ in range(n_sets)]
    top_k_ws = w.top_k if w.mode == "sample" else 0
    wsp = _workspace(sv, w, B, G, V, dev)
    stream = torch.cuda.Stream(device=dev)

    # default steps: about a second of timed work
    with torch.cuda.stream(stream):
        for i in range(n_sets):
            _call(sv, w, sets[i], outs[i], wsp, stream)
    torch.cuda.synchronize()
    all_kernels = sv.sv_last_kernels()       # what one call launches (the path the library chose)
    kernels_per_call = len(all_kernels) + (1 if w.ragged else 0)   # + the truncation kernel
    # the timing hook brackets the verify kernels; the kernels that form q
    # from draft logits (and clear it) run outside it and are timed with the
    # step only
    kernel_names = [k for k in all_kernels if k not in ("q_softmax_kernel", "q_truncate_kernel", "q_clear_kernel")]
    if kernels_per_call == 0:
        raise RuntimeError("the verify call launched no kernel")
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n_sets):
            _call(sv, w, sets[i], outs[i], wsp, stream)
    torch.cuda.synchronize()
    est = (time.perf_counter() - t0) / n_sets
    steps = args.steps if args.steps is not None else int(min(200_000, max(200, 1.0 / max(est, 1e-6))))
    warmup = args.warmup if args.warmup is not None else max(3, min(steps // 10, 1000))

    # a CUDA graph of n_sets calls (call i on input set i), replayed
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(n_sets):
            _call(sv, w, sets[i], outs[i], wsp, stream)
    torch.cuda.synchronize()

    def run_steps(k):
        full, rem = divmod(k, n_sets)
        for _ in range(full):
            graph.replay()
        if rem:
            with torch.cuda.stream(stream):
                for i in range(rem):
                    _call(sv, w, sets[i], outs[i], wsp, stream)

    with torch.cuda.stream(stream):
        run_steps(warmup)
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    _barrier(ws_n)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        run_steps(steps)
        e1.record(stream)
    torch.cuda.synchronize()
    _barrier(ws_n)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / steps
    ms_max = max_over_ranks(ms, ws_n, dev)
    value = positions * ws_n / (ms_max / 1e3)

    # per-kernel durations: events recorded before, between and after the
    # kernels of each call.  A fixed-length sleep kernel first keeps the GPU
    # busy while the host queues a batch of calls, so that the gaps between
    # events are device time, not host submission time.
    n_batch, batch = 4, 100
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_batch * batch)]
    with torch.cuda.stream(stream):
        for trio in evs:
            for e in trio:
                e.record(stream)          # torch creates the CUDA event on first record
        j = 0
        for _ in range(n_batch):
            torch.cuda._sleep(40_000_000)  # ~20 ms at 2 GHz
            for _ in range(batch):
                if sv.sv_set_timing_events(evs[j]) != sv.SV_OK:
                    raise RuntimeError("sv_set_timing_events failed")
                _call(sv, w, sets[j % n_sets], outs[j % n_sets], wsp, stream)
                j += 1
        sv.sv_set_timing_events(None)
    torch.cuda.synchronize()
    t_stream = float(np.mean([e[0].elapsed_time(e[1]) for e in evs])) * 1e-3
    t_final = float(np.mean([e[1].elapsed_time(e[2]) for e in evs])) * 1e-3 if len(kernel_names) == 2 else 0.0
    kernel_us = {kernel_names[0]: t_stream * 1e6}
    if len(kernel_names) == 2:
        kernel_us[kernel_names[1]] = t_final * 1e6

    # algorithmic bytes: average over the input sets (the final draw depends on the data)
    nacc = np.concatenate([o[1].cpu().numpy() for o in outs])
    gbs = np.concatenate([st["gamma_b"].cpu().numpy() for st in sets]) if w.ragged else None
    ab = algorithmic_bytes(w, nacc, gamma_b=gbs)
    if w.ragged:
        # a ragged round verifies sum_b (gamma_b + 1) positions (mean over the input sets)
        positions = float(np.sum(gbs)) / n_sets + B
        value = positions * ws_n / (ms_max / 1e3)
    ab = {k: v / n_sets for k, v in ab.items()}
    if len(kernel_names) == 1:
        # one kernel does the whole step (its final draw included)
        ab = {"stream": ab["stream"] + ab["final"], "final": 0.0}
    peak, peak_kind = _peaks()
    kern = "stream" if t_stream >= t_final else "final"
    kname = kernel_names[0] if kern == "stream" else kernel_names[1]
    t_k = t_stream if kern == "stream" else t_final
    achieved = ab[kern] / t_k / 1e9
    step_gbs = (ab["stream"] + ab["final"]) / (ms / 1e3) / 1e9

    # end to end: pinned host inputs -> device, the call, outputs -> host, every
    # step.  The step's inputs sit in one pinned host buffer and its outputs in
    # one device buffer (views at 256-byte offsets), so one copy moves each way;
    # copy in, call, copy out are captured in a CUDA graph replayed per step.
    ins = dict(sets[0])
    if w.mode == "greedy":
        ins["uniforms"] = None                     # greedy reads no uniforms
    host_in, dev_in_buf, dev_in = _packed(ins, dev)
    out_named = {str(i): x for i, x in enumerate(outs[0])}
    if w.mode == "greedy":
        out_named["2"] = None                      # greedy writes no accept_prob
    host_out, dev_out_buf, dev_out_v = _packed(out_named, dev)
    dev_out = tuple(dev_out_v[str(i)] for i in range(len(outs[0])))
    h2d = host_in.numel()
    d2h = host_out.numel()
    n_e2e = min(steps, 2000)
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for _ in range(3):
            dev_in_buf.copy_(host_in, non_blocking=True)
            _call(sv, w, dev_in, dev_out, wsp, stream)
            host_out.copy_(dev_out_buf, non_blocking=True)
    torch.cuda.synchronize()
    with torch.cuda.graph(g_e2e, stream=stream):
        dev_in_buf.copy_(host_in, non_blocking=True)
        _call(sv, w, dev_in, dev_out, wsp, stream)
        host_out.copy_(dev_out_buf, non_blocking=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(3):
            g_e2e.replay()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(n_e2e):
            g_e2e.replay()
        f1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(f0.elapsed_time(f1) / n_e2e, ws_n, dev)
    pos_e2e = float((sets[0]["gamma_b"].sum() + B).item()) if w.ragged else positions   # the input set used

    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": ws_n,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": w.name, "B": B, "gamma": G, "V": V, "logits_dtype": w.dtype, "mode": w.mode,
            "temperature": w.temperature, "top_k": w.top_k, "top_p": w.top_p,
            "parallelism": f"replicas x{ws_n} (batch per GPU fixed)",
            "l2": f"no flush: {n_sets} rotating input sets of {per_set / 1e6:.2f} MB (> 2x L2)",
            "timing": "CUDA graph of calls replayed, CUDA events on the launching stream",
        },
        "hbm_gbs": step_gbs,
        "hbm_frac_of_peak": step_gbs / peak,
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": _traffic(w.name, kname),
                     "algorithmic_bytes_per_launch": ab[kern], "avg_launch_us": t_k * 1e6,
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s"},
        "kernel_us": kernel_us,
        "e2e": {"value": pos_e2e * ws_n / (ms_e2e / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                "how": "inputs in one pinned host buffer, outputs in one device buffer; copy in, call, copy out "
                       "captured in a CUDA graph and replayed once per step"},
        "gpu_launches": steps * kernels_per_call,
        "clocks": clk,
    }
    return line, w


def other_workloads(args, local):
    """Short device-side runs of the other workloads (graph replay, rotating
    input sets, no flush), each ~0.3 s of timed work: value, ms/step, HBM GB/s
    and the fraction of the measured peak for the whole step."""
    import speculative_decoding_verification_46_gb300 as sv

    dev = torch.device("cuda", local)
    peak, _ = _peaks()
    out = {}
    for name, w in workloads.WORKLOADS.items():
        if name == args.workload:
            continue
        B, G, V = w.B, w.gamma, w.V
        per_set = B * (G + 1) * V * _elt_bytes(w) + B * G * V * _q_elt_bytes(w)
        n_sets = max(2, min(512, math.ceil(2 * L2_BYTES / per_set) + 1))
        sets = _input_sets(w, n_sets, dev)
        outs = [(torch.empty(B, G + 1, dtype=torch.int32, device=dev), torch.empty(B, dtype=torch.int32, device=dev),
                 torch.empty(B, G, dtype=torch.float32, device=dev) if w.mode == "sample" and G > 0 else None,
                 torch.empty(B, dtype=torch.int32, device=dev)) for _ in range(n_sets)]
        wsp = _workspace(sv, w, B, G, V, dev)
        stream = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(stream):
            for i in range(n_sets):
                _call(sv, w, sets[i], outs[i], wsp, stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(n_sets):
                _call(sv, w, sets[i], outs[i], wsp, stream)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        reps = max(1, int(0.3 / max(time.perf_counter() - t0, 1e-6)))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / (reps * n_sets)
        nacc = np.concatenate([o[1].cpu().numpy() for o in outs])
        gb_all = np.concatenate([st["gamma_b"].cpu().numpy() for st in sets]) if w.ragged else None
        ab = algorithmic_bytes(w, nacc, gamma_b=gb_all)
        gbs = (ab["stream"] + ab["final"]) / n_sets / (ms / 1e3) / 1e9
        pos = (float(np.sum(gb_all)) / n_sets + B) if w.ragged else B * (G + 1)   # positions in the round
        out[name] = {"value": pos / (ms / 1e3), "ms_per_step": ms, "hbm_gbs": gbs,
                     "frac_of_measured_peak": gbs / peak, "steps": reps * n_sets}
        del sets, outs, wsp, graph
        torch.cuda.empty_cache()
    return out


def oracle_throughput(w, budget_s: float, device="cpu"):
    """The CPU oracle on a bounded sample of the workload: whole batches of
    B sequences when they fit the budget, else a prefix of one batch."""
    from oracle import svref

    inp = workloads.make_inputs(w, seed=w.seed + 7, device="cuda" if torch.cuda.is_available() else "cpu")
    L = inp["logits"].float().cpu().numpy()
    d = inp["draft"].cpu().numpy()
    u = inp["uniforms"].cpu().numpy()
    q = inp["q"].cpu().numpy() if inp["q"] is not None else None
    qlg = inp["q_logits"].float().cpu().numpy() if w.qlogits else None
    gbh = inp["gamma_b"].cpu().numpy() if w.ragged else None
    stops = inp["stop_tokens"].cpu().numpy() if w.ragged else None
    mxh = inp["max_new"].cpu().numpy() if w.ragged else None
    done, seqs = 0.0, 0
    t0 = time.perf_counter()
    b = 0
    while True:
        sl = slice(b, b + 1)
        if w.mode == "greedy":
            svref.verify_greedy(L[sl], d[sl])
        elif w.ragged:
            r = svref.verify_sample_ragged(L[sl], q[sl] if q is not None else None, d[sl], u[sl], w.temperature,
                                           gbh[sl], w.top_k, w.top_p)
            svref.truncate_emitted(r["out_tokens"], r["n_accepted"], stops, mxh[sl])
        elif w.qlogits:
            svref.verify_sample_qlogits(L[sl], qlg[sl], d[sl], u[sl], w.temperature, w.top_k, w.top_p)
        else:
            svref.verify_sample(L[sl], q[sl] if q is not None else None, d[sl], u[sl], w.temperature, w.top_k,
                                w.top_p)
        seqs += 1
        b = (b + 1) % w.B
        done = time.perf_counter() - t0
        if done >= budget_s:
            break
    pos = seqs * (w.gamma + 1)
    return pos / done, f"{seqs} sequences of the workload ({pos} positions) in {done:.2f} s, numpy float64"


def main():
    args = _args()
    rank, ws_n, local = _dist()
    if args.impl == "reference":
        if rank != 0:
            return
        w = workloads.WORKLOADS[args.workload]
        steps = args.steps if args.steps is not None else 5
        warmup = args.warmup if args.warmup is not None else 1
        from oracle import svref

        inp = workloads.make_inputs(w, seed=w.seed + 7, device="cuda" if torch.cuda.is_available() else "cpu")
        L = inp["logits"].float().cpu().numpy()
        d = inp["draft"].cpu().numpy()
        u = inp["uniforms"].cpu().numpy()
        q = inp["q"].cpu().numpy() if inp["q"] is not None else None
        qlg = inp["q_logits"].float().cpu().numpy() if w.qlogits else None
        gbh = inp["gamma_b"].cpu().numpy() if w.ragged else None
        stops = inp["stop_tokens"].cpu().numpy() if w.ragged else None
        mxh = inp["max_new"].cpu().numpy() if w.ragged else None
        # one step = a bounded sample of the batch (at most ~2 s of oracle work)
        t0 = time.perf_counter()
        if w.mode == "greedy":
            svref.verify_greedy(L[:1], d[:1])
        elif w.ragged:
            r = svref.verify_sample_ragged(L[:1], q[:1] if q is not None else None, d[:1], u[:1], w.temperature,
                                           gbh[:1], w.top_k, w.top_p)
            svref.truncate_emitted(r["out_tokens"], r["n_accepted"], stops, mxh[:1])
        elif w.qlogits:
            svref.verify_sample_qlogits(L[:1], qlg[:1], d[:1], u[:1], w.temperature, w.top_k, w.top_p)
        else:
            svref.verify_sample(L[:1], q[:1] if q is not None else None, d[:1], u[:1], w.temperature, w.top_k,
                                w.top_p)
        per_seq = time.perf_counter() - t0
        per_step_budget = min(2.0, 120.0 / max(1, steps + warmup))
        nseq = int(max(1, min(w.B, per_step_budget / max(per_seq, 1e-6))))

        def step():
            if w.mode == "greedy":
                svref.verify_greedy(L[:nseq], d[:nseq])
            elif w.ragged:
                r = svref.verify_sample_ragged(L[:nseq], q[:nseq] if q is not None else None, d[:nseq], u[:nseq],
                                               w.temperature, gbh[:nseq], w.top_k, w.top_p)
                svref.truncate_emitted(r["out_tokens"], r["n_accepted"], stops, mxh[:nseq])
            elif w.qlogits:
                svref.verify_sample_qlogits(L[:nseq], qlg[:nseq], d[:nseq], u[:nseq], w.temperature, w.top_k,
                                            w.top_p)
            else:
                svref.verify_sample(L[:nseq], q[:nseq] if q is not None else None, d[:nseq], u[:nseq],
                                    w.temperature, w.top_k, w.top_p)

        for _ in range(warmup):
            step()
        t0 = time.perf_counter()
        for _ in range(steps):
            step()
        el = (time.perf_counter() - t0) / steps
        v = nseq * (w.gamma + 1) / el
        sample = f"{nseq} of {w.B} sequences per step, numpy float64, single thread"
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": ws_n, "steps": steps,
            "warmup": warmup, "ms_per_step": el * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "gamma": w.gamma, "V": w.V, "logits_dtype": w.dtype,
                       "mode": w.mode, "temperature": w.temperature, "top_k": w.top_k, "top_p": w.top_p},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }), flush=True)
        return

    line, w = run_gb300(args, rank, ws_n, local)
    if rank == 0 and ws_n == 1 and not args.no_other_workloads and args.batch is None:
        line["other_workloads"] = other_workloads(args, local)
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        v, sample = oracle_throughput(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
                                "host": platform.machine(), "host_cpus": os.cpu_count()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws_n > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
