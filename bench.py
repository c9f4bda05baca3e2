#!/usr/bin/env python
"""Benchmark of the speculative-decoding verify/sample step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one verify call (every kernel of the path) over one batch of
synthetic input.  Default workload: the largest single-GPU one, B=256
sequences, gamma=8 drafts, V=152064 bfloat16 logits, T=0.8, top-k 50 then
top-p 0.9 applied to p and q; --workload picks another entry of
workloads.WORKLOADS.  Inputs are resident in HBM before timing; each step uses
its own input set and the sets together exceed twice the 129 MB L2, so no
step starts with its inputs in L2.  The timed region replays CUDA graphs of
calls (one call per input set; a graph of n_sets calls replayed, plus one
graph of the remaining calls when K is not a multiple of n_sets) on one
stream, bracketed by CUDA events and a synchronize; ms_per_step = elapsed / K.

Printed as one JSON line (rank 0).  Under torchrun each rank runs an
independent replica on its own GPU (the path has no exchange step), the time
is the max over ranks and value = all ranks' positions / that time.

Besides the contract's keys the line carries: `roofline` for the step's
dominant kernel, `kernel_us` per kernel, `parity` (the GPU's outputs against
the CPU oracle on the cpu_baseline sample: draws, mismatches, boundary
draws), `acceptance` (empirical alpha and tokens per round against the
prediction from the same acceptance probabilities), and `other_workloads`
(the same measurements, shorter, for every other workload).
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
BOUNDARY_LIMIT = 1e-4      # boundary mismatches allowed, as a fraction of all draws


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


def algorithmic_bytes(w, n_accepted: np.ndarray, kept_rejected: int = 0, gamma_b=None):
    """Bytes the method must move for one step, split by kernel.

    streaming kernel: every logit once, plus the gathers of l(d_i) and q(d_i);
    final-draw kernel (untruncated sampling): one row of logits per sequence,
    plus the q row of a rejected sequence.  q as the draft's logits: every
    draft row once more (to form q) and q elements counted at the logits'
    size; the float32 q the library may form from them is the
    implementation's own traffic.  With top-k (then top-p) the final draw of a
    rejected sequence reads q only at the kept candidates of row n:
    kept_rejected is their total over the batch (read inside the streaming
    kernel's sequence finisher).  Top-p alone ranks the whole row: the final
    draw reads row n's logits again and q at its kept tokens (its own
    threshold passes over the rows are the implementation's traffic).
    Deterministic drafts (q one-hot, passed as None) read no q bytes.  A
    ragged round (gamma_b given) needs only rows 0..gamma_b of each
    sequence."""
    s = _elt_bytes(w)
    B, G, V = len(n_accepted), w.gamma, w.V
    qb = _q_elt_bytes(w)
    gsum = int(np.sum(gamma_b)) if gamma_b is not None else B * G
    if w.mode == "greedy":
        return {"stream": (gsum + B) * V * s, "final": 0}
    stream = (gsum + B) * V * s + gsum * (qb + s)
    if w.qlogits:
        stream += gsum * V * s           # the draft rows, read once to form their q
    if w.top_k > 0:
        return {"stream": stream + int(kept_rejected) * qb, "final": 0}
    gb = np.asarray(gamma_b) if gamma_b is not None else np.full(B, G)
    if w.top_p < 1.0:
        return {"stream": stream, "final": B * V * s + int(kept_rejected) * qb}
    rejected = int((n_accepted < gb).sum())
    final = rejected * V * (qb + s) + (B - rejected) * V * s
    return {"stream": stream, "final": final}


def kept_counts(logits_rows: torch.Tensor, temperature: float, top_k: int, top_p: float) -> torch.Tensor:
    """Number of tokens top-k then top-p keeps in each row (torch, on the
    rows' device): bench-side accounting of the kept candidates whose q the
    final draw reads; not part of the verify path."""
    z = logits_rows.float() / temperature
    V = z.shape[-1]
    k = V if top_k <= 0 else min(top_k, V)
    vals = torch.topk(z, k, dim=-1, sorted=True).values.double()
    pk = torch.softmax(vals, dim=-1)
    if top_p >= 1.0:
        return torch.full(z.shape[:-1], k, dtype=torch.int64, device=z.device)
    before = pk.cumsum(-1) - pk
    return (before < top_p).sum(-1)


def kept_rows_q(w, st, out):
    """Kept candidates over the rejected sequences' rows n (the q entries a
    truncated final draw reads), for one input set and its outputs."""
    if w.mode != "sample" or (w.top_k <= 0 and w.top_p >= 1.0) or _q_elt_bytes(w) == 0:
        return 0
    n = out[1].long()
    rej = n < w.gamma
    if not rej.any():
        return 0
    rows = st["logits"][torch.nonzero(rej).flatten(), n[rej]]
    return int(kept_counts(rows, w.temperature, w.top_k, w.top_p).sum().item())


def q_bytes_read(w, n_accepted: np.ndarray, st, kept_rejected: int) -> int:
    """Bytes of q the kernels read for one input set: q(d_i) at every tested
    position, then q at the kept candidates of each rejected sequence's row
    n (top-k / top-p) or that whole row (untruncated)."""
    qb = _q_elt_bytes(w)
    if w.mode != "sample" or qb == 0 or w.qlogits:
        return 0
    gb = st["gamma_b"].cpu().numpy() if w.ragged else np.full(len(n_accepted), w.gamma)
    gsum = int(gb.sum())
    if w.top_k > 0 or w.top_p < 1.0:
        return (gsum + int(kept_rejected)) * qb
    rejected = int((n_accepted < gb).sum())
    return (gsum + rejected * w.V) * qb


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


def _input_sets(w, n_sets: int, device, seed_offset: int = 1000):
    """n_sets independent input batches, generated as one batch of
    n_sets * B sequences and sliced (each slice is contiguous)."""
    big = workloads.make_inputs(w, seed=w.seed + seed_offset * (1 + int(os.environ.get("RANK", "0"))),
                                device=device, B=n_sets * w.B)
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


class Runner:
    """Input sets, outputs, workspace and CUDA graphs of one workload."""

    def __init__(self, sv, w, dev, max_sets: int = 1024):
        self.sv, self.w, self.dev = sv, w, dev
        B, G, V = w.B, w.gamma, w.V
        self.per_set = B * (G + 1) * V * _elt_bytes(w) + B * G * V * _q_elt_bytes(w)
        self.n_sets = max(2, min(max_sets, math.ceil(2 * L2_BYTES / self.per_set) + 1))
        self.sets = _input_sets(w, self.n_sets, dev)
        self.outs = [(torch.empty(B, G + 1, dtype=torch.int32, device=dev),
                      torch.empty(B, dtype=torch.int32, device=dev),
                      torch.empty(B, G, dtype=torch.float32, device=dev) if w.mode == "sample" and G > 0 else None,
                      torch.empty(B, dtype=torch.int32, device=dev)) for _ in range(self.n_sets)]
        self.ws = _workspace(sv, w, B, G, V, dev)
        self.stream = torch.cuda.Stream(device=dev)
        self.graphs = {}

    def call(self, i):
        return _call(self.sv, self.w, self.sets[i], self.outs[i], self.ws, self.stream)

    def eager(self, count):
        with torch.cuda.stream(self.stream):
            for i in range(count):
                self.call(i % self.n_sets)

    def graph(self, count):
        """A CUDA graph of `count` calls on input sets 0..count-1 (captured once)."""
        if count not in self.graphs:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                for i in range(count):
                    self.call(i)
            torch.cuda.synchronize()
            self.graphs[count] = g
        return self.graphs[count]

    def prepare(self, k):
        """Capture the graphs that run_steps(k) replays (outside any timing)."""
        full, rem = divmod(k, self.n_sets)
        if full:
            self.graph(self.n_sets)
        if rem:
            self.graph(rem)

    def run_steps(self, k):
        """k calls, every one replayed from a CUDA graph."""
        full, rem = divmod(k, self.n_sets)
        with torch.cuda.stream(self.stream):
            for _ in range(full):
                self.graph(self.n_sets).replay()
            if rem:
                self.graph(rem).replay()

    def kernel_times(self, n_batch: int, batch: int):
        """Mean device time of the call's kernels, from CUDA events the
        library records before its first kernel, after the kernel that streams
        the logits, and after its last kernel.  A fixed-length sleep kernel
        first keeps the GPU busy while the host queues a batch of calls, so
        that the gaps between events are device time, not host submission."""
        sv = self.sv
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_batch * batch)]
        with torch.cuda.stream(self.stream):
            for trio in evs:
                for e in trio:
                    e.record(self.stream)          # torch creates the CUDA event on first record
            j = 0
            for _ in range(n_batch):
                torch.cuda._sleep(40_000_000)  # ~20 ms at 2 GHz
                for _ in range(batch):
                    if sv.sv_set_timing_events(evs[j]) != sv.SV_OK:
                        raise RuntimeError("sv_set_timing_events failed")
                    self.call(j % self.n_sets)
                    j += 1
            sv.sv_set_timing_events(None)
        torch.cuda.synchronize()
        t_stream = float(np.mean([e[0].elapsed_time(e[1]) for e in evs])) * 1e-3
        t_final = float(np.mean([e[1].elapsed_time(e[2]) for e in evs])) * 1e-3
        return t_stream, t_final

    def kernels(self):
        """(all kernels of one call, the ones between the timing events)."""
        with torch.cuda.stream(self.stream):
            self.call(0)
        torch.cuda.synchronize()
        allk = self.sv.sv_last_kernels()
        # the kernels that form q from draft logits (and clear it) run outside
        # the timing hook's events
        timed = [k for k in allk if k not in ("q_softmax_kernel", "q_truncate_kernel", "q_clear_kernel")]
        return allk, timed

    def accounting(self):
        """Algorithmic bytes per step (mean over the input sets, after the
        last calls on every set), positions per step, and the acceptance
        statistics of the outputs."""
        w = self.w
        nacc = np.concatenate([o[1].cpu().numpy() for o in self.outs])
        gbs = np.concatenate([st["gamma_b"].cpu().numpy() for st in self.sets]) if w.ragged else None
        kept = 0
        if w.mode == "sample" and (w.top_k > 0 or w.top_p < 1.0) and _q_elt_bytes(w) > 0:
            for st, o in zip(self.sets, self.outs):
                n = o[1].long()
                rej = n < w.gamma
                if rej.any():
                    rows = st["logits"][torch.nonzero(rej).flatten(), n[rej]]
                    kept += int(kept_counts(rows, w.temperature, w.top_k, w.top_p).sum().item())
        ab = algorithmic_bytes(w, nacc, kept_rejected=kept, gamma_b=gbs)
        ab = {k: v / self.n_sets for k, v in ab.items()}
        ab["kept_q_reads_per_step"] = kept / self.n_sets
        if w.ragged:
            positions = float(np.sum(gbs)) / self.n_sets + w.B
        else:
            positions = float(w.B * (w.gamma + 1))
        return ab, positions, acceptance_stats(w, self.outs, self.sets)


def acceptance_stats(w, outs, sets):
    """Empirical alpha (the mean acceptance probability a_i over the tested
    positions: E[min(1, p/q)] under d ~ q is sum_v min(p, q), the overlap the
    notes call alpha) and tokens per round, mean n + 1 against
    1 + sum_{k=1..gamma_b} prod_{i<k} a_i (an unbiased estimate of the
    expected count when the rows' acceptances are independent).  Greedy
    reports the tokens per round only."""
    n = np.concatenate([o[1].cpu().numpy() for o in outs]).astype(np.float64)
    res = {"tokens_per_round": {"empirical": float(np.mean(n + 1))}}
    if w.mode != "sample" or w.gamma == 0 or outs[0][2] is None:
        return res
    a = np.concatenate([o[2].cpu().numpy() for o in outs]).astype(np.float64)
    G = w.gamma
    gb = (np.concatenate([st["gamma_b"].cpu().numpy() for st in sets]) if w.ragged
          else np.full(len(n), G))
    mask = np.arange(G)[None, :] < gb[:, None]
    prod = np.cumprod(np.where(mask, a, 0.0), axis=1)          # prod_{i<=j} a_i
    pred = 1.0 + prod.sum(1)
    res["alpha"] = float(a[mask].mean())
    res["tokens_per_round"]["predicted"] = float(pred.mean())
    res["tokens_per_round"]["std_err"] = float(np.std(n + 1, ddof=1) / np.sqrt(len(n))) if len(n) > 1 else None
    res["sequences"] = int(len(n))
    return res


def roofline_block(w, ab, t_stream, t_final, kernel_names, peak, peak_kind):
    """The dominant kernel (the longer of the two timed intervals), its
    algorithmic bytes per launch, average launch time and the fraction of
    the measured copy bandwidth."""
    if len(kernel_names) == 1:
        # one kernel does the whole step (its final draw included)
        ab = dict(ab, stream=ab["stream"] + ab["final"], final=0.0)
        t_final = 0.0
    kern = "stream" if t_stream >= t_final else "final"
    kname = kernel_names[0] if kern == "stream" else _final_name(kernel_names)
    t_k = t_stream if kern == "stream" else t_final
    achieved = ab[kern] / t_k / 1e9
    return {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": _traffic(w.name, kname),
            "algorithmic_bytes_per_launch": ab[kern], "avg_launch_us": t_k * 1e6,
            "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured"
            else "fallback 6.8 TB/s"}


def _final_name(kernel_names):
    """The kernels after the streaming one (timed together by the hook)."""
    return "+".join(kernel_names[1:])


def _kernel_us(kernel_names, t_stream, t_final):
    d = {kernel_names[0]: t_stream * 1e6}
    if len(kernel_names) >= 2:
        d[_final_name(kernel_names)] = t_final * 1e6
    return d


def run_gb300(args, rank, ws_n, local):
    import speculative_decoding_verification_46_gb300 as sv

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sv.load_library()
    w = workloads.WORKLOADS[args.workload]
    if args.batch is not None:
        w = w.with_(B=args.batch, name=f"{w.name}@B={args.batch}")
    B, G, V = w.B, w.gamma, w.V
    rn = Runner(sv, w, dev)
    stream = rn.stream

    all_kernels, kernel_names = rn.kernels()   # what one call launches (the path the library chose)
    kernels_per_call = len(all_kernels) + (1 if w.ragged else 0)   # + the truncation kernel
    if kernels_per_call == 0:
        raise RuntimeError("the verify call launched no kernel")
    rn.eager(rn.n_sets)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rn.eager(rn.n_sets)
    torch.cuda.synchronize()
    est = (time.perf_counter() - t0) / rn.n_sets
    steps = args.steps if args.steps is not None else int(min(200_000, max(200, 1.0 / max(est, 1e-6))))
    warmup = args.warmup if args.warmup is not None else max(3, min(steps // 10, 1000))

    rn.prepare(warmup)
    rn.prepare(steps)
    rn.run_steps(warmup)
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    _barrier(ws_n)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        rn.run_steps(steps)
        e1.record(stream)
    torch.cuda.synchronize()
    _barrier(ws_n)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / steps
    ms_max = max_over_ranks(ms, ws_n, dev)

    # per-kernel durations (timing hook), bytes, acceptance statistics
    t_stream, t_final = rn.kernel_times(4, 100)
    ab, positions, acc = rn.accounting()
    value = positions * ws_n / (ms_max / 1e3)
    peak, peak_kind = _peaks()
    roof = roofline_block(w, ab, t_stream, t_final, kernel_names, peak, peak_kind)
    step_gbs = (ab["stream"] + ab["final"]) / (ms / 1e3) / 1e9

    # end to end: pinned host inputs -> device, the call, outputs -> host, every
    # step.  The step's inputs sit in one pinned host buffer and its outputs in
    # one device buffer (views at 256-byte offsets), so one copy moves each way;
    # copy in, call, copy out are captured in a CUDA graph replayed per step.
    # q (the draft's probabilities) may stay in pinned host memory: the
    # kernels read it in place, only where the method needs it (q(d_i), the
    # kept candidates, a rejected sequence's residual row).  Both ways are
    # measured; the headline e2e leaves q on the host.
    def e2e_run(q_in_place):
        ins = dict(rn.sets[0])
        if w.mode == "greedy":
            ins["uniforms"] = None                 # greedy reads no uniforms
        q_host = None
        if q_in_place and ins.get("q") is not None:
            q_host = ins.pop("q").cpu().pin_memory()
        host_in, dev_in_buf, dev_in = _packed(ins, dev)
        if q_host is not None:
            dev_in["q"] = q_host
        out_named = {str(i): x for i, x in enumerate(rn.outs[0])}
        if w.mode == "greedy":
            out_named["2"] = None                  # greedy writes no accept_prob
        host_out, dev_out_buf, dev_out_v = _packed(out_named, dev)
        dev_out = tuple(dev_out_v[str(i)] for i in range(len(rn.outs[0])))
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for _ in range(3):
                dev_in_buf.copy_(host_in, non_blocking=True)
                _call(sv, w, dev_in, dev_out, rn.ws, stream)
                host_out.copy_(dev_out_buf, non_blocking=True)
        torch.cuda.synchronize()
        with torch.cuda.graph(g_e2e, stream=stream):
            dev_in_buf.copy_(host_in, non_blocking=True)
            _call(sv, w, dev_in, dev_out, rn.ws, stream)
            host_out.copy_(dev_out_buf, non_blocking=True)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for _ in range(3):
                g_e2e.replay()
        torch.cuda.synchronize()
        est_e2e = (time.perf_counter() - t0) / 3
        n_e2e = max(3, min(steps, 2000, int(2.0 / max(est_e2e, 1e-6))))
        with torch.cuda.stream(stream):
            f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            f0.record(stream)
            for _ in range(n_e2e):
                g_e2e.replay()
            f1.record(stream)
        torch.cuda.synchronize()
        ms_e2e = max_over_ranks(f0.elapsed_time(f1) / n_e2e, ws_n, dev)
        res = (ms_e2e, n_e2e, host_in.numel(), host_out.numel(), q_host is not None)
        del host_in, dev_in_buf, host_out, dev_out_buf, g_e2e, q_host
        return res

    pos_e2e = float((rn.sets[0]["gamma_b"].sum() + B).item()) if w.ragged else positions   # the input set used
    ms_e2e, n_e2e, h2d_copied, d2h, q_kept_on_host = e2e_run(True)
    ms_all, n_all, h2d_all = (e2e_run(False)[:3] if q_kept_on_host else (ms_e2e, n_e2e, h2d_copied))
    # q bytes the kernels read across the host link (the method's q reads,
    # for the input set used)
    q_link = 0
    if q_kept_on_host:
        q_link = q_bytes_read(w, rn.outs[0][1].cpu().numpy(), rn.sets[0], kept_rows_q(w, rn.sets[0], rn.outs[0]))
    e2e = {"value": pos_e2e * ws_n / (ms_e2e / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d_copied + q_link,
           "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e, "steps": n_e2e,
           "h2d_copied_bytes": h2d_copied, "q_read_in_place_bytes": q_link,
           "how": ("logits, drafts and uniforms in one pinned host buffer copied in; q left in pinned host "
                   "memory and read in place by the kernels; outputs in one device buffer copied out; "
                   "captured in a CUDA graph and replayed once per step") if q_kept_on_host else
                  ("inputs in one pinned host buffer, outputs in one device buffer; copy in, call, copy out "
                   "captured in a CUDA graph and replayed once per step"),
           "all_inputs_copied": {"value": pos_e2e * ws_n / (ms_all / 1e3), "ms_per_step": ms_all,
                                 "h2d_bytes_per_step": h2d_all, "steps": n_all}}

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
        "dtype_note": "float32 arithmetic (two-float sums where a draw is decided) on "
                      f"{w.dtype} logits",
        "data": "synthetic",
        "config": {
            "workload": w.name, "B": B, "gamma": G, "V": V, "logits_dtype": w.dtype, "mode": w.mode,
            "temperature": w.temperature, "top_k": w.top_k, "top_p": w.top_p,
            "parallelism": f"replicas x{ws_n} (batch per GPU fixed)",
            "l2": f"no flush: {rn.n_sets} rotating input sets of {rn.per_set / 1e6:.2f} MB (> 2x L2)",
            "timing": f"CUDA graphs of calls replayed ({steps // rn.n_sets} x {rn.n_sets} calls"
                      + (f" + 1 x {steps % rn.n_sets}" if steps % rn.n_sets else "")
                      + "), CUDA events on the launching stream",
        },
        "hbm_gbs": step_gbs,
        "hbm_frac_of_peak": step_gbs / peak,
        "roofline": roof,
        "kernel_us": _kernel_us(kernel_names, t_stream, t_final),
        "algorithmic_bytes_per_step": ab,
        "acceptance": acc,
        "e2e": e2e,
        "gpu_launches": steps * kernels_per_call,
        "clocks": clk,
    }
    del rn
    torch.cuda.empty_cache()
    return line, w


def other_workloads(args, local):
    """Short device-side runs of the other workloads (graph replay, rotating
    input sets, no flush), each ~0.3 s of timed work: value, ms/step, HBM GB/s
    and the fraction of the measured peak for the whole step, the roofline of
    the dominant kernel, the acceptance statistics and a parity sample."""
    import speculative_decoding_verification_46_gb300 as sv

    dev = torch.device("cuda", local)
    peak, peak_kind = _peaks()
    out = {}
    for name, w in workloads.WORKLOADS.items():
        if name == args.workload:
            continue
        rn = Runner(sv, w, dev, max_sets=512)
        _, kernel_names = rn.kernels()
        rn.prepare(rn.n_sets)
        rn.run_steps(rn.n_sets)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        rn.run_steps(rn.n_sets)
        torch.cuda.synchronize()
        reps = max(1, int(0.3 / max(time.perf_counter() - t0, 1e-6)))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(rn.stream):
            e0.record(rn.stream)
            rn.run_steps(reps * rn.n_sets)
            e1.record(rn.stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / (reps * rn.n_sets)
        t_stream, t_final = rn.kernel_times(2, 50)
        ab, pos, acc = rn.accounting()
        gbs = (ab["stream"] + ab["final"]) / (ms / 1e3) / 1e9
        out[name] = {"value": pos / (ms / 1e3), "ms_per_step": ms, "hbm_gbs": gbs,
                     "frac_of_measured_peak": gbs / peak, "steps": reps * rn.n_sets,
                     "roofline": roofline_block(w, ab, t_stream, t_final, kernel_names, peak, peak_kind),
                     "kernel_us": _kernel_us(kernel_names, t_stream, t_final), "acceptance": acc}
        del rn
        torch.cuda.empty_cache()
        if not args.no_cpu_baseline:
            out[name]["parity"] = parity_sample(w, 2.0, dev)[0]
    return out


# ---------------------------------------------------------------- the oracle legs

def _oracle_one(svref, w, h, b):
    """The oracle on sequence b of the host inputs h."""
    sl = slice(b, b + 1)
    if w.mode == "greedy":
        return svref.verify_greedy(h["L"][sl], h["d"][sl])
    if w.ragged:
        # the round ends at stop tokens / budgets, as the GPU call does
        r = svref.verify_sample_ragged(h["L"][sl], h["q"][sl] if h["q"] is not None else None, h["d"][sl],
                                       h["u"][sl], w.temperature, h["gb"][sl], w.top_k, w.top_p)
        r["out_tokens"], _ = svref.truncate_emitted(r["out_tokens"], r["n_accepted"], h["stops"], h["mx"][sl])
        return r
    if w.qlogits:
        return svref.verify_sample_qlogits(h["L"][sl], h["ql"][sl], h["d"][sl], h["u"][sl], w.temperature,
                                           w.top_k, w.top_p)
    return svref.verify_sample(h["L"][sl], h["q"][sl] if h["q"] is not None else None, h["d"][sl], h["u"][sl],
                               w.temperature, w.top_k, w.top_p)


def _host_inputs(inp, w):
    return {"L": inp["logits"].float().cpu().numpy(), "d": inp["draft"].cpu().numpy(),
            "u": inp["uniforms"].cpu().numpy(),
            "q": inp["q"].cpu().numpy() if inp.get("q") is not None else None,
            "ql": inp["q_logits"].float().cpu().numpy() if w.qlogits else None,
            "gb": inp["gamma_b"].cpu().numpy() if w.ragged else None,
            "stops": inp["stop_tokens"].cpu().numpy() if w.ragged else None,
            "mx": inp["max_new"].cpu().numpy() if w.ragged else None}


def parity_sample(w, budget_s: float, dev):
    """The GPU path and the oracle on the same inputs (seed + 7): the GPU call
    over the whole batch, the oracle on sequences 0, 1, ... for about
    budget_s seconds.  Returns (parity counts, oracle positions/s, sample
    description).  A draw is an evaluated accept test or the final draw; a
    boundary draw is one the oracle flags within 1e-6 of a decision boundary
    (with q from draft logits also within the wider absolute band on the final
    draw's CDF step, counted separately); a hard mismatch is a differing
    sequence with no boundary draw."""
    import speculative_decoding_verification_46_gb300 as sv
    from oracle import svref

    inp = workloads.make_inputs(w, seed=w.seed + 7, device=dev)
    G = w.gamma
    ws = _workspace(sv, w, w.B, G, w.V, dev)
    out = (torch.empty(w.B, G + 1, dtype=torch.int32, device=dev), torch.empty(w.B, dtype=torch.int32, device=dev),
           torch.empty(w.B, G, dtype=torch.float32, device=dev) if w.mode == "sample" and G > 0 else None,
           torch.empty(w.B, dtype=torch.int32, device=dev))
    stream = torch.cuda.current_stream(dev)
    _call(sv, w, inp, out, ws, stream)
    torch.cuda.synchronize()
    tok = out[0].cpu().numpy()
    n = out[1].cpu().numpy()
    a = out[2].cpu().numpy() if out[2] is not None else None
    h = _host_inputs(inp, w)
    del inp, ws
    c = dict(sequences=0, draws=0, hard_mismatches=0, boundary_flagged=0, boundary_mismatches=0,
             max_rel_err_accept_prob=0.0)
    if w.qlogits:
        c["widened_band_only"] = 0
    seqs, t0 = 0, time.perf_counter()
    while seqs < w.B:
        r = _oracle_one(svref, w, h, seqs)
        b = seqs
        seqs += 1
        rt = r["out_tokens"][0].copy()
        rn_ = int(r["n_accepted"][0])
        bad = (int(r["status"][0]) & svref.SEQ_BAD_ROW) != 0
        if not bad:
            gtok = tok[b]
            mism = (not np.array_equal(gtok, rt)) or int(n[b]) != rn_
            bnd = bool(r["boundary"][0]) if "boundary" in r else False
            c["sequences"] += 1
            gbb = int(h["gb"][b]) if w.ragged else G
            c["draws"] += (min(rn_ + 1, gbb) + 1) if w.mode == "sample" else 1
            c["boundary_flagged"] += int(bnd)
            c["hard_mismatches"] += int(mism and not bnd)
            c["boundary_mismatches"] += int(mism and bnd)
            if w.qlogits and "qlogits_band_only" in r:
                c["widened_band_only"] += int(r["qlogits_band_only"][0])
            if a is not None and "accept_prob" in r and gbb > 0:
                ar = r["accept_prob"][0][:gbb]
                ag = a[b][:gbb].astype(np.float64)
                rel = np.abs(ag - ar) / np.maximum(np.abs(ar), 1e-300)
                rel[(np.abs(ag - ar) <= 1e-30)] = 0.0
                c["max_rel_err_accept_prob"] = max(c["max_rel_err_accept_prob"], float(rel.max(initial=0.0)))
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    c["boundary_mismatch_frac"] = c["boundary_mismatches"] / max(c["draws"], 1)
    c["limit"] = BOUNDARY_LIMIT
    c["tolerance"] = ("greedy bit-exact" if w.mode == "greedy" else
                      "accept_prob 1e-5 relative; tokens and counts exact except draws within 1e-6 of a boundary")
    pos = seqs * (G + 1)
    return c, pos / el, f"sequences 0..{seqs - 1} of one batch ({pos} positions) in {el:.2f} s, numpy float64"


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
        h = _host_inputs(inp, w)
        del inp
        # one step = a bounded sample of the batch (at most ~2 s of oracle work)
        t0 = time.perf_counter()
        _oracle_one(svref, w, h, 0)
        per_seq = time.perf_counter() - t0
        per_step_budget = min(2.0, 120.0 / max(1, steps + warmup))
        nseq = int(max(1, min(w.B, per_step_budget / max(per_seq, 1e-6))))

        def step():
            for b in range(nseq):
                _oracle_one(svref, w, h, b)

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
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        par, v, sample = parity_sample(w, args.cpu_seconds, torch.device("cuda", local))
        line["parity"] = par
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
                                "host": platform.machine(), "host_cpus": os.cpu_count()}
    if rank == 0 and ws_n == 1 and not args.no_other_workloads and args.batch is None:
        line["other_workloads"] = other_workloads(args, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws_n > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
