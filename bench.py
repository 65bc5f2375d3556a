#!/usr/bin/env python
"""Benchmark of one EAGLE-style verify/accept step on GB300.

A step is one pass of the whole hot path over one batch: spec_select_topk x S,
spec_build_tree, spec_verify_attention, spec_verify_greedy (or
spec_verify_sampling) and spec_commit_kv.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--configs all|headline|a,b,..] [--impl ours|reference]

The headline workload is sampling_heavy (2048 verify tokens per step, the
largest of the five, on the sampling path).  At N=1 the other four workloads
are measured the same way and reported in the line's "configs" object.

Timing, per workload: W warm-up steps, then K steps replayed from CUDA graphs
of P consecutive steps each (P <= 4 divides K; consecutive steps use different
input replicas, whose combined size exceeds the 129 MB L2), bracketed by a
barrier and torch.cuda.synchronize() on both sides, CUDA events on the
launching stream, max over ranks.  Every kernel waits for the one before it
(the library's default): this is the step an EAGLE loop gets, where the draft
forward and the target's LM head run between the library's calls.  The same
steps with overlap allowed (spec_workspace_set_overlap: a select or a greedy
accept reads its input before the kernel ahead finishes) are timed too and
reported as step_us_overlap.  Per-call durations (for the roofline) come from
a separate pass right after the timed region: one-step graphs with CUDA
events between the calls, each step on its own replica and run alone (the
events remove the overlap of consecutive launches, so these durations are
upper bounds).  Under torchrun each rank verifies its own batch of the
headline workload (weak scaling, no collective on the data path).
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
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verify-step µs and verified tree tokens/s; % of GB300 HBM/tensor roofline"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
HEADLINE = "sampling_heavy"
ALL_CONFIGS = ["sampling_heavy", "llama8b_greedy", "long_context", "mtp_chain", "tiny"]
GROUPS = ["select", "build", "attention", "accept", "commit"]
L2_BYTES = 129e6


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=HEADLINE, help="the headline workload")
    ap.add_argument("--configs", default="all",
                    help="workloads measured at N=1: all (the five), headline, or a comma list")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--replicas", type=int, default=0, help="input replicas cycled by the timed steps (0: auto)")
    ap.add_argument("--graphs", type=int, default=64, help="distinct captured step graphs")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-overlap-variant", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=20.0,
                    help="seconds of oracle work for the headline's CPU baseline (a quarter for the others)")
    ap.add_argument("--reference-budget-s", type=float, default=100.0,
                    help="seconds of oracle work the reference arm spreads over its W + K steps")
    return ap.parse_args(argv)


# --------------------------------------------------------------- helpers

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def job_elapsed_ms(elapsed_ms, world, device, torch):
    """The job's elapsed time: the slowest rank's (every rank verifies its own
    batch; the job ends when the last one does)."""
    if world <= 1:
        return float(elapsed_ms)
    tt = torch.tensor([float(elapsed_ms)], device=device)
    torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
    return float(tt.item())


def job_tokens_per_s(b, n, steps, world, elapsed_ms):
    """Verified tree tokens of all ranks (weak scaling: b*n per rank per step)
    over the job's elapsed time."""
    return b * n * steps * world / (elapsed_ms / 1e3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while running (100 ms period)."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.samples.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        reasons = set()
        for s in self.samples:
            for name, val in zip(["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"], s[5:]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for_smi(torch, dev_index: int) -> str:
    try:
        u = torch.cuda.get_device_properties(dev_index).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[dev_index]
        return str(dev_index)


def steps_per_graph(replicas: int, steps: int) -> int:
    """Consecutive steps captured in one timed graph: at most 4 and at most the
    number of input replicas (consecutive steps then read different inputs),
    and a divisor of the timed step count, so that exactly `steps` run."""
    P = max(1, min(replicas, 4, steps))
    while steps % P:
        P -= 1
    return P


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


CSRC = "accept_select_top_gb300/csrc/"
# the sources each group's kernels compile from (common.cuh: helpers inlined in every kernel)
GROUP_SOURCES = {
    "select": [CSRC + "select_topk.cu", CSRC + "stream_records.cu", CSRC + "stream_records.cuh", CSRC + "common.cuh"],
    "build": [CSRC + "build_tree.cu", CSRC + "common.cuh"],
    "attention": [CSRC + "attention_tc.cu", CSRC + "common.cuh"],
    "accept": [CSRC + "verify_greedy.cu", CSRC + "verify_sampling.cu", CSRC + "stream_records.cu",
               CSRC + "stream_records.cuh", CSRC + "common.cuh"],
    "commit": [CSRC + "commit_kv.cu", CSRC + "common.cuh"],
}


def traffic_entry(group: str, workload: str):
    """DRAM bytes per step of a kernel group from the committed ncu summary,
    when it was taken on the current source of its kernels; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    e = table.get(f"{group}:{workload}")
    if not e or e.get("source_hash") != source_hash(GROUP_SOURCES[group]):
        return None
    return e


def selected_configs(args, world):
    if world > 1 or args.configs == "headline":
        return [args.workload]
    if args.configs == "all":
        names = [args.workload] + [c for c in ALL_CONFIGS if c != args.workload]
    else:
        names = [args.workload] + [c for c in args.configs.split(",") if c and c != args.workload]
    return names


# ------------------------------------------------------- workload setup

def accept_mode(wl):
    return "greedy" if wl.accept == "greedy" else "sampling"


def temps_mode(wl):
    return {"sampling": "sampling", "mixed": "mixed", "both": "sampling"}[wl.accept]


def prepare(wl, device, seed, torch):
    """Inputs on the device; the draft tree comes from one untimed GPU pass of
    select + build, and the target logits are drawn against that tree."""
    from accept_select_top_gb300 import workloads as W
    from accept_select_top_gb300.pipeline import DeviceInputs, VerifyStep

    mode = accept_mode(wl)
    drafts = [W.draft_logits(wl, i, device, seed) for i in range(wl.S)]
    lay = W.kv_layout(wl, seed)
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a)).to(device)
    att = W.attention_tensors(wl, int(lay["num_slots"]), device, seed)
    inp = DeviceInputs(drafts, W.bonus_tokens(wl, device, seed), t(lay["seq_lens"]), t(lay["req_pool_idx"]),
                       t(lay["req_to_token"]), t(lay["verify_loc"]), att["q"], att["k_pool"], att["v_pool"],
                       int(lay["seq_lens"].max()))
    probe = VerifyStep(wl, inp, mode, device=device)
    probe.select()
    probe.build()
    torch.cuda.synchronize()
    h = lambda x: x.detach().cpu().numpy()
    dt, nt, ns = h(probe.draft_tokens), h(probe.next_token), h(probe.next_sibling)
    all_d = torch.cat(drafts, 0)
    rows = W.draft_rows_of_nodes(wl, dt, nt, ns, h(probe.token_space), h(probe.parent_space))
    logits = W.target_logits(wl, rows, all_d, device, seed)
    if wl.agreement == "planted":
        logits = W.plant_agreement(wl, logits, dt, nt, ns, seed)
    inp.target_logits = logits
    if mode == "sampling":
        temps = W.request_temperatures(wl, temps_mode(wl))
        inp.temperatures = t(temps)
        inp.draft_probs = W.draft_probs(wl, rows, all_d, temps, device)
        inp.u, inp.u_final = W.coins(wl, device, seed)
    del probe
    return mode, inp, lay


def clone_inputs(inp, torch):
    from accept_select_top_gb300.pipeline import DeviceInputs
    c = lambda x: None if x is None else x.clone()
    return DeviceInputs([d.clone() for d in inp.drafts], c(inp.bonus), c(inp.seq_lens), c(inp.req_pool_idx),
                        c(inp.req_to_token), c(inp.verify_loc), c(inp.q), c(inp.k_pool), c(inp.v_pool),
                        inp.max_seq_len, c(inp.target_logits), c(inp.draft_probs), c(inp.temperatures), c(inp.u),
                        c(inp.u_final))


def group_bytes(wl, lay, mode, accept_lens):
    """Algorithmic bytes of each kernel group per step: what the method itself
    must move (each input read once, each output written once)."""
    es = 4 if wl.logits_dtype == "f32" else 2
    seq = lay["seq_lens"].astype(np.int64)
    b, n, k = wl.b, wl.n, wl.k
    kv_row = wl.Hkv * wl.D * 2
    out = {
        # every draft row once, plus each step's blocks
        "select": sum(wl.rows(i) * wl.V * es for i in range(wl.S)),
        # the score / token spaces and parent list in, the tree arrays and the mask out
        "build": b * (wl.C * 8 + wl.P * 4 + n * (4 * 5 + 8)),
        # the visible K/V rows once, Q in, O and LSE out, the slot ids
        "attention": int((seq.sum() + b * n) * kv_row * 2 + 2 * b * n * wl.Hq * wl.D * 2 + b * n * wl.Hq * 4
                         + (seq.sum() + b * n) * 4),
        # every verify row's logits once (argmax / softmax of all b*n rows)
        "accept": b * n * wl.V * es,
        # accepted K and V rows read and written
        "commit": int(np.sum(accept_lens)) * kv_row * 2 * 2,
    }
    if mode == "sampling":
        out["accept"] += b * n * 4 + b * wl.V * (es + 4)  # candidate q reads + one terminal row (logits and q)
    return out


def attention_flops(wl, lay, mask_bits):
    """4 * D per visible (query row, key) pair, over every q head."""
    seq = lay["seq_lens"].astype(np.int64)
    vis = np.array([bin(int(m) & ((1 << 64) - 1)).count("1") for m in mask_bits], np.int64).reshape(wl.b, wl.n)
    keys = (seq[:, None] + vis).sum()
    return float(4 * wl.D * wl.Hq * keys)


def roofline(group, t_us, bytes_, flops, peaks, peaks_kind):
    """The roofline object of one kernel group: HBM-bound unless it is the
    attention with an arithmetic intensity above the ridge."""
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if group == "attention" and flops / bytes_ > ridge:
        ach = flops / (t_us * 1e-6) / 1e12
        peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
        return {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                "peak_kind": f"{peaks_kind} bf16 (sustained)"}
    ach = bytes_ / (t_us * 1e-6) / 1e9
    peak = peaks["hbm_gbs"]
    return {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
            "peak_kind": f"{peaks_kind} copy bandwidth"}


# --------------------------------------------------------- one workload

class ConfigRun:
    """One workload on one GPU: R input replicas (each with its own KV pools),
    one VerifyStep per replica, a private stream."""

    def __init__(self, wl, device, seed, torch, replicas=0):
        from accept_select_top_gb300.pipeline import VerifyStep
        self.torch, self.wl, self.device = torch, wl, device
        self.mode, inp, self.lay = prepare(wl, device, seed, torch)
        nbytes = lambda x: 0 if x is None else x.numel() * x.element_size()
        per_replica = (sum(nbytes(d) for d in inp.drafts) + nbytes(inp.target_logits) + nbytes(inp.k_pool)
                       + nbytes(inp.v_pool) + nbytes(inp.q) + nbytes(inp.draft_probs))
        self.R = replicas or max(2, min(8, math.ceil(4 * L2_BYTES / per_replica)))
        self.inputs = [inp] + [clone_inputs(inp, torch) for _ in range(self.R - 1)]
        self.steps = [VerifyStep(wl, x, self.mode, device=device) for x in self.inputs]
        self.stream = torch.cuda.Stream(device=device)
        # inputs, clones and workspace zero fills were enqueued on the default
        # stream; the steps run on self.stream, which is not ordered after it
        torch.cuda.synchronize()

    def set_overlap(self, on):
        for s in self.steps:
            s.ws.set_overlap(on)

    def warmup(self, n):
        torch = self.torch
        with torch.cuda.stream(self.stream):
            for i in range(n):
                self.steps[i % self.R].run()
        torch.cuda.synchronize()
        assert self.steps[0].ws.last_error() == 0, "device error word set during warm-up"

    def capture(self, K, graphs_max):
        """Graphs of P consecutive steps (one per replica, so every step reads
        inputs the previous steps did not), holding only the kernels."""
        torch = self.torch
        P = steps_per_graph(self.R, K)
        G = max(1, min(graphs_max, K // P))
        graphs = []
        for j in range(G):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                for t in range(P):
                    self.steps[(j * P + t) % self.R].run()
            graphs.append(g)
        return graphs, P

    def replay(self, graphs, n):
        with self.torch.cuda.stream(self.stream):
            for i in range(n):
                graphs[i % len(graphs)].replay()

    def timed(self, graphs, P, K, world=1, barrier=None):
        torch = self.torch
        if barrier:
            barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            t0.record()
            for i in range(K // P):
                graphs[i % len(graphs)].replay()
            t1.record()
        torch.cuda.synchronize()
        if barrier:
            barrier()
        return t0.elapsed_time(t1)

    def per_call(self, M):
        """Per-call device durations (µs), each step alone on its replica, with
        events between the calls; averaged over M steps after one warm cycle."""
        torch = self.torch
        wl = self.wl
        try:
            torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return None
        names = [f"select{i}" for i in range(wl.S)] + ["build", "attention", "accept", "commit"]
        graphs, evs = [], []
        for j in range(self.R):
            s = self.steps[j]
            e = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(names) + 1)]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                e[0].record()
                s.select_step(0)
                e[1].record()
                for i in range(1, wl.S):
                    s.select_step(i)
                    e[i + 1].record()
                s.build()
                e[wl.S + 1].record()
                s.attention()
                e[wl.S + 2].record()
                s.accept()
                e[wl.S + 3].record()
                s.commit()
                e[wl.S + 4].record()
            graphs.append(g)
            evs.append(e)
        acc = {k: [] for k in names}
        with torch.cuda.stream(self.stream):
            for i in range(self.R + M):
                graphs[i % self.R].replay()
                torch.cuda.synchronize()
                if i >= self.R:
                    e = evs[i % self.R]
                    for c, k in enumerate(names):
                        acc[k].append(e[c].elapsed_time(e[c + 1]) * 1e3)
        per = {k: statistics.mean(v) for k, v in acc.items()}
        groups = {"select": sum(per[f"select{i}"] for i in range(wl.S)), "build": per["build"],
                  "attention": per["attention"], "accept": per["accept"], "commit": per["commit"]}
        return {"calls_us": per, "groups_us": groups}


def run_e2e(args, torch, wl, mode, step, stream, device):
    """Same step through the public API with host buffers: each step copies its
    inputs from pinned host memory to the device, runs the six calls eagerly,
    and copies its results back to pinned host memory.  Steps are pipelined the
    way a server would run them: two device input sets (sharing the resident KV
    pools and tables), a copy stream that fills set (i+1) % 2 while the compute
    stream runs step i on set i % 2, and events so that a set is overwritten
    only after the step that read it has finished."""
    import copy as _copy
    from accept_select_top_gb300.pipeline import VerifyStep
    inp = step.inp
    names = ["target_logits", "q", "bonus", "seq_lens"] + (["draft_probs", "u", "u_final", "temperatures"]
                                                             if mode == "sampling" else [])
    h_in = {k: getattr(inp, k).cpu().pin_memory() for k in names}
    h_drafts = [d.cpu().pin_memory() for d in inp.drafts]
    outs = ["accept_index", "accept_lens", "accepted_tokens", "next_root", "new_seq_lens", "free_ids", "n_free"]
    h_out = {k: torch.empty_like(getattr(step, k), device="cpu").pin_memory() for k in outs}
    h2d = sum(v.numel() * v.element_size() for v in h_in.values()) + sum(d.numel() * d.element_size()
                                                                         for d in h_drafts)
    d2h = sum(v.numel() * v.element_size() for v in h_out.values())
    K = max(8, min(args.steps, 50))

    inp1 = _copy.copy(inp)  # the copied inputs get buffers of their own; the rest is shared
    for k in names:
        setattr(inp1, k, torch.empty_like(getattr(inp, k)))
    inp1.drafts = [torch.empty_like(d) for d in inp.drafts]
    sets = [(inp, step), (inp1, VerifyStep(wl, inp1, mode, device=device))]
    torch.cuda.synchronize()  # the new step's workspace zero fill ran on the default stream
    copy_stream = torch.cuda.Stream(device)
    ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    for e in done:
        e.record(stream)

    def one(i):
        ip, st = sets[i % 2]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(done[i % 2])  # the step that last read this set is over
            for d, hd in zip(ip.drafts, h_drafts):
                d.copy_(hd, non_blocking=True)
            for k in names:
                getattr(ip, k).copy_(h_in[k], non_blocking=True)
            ready[i % 2].record(copy_stream)
        with torch.cuda.stream(stream):
            stream.wait_event(ready[i % 2])
            st.run()
            done[i % 2].record(stream)
            for k in outs:
                h_out[k].copy_(getattr(st, k), non_blocking=True)

    for i in range(4):
        one(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    copy_stream.wait_event(t0)  # no copy of the timed steps starts before the clock does
    for i in range(K):
        one(i)
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    return {"value": wl.b * wl.n * K / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": K, "ms_per_step": ms / K,
            "path": "ops.spec_* calls eagerly from Python, pinned host buffers; step i+1's host-to-device "
                    "copies (a copy stream, two device input sets) overlap step i's compute"}


def measure_config(name, args, torch, device, seed, world, peaks, peaks_kind, headline):
    """Everything measured for one workload: the timed steps (and the clocks
    around them for the headline), the same steps with overlap allowed, the
    per-call pass, e2e and the CPU baseline."""
    from accept_select_top_gb300 import workloads as W
    from accept_select_top_gb300.pipeline import launches_per_step, sampling_launches, select_launches
    rank = int(os.environ.get("RANK", 0))
    wl = W.WORKLOADS[name]
    run = ConfigRun(wl, device, seed, torch, args.replicas)
    W0 = max(3, args.warmup)
    run.warmup(W0)
    s0 = run.steps[0]
    mask_bits = s0.mask_bits.cpu().numpy()
    accept_lens = s0.accept_lens.cpu().numpy()
    K = args.steps
    graphs, P = run.capture(K, args.graphs)
    run.replay(graphs, W0)
    torch.cuda.synchronize()
    barrier = (lambda: torch.distributed.barrier()) if world > 1 else None
    sampler = None
    if headline and not args.no_clocks:
        sampler = ClockSampler(gpu_id_for_smi(torch, torch.cuda.current_device()))
        time.sleep(0.3)
    elapsed = run.timed(graphs, P, K, world, barrier)
    clocks = sampler.stop() if sampler is not None else None
    elapsed = job_elapsed_ms(elapsed, world, device, torch)
    assert s0.ws.last_error() == 0, "device error word set during the timed region"
    del graphs
    overlap_ms = None
    if not args.no_overlap_variant:
        run.set_overlap(True)
        og, OP_ = run.capture(K, args.graphs)
        run.replay(og, W0)
        overlap_ms = run.timed(og, OP_, K)
        run.set_overlap(False)
        del og
    calls = run.per_call(max(2 * run.R, min(K, 50)))
    bytes_ = group_bytes(wl, run.lay, run.mode, accept_lens)
    flops = attention_flops(wl, run.lay, mask_bits)
    kernels = None
    roof = None
    if calls is not None:
        kernels = {}
        for g in GROUPS:
            r = roofline(g, calls["groups_us"][g], bytes_[g], flops, peaks, peaks_kind)
            r.update({"us": calls["groups_us"][g], "algorithmic_bytes": int(bytes_[g])})
            kernels[g] = r
        dom = max(GROUPS, key=lambda g: calls["groups_us"][g])
        roof = {k: kernels[dom][k] for k in ("bound", "achieved", "peak", "unit", "frac")}
        tr = traffic_entry(dom, name)
        roof.update({"traffic": None if tr is None else tr["dram_bytes_per_launch"], "kernel": dom,
                     "kernel_us": kernels[dom]["us"], "algorithmic_bytes": kernels[dom]["algorithmic_bytes"],
                     "peak_kind": kernels[dom]["peak_kind"],
                     "launches": sum(select_launches(wl, i) for i in range(wl.S)) if dom == "select" else
                     (sampling_launches(wl) if dom == "accept" and run.mode == "sampling" else 1)})
        if dom == "attention":
            roof["flops"] = flops
    e2e = None if args.no_e2e else run_e2e(args, torch, wl, run.mode, s0, run.stream, device)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        budget = args.cpu_budget_s if headline else args.cpu_budget_s / 4
        cpu = cpu_baseline(wl, run.mode, s0, budget)
    ms_per_step = elapsed / K
    out = {
        "workload": name, "b": wl.b, "topk": wl.k, "num_steps": wl.S, "num_draft_tokens": wl.n, "vocab": wl.V,
        "heads": f"{wl.Hq}/{wl.Hkv}", "head_dim": wl.D, "page_size": wl.page_size, "context": list(wl.ctx),
        "accept": run.mode, "step_us": ms_per_step * 1e3,
        "tokens_per_s": job_tokens_per_s(wl.b, wl.n, K, world, elapsed),
        "step_us_overlap": None if overlap_ms is None else overlap_ms / K * 1e3,
        "mean_accept_lens": float(np.mean(accept_lens)),
        "kernels": kernels, "calls_us": None if calls is None else calls["calls_us"],
        "roofline": roof, "e2e": e2e, "cpu_baseline": cpu,
        "gpu_launches_per_step": launches_per_step(wl, run.mode),
        "replicas": run.R, "steps_per_graph": P, "steps": K,
        "l2": f"{run.R} rotating input replicas, each with its own KV pools (> 4x the 129 MB L2 per cycle)",
    }
    del run
    torch.cuda.empty_cache()
    return out, elapsed, clocks


# ------------------------------------------------- oracle (CPU baseline)

def oracle_sample(wl, mode, host, reqs, pair_frac, seed=0):
    """Runs the oracle over requests `reqs` end to end, the attention on a
    fraction of their (row, head) pairs, and returns per-stage seconds and the
    pairs done."""
    import oracle
    from accept_select_top_gb300.workloads import scaled
    n, V = wl.n, wl.V
    times = {"select_build": 0.0, "attention": 0.0, "accept_commit": 0.0}
    npairs_total = 0
    w1 = scaled(wl, b=1)
    rng = np.random.default_rng(seed)
    for r in reqs:
        rows = slice(r * n, (r + 1) * n)
        t = time.perf_counter()
        chain_steps, scores = [], None
        for i in range(wl.S):
            rr = slice(r * w1.rows(i), (r + 1) * w1.rows(i))
            o = oracle.select_topk(i, 1, wl.k, host["drafts"][i][rr], 1.0, scores)
            chain_steps.append(o)
            scores = o["scores_out"]
        score_space = np.ascontiguousarray(np.concatenate([s["score_blk"] for s in chain_steps], axis=1))
        token_space = np.ascontiguousarray(np.concatenate([s["token_blk"] for s in chain_steps], axis=1))
        parent_space = (np.ascontiguousarray(np.concatenate([s["parent_blk"] for s in chain_steps[:-1]], axis=1))
                        if wl.S > 1 else np.full((1, 1), -1, np.int32))
        tree = oracle.build_tree(1, wl.k, wl.S, n, score_space, token_space, parent_space,
                                 host["bonus"][r:r + 1], host["seq_lens"][r:r + 1])
        times["select_build"] += time.perf_counter() - t
        npairs = max(1, int(round(n * wl.Hq * pair_frac)))
        flat = rng.choice(n * wl.Hq, size=npairs, replace=False)
        pairs = np.stack([flat // wl.Hq, flat % wl.Hq], 1).astype(np.int32)
        t = time.perf_counter()
        oracle.verify_attention(1, n, wl.Hq, wl.Hkv, wl.D, host["q"][rows], host["k_pool"], host["v_pool"],
                                host["req_to_token"], host["req_pool_idx"][r:r + 1], host["seq_lens"][r:r + 1],
                                host["verify_loc"][rows], tree["mask_bits"], 1.0 / math.sqrt(wl.D), pairs=pairs)
        times["attention"] += time.perf_counter() - t
        npairs_total += npairs
        t = time.perf_counter()
        args = (tree["draft_tokens"], np.arange(n, dtype=np.int32), tree["next_token"], tree["next_sibling"])
        if mode == "greedy":
            acc = oracle.verify_greedy(1, n, wl.S, host["logits"][rows], *args)
        else:
            acc = oracle.verify_sampling(1, n, wl.S, host["logits"][rows], host["q_probs"][rows],
                                         host["temps"][r:r + 1], host["u"][rows], host["u_final"][r:r + 1], *args)
        oracle.commit_kv(1, n, wl.W, wl.Hkv, wl.D, wl.page_size, [host["k_pool"]], [host["v_pool"]],
                         host["req_to_token"], host["req_pool_idx"][r:r + 1], host["seq_lens"][r:r + 1],
                         host["verify_loc"][rows], acc["accept_index"], acc["accept_lens"])
        times["accept_commit"] += time.perf_counter() - t
    return times, npairs_total


def host_inputs(step, mode):
    from accept_select_top_gb300 import workloads as W
    inp = step.inp
    h = {"drafts": [W.host(d) for d in inp.drafts], "bonus": W.host(inp.bonus), "seq_lens": W.host(inp.seq_lens),
         "req_pool_idx": W.host(inp.req_pool_idx), "req_to_token": W.host(inp.req_to_token),
         "verify_loc": W.host(inp.verify_loc), "q": W.host(inp.q), "k_pool": W.host(inp.k_pool).copy(),
         "v_pool": W.host(inp.v_pool).copy(), "logits": W.host(inp.target_logits)}
    if mode == "sampling":
        h.update(q_probs=W.host(inp.draft_probs), temps=W.host(inp.temperatures), u=W.host(inp.u),
                 u_final=W.host(inp.u_final))
    return h


def pair_seconds(wl):
    """A rough cost of one (row, head) pair of the oracle's fp64 attention."""
    ctx = wl.ctx[1] if wl.ctx[0] == "fixed" else (wl.ctx[2] if wl.ctx[0] == "uniform" else max(wl.ctx[1]))
    return 4.0 * wl.D * (ctx + wl.n) * 2.5e-9


def pair_fraction(wl, budget_s, reqs):
    """The fraction of a request's (row, head) pairs whose attention fits in
    about half the budget for `reqs` requests."""
    return min(1.0, 0.5 * budget_s / max(1e-9, pair_seconds(wl) * reqs * wl.n * wl.Hq))


def scale_to_request(wl, times, nreq, npairs):
    """Seconds one full request costs the oracle: select/build and
    accept/commit per request, attention per (row, head) pair."""
    return ((times["select_build"] + times["accept_commit"]) / nreq
            + times["attention"] / npairs * wl.n * wl.Hq)


def cpu_baseline(wl, mode, step, budget_s):
    host = host_inputs(step, mode)
    reqs = list(range(min(wl.b, 2)))
    frac = pair_fraction(wl, budget_s, len(reqs))
    times, npairs = oracle_sample(wl, mode, host, reqs, frac)
    per_req = scale_to_request(wl, times, len(reqs), npairs)
    return {"value": wl.n / per_req, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"requests {reqs} of {wl.b} end to end, attention on {npairs} of "
                      f"{len(reqs) * wl.n * wl.Hq} (row, head) pairs; scaled by request and by pair",
            "sample_seconds": round(sum(times.values()), 2), "full_step_seconds_est": round(per_req * wl.b, 3)}


# ---------------------------------------------------------- reference arm

def host_prepare(wl, seed=0):
    """The workload's inputs drawn on the host, the draft tree and the target
    agreement from the oracle's own select chain: no GPU and no CUDA library."""
    import torch
    from accept_select_top_gb300 import workloads as W
    from oracle import pipeline as OP
    mode = accept_mode(wl)
    drafts_t = [W.draft_logits(wl, i, "cpu", seed) for i in range(wl.S)]
    drafts = [W.host(d) for d in drafts_t]
    lay = W.kv_layout(wl, seed)
    bonus = W.host(W.bonus_tokens(wl, "cpu", seed))
    chain = OP.select_chain(wl, drafts)
    tree = OP.tree_from_chain(wl, chain, bonus, lay["seq_lens"])
    rows = W.draft_rows_of_nodes(wl, tree["draft_tokens"], tree["next_token"], tree["next_sibling"],
                                 chain["token_space"], chain["parent_space"])
    all_d = torch.cat(drafts_t, 0)
    logits = W.target_logits(wl, rows, all_d, "cpu", seed)
    if wl.agreement == "planted":
        logits = W.plant_agreement(wl, logits, tree["draft_tokens"], tree["next_token"], tree["next_sibling"], seed)
    att = W.attention_tensors(wl, int(lay["num_slots"]), "cpu", seed)
    host = {"drafts": drafts, "bonus": bonus, "seq_lens": lay["seq_lens"], "req_pool_idx": lay["req_pool_idx"],
            "req_to_token": lay["req_to_token"], "verify_loc": lay["verify_loc"], "q": W.host(att["q"]),
            "k_pool": W.host(att["k_pool"]).copy(), "v_pool": W.host(att["v_pool"]).copy(),
            "logits": W.host(logits)}
    if mode == "sampling":
        temps = W.request_temperatures(wl, temps_mode(wl))
        u, uf = W.coins(wl, "cpu", seed)
        host.update(q_probs=W.host(W.draft_probs(wl, rows, all_d, temps, "cpu")), temps=temps, u=W.host(u),
                    u_final=W.host(uf))
    return mode, host


def run_reference(args):
    """The oracle, as it stands, on the host cores (one thread) for the same
    workload, metric and unit.  Each of the W + K steps is one request of the
    batch (cycling through a few) end to end, with the attention on a fraction
    of its (row, head) pairs sized so that the whole run spends about
    --reference-budget-s seconds; every step's wall time is measured.  The
    value scales each step's stages to one full request (select/build and
    accept/commit per request, attention per pair) and counts its n tokens."""
    from accept_select_top_gb300 import workloads as W
    wl_full = W.WORKLOADS[args.workload]
    nreq = min(wl_full.b, 4)
    wl = W.scaled(wl_full, b=nreq)  # a few requests of the same recipe, drawn on the host
    t_setup = time.perf_counter()
    mode, host = host_prepare(wl, 0)
    setup_s = time.perf_counter() - t_setup
    Wn, K = max(3, args.warmup), args.steps
    per_step = args.reference_budget_s / (Wn + K)
    frac = pair_fraction(wl, per_step, 1)
    walls, per_req = [], []
    for i in range(Wn + K):
        t = time.perf_counter()
        times, npairs = oracle_sample(wl, mode, host, [i % nreq], frac, seed=i)
        wall = time.perf_counter() - t
        if i >= Wn:
            walls.append(wall)
            per_req.append(scale_to_request(wl, times, 1, npairs))
    sec_per_req = sum(per_req) / len(per_req)
    sample = (f"each step one request (of {nreq} drawn on the host with the {args.workload} recipe) end to end, "
              f"attention on {npairs} of {wl.n * wl.Hq} (row, head) pairs; value scales each step to one full "
              f"request ({wl.n} tokens)")
    return wl_full, sec_per_req, sum(walls) / len(walls), sample, setup_s


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    peaks, peaks_kind = load_peaks()
    if args.impl == "reference":
        if rank != 0:
            return 0
        wl, sec_req, wall, sample, setup_s = run_reference(args)
        val = wl.n / sec_req
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": wall * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (drawn on the host)",
            "config": {"workload": args.workload, "b": wl.b, "topk": wl.k, "num_steps": wl.S,
                       "num_draft_tokens": wl.n, "vocab": wl.V},
            "full_batch_step_s_est": sec_req * wl.b, "setup_s": round(setup_s, 2),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return 0

    import torch
    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    names = selected_configs(args, world)
    results, head_elapsed, head_clocks = {}, None, None
    for name in names:
        headline = name == names[0]
        out, elapsed, clocks = measure_config(name, args, torch, device, rank, world, peaks, peaks_kind, headline)
        results[name] = out
        if headline:
            head_elapsed, head_clocks = elapsed, clocks
    if rank != 0:
        return 0
    h = results[names[0]]
    line = {
        "metric": METRIC, "value": h["tokens_per_s"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": head_elapsed / args.steps, "step_us": h["step_us"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded draws; target agreement planted / correlated per the workload recipe)",
        "config": {"workload": names[0], "b": h["b"], "topk": h["topk"], "num_steps": h["num_steps"],
                   "num_draft_tokens": h["num_draft_tokens"], "vocab": h["vocab"], "heads": h["heads"],
                   "head_dim": h["head_dim"], "page_size": h["page_size"], "context": h["context"],
                   "accept": h["accept"], "parallelism": f"replicas x{world}", "l2": h["l2"],
                   "steps_per_graph": h["steps_per_graph"],
                   "timing": "every kernel waits for the one before it (no overlap: the EAGLE-loop step); "
                             "step_us_overlap: the same steps with overlap allowed",
                   "kernel_timing": "separate pass after the timed region: one-step graphs with events between "
                                    "the calls, each step alone on its replica"},
        "step_us_overlap": h["step_us_overlap"], "mean_accept_lens": h["mean_accept_lens"],
        "roofline": h["roofline"], "kernels": h["kernels"], "cpu_baseline": h["cpu_baseline"], "e2e": h["e2e"],
        "gpu_launches": h["gpu_launches_per_step"] * args.steps, "clocks": head_clocks,
        "configs": {k: v for k, v in results.items() if k != names[0]},
    }
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
