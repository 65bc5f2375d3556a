#!/usr/bin/env python
"""Benchmark of one EAGLE-style verify/accept step on GB300.

A step is one pass of the whole hot path over one batch: spec_select_topk x S,
spec_build_tree, spec_verify_attention, spec_verify_greedy (or
spec_verify_sampling) and spec_commit_kv.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Timing: W warm-up steps, then K steps replayed from CUDA graphs of P
consecutive steps each (P <= 4 divides K; consecutive steps use different
input replicas, whose combined size exceeds the 129 MB L2), bracketed by a
barrier and torch.cuda.synchronize() on both sides, CUDA events on the
launching stream, max over ranks.  The timed graphs hold only the kernels, so
consecutive kernels overlap as they do for a caller running steps back to
back.  Stage durations (for the roofline) come from a second pass right after
the timed region: one-step graphs with CUDA events at the stage boundaries,
each step run alone (the events and the per-step synchronisation remove the
overlap across stages, so these durations are upper bounds).  Under torchrun
each rank verifies its own batch (weak scaling, no collective on the data
path).
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


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="llama8b_greedy")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--replicas", type=int, default=0, help="input replicas cycled by the timed steps (0: auto)")
    ap.add_argument("--graphs", type=int, default=64, help="distinct captured step graphs")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
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


def traffic_entry(kernel_key: str, sources):
    """DRAM bytes per launch from the committed ncu summary, when it was taken
    on the current source of the kernel; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    e = table.get(kernel_key)
    if not e or e.get("source_hash") != source_hash(sources):
        return None
    return e


# ------------------------------------------------------- workload setup

def prepare(wl, device, seed, torch):
    """Inputs on the device; the draft tree comes from one untimed GPU pass of
    select + build, and the target logits are drawn against that tree."""
    from accept_select_top_gb300 import workloads as W
    from accept_select_top_gb300.pipeline import DeviceInputs, VerifyStep

    mode = "greedy" if wl.accept == "greedy" else "sampling"
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
        temps = W.request_temperatures(wl, {"sampling": "sampling", "mixed": "mixed", "both": "sampling"}[wl.accept])
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


def step_bytes(wl, inp, lay, mode):
    """Algorithmic bytes of each stage per step (what the method itself moves)."""
    es = 4 if wl.logits_dtype == "f32" else 2
    seq = lay["seq_lens"].astype(np.int64)
    b, n = wl.b, wl.n
    select = sum(wl.rows(i) * wl.V * es for i in range(wl.S))
    kv_row = wl.Hkv * wl.D * 2
    attention = int((seq.sum() + b * n) * kv_row * 2 + 2 * b * n * wl.Hq * wl.D * 2 + b * n * wl.Hq * 4
                    + (seq.sum() + b * n) * 4)
    accept = b * n * wl.V * es
    if mode == "sampling":
        accept += b * n * 4 * 2 + b * wl.V * (es + 4)  # candidate q reads + one terminal row (p and q)
    return {"select_build": select, "attention": attention, "accept_commit": accept + 4 * b * wl.W * kv_row}


def attention_flops(wl, lay, mask_bits):
    """4 * D per visible (query row, key) pair, over every q head."""
    seq = lay["seq_lens"].astype(np.int64)
    vis = np.array([bin(int(m) & ((1 << 64) - 1)).count("1") for m in mask_bits], np.int64).reshape(wl.b, wl.n)
    keys = (seq[:, None] + vis).sum()
    return float(4 * wl.D * wl.Hq * keys)


# ------------------------------------------------------------- our arm

def run_ours(args, torch):
    from accept_select_top_gb300 import workloads as W
    from accept_select_top_gb300.pipeline import VerifyStep

    rank, world, local = dist_env()
    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    wl = W.WORKLOADS[args.workload]
    mode, inp, lay = prepare(wl, device, seed=rank, torch=torch)
    per_replica = sum(d.numel() * d.element_size() for d in inp.drafts) + inp.target_logits.numel() * \
        inp.target_logits.element_size() + 2 * inp.k_pool.numel() * 2 + inp.q.numel() * 2 + \
        (inp.draft_probs.numel() * 4 if inp.draft_probs is not None else 0)
    R = args.replicas or max(2, min(8, math.ceil(4 * 129e6 / per_replica)))
    replicas = [inp] + [clone_inputs(inp, torch) for _ in range(R - 1)]
    steps = [VerifyStep(wl, x, mode, device=device) for x in replicas]
    stream = torch.cuda.Stream(device=device)

    # warm-up, eager
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            steps[i % R].run()
    torch.cuda.synchronize()
    mask_bits = steps[0].mask_bits.cpu().numpy()
    accept_lens = steps[0].accept_lens.cpu().numpy()
    assert steps[0].ws.last_error() == 0, "device error word set during warm-up"

    # Timed graphs: P consecutive steps each (one per input replica, so every
    # step reads inputs the previous steps did not), with nothing but the
    # kernels inside, so that consecutive kernels overlap as they do when a
    # caller runs steps back to back (programmatic dependent launch does not
    # cross a graph launch or an event node).  P divides K.
    P = steps_per_graph(R, args.steps)
    G = max(1, min(args.graphs, args.steps // P))
    graphs = []
    for j in range(G):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for t in range(P):
                steps[(j * P + t) % R].run()
        graphs.append(g)
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            graphs[i % G].replay()
    torch.cuda.synchronize()

    sampler = None if args.no_clocks else ClockSampler(gpu_id_for_smi(torch, local))
    if sampler is not None:
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record()
        for i in range(args.steps // P):
            graphs[i % G].replay()
        t1.record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler is not None else None
    elapsed_ms = job_elapsed_ms(t0.elapsed_time(t1), world, device, torch)
    assert steps[0].ws.last_error() == 0, "device error word set during the timed region"

    # Stage breakdown (diagnostic, after the timed region): one-step graphs
    # with timing events captured at the stage boundaries.
    stage = None
    try:
        torch.cuda.Event(enable_timing=True, external=True)
        external = True
    except TypeError:
        external = False
    if external:
        evs, sgraphs = [], []
        for j in range(R):
            e = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                s = steps[j]
                e[0].record()
                s.select()
                s.build()
                e[1].record()
                s.attention()
                e[2].record()
                s.accept()
                s.commit()
                e[3].record()
            sgraphs.append(g)
            evs.append(e)
        sel, att, acc = [], [], []
        with torch.cuda.stream(stream):
            for i in range(max(2 * R, min(args.steps, 200))):
                sgraphs[i % R].replay()
                if i >= R:  # warm
                    torch.cuda.synchronize()
                    e = evs[i % R]
                    sel.append(e[0].elapsed_time(e[1]))
                    att.append(e[1].elapsed_time(e[2]))
                    acc.append(e[2].elapsed_time(e[3]))
        torch.cuda.synchronize()
        stage = {"select_build": statistics.mean(sel), "attention": statistics.mean(att),
                 "accept_commit": statistics.mean(acc)}

    e2e = None if args.no_e2e else run_e2e(args, torch, wl, mode, steps[0], stream, device)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, mode, steps[0], lay, torch)
    return wl, mode, lay, elapsed_ms, stage, mask_bits, accept_lens, clocks, e2e, cpu, world, G, R, external, P


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
    K = min(args.steps, 200)

    inp1 = _copy.copy(inp)  # the copied inputs get buffers of their own; the rest is shared
    for k in names:
        setattr(inp1, k, torch.empty_like(getattr(inp, k)))
    inp1.drafts = [torch.empty_like(d) for d in inp.drafts]
    sets = [(inp, step), (inp1, VerifyStep(wl, inp1, mode, device=device))]
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


# ------------------------------------------------- oracle (CPU baseline)

def oracle_sample(wl, mode, host, r, pair_frac):
    """Runs the oracle over requests [0, r) (attention on a fraction of their
    (row, head) pairs) and returns per-stage seconds and the units done."""
    import oracle
    from oracle import pipeline as OP
    sub = dict(wl.__dict__)
    sub["b"] = r
    from accept_select_top_gb300.workloads import Workload
    w = Workload(**sub)
    n = wl.n
    times = {}
    t = time.perf_counter()
    chain = OP.select_chain(w, [d[: w.rows(i)] for i, d in enumerate(host["drafts"])])
    tree = OP.tree_from_chain(w, chain, host["bonus"][:r], host["seq_lens"][:r])
    times["select_build"] = time.perf_counter() - t
    rows = r * n
    npairs = max(1, int(rows * wl.Hq * pair_frac))
    rng = np.random.default_rng(0)
    flat = rng.choice(rows * wl.Hq, size=npairs, replace=False)
    pairs = np.stack([flat // wl.Hq, flat % wl.Hq], 1).astype(np.int32)
    t = time.perf_counter()
    oracle.verify_attention(r, n, wl.Hq, wl.Hkv, wl.D, host["q"][: rows], host["k_pool"], host["v_pool"],
                            host["req_to_token"], host["req_pool_idx"][:r], host["seq_lens"][:r],
                            host["verify_loc"][: rows], tree["mask_bits"], 1.0 / math.sqrt(wl.D), pairs=pairs)
    times["attention"] = time.perf_counter() - t
    t = time.perf_counter()
    if mode == "greedy":
        acc = OP.accept(w, "greedy", tree, host["logits"][: rows])
    else:
        acc = OP.accept(w, "sampling", tree, host["logits"][: rows], host["q_probs"][: rows], host["temps"][:r],
                        host["u"][: rows], host["u_final"][:r])
    OP.commit(w, {"req_to_token": host["req_to_token"], "req_pool_idx": host["req_pool_idx"][:r],
                  "seq_lens": host["seq_lens"][:r], "verify_loc": host["verify_loc"][: rows]},
              host["k_pool"], host["v_pool"], acc)
    times["accept_commit"] = time.perf_counter() - t
    return times, npairs


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


def sample_plan(wl):
    """(requests, attention pair fraction) of the bounded oracle sample."""
    ctx = wl.ctx[1] if wl.ctx[0] == "fixed" else (wl.ctx[2] if wl.ctx[0] == "uniform" else max(wl.ctx[1]))
    per_pair = 4.0 * wl.D * (ctx + wl.n) * 2.5e-9  # ~ seconds of fp64 work per (row, head) pair
    r = max(1, min(wl.b, 2))
    frac = min(1.0, 6.0 / max(1e-9, per_pair * r * wl.n * wl.Hq))
    return r, frac


def cpu_baseline(wl, mode, step, lay, torch):
    host = host_inputs(step, mode)
    r, frac = sample_plan(wl)
    times, npairs = oracle_sample(wl, mode, host, r, frac)
    # scale each stage to the whole batch: select/build and accept/commit by
    # requests, attention by (row, head) pairs
    full = (times["select_build"] + times["accept_commit"]) * (wl.b / r) + \
        times["attention"] * (wl.b * wl.n * wl.Hq / npairs)
    return {"value": wl.b * wl.n / full, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{r} of {wl.b} requests end to end, attention on {npairs} of {r * wl.n * wl.Hq} "
                      f"(row, head) pairs; stages scaled to the full batch",
            "sample_seconds": round(sum(times.values()), 2), "full_step_seconds_est": round(full, 3)}


# ---------------------------------------------------------- reference arm

def run_reference(args, torch):
    """The oracle, as it stands, timed on the host cores for the same workload,
    metric and unit; each step is a bounded sample (one request, a fraction of
    the attention pairs) scaled to the full batch."""
    from accept_select_top_gb300 import workloads as W
    from accept_select_top_gb300.pipeline import VerifyStep
    wl = W.WORKLOADS[args.workload]
    device = "cuda:0" if torch.cuda.is_available() else "cpu"
    if device == "cpu":
        return None
    mode, inp, lay = prepare(wl, device, 0, torch)
    step = VerifyStep(wl, inp, mode, device=device)
    host = host_inputs(step, mode)
    del step
    r, frac = 1, sample_plan(wl)[1] / 2
    tot = []
    for i in range(max(3, args.warmup) + args.steps):
        times, npairs = oracle_sample(wl, mode, host, r, frac)
        if i >= max(3, args.warmup):
            tot.append((times["select_build"] + times["accept_commit"]) * wl.b / r +
                       times["attention"] * (wl.b * wl.n * wl.Hq / npairs))
    sec = sum(tot) / len(tot)
    return wl, sec, f"1 of {wl.b} requests per step, attention on {npairs} (row, head) pairs; scaled to the batch"


def main(argv=None):
    args = parse_args(argv)
    import torch
    rank, world, _ = dist_env()
    peaks, peaks_kind = load_peaks()
    if args.impl == "reference":
        if rank != 0:
            return 0
        res = run_reference(args, torch)
        if res is None:
            print(json.dumps({"impl": "reference", "unavailable": "no CUDA device to prepare the inputs"}))
            return 0
        wl, sec, sample = res
        val = wl.b * wl.n / sec
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "b": wl.b, "topk": wl.k, "num_steps": wl.S,
                       "num_draft_tokens": wl.n, "vocab": wl.V},
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return 0

    (wl, mode, lay, elapsed_ms, stage, mask_bits, accept_lens, clocks, e2e, cpu, world, G, R,
     external, P) = run_ours(args, torch)
    if rank != 0:
        return 0
    from accept_select_top_gb300.pipeline import launches_per_step
    ms_per_step = elapsed_ms / args.steps
    value = job_tokens_per_s(wl.b, wl.n, args.steps, world, elapsed_ms)
    bytes_ = step_bytes(wl, None, lay, mode)
    roof = None
    if stage is not None:
        dom = max(stage, key=stage.get)
        common = "accept_select_top_gb300/csrc/common.cuh"  # helpers compiled into every kernel
        sources = {"attention": ["accept_select_top_gb300/csrc/attention_tc.cu", common],
                   "select_build": ["accept_select_top_gb300/csrc/select_topk.cu",
                                    "accept_select_top_gb300/csrc/build_tree.cu", common],
                   "accept_commit": ["accept_select_top_gb300/csrc/verify_greedy.cu",
                                     "accept_select_top_gb300/csrc/verify_sampling.cu",
                                     "accept_select_top_gb300/csrc/commit_kv.cu", common]}[dom]
        flops = attention_flops(wl, lay, mask_bits)
        tensor_bound = dom == "attention" and flops / bytes_["attention"] > \
            peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
        ms = stage[dom]
        if tensor_bound:
            ach = flops / (ms / 1e3) / 1e12
            peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
            roof = {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak}
        else:
            ach = bytes_[dom] / (ms / 1e3) / 1e9
            peak = peaks["hbm_gbs"]
            roof = {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak}
        tr = traffic_entry(f"{dom}:{args.workload}", sources)
        roof.update({"traffic": None if tr is None else tr["dram_bytes_per_launch"], "stage": dom,
                     "stage_us": ms * 1e3, "algorithmic_bytes": bytes_[dom],
                     "peak_kind": f"{peaks_kind} ({'sustained' if tensor_bound else 'copy'})"})
    launches = launches_per_step(wl, mode, int(lay["seq_lens"].max()))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "step_us": ms_per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded draws; target agreement planted / correlated per the workload recipe)",
        "config": {"workload": args.workload, "b": wl.b, "topk": wl.k, "num_steps": wl.S, "num_draft_tokens": wl.n,
                   "vocab": wl.V, "heads": f"{wl.Hq}/{wl.Hkv}", "head_dim": wl.D, "page_size": wl.page_size,
                   "context": list(wl.ctx), "accept": mode, "parallelism": f"replicas x{world}",
                   "l2": f"{R} rotating input replicas (> 4x the 129 MB L2 per cycle)",
                   "graphs": G, "steps_per_graph": P,
                   "stage_timing": ("separate pass after the timed region: one-step graphs, events at the stage "
                                    "boundaries, each step alone" if external else "none")},
        "stages_us": None if stage is None else {k: v * 1e3 for k, v in stage.items()},
        "mean_accept_lens": float(np.mean(accept_lens)),
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches * args.steps, "clocks": clocks,
    }
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
