#!/usr/bin/env python
"""Benchmark: emulated context-parallel causal THD attention, fwd + bwd.

Workload (the headline configuration): 32768 packed tokens in 16 documents
(lengths multiples of 16 drawn uniformly in [256, 4096], the last one
adjusted), cp_size=4, H=16, D=128, bf16 ~N(0,1), causal fwd+bwd, both
DUAL_CHUNK_SWAP and NO_LOAD_BALANCE.  One step = the whole hot path for both
strategies: partition index for every rank, partition gather of Q/K/V/dO,
K/V restore, attention forward of every rank, attention backward of every
rank with fp32 dK/dV accumulation, the emulated reduce-scatter epilogue and
the gated tail-zeroing.

value = algorithmic attention FLOP per step (4*D*H*pairs fwd + 10*D*H*pairs
bwd, summed over ranks and strategies) / device time per step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl own|reference]

--impl reference times the fp64 CPU oracle on the host cores (a bounded
sample of the same workload per step).  With torchrun (N>1) every rank runs
the same workload on its own GPU (replicas: the path has no cross-GPU step
when every CP rank is emulated on one GPU); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CP-rank causal THD attention TFLOP/s (% BF16 peak); THD gather GB/s (% HBM)"
WORKLOAD = "THD packed 32768 tokens: 16 docs, cp_size=4, H=16, D=128, bf16, causal fwd+bwd, both strategies"


# DRAM bytes (read + write) of one attn_bwd call from an ncu capture.  The last capture
# (attn_dq_tc 495.0 + 22.9 MB, attn_dkdv_tc 467.9 + 478.9 MB for the DUAL_CHUNK_SWAP rank-0 call)
# predates the dK/dV epilogue's move to bulk tensor reduce / store, so the figure is not
# reported until the counters are taken again on the current kernel.
BWD_TRAFFIC_BYTES = None
BWD_TRAFFIC_NOTE = ("not re-captured since the dK/dV epilogue changed; the previous capture of the "
                    "DUAL_CHUNK_SWAP rank-0 call read 963 MB and wrote 502 MB (dq + dkdv)")


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), \
            d.get("bf16_tflops_sustained", 1700.0), "measured"
    except OSError:
        return 6800.0, 1900.0, 1700.0, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    return ws, rank


def _max_over_ranks(values, device):
    """Element-wise maximum of per-rank timings over the process group (the
    slowest replica sets the time); the values themselves with one process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def _whole_job_value(ws, flop_per_step, ms_per_step):
    """TFLOP/s of all replicas together: each of the ws replicas does
    flop_per_step per step, and a step lasts the slowest replica's time."""
    return ws * flop_per_step / (ms_per_step * 1e-3) / 1e12


def _workload():
    from context_packed_sequence_thd_gb300 import inputs
    return inputs.cfg2()


def _pairs_all(wl, strategies):
    from context_packed_sequence_thd_gb300 import pipeline
    return sum(pipeline.rank_pairs(wl.cu, wl.cup, wl.cp, r, s, wl.pad_between_seqs)
               for s in strategies for r in range(wl.cp))


class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        self.gpu = gpu_index

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def run_own(args):
    import torch
    import torch.distributed as dist

    ws, rank = _dist()
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())

    import __graft_entry__
    __graft_entry__.build()
    from context_packed_sequence_thd_gb300 import api, pipeline

    hbm, bf16_burst, bf16_sust, peak_src = _peaks()
    wl = _workload()
    strategies = (pipeline.DCS, pipeline.NLB)
    host = wl.tensors()
    pinned = {k: v.pin_memory() for k, v in host.items()}
    g = {k: v.to(dev) for k, v in host.items()}
    atts = [pipeline.CPAttention(pipeline.CPPlan(wl.cu, wl.cup, wl.cp, s, wl.pad_between_seqs,
                                                 wl.H, wl.D, dev)) for s in strategies]
    pairs = _pairs_all(wl, strategies)
    flop_fwd = 4.0 * wl.D * wl.H * pairs
    flop_bwd = 10.0 * wl.D * wl.H * pairs
    flop_step = flop_fwd + flop_bwd

    def step():
        for a in atts:
            a.step(g["q"], g["k"], g["v"], g["do"])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert api.cp_device_status() == 0, "device status after warm-up"

    for a in atts:
        a.launches = 0
        a.events = {}
    stream = torch.cuda.current_stream()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index if os.environ.get("CUDA_VISIBLE_DEVICES") is None else 0) as clk:
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    ms = _max_over_ranks([t0.elapsed_time(t1) / args.steps], dev)[0]
    launches = sum(a.launches for a in atts)

    # per-call breakdown from the events recorded inside the timed region
    per = {}
    for a, s in zip(atts, strategies):
        for cat, vals in a.event_ms().items():
            per.setdefault(cat, []).extend(vals)
    cat_total = {k: sum(v) / args.steps for k, v in per.items()}
    bwd_calls = per.get("attn_bwd", [])
    fwd_calls = per.get("attn_fwd", [])
    n_rank_calls = len(strategies) * wl.cp
    # algorithmic FLOP per launch: average over the per-rank calls of a step
    bwd_flop_per_call = flop_bwd / n_rank_calls
    fwd_flop_per_call = flop_fwd / n_rank_calls
    bwd_ms = statistics.mean(bwd_calls) if bwd_calls else float("nan")
    fwd_ms = statistics.mean(fwd_calls) if fwd_calls else float("nan")
    dominant = "attn_bwd" if sum(bwd_calls) >= sum(fwd_calls) else "attn_fwd"
    if dominant == "attn_bwd":
        ach = bwd_flop_per_call / (bwd_ms * 1e-3) / 1e12
    else:
        ach = fwd_flop_per_call / (fwd_ms * 1e-3) / 1e12
    # gather bandwidth: partition gather of Q/K/V/dO for every rank (DCS) + K/V restore
    row_bytes = wl.H * wl.D * 2
    pg = per.get("partition_gather", [])
    pg_bytes = 4 * 2 * wl.total_tokens * row_bytes + 4 * wl.total_tokens  # all ranks, one launch
    rg = per.get("restore_gather", [])
    rg_bytes = 2 * 2 * wl.total_tokens * row_bytes + 4 * wl.total_tokens
    gather_gbs = pg_bytes / (statistics.mean(pg) * 1e-3) / 1e9 if pg else None
    restore_gbs = rg_bytes / (statistics.mean(rg) * 1e-3) / 1e9 if rg else None

    # end to end: pinned host inputs -> device, step, outputs -> pinned host.
    # Serial form first (copy in, step, copy out, one after another), then the
    # pipelined form the public API allows: two sets of device inputs and of
    # attention objects (outputs), the next step's inputs copied in and the
    # previous step's outputs copied out on their own streams while a step
    # computes.  Every step's copies are inside the timed region in both.
    e2e_steps = max(2, min(args.steps, 40))
    outs = [t for a in atts for t in (a.oc, a.dqc, a.dkc, a.dvc)]
    host_outs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = sum(t.numel() * t.element_size() for t in outs)
    for a in atts:
        a.events = None
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        for kname in ("q", "k", "v", "do"):
            g[kname].copy_(pinned[kname], non_blocking=True)
        step()
        for h, d in zip(host_outs, outs):
            h.copy_(d, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_serial_ms = e0.elapsed_time(e1) / e2e_steps

    g2 = {k: torch.empty_like(v) for k, v in g.items()}
    atts2 = [pipeline.CPAttention(pipeline.CPPlan(wl.cu, wl.cup, wl.cp, s, wl.pad_between_seqs,
                                                  wl.H, wl.D, dev)) for s in strategies]
    sets = [(g, atts), (g2, atts2)]
    outs_of = [[t for a in aa for t in (a.oc, a.dqc, a.dkc, a.dvc)] for _, aa in sets]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()                                        # noqa: E731
    in_ready = [ev(), ev()]
    computed = [ev(), ev()]
    out_done = [ev(), ev()]

    def copy_in(b):
        s_in.wait_event(computed[b])            # the set's previous step has read its inputs
        with torch.cuda.stream(s_in):
            for kname in ("q", "k", "v", "do"):
                sets[b][0][kname].copy_(pinned[kname], non_blocking=True)
        in_ready[b].record(s_in)

    for b in (0, 1):
        computed[b].record(stream)
        out_done[b].record(stream)
    torch.cuda.synchronize()
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    copy_in(0)
    copy_in(1)
    for i in range(e2e_steps):
        b = i & 1
        gb, ab = sets[b]
        stream.wait_event(in_ready[b])
        stream.wait_event(out_done[b])           # this set's previous outputs are copied out
        for a in ab:
            a.step(gb["q"], gb["k"], gb["v"], gb["do"], stream=stream)
        computed[b].record(stream)
        s_out.wait_event(computed[b])
        with torch.cuda.stream(s_out):
            for h, d in zip(host_outs, outs_of[b]):
                h.copy_(d, non_blocking=True)
        out_done[b].record(s_out)
        if i + 2 < e2e_steps:
            copy_in(b)
    stream.wait_event(out_done[(e2e_steps - 1) & 1])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms, e2e_serial_ms = _max_over_ranks([e0.elapsed_time(e1) / e2e_steps, e2e_serial_ms], dev)
    assert api.cp_device_status() == 0, "device status after timing"

    result = None
    if rank == 0:
        value = _whole_job_value(ws, flop_step, ms)
        peak = bf16_sust
        result = {
            "metric": METRIC,
            "value": round(value, 3),
            "unit": "TFLOP/s",
            "n_gpus": ws,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "total_tokens": wl.total_tokens,
                       "n_docs": wl.n_docs, "cp_size": wl.cp, "H": wl.H, "D": wl.D,
                       "strategies": ["dual_chunk_swap", "no_load_balance"],
                       "parallelism": f"replicas{ws}" if ws > 1 else "cp4 emulated on 1 GPU",
                       "l2": "inputs larger than L2 (4 x 134 MB bf16 inputs, ~2 GB touched per step)"},
            "roofline": {"bound": "tensor", "kernel": dominant, "achieved": round(ach, 2),
                         "peak": peak, "unit": "TFLOP/s", "frac": round(ach / peak, 4),
                         "peak_source": f"{peak_src} bf16 sustained",
                         "traffic": BWD_TRAFFIC_BYTES if dominant == "attn_bwd" else None,
                         "traffic_note": BWD_TRAFFIC_NOTE if dominant == "attn_bwd" else None},
            "gpu_launches": launches,
            "clocks": clk.summary(),
            "e2e": {"value": round(_whole_job_value(ws, flop_step, e2e_ms), 3),
                    "unit": "TFLOP/s", "ms_per_step": round(e2e_ms, 4),
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps,
                    "copies": "pinned host; next step's inputs in and previous step's outputs "
                              "out on copy streams, overlapped with the step",
                    "serial": {"value": round(_whole_job_value(ws, flop_step, e2e_serial_ms), 3),
                               "ms_per_step": round(e2e_serial_ms, 4)}},
            "breakdown_ms_per_step": {k: round(v, 4) for k, v in cat_total.items()},
            "attn_fwd_tflops": round(fwd_flop_per_call / (fwd_ms * 1e-3) / 1e12, 2),
            "attn_bwd_tflops": round(bwd_flop_per_call / (bwd_ms * 1e-3) / 1e12, 2),
            "gather": {"partition_gather_gbs": None if gather_gbs is None else round(gather_gbs, 1),
                       "restore_gather_gbs": None if restore_gbs is None else round(restore_gbs, 1),
                       "hbm_peak_gbs": hbm,
                       "frac": None if gather_gbs is None else round(gather_gbs / hbm, 4)},
            "pairs_per_step": pairs,
        }
        if not args.no_cpu_baseline and ws == 1:
            result["cpu_baseline"] = cpu_baseline(wl)
        else:
            result["cpu_baseline"] = None
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    if result is not None:
        print(json.dumps(result), flush=True)


def _oracle_sample(wl, heads, row_stride):
    """fwd + bwd of the oracle on a sample: the given heads, every
    `row_stride`-th query row.  Returns (seconds, algorithmic FLOP)."""
    import numpy as np
    import oracle
    t = wl.tensors()
    sel = {k: v[:, heads].contiguous() for k, v in t.items()}
    qm = np.zeros(wl.total_tokens, dtype=bool)
    qm[::row_stride] = True
    t0 = time.perf_counter()
    o, lse = oracle.attn_fwd(sel["q"], sel["k"], sel["v"], wl.cu, wl.cup, wl.pad_between_seqs,
                             qmask=qm)
    oracle.attn_bwd(sel["q"], sel["k"], sel["v"], np.nan_to_num(o), np.nan_to_num(lse),
                    sel["do"], wl.cu, wl.cup, wl.pad_between_seqs, qmask=qm)
    dt = time.perf_counter() - t0
    pairs = oracle.causal_pairs(wl.cu, wl.cup, wl.pad_between_seqs, np.nonzero(qm)[0])
    return dt, 14.0 * wl.D * len(heads) * pairs


def cpu_baseline(wl):
    import oracle
    oracle.build()
    heads = [0, 1]
    dt, flop = _oracle_sample(wl, heads, 1)
    return {"value": round(flop / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"fp64 C oracle fwd+bwd, heads {heads} of {wl.H}, all {wl.total_tokens} "
                      f"query rows ({dt:.1f} s); same FLOP accounting as the GPU line"}


def run_reference(args):
    ws, rank = _dist()
    if rank != 0:
        return
    import oracle
    oracle.build()
    wl = _workload()
    for _ in range(args.warmup):
        _oracle_sample(wl, [0], 64)
    secs, flops = [], []
    for _ in range(args.steps):
        dt, f = _oracle_sample(wl, [0], 64)
        secs.append(dt)
        flops.append(f)
    v = sum(flops) / sum(secs) / 1e12
    ms = 1e3 * sum(secs) / len(secs)
    sample = (f"fp64 C oracle fwd+bwd per step: head 0 of {wl.H}, every 64th query row "
              f"of the {wl.total_tokens}-token workload")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["own", "reference"], default="own")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_own(args)


if __name__ == "__main__":
    main()
