#!/usr/bin/env python
"""Benchmark: emulated context-parallel causal THD attention, fwd + bwd.

Headline workload: 65536 padded tokens in 24 documents (lognormal lengths,
median 1656, sigma 1, each padded up to a multiple of 2*cp_size; the last
document keeps a 3-row tail), cp_size=4, H=32, D=128, bf16 ~N(0,1),
pad_between_seqs=1, causal fwd+bwd, both DUAL_CHUNK_SWAP and NO_LOAD_BALANCE.
One step = the whole hot path for both strategies: partition index for every
rank, partition gather of Q/K/V/dO, K/V restore, attention forward of every
rank, attention backward of every rank with fp32 dK/dV accumulation, the
emulated reduce-scatter epilogue and the gated tail-zeroing (one rank holds
the tail, so the tail-zero kernel runs in the step).

value = algorithmic attention FLOP per step (4*D*H*pairs fwd + 10*D*H*pairs
bwd, summed over ranks and strategies) / device time per step.

The same JSON line carries, measured outside the headline's timed region:
per-rank forward / backward times with their sum and max over ranks (the CP
critical path), the other workloads' throughput, the padding arms of the
headline workload (A: padded metadata; B: value-equal metadata; C: no tail),
and a per-rank partition / restore / unrestore gather sweep on the
single-sequence shapes.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl own|reference]
                  [--no-secondary] [--no-cpu-baseline] [--no-e2e]

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
WORKLOAD = ("THD fwd+bwd with inter-sequence padding: 65536 padded tokens, 24 lognormal docs "
            "padded to multiples of 2*cp, cp_size=4, H=32, D=128, bf16, pad_between_seqs=1, "
            "both strategies")

# DRAM bytes (read + write) per backward call (cp_attn_bwd_grouped_rs: every rank's
# attn_delta and attn_dq_tc, one attn_dkdv_tc that also writes the reduce-scatter's bf16 rows),
# averaged over the 2 calls of a step (2 strategies), from the ncu capture named in
# BWD_TRAFFIC_NOTE; None until a capture of the current kernels exists.
BWD_TRAFFIC_BYTES = 19984964352
BWD_TRAFFIC_NOTE = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of the kernels of the timed "
                    "step's two cp_attn_bwd_grouped_rs calls (DCS 22.67 GB, NLB 17.30 GB), full "
                    "size, one pass; profiles/attn_bwd_dram_cfg5.md")

# without clock samples, a timed region shorter than this is a burst (burst
# peak as the denominator), a longer one sustained
BURST_REGION_S = 1.0


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


def _workload(name="cfg5"):
    from context_packed_sequence_thd_gb300 import inputs
    return {"cfg5": inputs.cfg5, "cfg2": inputs.cfg2, "cfg3": inputs.cfg3}[name]()


def _pairs_all(wl, strategies):
    from context_packed_sequence_thd_gb300 import pipeline
    return sum(pipeline.rank_pairs(wl.cu, wl.cup, wl.cp, r, s, wl.pad_between_seqs)
               for s in strategies for r in range(wl.cp))


def _pick_peak(region_s, clocks, burst, sustained):
    """The measured peak of the regime the kernel ran in.  The sustained
    figure was taken with the SM clock pulled far below its maximum by the
    power limit; a region whose median SM clock stays within 10% of the
    maximum runs in the burst regime (whatever its length or a power-cap flag
    that barely binds), so its denominator is the burst peak.  Without clock
    samples the region's length decides."""
    sm, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    if sm is None or mx is None:
        return (burst, "burst") if region_s < BURST_REGION_S else (sustained, "sustained")
    if sm >= 0.9 * mx:
        return burst, "burst"
    return sustained, "sustained"


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
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_max": max(pw) if pw else None, "samples": len(rows)}


# ---------------------------------------------------------------------------
# measurements outside the headline's timed region
# ---------------------------------------------------------------------------

def _time_ms(fn, reps, flush=None):
    """Median CUDA-event time of fn over reps calls (after one untimed call);
    with `flush`, a buffer larger than L2 is overwritten before every call."""
    import torch
    fn()
    ms = []
    for _ in range(reps):
        if flush is not None:
            flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    return statistics.median(ms)


def _per_rank(att, steps, cp):
    """Per-rank forward / backward times (ms) from the events of `steps` steps,
    with their sum and max over ranks (the critical path of a real CP group)."""
    ev = att.event_ms()
    out = {}
    for cat, key in (("attn_fwd", "fwd"), ("attn_bwd", "bwd")):
        vals = ev.get(cat, [])
        if len(vals) != steps * cp:
            continue
        per = [statistics.mean(vals[r::cp]) for r in range(cp)]
        out[f"{key}_ms"] = [round(x, 4) for x in per]
        out[f"{key}_sum_ms"] = round(sum(per), 4)
        out[f"{key}_max_ms"] = round(max(per), 4)
    return out


def _workload_line(wl, strategies, dev, reps=5, bwd=True, grouped_bwd=True):
    """Step time and attention TFLOP/s of one workload, every strategy
    (grouped_bwd=False: the rank-by-rank backward, whose per-rank times are
    then reported too)."""
    import torch
    from context_packed_sequence_thd_gb300 import pipeline
    g = {k: v.to(dev) for k, v in wl.tensors(with_grad=bwd).items()}
    res = {}
    for s in strategies:
        att = pipeline.CPAttention(pipeline.CPPlan(wl.cu, wl.cup, wl.cp, s, wl.pad_between_seqs,
                                                   wl.H, wl.D, dev), grouped_bwd=grouped_bwd)
        run = lambda: att.step(g["q"], g["k"], g["v"], g.get("do"))   # noqa: E731
        step_ms = _time_ms(run, reps)
        att.events = {}
        for _ in range(reps):
            run()
        torch.cuda.synchronize()
        ev = att.event_ms()
        f = att.flops(bwd)
        fwd_ms = sum(ev["attn_fwd"]) / reps
        r = {"step_ms": round(step_ms, 4), "attn_fwd_ms": round(fwd_ms, 4),
             "attn_fwd_tflops": round(f["fwd"] / (fwd_ms * 1e-3) / 1e12, 1)}
        if bwd:
            bwd_ms = sum(ev["attn_bwd"]) / reps
            r["attn_bwd_ms"] = round(bwd_ms, 4)
            r["attn_bwd_tflops"] = round(f["bwd"] / (bwd_ms * 1e-3) / 1e12, 1)
        r["per_rank"] = _per_rank(att, reps, wl.cp)
        res[pipeline.STRATEGY_NAMES[s]] = r
        del att
    del g
    torch.cuda.empty_cache()
    return res


def _padding_arms(dev, reps=5):
    """Step time of the headline workload under its three metadata arms:
    A padded metadata (pad_between_seqs=1, a tail on one rank), B value-equal
    metadata (cu_seqlens a copy of cu_seqlens_padded, flag decided 0 from
    values), C padded metadata whose last document has no tail (the tail-zero
    launches nothing)."""
    import torch
    from context_packed_sequence_thd_gb300 import api, inputs, pipeline
    out = {}
    for arm, wl in (("A_padded", inputs.cfg5()), ("B_value_equal", inputs.cfg5(value_equal=True)),
                    ("C_no_tail", inputs.cfg5(tail=False))):
        g = {k: v.to(dev) for k, v in wl.tensors().items()}
        r = {"pad_between_seqs": int(api.cp_detect_pad_between_seqs(wl.cu, wl.cup))}
        for s in (pipeline.DCS, pipeline.NLB):
            att = pipeline.CPAttention(pipeline.CPPlan(wl.cu, wl.cup, wl.cp, s,
                                                       wl.pad_between_seqs, wl.H, wl.D, dev))
            att.launches = 0
            att.step(g["q"], g["k"], g["v"], g["do"])
            launches = att.launches
            r[pipeline.STRATEGY_NAMES[s]] = {
                "step_ms": round(_time_ms(lambda: att.step(g["q"], g["k"], g["v"], g["do"]),
                                          reps), 4),
                "launches": launches}
            del att
        out[arm] = r
        del g
    torch.cuda.empty_cache()
    return out


def _gather_sweep(dev, hbm, reps=10):
    """The single-sequence shapes of the a2a measurement (cp=8, H=40, D=128,
    s in {8192, 32768, 75600}): for every rank r, the partition gather of
    Q/K/V (three tensors, one launch), and the restore gather of K/V and the
    unrestore of dK/dV (the reduce-scatter cast: fp32 sums gathered by the
    rank's index, rounded to bf16) -- GB/s, L2 flushed before every call."""
    import torch
    from context_packed_sequence_thd_gb300 import api, inputs, pipeline
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    out = {}
    for s in (8192, 32768, 75600):
        wl = inputs.cfg3(s)
        T, H, D, cp = wl.total_tokens, wl.H, wl.D, wl.cp
        S = T // cp
        rb = H * D * 2
        gen = torch.Generator(device="cpu").manual_seed(7)
        src = [torch.randn(T, H, D, generator=gen).bfloat16().to(dev) for _ in range(3)]
        dst = [torch.empty(S, H, D, dtype=torch.bfloat16, device=dev) for _ in range(3)]
        acc = [torch.randn(T, H, D, generator=gen).to(dev) for _ in range(2)]
        full = [torch.empty(T, H, D, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        r_s = {}
        for st in (pipeline.DCS, pipeline.NLB):
            plan = pipeline.CPPlan(wl.cu, wl.cup, cp, st, 0, H, D, dev)
            per = []
            for r in range(cp):
                idx = plan.ranks[r].idx
                t_g = _time_ms(lambda: api.cp_thd_gather(src, dst, idx), reps, flush)
                t_u = _time_ms(lambda: api.cp_reduce_scatter_emul(acc, dst[:2], idx, 0, S), reps,
                               flush)
                per.append({"rank": r,
                            "partition_gather_gbs": round((3 * 2 * S * rb + 4 * S) / t_g / 1e6, 1),
                            "unrestore_gbs": round((2 * S * H * D * 6 + 4 * S) / t_u / 1e6, 1)})
            t_r = _time_ms(lambda: api.cp_thd_gather(src[:2], full, plan.restore), reps, flush)
            r_s[pipeline.STRATEGY_NAMES[st]] = {
                "per_rank": per,
                "restore_kv_gbs": round((2 * 2 * T * rb + 4 * T) / t_r / 1e6, 1),
                "partition_gather_frac_min": round(min(p["partition_gather_gbs"] for p in per) / hbm, 4)}
        out[f"s{s}"] = r_s
        del src, dst, acc, full
    del flush
    torch.cuda.empty_cache()
    return out


def _comm_types(wl, dev, reps=3):
    """Forward / backward TFLOP/s of the emulated a2a and P2P (ring) comm types
    on one workload, every strategy (their exchanges, merges and casts
    included): the ring as one pass per rank and gradient (default) and step
    by step, with all-gather CP beside them."""
    import torch
    from context_packed_sequence_thd_gb300 import pipeline
    g = {k: v.to(dev) for k, v in wl.tensors().items()}
    out = {}
    variants = (("a2a", pipeline.CPA2AAttention),
                ("p2p", pipeline.CPP2PAttention),   # one pass per rank and gradient
                ("p2p_per_step", lambda plan: pipeline.CPP2PAttention(plan, fused_ring=False)),
                ("allgather", pipeline.CPAttention))
    for name, cls in variants:
        for s in (pipeline.DCS, pipeline.NLB):
            plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, s, wl.pad_between_seqs, wl.H, wl.D, dev)
            att = cls(plan)
            att.shard_inputs(g["q"], g["k"], g["v"], g["do"])
            f = att.flops(True)
            kv = att.forward()
            kv = kv if isinstance(kv, tuple) else (None, None)
            t_f = _time_ms(lambda: att.forward(), reps)
            t_b = _time_ms(lambda: att.backward(*kv), reps)
            out[f"{name}_{pipeline.STRATEGY_NAMES[s]}"] = {
                "fwd_ms": round(t_f, 4), "fwd_tflops": round(f["fwd"] / t_f / 1e9, 1),
                "bwd_ms": round(t_b, 4), "bwd_tflops": round(f["bwd"] / t_b / 1e9, 1)}
            del att
    del g
    torch.cuda.empty_cache()
    return out


def _a2a_exchange(dev, hbm, reps=10):
    """The a2a page's exchange shapes (cp=8, H=40, D=128): GB/s of the
    seq->head exchange of Q, K, V; under DUAL_CHUNK_SWAP the dual-chunk reorder
    is folded into the same pass, timed against the exchange followed by a
    separate reorder gather."""
    import torch
    from context_packed_sequence_thd_gb300 import api, inputs, pipeline
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    out = {}
    cp, H, D = 8, 40, 128
    for T in (8192, 32768, 75600):
        wl = inputs.custom([T], cp=cp, H=H, D=D, seed=7)
        gen = torch.Generator(device="cpu").manual_seed(7)
        seq = [torch.randn(T, H, D, generator=gen).bfloat16().to(dev) for _ in range(3)]
        head = [torch.empty(cp, T, H // cp, D, dtype=torch.bfloat16, device=dev) for _ in range(3)]
        nbytes = 3 * 2 * T * H * D * 2
        r = {}
        for s in (pipeline.DCS, pipeline.NLB):
            plan = pipeline.CPPlan(wl.cu, wl.cup, cp, s, 0, H, D, dev)
            perm = plan.restore if s == pipeline.DCS else None
            t = _time_ms(lambda: api.cp_a2a_exchange(seq, head, perm, cp, api.A2A_SEQ_TO_HEAD),
                         reps, flush)
            gbs = (nbytes + (4 * T if perm is not None else 0)) / t / 1e6
            r[pipeline.STRATEGY_NAMES[s]] = {"us": round(t * 1e3, 1), "gbs": round(gbs, 1),
                                             "frac": round(gbs / hbm, 4)}
            if perm is not None:
                tmp = [torch.empty_like(h) for h in head]
                rows = (torch.arange(cp, device=dev, dtype=torch.int64)[:, None] * T +
                        perm.to(torch.int64)[None, :]).reshape(-1).to(torch.int32)
                flat_t = [x.view(cp * T, H // cp, D) for x in tmp]
                flat_h = [x.view(cp * T, H // cp, D) for x in head]

                def unfused():
                    api.cp_a2a_exchange(seq, tmp, None, cp, api.A2A_SEQ_TO_HEAD)
                    api.cp_thd_gather(flat_t, flat_h, rows)
                t2 = _time_ms(unfused, reps, flush)
                r["dual_chunk_swap_exchange_then_reorder_us"] = round(t2 * 1e3, 1)
                del tmp
        out[f"s{T}"] = r
        del seq, head
    del flush
    torch.cuda.empty_cache()
    return out


def _fused_q_gather(dev, reps=5):
    """Forward-only DUAL_CHUNK_SWAP step on the single 32768-token sequence
    (cp=8, H=40): the Q shard gathered by the copy kernel, and by the
    attention's own loads through the partition index (cp_attn_fwd_gather)."""
    import torch
    from context_packed_sequence_thd_gb300 import inputs, pipeline
    wl = inputs.cfg3()
    g = {k: v.to(dev) for k, v in wl.tensors(with_grad=False).items()}
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, pipeline.DCS, 0, wl.H, wl.D, dev)
    out = {}
    for fuse in (False, True):   # the fused gather reads the bf16 batch: bf16 operands both
        att = pipeline.CPAttention(plan, fuse_q_gather=fuse, operand_dtype=torch.bfloat16)
        t = _time_ms(lambda: att.step(g["q"], g["k"], g["v"], rebuild_index=False), reps)
        out["fused_gather_ms" if fuse else "copy_gather_ms"] = round(t, 4)
        del att
    del g
    torch.cuda.empty_cache()
    return out


def _secondary(dev, hbm):
    from context_packed_sequence_thd_gb300 import inputs, pipeline
    both = (pipeline.DCS, pipeline.NLB)
    return {
        "cfg2_32k_16docs_cp4_h16": _workload_line(inputs.cfg2(), both, dev),
        # the headline workload with the rank-by-rank backward (cp_attn_bwd per
        # rank, partial dK/dV added into the fp32 sums): per-rank backward times
        "headline_workload_rank_by_rank_bwd": _workload_line(inputs.cfg5(), both, dev, reps=3,
                                                             grouped_bwd=False),
        "cfg4_75600_nlb_cp8_h40": _workload_line(inputs.cfg4(), (pipeline.NLB,), dev, reps=3),
        "cfg3_32k_single_seq_cp8_h40_fwd": _workload_line(inputs.cfg3(), both, dev, reps=3,
                                                          bwd=False),
        "padding_arms_ms": _padding_arms(dev),
        "gather_sweep_cp8_h40": _gather_sweep(dev, hbm),
        "comm_types_headline_workload": _comm_types(inputs.cfg5(), dev),
        "a2a_exchange_cp8_h40": _a2a_exchange(dev, hbm),
        "fused_q_gather_fwd_cfg3": _fused_q_gather(dev),
    }


# ---------------------------------------------------------------------------
# the headline
# ---------------------------------------------------------------------------

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
    wl = _workload(args.workload)
    strategies = (pipeline.DCS, pipeline.NLB)
    host = wl.tensors(with_grad=wl.bwd)
    g = {k: v.to(dev) for k, v in host.items()}
    atts = [pipeline.CPAttention(pipeline.CPPlan(wl.cu, wl.cup, wl.cp, s, wl.pad_between_seqs,
                                                 wl.H, wl.D, dev)) for s in strategies]
    pairs = _pairs_all(wl, strategies)
    flop_fwd = 4.0 * wl.D * wl.H * pairs
    flop_bwd = 10.0 * wl.D * wl.H * pairs
    flop_step = flop_fwd + flop_bwd

    def step():
        for a in atts:
            a.step(g["q"], g["k"], g["v"], g.get("do"))  # (forward-only workloads: no dO)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert api.cp_device_status() == 0, "device status after warm-up"
    if args.capture:
        # a fixed number of headline steps and nothing else, for ncu captures
        for _ in range(args.steps):
            step()
        torch.cuda.synchronize()
        assert api.cp_device_status() == 0
        print("capture steps done", flush=True)
        return

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
    clocks = clk.summary()

    # per-call breakdown from the events recorded inside the timed region
    per = {}
    for a in atts:
        for cat, vals in a.event_ms().items():
            per.setdefault(cat, []).extend(vals)
    cat_total = {k: sum(v) / args.steps for k, v in per.items()}
    per_rank = {pipeline.STRATEGY_NAMES[s]: _per_rank(a, args.steps, wl.cp)
                for a, s in zip(atts, strategies)}
    bwd_calls = per.get("attn_bwd", [])
    fwd_calls = per.get("attn_fwd", [])
    # algorithmic FLOP per call, averaged over a step's calls: the forward is one
    # cp_attn_fwd per rank and strategy, the backward one cp_attn_bwd_grouped_rs
    # per strategy (every rank's Delta and dQ launches and one dK/dV launch)
    n_bwd_calls = max(1, len(bwd_calls) // args.steps)
    n_fwd_calls = max(1, len(fwd_calls) // args.steps)
    bwd_flop_per_call = flop_bwd / n_bwd_calls
    fwd_flop_per_call = flop_fwd / n_fwd_calls
    bwd_ms = statistics.mean(bwd_calls) if bwd_calls else float("nan")
    fwd_ms = statistics.mean(fwd_calls) if fwd_calls else float("nan")
    dominant = "attn_bwd" if sum(bwd_calls) >= sum(fwd_calls) else "attn_fwd"
    if dominant == "attn_bwd":
        ach = bwd_flop_per_call / (bwd_ms * 1e-3) / 1e12
    else:
        ach = fwd_flop_per_call / (fwd_ms * 1e-3) / 1e12
    region_s = ms * args.steps * 1e-3
    peak, peak_kind = _pick_peak(region_s, clocks, bf16_burst, bf16_sust)
    # gather bandwidth: partition gather of Q/K/V/dO for every rank (DCS) + K/V restore
    row_bytes = wl.H * wl.D * 2
    pg = per.get("partition_gather", [])
    pg_bytes = 4 * 2 * wl.total_tokens * row_bytes + 4 * wl.total_tokens  # all ranks, one launch
    rg = per.get("restore_gather", [])
    rg_bytes = 2 * 2 * wl.total_tokens * row_bytes + 4 * wl.total_tokens
    gather_gbs = pg_bytes / (statistics.mean(pg) * 1e-3) / 1e9 if pg else None
    restore_gbs = rg_bytes / (statistics.mean(rg) * 1e-3) / 1e9 if rg else None
    for a in atts:
        a.events = None

    e2e = None
    if not args.no_e2e:
        e2e = _e2e(args, wl, strategies, host, g, atts, step, flop_step, ws, dev)
    assert api.cp_device_status() == 0, "device status after timing"

    secondary = None
    if not args.no_secondary and rank == 0:
        del g, atts
        torch.cuda.empty_cache()
        secondary = _secondary(dev, hbm)
        assert api.cp_device_status() == 0, "device status after the secondary measurements"

    result = None
    if rank == 0:
        value = _whole_job_value(ws, flop_step, ms)
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
                       "pad_between_seqs": wl.pad_between_seqs,
                       "operands": "bf16 inputs; fp16 tensor-core operands (converted in the shard "
                                   "gather), fp32 accumulation, bf16 outputs",
                       "strategies": ["dual_chunk_swap", "no_load_balance"],
                       "parallelism": f"replicas{ws}" if ws > 1 else "cp4 emulated on 1 GPU",
                       "l2": "inputs larger than L2 (4 x 537 MB bf16 inputs, ~25 GB touched "
                             "per step)"},
            "roofline": {"bound": "tensor", "kernel": dominant,
                         "kernels": "cp_attn_bwd_grouped_rs: attn_delta + attn_dq_tc per rank, "
                                    "one rank-grouped attn_dkdv_tc writing the reduce-scatter's "
                                    "bf16 rows"
                         if dominant == "attn_bwd" else "attn_fwd_tc",
                         "achieved": round(ach, 2), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(ach / peak, 4),
                         "peak_source": f"{peak_src} bf16 {peak_kind} (timed region "
                                        f"{region_s:.2f} s at median {clocks.get('sm_mhz')} MHz)",
                         "traffic": BWD_TRAFFIC_BYTES if dominant == "attn_bwd" else None,
                         "traffic_note": BWD_TRAFFIC_NOTE if dominant == "attn_bwd" else None},
            "gpu_launches": launches,
            "clocks": clocks,
            "e2e": e2e,
            "breakdown_ms_per_step": {k: round(v, 4) for k, v in cat_total.items()},
            "attn_fwd_tflops": round(fwd_flop_per_call / (fwd_ms * 1e-3) / 1e12, 2),
            "attn_bwd_tflops": round(bwd_flop_per_call / (bwd_ms * 1e-3) / 1e12, 2),
            "attn_fwd_frac": round(fwd_flop_per_call / (fwd_ms * 1e-3) / 1e12 / peak, 4),
            "per_rank": per_rank,
            "gather": {"partition_gather_gbs": None if gather_gbs is None else round(gather_gbs, 1),
                       "restore_gather_gbs": None if restore_gbs is None else round(restore_gbs, 1),
                       "hbm_peak_gbs": hbm,
                       "frac": None if gather_gbs is None else round(gather_gbs / hbm, 4)},
            "pairs_per_step": pairs,
            "secondary": secondary,
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


def _e2e(args, wl, strategies, host, g, atts, step, flop_step, ws, dev):
    """End to end through the public API: pinned host inputs -> device, step,
    outputs -> pinned host, every step's copies inside the timed region.
    Serial form first (copy in, step, copy out, one after another), then the
    pipelined form the API allows: two sets of device inputs and of attention
    objects, the next step's inputs copied in and the previous step's outputs
    copied out on their own streams while a step computes."""
    import torch
    from context_packed_sequence_thd_gb300 import pipeline
    stream = torch.cuda.current_stream()
    pinned = {k: v.pin_memory() for k, v in host.items()}
    e2e_steps = max(2, min(args.steps, 20))
    outs = [t for a in atts for t in (a.oc, a.dqc, a.dkc, a.dvc)]
    host_outs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = sum(t.numel() * t.element_size() for t in outs)
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
    del g2, atts2, sets, outs_of, host_outs, pinned
    torch.cuda.empty_cache()
    return {"value": round(_whole_job_value(ws, flop_step, e2e_ms), 3),
            "unit": "TFLOP/s", "ms_per_step": round(e2e_ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": e2e_steps,
            "copies": "pinned host; next step's inputs in and previous step's outputs "
                      "out on copy streams, overlapped with the step",
            "serial": {"value": round(_whole_job_value(ws, flop_step, e2e_serial_ms), 3),
                       "ms_per_step": round(e2e_serial_ms, 4)}}


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
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["own", "reference"], default="own")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--capture", action="store_true",
                    help="run warm-up + --steps headline steps only (for ncu captures)")
    ap.add_argument("--workload", choices=["cfg5", "cfg2", "cfg3"], default="cfg5",
                    help="with --capture only: cfg2 (32768 tokens, H=16, fwd+bwd) or cfg3 (one "
                         "32768-token sequence, cp=8, H=40, forward only) for smaller ncu captures")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload != "cfg5" and not args.capture:
        ap.error("--workload cfg2 / cfg3 are for --capture runs only")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_own(args)


if __name__ == "__main__":
    main()
