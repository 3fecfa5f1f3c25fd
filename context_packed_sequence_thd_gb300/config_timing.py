"""Per-workload attention throughput of the C-ABI entry points (GB300), and
the emulated a2a and P2P comm types (exchange GB/s, attention TFLOP/s).

    python -m context_packed_sequence_thd_gb300.config_timing

For each workload and strategy: every rank's forward (``cp_attn_fwd``) and backward
(``cp_attn_bwd`` plus the fp32 accumulator clear and the reduce-scatter cast), timed with CUDA
events over 10 repetitions after one warm-up pass, reported as algorithmic TFLOP/s
(4·D·H·pairs for the forward, 10·D·H·pairs for the backward).
"""
import torch

from . import api, inputs, pipeline


def run(wl, strategies, label, bwd=True, reps=10, dev=None):
    dev = dev or torch.device("cuda", torch.cuda.current_device())
    t = {k: v.to(dev) for k, v in wl.tensors(with_grad=bwd).items()}
    rows = []
    for s in strategies:
        plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, s, wl.pad_between_seqs, wl.H, wl.D, dev)
        att = pipeline.CPAttention(plan)
        att.shard_inputs(t["q"], t["k"], t["v"], t.get("do"))
        kf, vf = att.forward()
        if bwd:
            att.backward(kf, vf)
        torch.cuda.synchronize()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        for _ in range(reps):
            att.forward()
        e[1].record()
        if bwd:
            for _ in range(reps):
                att.backward(kf, vf)
        e[2].record()
        torch.cuda.synchronize()
        f = att.flops(bwd)
        tf = f["fwd"] / (e[0].elapsed_time(e[1]) / reps) / 1e9
        tb = f["bwd"] / (e[1].elapsed_time(e[2]) / reps) / 1e9 if bwd else None
        rows.append((label, s, tf, tb))
        msg = f"{label:32s} strategy {s}: fwd {tf:7.1f} TFLOP/s"
        if bwd:
            msg += f"   bwd {tb:7.1f} TFLOP/s"
        print(msg, flush=True)
    return rows


def a2a_exchange(T, cp, H, D, strategy, reps=20, dev=None):
    """GB/s of the seq->head exchange of Q, K and V (the a2a page's before_attn
    exchange) for one document of T tokens; under DUAL_CHUNK_SWAP the restore
    reorder is part of the same pass."""
    dev = dev or torch.device("cuda", torch.cuda.current_device())
    wl = inputs.custom([T], cp=cp, H=H, D=D, seed=7)
    plan = pipeline.CPPlan(wl.cu, wl.cup, cp, strategy, 0, H, D, dev)
    g = torch.Generator(device="cpu").manual_seed(7)
    seq = [torch.randn(T, H, D, generator=g).bfloat16().to(dev) for _ in range(3)]
    head = [torch.empty(cp, T, H // cp, D, dtype=torch.bfloat16, device=dev) for _ in range(3)]
    perm = plan.restore if strategy == pipeline.DCS else None
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # larger than L2

    def timed(fn):
        fn()
        ms = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        ms.sort()
        return ms[len(ms) // 2]

    t = timed(lambda: api.cp_a2a_exchange(seq, head, perm, cp, api.A2A_SEQ_TO_HEAD))
    nbytes = 3 * 2 * T * H * D * 2 + (4 * T if perm is not None else 0)
    gbs = nbytes / (t * 1e-3) / 1e9
    name = "dual_chunk_swap" if strategy == pipeline.DCS else "no_load_balance"
    print(f"a2a q+k+v exchange, s={T:6d} cp={cp} H={H} D={D} {name:16s}: "
          f"{t * 1e3:8.1f} us  {gbs:7.1f} GB/s", flush=True)
    if perm is not None:
        # the pages' dual-chunk path: the exchange in rank order, then a
        # separate index_select to the original order (per head slice)
        tmp = [torch.empty_like(h) for h in head]
        rows = (torch.arange(cp, device=dev, dtype=torch.int64)[:, None] * T +
                perm.to(torch.int64)[None, :]).reshape(-1).to(torch.int32)
        flat_t = [x.view(cp * T, H // cp, D) for x in tmp]
        flat_h = [x.view(cp * T, H // cp, D) for x in head]

        def unfused():
            api.cp_a2a_exchange(seq, tmp, None, cp, api.A2A_SEQ_TO_HEAD)
            api.cp_thd_gather(flat_t, flat_h, rows)
        t2 = timed(unfused)
        print(f"a2a q+k+v exchange, s={T:6d} cp={cp} H={H} D={D} {'dual_chunk_swap, exchange + separate reorder':16s}: "
              f"{t2 * 1e3:8.1f} us  ({t2 / t:.2f}x the fused pass)", flush=True)
    return t, gbs


COMM_TYPES = {"a2a": pipeline.CPA2AAttention, "p2p": pipeline.CPP2PAttention}


def run_comm(wl, strategies, label, comm, reps=10, dev=None):
    """Forward / backward TFLOP/s of the emulated a2a or P2P comm type (its
    exchanges, merges and casts included), with the time of each phase."""
    dev = dev or torch.device("cuda", torch.cuda.current_device())
    t = {k: v.to(dev) for k, v in wl.tensors(with_grad=True).items()}
    for s in strategies:
        plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, s, wl.pad_between_seqs, wl.H, wl.D, dev)
        att = COMM_TYPES[comm](plan)
        att.shard_inputs(t["q"], t["k"], t["v"], t["do"])
        att.forward()
        att.backward()
        torch.cuda.synchronize()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        for _ in range(reps):
            att.forward()
        e[1].record()
        for _ in range(reps):
            att.backward()
        e[2].record()
        torch.cuda.synchronize()
        f = att.flops(True)
        tf = f["fwd"] / (e[0].elapsed_time(e[1]) / reps) / 1e9
        tb = f["bwd"] / (e[1].elapsed_time(e[2]) / reps) / 1e9
        att.events = {}
        att.forward()
        att.backward()
        torch.cuda.synchronize()
        phases = "  ".join(f"{k} {sum(v):.3f} ms" for k, v in att.event_ms().items())
        print(f"{label:32s} {comm} strategy {s}: fwd {tf:7.1f} TFLOP/s   bwd {tb:7.1f} TFLOP/s"
              f"   [{phases}]", flush=True)


def p2p_index_time(wl, strategy, reps=20, dev=None):
    """Time of the ring metadata of every rank: one cp_p2p_index launch per rank."""
    dev = dev or torch.device("cuda", torch.cuda.current_device())
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, strategy, wl.pad_between_seqs, wl.H, wl.D, dev)
    att = pipeline.CPP2PAttention(plan)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        att.build_p2p_index()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) / reps * 1e3
    print(f"{wl.name:32s} p2p metadata, {wl.cp} ranks x {wl.cp} steps, strategy {strategy}: "
          f"{us:7.1f} us ({wl.cp} launches)", flush=True)


def fused_gather_timing(wl, reps=10, dev=None):
    """Forward-only DUAL_CHUNK_SWAP step (shard gather + restore + every rank's
    forward) with the Q shard gathered by a copy kernel and with the gather
    fused into the attention's loads (cp_attn_fwd_gather)."""
    dev = dev or torch.device("cuda", torch.cuda.current_device())
    t = {k: v.to(dev) for k, v in wl.tensors(with_grad=False).items()}
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, pipeline.DCS, wl.pad_between_seqs, wl.H, wl.D,
                           dev)
    out = {}
    for fuse in (False, True):
        att = pipeline.CPAttention(plan, fuse_q_gather=fuse)
        att.step(t["q"], t["k"], t["v"], rebuild_index=False)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            att.step(t["q"], t["k"], t["v"], rebuild_index=False)
        e1.record()
        torch.cuda.synchronize()
        out[fuse] = e0.elapsed_time(e1) / reps
        att.events = {}
        att.step(t["q"], t["k"], t["v"], rebuild_index=False)
        torch.cuda.synchronize()
        phases = "  ".join(f"{k} {sum(v):.3f} ms" for k, v in att.event_ms().items())
        tf = att.flops(False)["fwd"] / (out[fuse] * 1e-3) / 1e12
        print(f"{wl.name:32s} fwd-only DCS step, {'fused Q gather' if fuse else 'Q shard copy  '}: "
              f"{out[fuse]:.3f} ms ({tf:6.1f} TFLOP/s)  [{phases}]", flush=True)
    return out


def main():
    run(inputs.cfg2(), (pipeline.DCS, pipeline.NLB), "cfg2 32k tokens, 16 docs, cp4 H16")
    run(inputs.custom([32768], cp=1, H=16, D=128, seed=5), (pipeline.NLB,), "one 32k doc, cp1 H16")
    run(inputs.custom([32768], cp=8, H=16, D=128, seed=5), (pipeline.DCS, pipeline.NLB),
        "one 32k doc, cp8 H16")
    run(inputs.cfg3(), (pipeline.DCS, pipeline.NLB), "cfg3 32k seq, cp8 H40", bwd=False)
    for s in (8192, 32768, 75600):
        fused_gather_timing(inputs.cfg3(s))
    run_comm(inputs.cfg2(), (pipeline.DCS, pipeline.NLB), "cfg2 32k tokens, 16 docs, cp4 H16",
             "a2a")
    run_comm(inputs.cfg2(), (pipeline.DCS, pipeline.NLB), "cfg2 32k tokens, 16 docs, cp4 H16",
             "p2p")
    for wl in (inputs.cfg5(), inputs.cfg5(value_equal=True)):
        label = f"{wl.name} 64k padded, 24 docs, cp4 H32"
        run(wl, (pipeline.DCS, pipeline.NLB), label)
        run_comm(wl, (pipeline.DCS, pipeline.NLB), label, "p2p")
        for s in (pipeline.DCS, pipeline.NLB):
            p2p_index_time(wl, s)
    for T in (8192, 32768, 75600):
        for s in (pipeline.DCS, pipeline.NLB):
            a2a_exchange(T, 8, 40, 128, s)


if __name__ == "__main__":
    main()
