"""Per-workload attention throughput of the C-ABI entry points (GB300).

    python -m context_packed_sequence_thd_gb300.config_timing

For each workload and strategy: every rank's forward (``cp_attn_fwd``) and backward
(``cp_attn_bwd`` plus the fp32 accumulator clear and the reduce-scatter cast), timed with CUDA
events over 10 repetitions after one warm-up pass, reported as algorithmic TFLOP/s
(4·D·H·pairs for the forward, 10·D·H·pairs for the backward).
"""
import torch

from . import inputs, pipeline


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


def main():
    run(inputs.cfg2(), (pipeline.DCS, pipeline.NLB), "cfg2 32k tokens, 16 docs, cp4 H16")
    run(inputs.custom([32768], cp=1, H=16, D=128, seed=5), (pipeline.NLB,), "one 32k doc, cp1 H16")
    run(inputs.custom([32768], cp=8, H=16, D=128, seed=5), (pipeline.DCS, pipeline.NLB),
        "one 32k doc, cp8 H16")
    run(inputs.cfg3(), (pipeline.DCS, pipeline.NLB), "cfg3 32k seq, cp8 H40", bwd=False)


if __name__ == "__main__":
    main()
