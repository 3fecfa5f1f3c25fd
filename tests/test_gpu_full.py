"""Parity at the full workload sizes, in the launch configuration bench.py
times (every rank of the emulated CP group, both strategies where the
workload has them).  For the forward+backward workloads the oracle computes
every head exactly and the GPU result is compared element by element; the
single-sequence forward and the ring are checked on a head the oracle computes
(heads are independent); the integer parts are checked for every row.  The
worst errors per tensor are printed (pytest -s) for the record."""
import numpy as np
import pytest
import torch

import oracle
from context_packed_sequence_thd_gb300 import api, inputs, pipeline
from gpu_util import assert_close, assert_lse_close, dev, to_np

pytestmark = pytest.mark.gpu


def _heads_slice(t, heads):
    return {k: v[:, heads].contiguous() for k, v in t.items()}


def _run_all(wl, strategy, d, g, bwd, cls=pipeline.CPAttention, operand_dtype=None, **kw):
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, strategy, wl.pad_between_seqs, wl.H, wl.D, d)
    att = cls(plan, operand_dtype=operand_dtype, **kw)
    att.step(g["q"], g["k"], g["v"], g["do"] if bwd else None)
    torch.cuda.synchronize()
    assert api.cp_device_status() == 0
    return plan, att


def _worst(acc, name, err):
    acc[name] = max(acc.get(name, 0.0), err[0])


def _compare(wl, plan, att, heads, o, lse, grads, rows_of_interest=None, acc=None):
    acc = {} if acc is None else acc
    for r in range(wl.cp):
        rows = oracle.partition_index(wl.cup, wl.cp, r, plan.strategy)
        np.testing.assert_array_equal(plan.ranks[r].idx.cpu().numpy(), rows)
        sel = slice(None) if rows_of_interest is None else rows_of_interest[rows]
        _worst(acc, "O", assert_close(to_np(plan.local(att.oc, r)[:, heads])[sel], o[rows][sel],
                                      f"O rank {r}"))
        assert_lse_close(to_np(att.lse[r][heads])[:, sel], lse[:, rows][:, sel], f"LSE rank {r}")
        if grads is not None:
            dq, dk, dv = grads
            for name, buf, ref in (("dQ", att.dqc, dq), ("dK", att.dkc, dk), ("dV", att.dvc, dv)):
                _worst(acc, name, assert_close(to_np(plan.local(buf, r)[:, heads])[sel],
                                               ref[rows][sel], f"{name} rank {r} heads {heads}"))
    return acc


def _compare_acc(att, heads, dk, dv, what, acc):
    """The fp32 dK/dV sums over ranks (original order) before the bf16 cast."""
    _worst(acc, "dK fp32", assert_close(to_np(att.dk_acc[:, heads]), dk, f"{what} dK fp32 sum"))
    _worst(acc, "dV fp32", assert_close(to_np(att.dv_acc[:, heads]), dv, f"{what} dV fp32 sum"))


# Every head of every workload with a backward: the heads are independent, so
# the oracle computes them in groups of 8 while the GPU results of both
# strategies and both tensor-core operand types (fp16, the default, with the
# reduce-scatter inside the dK/dV kernel as timed; bf16 with two-term P and dS,
# with the reduce-scatter as its own pass over fp32 sums, which are checked
# too) stay on the device.  No head is left out, so no head can hide an
# out-of-tolerance element.
@pytest.mark.parametrize("make", [inputs.cfg2, inputs.cfg4, inputs.cfg5], ids=["cfg2", "cfg4", "cfg5"])
def test_full_size_fwd_bwd_all_heads(make):
    d = dev()
    wl = make()
    t = wl.tensors()
    g = {k: v.to(d) for k, v in t.items()}
    pad = wl.pad_between_seqs
    runs = [_run_all(wl, strategy, d, g, True, operand_dtype=dt, fused_rs=dt == torch.float16)
            for strategy in wl.strategies for dt in (torch.float16, torch.bfloat16)]
    worst = [{} for _ in runs]
    for h0 in range(0, wl.H, 8):
        heads = list(range(h0, min(h0 + 8, wl.H)))
        s = _heads_slice(t, heads)
        o, lse = oracle.attn_fwd(s["q"], s["k"], s["v"], wl.cu, wl.cup, pad)
        grads = oracle.attn_bwd(s["q"], s["k"], s["v"], o, lse, s["do"], wl.cu, wl.cup, pad)
        for (plan, att), acc in zip(runs, worst):
            _compare(wl, plan, att, heads, o, lse, grads, acc=acc)
            if att.dk_acc is not None:
                _compare_acc(att, heads, grads[1], grads[2], f"heads {heads}", acc)
    for (plan, att), acc in zip(runs, worst):
        print(f"\n{wl.name} {pipeline.STRATEGY_NAMES[plan.strategy]} {att.operand_dtype} worst "
              f"max-abs over all {wl.H} heads: " + ", ".join(f"{k} {v:.5f}" for k, v in acc.items()))


@pytest.mark.parametrize("make,heads", [(inputs.cfg2, [3]), (inputs.cfg5, [0])],
                         ids=["cfg2", "cfg5"])
def test_full_size_p2p_ring(make, heads):
    """The emulated P2P ring (per-step attention, LSE merge, per-step backward,
    fp32 dQ/dK/dV sums) at full size, both strategies, against the oracle on
    a subset of heads."""
    d = dev()
    wl = make()
    t = wl.tensors()
    g = {k: v.to(d) for k, v in t.items()}
    s = _heads_slice(t, heads)
    pad = wl.pad_between_seqs
    o, lse = oracle.attn_fwd(s["q"], s["k"], s["v"], wl.cu, wl.cup, pad)
    grads = oracle.attn_bwd(s["q"], s["k"], s["v"], o, lse, s["do"], wl.cu, wl.cup, pad)
    for strategy in wl.strategies:
        plan, att = _run_all(wl, strategy, d, g, True, cls=pipeline.CPP2PAttention)
        _compare(wl, plan, att, heads, o, lse, grads)
        del att


def test_cfg3_single_sequence_fwd_sampled_rows():
    """One 32768-token sequence, cp=8, H=40: forward of all 8 ranks for both
    strategies; the oracle computes head 17 on every 16th query row."""
    d = dev()
    wl = inputs.cfg3()
    t = wl.tensors(with_grad=False)
    g = {k: v.to(d) for k, v in t.items()}
    heads = [17]
    s = _heads_slice(t, heads)
    qm = np.zeros(wl.total_tokens, dtype=bool)
    qm[::16] = True
    qm[-3:] = True
    o, lse = oracle.attn_fwd(s["q"], s["k"], s["v"], wl.cu, wl.cup, 0, qmask=qm)
    for strategy in wl.strategies:
        plan, att = _run_all(wl, strategy, d, g, False)
        _compare(wl, plan, att, heads, o, lse, None, rows_of_interest=qm)


def test_cfg5_padding_arms():
    """pad_between_seqs with cu != cu_padded (arm A) against value-equal,
    no-padding metadata (arm B: cu := clone of cu_padded, detector -> 0, dO
    zero on the former padding rows): every real-token row agrees.  Arm C (no
    tail) launches no tail-zero kernel, arm A launches one on the rank that
    holds the tail."""
    d = dev()
    A = inputs.cfg5()
    B = inputs.cfg5(value_equal=True)
    assert api.cp_detect_pad_between_seqs(B.cu, B.cup) == 0 and B.pad_between_seqs == 0
    t = A.tensors()
    valid = oracle.valid_mask(A.cu, A.cup, 1)
    gA = {k: v.to(d) for k, v in t.items()}
    gB = dict(gA)
    gB["do"] = gA["do"].clone()
    gB["do"][torch.from_numpy(~valid).to(d)] = 0
    for strategy in A.strategies:
        pA, aA = _run_all(A, strategy, d, gA, True)
        pB, aB = _run_all(B, strategy, d, gB, True)
        for r in range(A.cp):
            rows = pA.ranks[r].idx.cpu().numpy()
            v = torch.from_numpy(valid[rows]).to(d)
            for name in ("oc", "dqc", "dkc", "dvc"):
                x = pA.local(getattr(aA, name), r)[v]
                y = pB.local(getattr(aB, name), r)[v]
                assert_close(to_np(x), to_np(y), f"{name} rank {r} arm A vs B",
                             max_abs=2e-2, mean_abs=2e-4)
        tail_ranks = [r for r, rm in enumerate(pA.ranks) if rm.valid_end < pA.s_local]
        assert len(tail_ranks) == 1
        del aA, aB
    C = inputs.cfg5(tail=False)
    for strategy in C.strategies:
        plan = pipeline.CPPlan(C.cu, C.cup, C.cp, strategy, 1, C.H, C.D, d)
        assert all(rm.valid_end == plan.s_local for rm in plan.ranks)
        x = torch.zeros(plan.s_local, 1, 64, dtype=torch.bfloat16, device=d)
        assert api.cp_zero_tail([x], plan.ranks[0].valid_end) is False
