"""Parity at the full workload sizes, in the launch configuration bench.py
times (every rank of the emulated CP group, both strategies where the
workload has them).  The oracle computes a subset of heads exactly (heads are
independent), and the GPU result for those heads is compared element by
element; the integer parts are checked for every row."""
import numpy as np
import pytest
import torch

import oracle
from context_packed_sequence_thd_gb300 import api, inputs, pipeline
from gpu_util import assert_close, assert_lse_close, dev, to_np

pytestmark = pytest.mark.gpu


def _heads_slice(t, heads):
    return {k: v[:, heads].contiguous() for k, v in t.items()}


def _run_all(wl, strategy, d, g, bwd, cls=pipeline.CPAttention):
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, strategy, wl.pad_between_seqs, wl.H, wl.D, d)
    att = cls(plan)
    att.step(g["q"], g["k"], g["v"], g["do"] if bwd else None)
    torch.cuda.synchronize()
    assert api.cp_device_status() == 0
    return plan, att


def _compare(wl, plan, att, heads, o, lse, grads, rows_of_interest=None):
    for r in range(wl.cp):
        rows = oracle.partition_index(wl.cup, wl.cp, r, plan.strategy)
        np.testing.assert_array_equal(plan.ranks[r].idx.cpu().numpy(), rows)
        sel = slice(None) if rows_of_interest is None else rows_of_interest[rows]
        assert_close(to_np(plan.local(att.oc, r)[:, heads])[sel], o[rows][sel], f"O rank {r}")
        assert_lse_close(to_np(att.lse[r][heads])[:, sel], lse[:, rows][:, sel], f"LSE rank {r}")
        if grads is not None:
            dq, dk, dv = grads
            assert_close(to_np(plan.local(att.dqc, r)[:, heads])[sel], dq[rows][sel], f"dQ rank {r}")
            assert_close(to_np(plan.local(att.dkc, r)[:, heads])[sel], dk[rows][sel], f"dK rank {r}")
            assert_close(to_np(plan.local(att.dvc, r)[:, heads])[sel], dv[rows][sel], f"dV rank {r}")


@pytest.mark.parametrize("make,heads,bwd", [
    (inputs.cfg2, [0, 15], True),
    (inputs.cfg4, [39], True),
    (inputs.cfg5, [0], True),
], ids=["cfg2", "cfg4", "cfg5"])
def test_full_size_fwd_bwd(make, heads, bwd):
    d = dev()
    wl = make()
    t = wl.tensors()
    g = {k: v.to(d) for k, v in t.items()}
    s = _heads_slice(t, heads)
    pad = wl.pad_between_seqs
    o, lse = oracle.attn_fwd(s["q"], s["k"], s["v"], wl.cu, wl.cup, pad)
    grads = oracle.attn_bwd(s["q"], s["k"], s["v"], o, lse, s["do"], wl.cu, wl.cup, pad)
    for strategy in wl.strategies:
        plan, att = _run_all(wl, strategy, d, g, bwd)
        _compare(wl, plan, att, heads, o, lse, grads)
        del att


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
