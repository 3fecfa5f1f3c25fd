"""The allocation-free backward entry point, cp_attn_bwd_noalloc.

It exists for callers that cannot allocate device memory where they run the
backward (a runtime that only hands out memory from a pre-planned arena, a
plugin whose host framework owns the allocator, code that must not pay the
device synchronisation of cudaMalloc/cudaFree).  Its scratch is a fixed
array inside the library, so these tests check, through the C ABI, that it
gives the same dQ and dK/dV as cp_attn_bwd with a caller workspace on two
calls in a row (the second call sees the first call's scratch contents), and
that an oversized problem is refused before anything is launched.

This file is collected last on purpose: if it fails, every other test has
already run.
"""
import ctypes

import pytest
import torch

from context_packed_sequence_thd_gb300 import api, inputs, pipeline
from gpu_util import assert_close, dev, to_np

pytestmark = pytest.mark.gpu


def _forward(wl, strategy, d, seed_shift, operand_dtype):
    t = wl.tensors()
    if seed_shift:
        g = torch.Generator().manual_seed(wl.seed + seed_shift)
        t["do"] = torch.randn(t["do"].shape, generator=g).bfloat16()
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, strategy, wl.pad_between_seqs, wl.H, wl.D, d)
    att = pipeline.CPAttention(plan, operand_dtype=operand_dtype)
    g = {k: v.to(d) for k, v in t.items()}
    att.shard_inputs(g["q"], g["k"], g["v"], g["do"])
    kf, vf = att.forward()
    return plan, att, kf, vf


def _backward(plan, att, kf, vf, noalloc):
    T, H, D = att.dqc.shape
    dq = torch.zeros_like(att.dqc)
    dk = torch.zeros(T, H, D, dtype=torch.float32, device=dq.device)
    dv = torch.zeros_like(dk)
    for r in range(plan.cp):
        args = (plan.local(att.qc, r), kf, vf, plan.local(att.oc, r), att.lse[r],
                plan.local(att.doc, r), plan.local(dq, r), dk, dv, plan.ranks[r].meta, plan.T,
                plan.cp, r, plan.strategy, plan.scale)
        o_resid = plan.local(att.oc_resid, r)
        if noalloc:
            api.cp_attn_bwd_noalloc(*args, o_resid=o_resid)
        else:
            api.cp_attn_bwd(*args, att.ws, o_resid=o_resid)
    torch.cuda.synchronize()
    assert api.cp_device_status() == 0
    return dq, dk, dv


@pytest.mark.parametrize("operand_dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("strategy", [pipeline.DCS, pipeline.NLB], ids=["dcs", "nlb"])
def test_noalloc_backward_matches_workspace_backward_twice(strategy, operand_dtype):
    d = dev()
    cases = [inputs.custom([176, 272, 64], cp=4, H=3, D=128, seed=81),
             inputs.custom([100, 7, 250, 33], padded=[112, 16, 256, 48], cp=4, H=2, D=64, seed=82)]
    for wl in cases:
        for call in range(2):  # two calls in a row: the scratch keeps the previous contents
            plan, att, kf, vf = _forward(wl, strategy, d, call, operand_dtype)
            ref = _backward(plan, att, kf, vf, noalloc=False)
            got = _backward(plan, att, kf, vf, noalloc=True)
            for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
                assert_close(to_np(a), to_np(b), f"{name} call {call}")
                assert torch.equal(a, b), f"{name} call {call}: same kernels, same order"


def test_noalloc_rejects_sizes_beyond_the_scratch():
    """s_local * H above CP_NOALLOC_MAX_SCRATCH_FLOATS is refused before any
    launch (the pointers below are never dereferenced)."""
    api.lib()
    L = api.lib()
    fake = 0x10000
    T = 2 * api.NOALLOC_MAX_SCRATCH_FLOATS  # cp=1, H=1: s_local*H = 2x the maximum
    st = L.cp_attn_bwd_noalloc(fake, fake, fake, fake, None, fake, fake, fake, fake, fake, fake,
                               1 << 20, T, 1, 64, 1, 0, 1, ctypes.c_float(0.125), 0, None)
    assert st == -6
    assert api.status_string(st) == "CP_ERR_WORKSPACE"
