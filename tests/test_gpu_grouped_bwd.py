"""The rank-grouped backward (cp_attn_bwd_grouped) against the rank-by-rank one
(cp_attn_bwd_ex: rank 0 stores its partial dK/dV, the others add theirs) and
against the fp64 oracle.

"[PyTorch] Add no-load-balance THD all-gather CP", §Sequence Diagram: every
rank computes a partial dK/dV over the all-gathered keys and the group sums
them (reduce-scatter).  The grouped call forms the same sum inside one dK/dV
launch, each key block accumulating the terms of every rank's attending query
tiles in its tensor-core accumulator.  dQ is computed by the same per-rank dQ
launches in both paths (bitwise equal); the fp32 dK/dV sums differ only in
rounding order.  The fused form (cp_attn_bwd_grouped_rs) also does the
reduce-scatter's scatter and bf16 cast in the dK/dV kernel's epilogue; its
rank-concatenated dK/dV must be bitwise those of the grouped call followed by
cp_reduce_scatter_emul."""
import numpy as np
import pytest
import torch

import oracle
from context_packed_sequence_thd_gb300 import api, inputs, pipeline
from gpu_util import assert_close, dev, to_np

pytestmark = pytest.mark.gpu

CASES = {
    # several documents per tile, ragged tail, padding between sequences
    "docs_cp4_d128": lambda: inputs.custom([176, 272, 64, 400, 112], cp=4, H=3, D=128, seed=91),
    "docs_cp2_d64": lambda: inputs.custom([300, 44, 212, 60], cp=2, H=2, D=64, seed=92),
    # one long document: every key block attended by every rank's later rows
    "long_cp8_d128": lambda: inputs.custom([2048], cp=8, H=2, D=128, seed=93, pad_between_seqs=0),
}


def _step(wl, t, strategy, grouped, operand_dtype, fused_rs=False):
    d = dev()
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, strategy, wl.pad_between_seqs, wl.H, wl.D, d)
    att = pipeline.CPAttention(plan, operand_dtype=operand_dtype, grouped_bwd=grouped,
                               fused_rs=fused_rs)
    g = {k: v.to(d) for k, v in t.items()}
    att.step(g["q"], g["k"], g["v"], g["do"])
    torch.cuda.synchronize()
    assert api.cp_device_status() == 0
    return plan, att


@pytest.mark.parametrize("operand_dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("strategy", [pipeline.DCS, pipeline.NLB])
@pytest.mark.parametrize("case", sorted(CASES))
def test_grouped_matches_rank_by_rank_and_oracle(case, strategy, operand_dtype):
    wl = CASES[case]()
    t = wl.tensors()
    plan_g, g = _step(wl, t, strategy, True, operand_dtype)
    plan_r, r = _step(wl, t, strategy, False, operand_dtype)
    _, f = _step(wl, t, strategy, True, operand_dtype, fused_rs=True)
    # dQ: the same per-rank launches
    assert torch.equal(g.dqc, r.dqc)
    # the fused reduce-scatter: bitwise the grouped sums cast by the separate pass
    for name in ("dqc", "dkc", "dvc"):
        assert torch.equal(getattr(f, name).view(torch.int16),
                           getattr(g, name).view(torch.int16)), name
    # dK / dV fp32 sums: the same terms, another rounding order
    for name in ("dk_acc", "dv_acc"):
        a, b = to_np(getattr(g, name)), to_np(getattr(r, name))
        scale = max(1.0, float(np.abs(b).max()))
        assert np.abs(a - b).max() <= 1e-5 * scale, (name, float(np.abs(a - b).max()))
    # and both within the bound of the fp64 oracle
    pad = wl.pad_between_seqs
    o, lse = oracle.attn_fwd(t["q"], t["k"], t["v"], wl.cu, wl.cup, pad)
    dq, dk, dv = oracle.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], wl.cu, wl.cup, pad)
    assert_close(to_np(g.dk_acc), dk, "dK fp32 (grouped)")
    assert_close(to_np(g.dv_acc), dv, "dV fp32 (grouped)")
    for rk in range(wl.cp):
        rows = oracle.partition_index(wl.cup, wl.cp, rk, strategy)
        assert_close(to_np(plan_g.local(g.dkc, rk)), dk[rows], f"dK rank {rk}")
        assert_close(to_np(plan_g.local(g.dvc, rk)), dv[rows], f"dV rank {rk}")
        assert_close(to_np(plan_g.local(g.dqc, rk)), dq[rows], f"dQ rank {rk}")


def test_grouped_is_deterministic():
    wl = CASES["docs_cp4_d128"]()
    t = wl.tensors()
    _, a = _step(wl, t, pipeline.DCS, True, torch.float16)
    _, b = _step(wl, t, pipeline.DCS, True, torch.float16)
    assert torch.equal(a.dk_acc, b.dk_acc) and torch.equal(a.dv_acc, b.dv_acc)
    _, a = _step(wl, t, pipeline.DCS, True, torch.float16, fused_rs=True)
    _, b = _step(wl, t, pipeline.DCS, True, torch.float16, fused_rs=True)
    assert torch.equal(a.dkc, b.dkc) and torch.equal(a.dvc, b.dvc)


def test_grouped_refuses_metadata_of_another_strategy():
    """Every rank's metadata is checked on the device: the other strategy's
    set writes nothing and reports CP_ERR_METADATA."""
    d = dev()
    wl = CASES["docs_cp4_d128"]()
    t = wl.tensors()
    plan, att = _step(wl, t, pipeline.DCS, True, torch.float16)
    other = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, pipeline.NLB, wl.pad_between_seqs, wl.H, wl.D, d)
    sentinel = 3.0
    dk = torch.full_like(att.dk_acc, sentinel)
    dv = torch.full_like(att.dv_acc, sentinel)
    api.cp_attn_bwd_grouped(att.qc, att.k_full, att.v_full, att.oc, att.lse, att.doc, att.dqc,
                            dk, dv, other.meta_all, other.meta_stride, plan.T, plan.cp,
                            pipeline.DCS, plan.scale, att.ws_grouped, o_resid_all=att.oc_resid)
    torch.cuda.synchronize()
    assert api.cp_device_status(reset=True) == -7  # CP_ERR_METADATA
    assert torch.all(dk == sentinel) and torch.all(dv == sentinel)


def test_fused_reduce_scatter_refuses_metadata_of_another_strategy():
    """The fused form checks every rank's metadata on the device too: the
    other strategy's set leaves dK/dV unwritten and reports CP_ERR_METADATA."""
    d = dev()
    wl = CASES["docs_cp4_d128"]()
    t = wl.tensors()
    plan, att = _step(wl, t, pipeline.DCS, True, torch.float16, fused_rs=True)
    other = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, pipeline.NLB, wl.pad_between_seqs, wl.H, wl.D, d)
    dk = torch.full_like(att.dkc, 3.0)
    dv = torch.full_like(att.dvc, 3.0)
    api.cp_attn_bwd_grouped_rs(att.qc, att.k_full, att.v_full, att.oc, att.lse, att.doc,
                               att.dqc, dk, dv, plan.restore, other.meta_all, other.meta_stride,
                               plan.T, plan.cp, pipeline.DCS, plan.scale, att.ws_grouped,
                               o_resid_all=att.oc_resid)
    torch.cuda.synchronize()
    assert api.cp_device_status(reset=True) == -7  # CP_ERR_METADATA
    assert torch.all(dk == 3.0) and torch.all(dv == 3.0)


def test_fused_reduce_scatter_skips_rows_of_a_bad_index():
    """Restore-index entries outside [0, T) (made on the host) are skipped and
    reported (CP_ERR_INVALID_ARG on the status word); every other row is
    written as with the valid index."""
    d = dev()
    wl = CASES["docs_cp2_d64"]()
    t = wl.tensors()
    plan, att = _step(wl, t, pipeline.DCS, True, torch.float16, fused_rs=True)
    bad = plan.restore.clone()
    rows = [3, plan.T - 1]
    bad[rows[0]] = -1
    bad[rows[1]] = plan.T
    dk = torch.full_like(att.dkc, 3.0)
    dv = torch.full_like(att.dvc, 3.0)
    api.cp_attn_bwd_grouped_rs(att.qc, att.k_full, att.v_full, att.oc, att.lse, att.doc,
                               att.dqc, dk, dv, bad, plan.meta_all, plan.meta_stride, plan.T,
                               plan.cp, pipeline.DCS, plan.scale, att.ws_grouped,
                               o_resid_all=att.oc_resid)
    torch.cuda.synchronize()
    assert api.cp_device_status(reset=True) == -1  # CP_ERR_INVALID_ARG
    skipped = plan.restore[rows].long()
    keep = torch.ones(plan.T, dtype=torch.bool, device=d)
    keep[skipped] = False
    assert torch.equal(dk[keep], att.dkc[keep]) and torch.equal(dv[keep], att.dvc[keep])
    assert torch.all(dk[skipped] == 3.0) and torch.all(dv[skipped] == 3.0)
