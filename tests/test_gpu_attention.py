"""GPU parity of the emulated context-parallel attention (fwd + bwd) against
the fp64 oracle, element by element, at sizes the oracle finishes in seconds
that still span several tiles and a ragged tail; plus the invariants the
pages fix: document isolation, padded vs value-equal metadata, the cp=1
equivalence of both strategies, and determinism."""
import numpy as np
import pytest
import torch

import oracle
from context_packed_sequence_thd_gb300 import api, inputs, pipeline
from gpu_util import assert_close, assert_lse_close, dev, to_np

pytestmark = pytest.mark.gpu


def run(wl, strategy, d, tensors=None, bwd=True, operand_dtype=None, fused_rs=True):
    t = wl.tensors() if tensors is None else tensors
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, strategy, wl.pad_between_seqs, wl.H, wl.D, d)
    att = pipeline.CPAttention(plan, operand_dtype=operand_dtype, fused_rs=fused_rs)
    g = {k: v.to(d) for k, v in t.items()}
    att.step(g["q"], g["k"], g["v"], g["do"] if bwd else None)
    torch.cuda.synchronize()
    assert api.cp_device_status() == 0
    return plan, att


def oracle_all(wl, t, bwd=True):
    pad = wl.pad_between_seqs
    o, lse = oracle.attn_fwd(t["q"], t["k"], t["v"], wl.cu, wl.cup, pad)
    if not bwd:
        return o, lse, None
    return o, lse, oracle.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], wl.cu, wl.cup, pad)


def check_against_oracle(wl, strategy, bwd=True, operand_dtype=None):
    d = dev()
    t = wl.tensors()
    o, lse, grads = oracle_all(wl, t, bwd)
    plan, att = run(wl, strategy, d, t, bwd, operand_dtype)
    for r in range(wl.cp):
        rows = oracle.partition_index(wl.cup, wl.cp, r, strategy)
        np.testing.assert_array_equal(plan.ranks[r].idx.cpu().numpy(), rows)
        assert_close(to_np(plan.local(att.oc, r)), o[rows], f"O rank {r}")
        assert_lse_close(to_np(att.lse[r]), lse[:, rows], f"LSE rank {r}")
        if bwd:
            dq, dk, dv = grads
            assert_close(to_np(plan.local(att.dqc, r)), dq[rows], f"dQ rank {r}")
            assert_close(to_np(plan.local(att.dkc, r)), dk[rows], f"dK rank {r}")
            assert_close(to_np(plan.local(att.dvc, r)), dv[rows], f"dV rank {r}")
    if bwd:
        # the reduce-scatter as a separate pass: its fp32 sums hold the cp=1
        # gradient before the cast, and its bf16 rows are bitwise the ones the
        # dK/dV kernel writes itself
        _, sep = run(wl, strategy, d, t, bwd, operand_dtype, fused_rs=False)
        assert_close(to_np(sep.dk_acc), grads[1], "dK fp32 accumulator")
        assert_close(to_np(sep.dv_acc), grads[2], "dV fp32 accumulator")
        for name in ("dqc", "dkc", "dvc"):
            assert torch.equal(getattr(att, name).view(torch.int16),
                               getattr(sep, name).view(torch.int16)), name


SMALL = {
    "tiny_fwd": (inputs.tiny, False),
    "tiny_fwdbwd": (inputs.tiny, True),
    "three_docs_d128": (lambda: inputs.custom([176, 272, 64], cp=4, H=3, D=128, seed=61), True),
    "padded_d64": (lambda: inputs.custom([100, 7, 250, 33], padded=[112, 16, 256, 48], cp=4,
                                         H=2, D=64, seed=62), True),
    "padded_d128_cp2": (lambda: inputs.custom([61, 190, 1, 300], padded=[64, 192, 4, 308], cp=2,
                                              H=2, D=128, seed=63), True),
    "empty_docs": (lambda: inputs.custom([0, 6, 0, 10, 0], padded=[4, 8, 0, 12, 8], cp=2, H=1,
                                         D=64, seed=64), True),
    "one_long_doc_cp8": (lambda: inputs.custom([1024], cp=8, H=2, D=128, seed=65), True),
    "cp1": (lambda: inputs.custom([130, 126], cp=1, H=2, D=64, seed=66), True),
}


# both tensor-core operand types: fp16 (the pipeline's default) and bf16
# (P and dS as two bf16 terms)
@pytest.mark.parametrize("operand_dtype", [torch.float16, torch.bfloat16], ids=["f16", "bf16"])
@pytest.mark.parametrize("strategy", [pipeline.DCS, pipeline.NLB], ids=["dcs", "nlb"])
@pytest.mark.parametrize("name", list(SMALL))
def test_parity_small(name, strategy, operand_dtype):
    make, bwd = SMALL[name]
    check_against_oracle(make(), strategy, bwd, operand_dtype)


def test_nlb_documents_not_divisible():
    """NO_LOAD_BALANCE needs no per-document divisibility (cfg4's property)."""
    wl = inputs.custom([101, 37, 211, 35], cp=4, H=2, D=128, seed=67)
    check_against_oracle(wl, pipeline.NLB, True)


def test_rank_partial_accumulators():
    """After each rank's backward the fp32 accumulators equal the oracle's sum
    of the partials of ranks 0..r (per-rank query masks)."""
    d = dev()
    wl = inputs.custom([200, 56, 128], cp=4, H=2, D=64, seed=68)
    t = wl.tensors()
    o, lse = oracle.attn_fwd(t["q"], t["k"], t["v"], wl.cu, wl.cup, 0)
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, pipeline.DCS, 0, wl.H, wl.D, d)
    att = pipeline.CPAttention(plan, fused_rs=False)
    g = {k: v.to(d) for k, v in t.items()}
    att.shard_inputs(g["q"], g["k"], g["v"], g["do"])
    kf, vf = att.forward()
    api.cp_zero_tail([att.dk_acc, att.dv_acc], 0)
    qm = np.zeros(wl.total_tokens, dtype=bool)
    for r in range(wl.cp):
        api.cp_attn_bwd(plan.local(att.qc, r), kf, vf, plan.local(att.oc, r), att.lse[r],
                        plan.local(att.doc, r), plan.local(att.dqc, r), att.dk_acc, att.dv_acc,
                        plan.ranks[r].meta, plan.T, plan.cp, r, plan.strategy, plan.scale, att.ws)
        torch.cuda.synchronize()
        qm[oracle.partition_index(wl.cup, wl.cp, r, pipeline.DCS)] = True
        _, dk_p, dv_p = oracle.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], wl.cu, wl.cup, 0,
                                        qmask=qm)
        assert_close(to_np(att.dk_acc), dk_p, f"dK partial through rank {r}")
        assert_close(to_np(att.dv_acc), dv_p, f"dV partial through rank {r}")


@pytest.mark.parametrize("strategy", [pipeline.DCS, pipeline.NLB], ids=["dcs", "nlb"])
def test_store_mode_starts_the_sum_bitwise(strategy):
    """Rank 0 in store mode over NaN-filled accumulators, then ranks 1.. adding,
    gives bitwise the accumulators of clear-then-add-all: every element is
    written, and the stored partial is what the first addition would give."""
    d = dev()
    wl = inputs.custom([200, 56, 128, 640], cp=4, H=2, D=64, seed=71)
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, strategy, 0, wl.H, wl.D, d)
    att = pipeline.CPAttention(plan, fused_rs=False)
    g = {k: v.to(d) for k, v in wl.tensors().items()}
    att.shard_inputs(g["q"], g["k"], g["v"], g["do"])
    kf, vf = att.forward()

    def run(first_mode):
        for r in range(wl.cp):
            api.cp_attn_bwd(plan.local(att.qc, r), kf, vf, plan.local(att.oc, r), att.lse[r],
                            plan.local(att.doc, r), plan.local(att.dqc, r), att.dk_acc, att.dv_acc,
                            plan.ranks[r].meta, plan.T, plan.cp, r, plan.strategy, plan.scale,
                            att.ws, mode=first_mode if r == 0 else api.BWD_ACCUMULATE)
        torch.cuda.synchronize()
        return att.dk_acc.clone(), att.dv_acc.clone()

    api.cp_zero_tail([att.dk_acc, att.dv_acc], 0)
    want = run(api.BWD_ACCUMULATE)
    att.dk_acc.fill_(float("nan"))
    att.dv_acc.fill_(float("nan"))
    got = run(api.BWD_STORE)
    assert api.cp_device_status() == 0
    for w, x in zip(want, got):
        assert torch.equal(w.view(torch.int32), x.view(torch.int32))


def test_document_isolation_bitwise():
    """Perturbing the other documents' K/V leaves a document's O, LSE and dQ
    bitwise unchanged on the GPU."""
    d = dev()
    wl = inputs.custom([192, 320, 128], cp=2, H=2, D=128, seed=69)
    t = wl.tensors()
    t2 = {k: v.clone() for k, v in t.items()}
    t2["k"][:192] = -t2["k"][:192]
    t2["v"][512:] = t2["v"][512:] * 2
    for s in (pipeline.DCS, pipeline.NLB):
        p1, a1 = run(wl, s, d, t)
        p2, a2 = run(wl, s, d, t2)
        for r in range(wl.cp):
            rows = p1.ranks[r].idx.cpu().numpy()
            sel = np.nonzero((rows >= 192) & (rows < 512))[0]
            for x1, x2 in ((a1.oc, a2.oc), (a1.dqc, a2.dqc)):
                assert torch.equal(p1.local(x1, r)[sel], p2.local(x2, r)[sel])
            assert torch.equal(a1.lse[r][:, sel], a2.lse[r][:, sel])


def test_value_equal_metadata_bitwise():
    """cu_seqlens_padded a value-equal clone of cu_seqlens: the detector says 0
    and pad_between_seqs=1 / 0 give bitwise identical results."""
    d = dev()
    base = inputs.custom([96, 160, 64], cp=2, H=2, D=64, seed=70)
    cup = base.cu.copy()
    assert api.cp_detect_pad_between_seqs(base.cu, cup) == 0
    t = base.tensors()
    outs = []
    for flag in (1, 0):
        wl = inputs.custom([96, 160, 64], cp=2, H=2, D=64, seed=70, pad_between_seqs=flag)
        wl.cup = cup
        outs.append(run(wl, pipeline.DCS, d, t))
    (_, a), (_, b) = outs
    for name in ("oc", "dqc", "dkc", "dvc"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert torch.equal(a.lse, b.lse)


def test_strategies_equal_cp1_result():
    """Both strategies' per-rank outputs, put back in original order, equal the
    cp=1 result (within the bf16 tolerance; tiling differs)."""
    d = dev()
    wl = inputs.custom([320, 192, 256], cp=4, H=2, D=128, seed=71)
    t = wl.tensors()
    wl1 = inputs.custom([320, 192, 256], cp=1, H=2, D=128, seed=71)
    _, a1 = run(wl1, pipeline.NLB, d, t)
    for s in (pipeline.DCS, pipeline.NLB):
        plan, a = run(wl, s, d, t)
        G = torch.cat([plan.ranks[r].idx.long() for r in range(wl.cp)])
        for name in ("oc", "dqc", "dkc", "dvc"):
            full = torch.empty_like(getattr(a, name))
            full[G] = getattr(a, name)
            assert_close(to_np(full), to_np(getattr(a1, name)), f"{name} strategy {s} vs cp=1")


def test_deterministic():
    d = dev()
    wl = inputs.custom([300, 212], cp=2, H=2, D=128, seed=72)
    t = wl.tensors()
    _, a = run(wl, pipeline.DCS, d, t)
    _, b = run(wl, pipeline.DCS, d, t)
    for name in ("oc", "dqc", "dkc", "dvc"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    _, a = run(wl, pipeline.DCS, d, t, fused_rs=False)
    _, b = run(wl, pipeline.DCS, d, t, fused_rs=False)
    for name in ("dk_acc", "dv_acc"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


def test_tail_zeroing_gated_in_pipeline():
    """With padding at the end (a tail) the pipeline clears it; without a tail
    no tail-zero kernel is launched."""
    d = dev()
    with_tail = inputs.custom([100, 57], padded=[104, 64], cp=2, H=1, D=64, seed=73)
    no_tail = inputs.custom([100, 64], padded=[104, 64], cp=2, H=1, D=64, seed=73)
    for wl, expect in ((with_tail, True), (no_tail, False)):
        plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, pipeline.NLB, 1, wl.H, wl.D, d)
        ends = [rm.valid_end for rm in plan.ranks]
        assert (ends[-1] < plan.s_local) == expect
        att = pipeline.CPAttention(plan)
        t = {k: v.to(d) for k, v in wl.tensors().items()}
        att.dqc.fill_(3.0)
        att.step(t["q"], t["k"], t["v"], t["do"])
        torch.cuda.synchronize()
        last = plan.local(att.dqc, wl.cp - 1)
        assert torch.all(last[ends[-1]:] == 0)

