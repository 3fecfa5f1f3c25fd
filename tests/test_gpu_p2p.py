"""GPU parity of the emulated P2P (ring) comm type ("THD P2P context-parallel
regression when padded cu_seqlens are value-equal but not object-identical",
§Describe the bug): the per-step metadata of every ring step bit-exact
against the oracle's brute force, the log-sum-exp merge against the oracle's
fp64 merge, and the full ring forward/backward against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from context_packed_sequence_thd_gb300 import api, inputs, pipeline
from gpu_util import assert_close, assert_lse_close, check_block_lists, dev, to_np

pytestmark = pytest.mark.gpu

META_CASES = {
    "tiny": inputs.tiny,
    "cfg2": inputs.cfg2,
    "padded_cp4": lambda: inputs.custom([1000, 3, 2500, 600, 77, 900],
                                        padded=[1008, 8, 2504, 608, 80, 904], cp=4),
    "value_equal_cp4": lambda: inputs.custom([1008, 8, 2504, 608, 80, 904],
                                             padded=[1008, 8, 2504, 608, 80, 904], cp=4),
    "ragged_padded_cp4": lambda: inputs.custom([7, 33, 1, 90], cp=4, padded=[8, 40, 8, 96]),
    "empty_docs_cp2": lambda: inputs.custom([0, 6, 0, 10], padded=[4, 8, 0, 12], cp=2),
    "cp1": lambda: inputs.custom([3, 5], padded=[4, 12], cp=1),
}


def _hdr(meta: torch.Tensor) -> np.ndarray:
    return meta[:64].cpu().numpy().view(np.int32)


@pytest.mark.parametrize("name", list(META_CASES))
def test_p2p_step_metadata_bit_exact(name):
    """Every ring step's row tables equal the oracle's brute-force visible key
    range, its header is the cp_size = 1 call's, and its block lists and work
    order agree with the row tables."""
    d = dev()
    wl = META_CASES[name]()
    pad = wl.pad_between_seqs
    S = wl.s_local
    for s in wl.strategies:
        nbytes = api.cp_p2p_meta_bytes(wl.n_docs, wl.total_tokens, wl.cp)
        assert nbytes > 0 and nbytes % 16 == 0
        d_cu = torch.from_numpy(np.asarray(wl.cu, dtype=np.int32)).to(d)
        d_cup = torch.from_numpy(np.asarray(wl.cup, dtype=np.int32)).to(d)
        for r in range(wl.cp):
            meta = torch.full((wl.cp * nbytes,), 0xAB, dtype=torch.uint8, device=d)
            api.cp_p2p_index(d_cu if pad else None, d_cup, wl.total_tokens, wl.cp, r, s, pad, meta)
            torch.cuda.synchronize()
            assert api.cp_device_status() == 0
            for i, j in enumerate(oracle.p2p_schedule(wl.cp, r)):
                m = meta[i * nbytes:(i + 1) * nbytes]
                h = _hdr(m)
                assert h[0] == 0x43505448 and h[1] == 0           # magic, status
                assert (h[2], h[3], h[4], h[6], h[10]) == (s, 1, 0, S, S)
                rows_off = int(h[13])
                tabs = m[rows_off:rows_off + 8 * S].cpu().numpy().view(np.int32)
                lo, hi = oracle.p2p_step_rows(wl.cu, wl.cup, wl.cp, r, j, s, pad)
                np.testing.assert_array_equal(tabs[:S], lo, err_msg=f"row_lo r={r} step={i}")
                np.testing.assert_array_equal(tabs[S:], hi, err_msg=f"row_hi r={r} step={i}")
                check_block_lists(m, h, lo, hi, S)


def test_p2p_index_flags_bad_offsets():
    """A document length not divisible by 2*cp_size under DUAL_CHUNK_SWAP sets
    the header status of every step and the device status word."""
    d = dev()
    cup = torch.tensor([0, 10, 24], dtype=torch.int32, device=d)
    nbytes = api.cp_p2p_meta_bytes(2, 24, 2)
    meta = torch.zeros(2 * nbytes, dtype=torch.uint8, device=d)
    api.cp_p2p_index(None, cup, 24, 2, 0, pipeline.DCS, 0, meta)
    torch.cuda.synchronize()
    assert api.cp_device_status(reset=True) == -2
    for i in range(2):
        assert _hdr(meta[i * nbytes:])[1] == -2
    assert api.cp_device_status() == 0


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("n", [1, 3, 8])
def test_p2p_merge_matches_oracle(n, D):
    """cp_p2p_merge against the oracle's fp64 merge of the same bf16 partials,
    including rows that some or all steps did not see (LSE = -inf)."""
    d = dev()
    S, H = 777, 5
    g = torch.Generator().manual_seed(100 + n + D)
    o = torch.randn(n, S, H, D, generator=g).bfloat16()
    lse = torch.randn(n, H, S, generator=g) * 4.0
    lse[torch.rand(n, H, S, generator=g) < 0.3] = -float("inf")
    lse[:, :, :9] = -float("inf")                        # rows no step saw
    want_o, want_l = oracle.lse_merge(o.float().numpy(), lse.numpy())
    out = torch.empty(S, H, D, dtype=torch.bfloat16, device=d)
    l_out = torch.empty(H, S, dtype=torch.float32, device=d)
    api.cp_p2p_merge(o.to(d), lse.to(d), out, l_out)
    torch.cuda.synchronize()
    got = to_np(out)
    # one bf16 rounding of the fp32 combination
    assert np.all(np.abs(got - want_o) <= np.abs(want_o) * 2.0 ** -8 + 1e-5)
    assert np.all(got[:9] == 0)
    assert_lse_close(l_out.cpu().numpy(), want_l, "merged LSE", tol=1e-5)


P2P_CASES = {
    "three_docs_d128": lambda: inputs.custom([176, 272, 64], cp=4, H=4, D=128, seed=71),
    "padded_d64": lambda: inputs.custom([100, 7, 250, 33], padded=[112, 16, 256, 48], cp=4, H=8,
                                        D=64, seed=72),
    "one_doc_cp8": lambda: inputs.custom([1024], cp=8, H=2, D=128, seed=73),
    "tiny": inputs.tiny,
}


@pytest.mark.parametrize("fused", [True, False], ids=["one_pass", "per_step"])
@pytest.mark.parametrize("strategy", [pipeline.DCS, pipeline.NLB], ids=["dcs", "nlb"])
@pytest.mark.parametrize("name", list(P2P_CASES))
def test_p2p_attention_matches_oracle(name, strategy, fused):
    """Every rank's O, LSE, dQ, dK, dV after the emulated ring equal the fp64
    oracle's causal attention at the rank's rows, with the forward as one pass
    per rank over its ring steps (cp_attn_fwd_ring) or step by step with the
    merge (cp_attn_fwd + cp_p2p_merge)."""
    d = dev()
    wl = P2P_CASES[name]()
    if strategy not in wl.strategies:
        pytest.skip("strategy not valid for these lengths")
    t = wl.tensors()
    pad = wl.pad_between_seqs
    o, lse = oracle.attn_fwd(t["q"], t["k"], t["v"], wl.cu, wl.cup, pad)
    dq, dk, dv = oracle.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], wl.cu, wl.cup, pad)
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, strategy, pad, wl.H, wl.D, d)
    att = pipeline.CPP2PAttention(plan, fused_ring=fused)
    g = {k: v.to(d) for k, v in t.items()}
    att.step(g["q"], g["k"], g["v"], g["do"])
    torch.cuda.synchronize()
    assert api.cp_device_status() == 0
    for r in range(wl.cp):
        rows = oracle.partition_index(wl.cup, wl.cp, r, strategy)
        assert_close(to_np(plan.local(att.oc, r)), o[rows], f"O rank {r}")
        assert_lse_close(att.lse[r].cpu().numpy(), lse[:, rows], f"LSE rank {r}")
        assert_close(to_np(plan.local(att.dqc, r)), dq[rows], f"dQ rank {r}")
        assert_close(to_np(plan.local(att.dkc, r)), dk[rows], f"dK rank {r}")
        assert_close(to_np(plan.local(att.dvc, r)), dv[rows], f"dV rank {r}")


def test_p2p_step_is_deterministic():
    """Two ring steps on the same inputs give bitwise equal results (fixed
    order of every fp32 sum)."""
    d = dev()
    wl = inputs.custom([304, 216, 504], cp=4, H=4, D=128, seed=74)
    g = {k: v.to(d) for k, v in wl.tensors().items()}
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, pipeline.DCS, 0, wl.H, wl.D, d)
    att = pipeline.CPP2PAttention(plan)
    outs = []
    for _ in range(2):
        att.step(g["q"], g["k"], g["v"], g["do"])
        torch.cuda.synchronize()
        outs.append([x.clone() for x in (att.oc, att.dqc, att.dkc, att.dvc)])
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("strategy", [pipeline.DCS, pipeline.NLB], ids=["dcs", "nlb"])
def test_ring_one_pass_matches_per_step(strategy):
    """The one-pass ring forward and backward (cp_attn_fwd_ring, cp_attn_bwd_ring)
    against the per-step path (cp_attn_fwd + cp_p2p_merge, cp_attn_bwd_ex per
    step with fp32 sums) on the same inputs: outputs and gradients within two
    bf16 roundings of each other, LSE within 1e-4 (the same terms summed in
    another order)."""
    d = dev()
    # s_local = 384: lse rows 16-byte aligned, a multiple of 32 (one-pass backward)
    wl = inputs.custom([304, 216, 504, 96, 416], cp=4, H=3, D=128, seed=75)
    assert wl.total_tokens // wl.cp % 32 == 0
    g = {k: v.to(d) for k, v in wl.tensors().items()}
    res = []
    for fused in (True, False):
        plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, strategy, wl.pad_between_seqs, wl.H, wl.D, d)
        att = pipeline.CPP2PAttention(plan, fused_ring=fused)
        att.launches = 0
        att.step(g["q"], g["k"], g["v"], g["do"])
        torch.cuda.synchronize()
        assert api.cp_device_status() == 0
        res.append({"o": att.oc.float().clone(), "lse": att.lse.clone(), "dq": att.dqc.float().clone(),
                    "dk": att.dkc.float().clone(), "dv": att.dvc.float().clone(),
                    "launches": att.launches})
    a, b = res
    assert a["launches"] < b["launches"]  # the one-pass path ran
    assert torch.equal(torch.isneginf(a["lse"]), torch.isneginf(b["lse"]))
    fin = ~torch.isneginf(a["lse"])
    assert (a["lse"][fin] - b["lse"][fin]).abs().max().item() <= 1e-4
    for k in ("o", "dq", "dk", "dv"):
        scale = max(1.0, b[k].abs().max().item())
        assert (a[k] - b[k]).abs().max().item() <= 2.0 ** -6 * scale, k


@pytest.mark.parametrize("strategy", [pipeline.DCS, pipeline.NLB], ids=["dcs", "nlb"])
def test_ring_cast_in_epilogue_is_bitwise_the_separate_cast(strategy):
    """cp_attn_bwd_ring_rs (the pipeline's one-pass backward) writes dK/dV as
    bf16 from the dK/dV kernel's epilogue: bitwise cp_attn_bwd_ring's fp32 sums
    cast by cp_reduce_scatter_emul, and the same dQ."""
    d = dev()
    wl = inputs.custom([304, 216, 504, 96, 416], cp=4, H=3, D=128, seed=77)
    g = {k: v.to(d) for k, v in wl.tensors().items()}
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, strategy, wl.pad_between_seqs, wl.H, wl.D, d)
    att = pipeline.CPP2PAttention(plan)
    att.step(g["q"], g["k"], g["v"], g["do"])
    dq = torch.empty_like(att.dqc)
    dk = torch.empty_like(att.dkc)
    dv = torch.empty_like(att.dvc)
    api.cp_attn_bwd_ring(att.qc, att.kc, att.vc, att.oc, att.lse, att.doc, dq, att.dk_acc,
                         att.dv_acc, att.p2p_meta_all, att.step_bytes, att.rank_stride, plan.cp,
                         plan.strategy, plan.scale, att.ws_ring_bwd, o_resid_all=att.oc_resid)
    api.cp_reduce_scatter_emul([att.dk_acc, att.dv_acc], [dk, dv], None, 0, plan.T)
    for r, rm in enumerate(plan.ranks):
        api.cp_zero_tail([plan.local(dq, r), plan.local(dk, r), plan.local(dv, r)], rm.valid_end)
    torch.cuda.synchronize()
    assert api.cp_device_status() == 0
    for name, sep in (("dqc", dq), ("dkc", dk), ("dvc", dv)):
        assert torch.equal(getattr(att, name).view(torch.int16), sep.view(torch.int16)), name


def test_ring_one_pass_refuses_other_metadata():
    """Every step's header is checked on the device: the other strategy's step
    metadata writes nothing and reports CP_ERR_METADATA."""
    d = dev()
    wl = inputs.custom([304, 216, 504], cp=4, H=2, D=64, seed=76)
    g = {k: v.to(d) for k, v in wl.tensors().items()}
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, pipeline.DCS, 0, wl.H, wl.D, d)
    att = pipeline.CPP2PAttention(plan)
    att.step(g["q"], g["k"], g["v"])
    other = pipeline.CPP2PAttention(pipeline.CPPlan(wl.cu, wl.cup, wl.cp, pipeline.NLB, 0,
                                                    wl.H, wl.D, d))
    torch.cuda.synchronize()
    sentinel = 3.0
    o = torch.full_like(plan.local(att.oc, 1), sentinel)
    lse = torch.full_like(att.lse[1], sentinel)
    api.cp_attn_fwd_ring(plan.local(att.qc, 1), att.kc, att.vc, o, lse, other.p2p_meta[1],
                         other.step_bytes, 2, plan.cp, 1, pipeline.DCS, plan.scale, att.ws_ring)
    torch.cuda.synchronize()
    assert api.cp_device_status(reset=True) == -7  # CP_ERR_METADATA
    assert torch.all(o == sentinel) and torch.all(lse == sentinel)
