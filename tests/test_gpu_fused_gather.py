"""GPU parity of the forward with the partition gather fused into its loads
(cp_attn_fwd_gather: query row t read from q_src[idx[t]] by the attention
kernel itself, the index_select of "[PyTorch] Add no-load-balance THD
all-gather CP", §Sequence Diagram, folded into the attention).  The result
must be bitwise that of cp_attn_fwd on the gathered rows, and match the fp64
oracle."""
import numpy as np
import pytest
import torch

import oracle
from context_packed_sequence_thd_gb300 import api, inputs, pipeline
from gpu_util import assert_close, assert_lse_close, dev, to_np

pytestmark = pytest.mark.gpu

CASES = {
    "tiny_d64": inputs.tiny,
    "ragged_padded": lambda: inputs.custom([100, 7, 250, 33], padded=[112, 16, 256, 48], cp=4,
                                           H=8, D=64, seed=61),
    "cfg2": inputs.cfg2,
    "one_doc_cp8": lambda: inputs.custom([4096], cp=8, H=4, D=128, seed=62),
    # s_local = 1000: odd ranks' index slices start 8 bytes past a 16-byte boundary
    "odd_slices_cp4": lambda: inputs.custom([2000, 1008, 992], cp=4, H=2, D=128, seed=65),
}


@pytest.mark.parametrize("strategy", [pipeline.DCS, pipeline.NLB], ids=["dcs", "nlb"])
@pytest.mark.parametrize("name", list(CASES))
def test_fused_gather_bitwise_equals_gathered_forward(name, strategy):
    d = dev()
    wl = CASES[name]()
    t = {k: v.to(d) for k, v in wl.tensors(with_grad=False).items()}
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, strategy, wl.pad_between_seqs, wl.H, wl.D, d)
    ref = pipeline.CPAttention(plan, operand_dtype=torch.bfloat16)
    ref.step(t["q"], t["k"], t["v"])
    kf, vf = (ref.k_full, ref.v_full) if strategy == pipeline.DCS else (t["k"], t["v"])
    o = torch.empty_like(ref.oc)
    lse = torch.empty_like(ref.lse)
    for r in range(wl.cp):
        api.cp_attn_fwd_gather(t["q"], plan.ranks[r].idx, kf, vf, plan.local(o, r), lse[r],
                               plan.ranks[r].meta, plan.T, plan.cp, r, strategy, plan.scale)
    torch.cuda.synchronize()
    assert api.cp_device_status() == 0
    assert torch.equal(o.view(torch.int16), ref.oc.view(torch.int16))
    assert torch.equal(lse, ref.lse)


def test_fused_gather_pipeline_matches_oracle():
    """A forward-only DUAL_CHUNK_SWAP step with the fused gather (no Q shard
    copy) against the fp64 oracle, every rank."""
    d = dev()
    wl = inputs.custom([176, 272, 64, 512], cp=4, H=4, D=128, seed=63)
    t = wl.tensors(with_grad=False)
    o, lse = oracle.attn_fwd(t["q"], t["k"], t["v"], wl.cu, wl.cup, 0)
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, pipeline.DCS, 0, wl.H, wl.D, d)
    att = pipeline.CPAttention(plan, fuse_q_gather=True)
    g = {k: v.to(d) for k, v in t.items()}
    att.step(g["q"], g["k"], g["v"])
    torch.cuda.synchronize()
    assert att.q_src is not None and api.cp_device_status() == 0
    for r in range(wl.cp):
        rows = oracle.partition_index(wl.cup, wl.cp, r, pipeline.DCS)
        assert_close(to_np(plan.local(att.oc, r)), o[rows], f"O rank {r}")
        assert_lse_close(att.lse[r].cpu().numpy(), lse[:, rows], f"LSE rank {r}")


def test_fused_gather_from_a_larger_source_with_any_rows():
    """The source may have more rows than the layout and the index any rows of
    it (repeats allowed): the result is the forward on the rows it names."""
    d = dev()
    T, H, D, cp = 512, 4, 128, 2
    cu = np.array([0, 300, 512], dtype=np.int32)
    g = torch.Generator().manual_seed(64)
    src = torch.randn(3000, H, D, generator=g).bfloat16().to(d)
    k = torch.randn(T, H, D, generator=g).bfloat16().to(d)
    v = torch.randn(T, H, D, generator=g).bfloat16().to(d)
    plan = pipeline.CPPlan(cu, cu, cp, pipeline.NLB, 0, H, D, d)
    S = plan.s_local
    idx = torch.randint(0, 3000, (S,), generator=g, dtype=torch.int32)
    idx[:5] = idx[5]                                   # repeated rows
    q_local = src[idx.long().to(d)].contiguous()
    for r in range(cp):
        o1 = torch.empty(S, H, D, dtype=torch.bfloat16, device=d)
        o2 = torch.empty_like(o1)
        l1 = torch.empty(H, S, dtype=torch.float32, device=d)
        l2 = torch.empty_like(l1)
        api.cp_attn_fwd(q_local, k, v, o1, l1, plan.ranks[r].meta, T, cp, r, pipeline.NLB,
                        plan.scale)
        api.cp_attn_fwd_gather(src, idx.to(d), k, v, o2, l2, plan.ranks[r].meta, T, cp, r,
                               pipeline.NLB, plan.scale)
        torch.cuda.synchronize()
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
        assert torch.equal(l1, l2)
    assert api.cp_device_status() == 0


def test_fused_gather_out_of_range_index_is_reported():
    """An index outside the source is caught by the kernel's own bounds check:
    it reads row 0 instead and sets the device status word."""
    d = dev()
    T, H, D = 256, 2, 64
    cu = np.array([0, 256], dtype=np.int32)
    plan = pipeline.CPPlan(cu, cu, 1, pipeline.NLB, 0, H, D, d)
    q = torch.zeros(T, H, D, dtype=torch.bfloat16, device=d)
    idx = torch.arange(T, dtype=torch.int32, device=d)
    idx[7] = T + 5
    o = torch.empty(T, H, D, dtype=torch.bfloat16, device=d)
    lse = torch.empty(H, T, dtype=torch.float32, device=d)
    api.cp_attn_fwd_gather(q, idx, q, q, o, lse, plan.ranks[0].meta, T, 1, 0, pipeline.NLB,
                           plan.scale)
    torch.cuda.synchronize()
    assert api.cp_device_status(reset=True) == -1
    assert api.cp_device_status() == 0
