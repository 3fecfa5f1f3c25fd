"""GPU parity of the emulated a2a comm type ("[PyTorch] Extend no-load-balance
CP to the a2a comm type"): the all-to-all exchange bit-exact against the
oracle's numpy restatement, and the full a2a attention forward/backward --
exchange, per-rank attention on the whole sequence with its head slice,
exchange back -- against the fp64 oracle, for flat and dual-chunk sharding."""
import numpy as np
import pytest
import torch

import oracle
from context_packed_sequence_thd_gb300 import api, inputs, pipeline
from gpu_util import assert_close, dev, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("perm_kind", ["none", "random"])
@pytest.mark.parametrize("shape", [(96, 8, 64), (1000, 40, 128)])
def test_a2a_exchange_bit_exact(shape, perm_kind):
    d = dev()
    T, H, D = shape
    cp = 4 if H % 8 else 8
    g = torch.Generator().manual_seed(11)
    xs = [torch.randn(T, H, D, generator=g).bfloat16() for _ in range(3)]
    perm = None if perm_kind == "none" else torch.randperm(T, generator=g).to(torch.int32)
    p_np = None if perm is None else perm.numpy()
    heads = [torch.empty(cp, T, H // cp, D, dtype=torch.bfloat16, device=d) for _ in range(3)]
    api.cp_a2a_exchange([x.to(d) for x in xs], heads, None if perm is None else perm.to(d), cp,
                        api.A2A_SEQ_TO_HEAD)
    for x, h in zip(xs, heads):
        want = oracle.a2a_seq_to_head(x.view(torch.int16).numpy(), cp, p_np)
        np.testing.assert_array_equal(h.cpu().view(torch.int16).numpy(), want)
    back = [torch.empty(T, H, D, dtype=torch.bfloat16, device=d) for _ in range(3)]
    api.cp_a2a_exchange(heads, back, None if perm is None else perm.to(d), cp, api.A2A_HEAD_TO_SEQ)
    for x, b in zip(xs, back):
        np.testing.assert_array_equal(b.cpu().view(torch.int16).numpy(), x.view(torch.int16).numpy())
    assert api.cp_device_status() == 0


def test_a2a_exchange_rejects_bad_shapes():
    d = dev()
    x = torch.zeros(16, 6, 64, dtype=torch.bfloat16, device=d)
    h = torch.zeros(4, 16, 1, 64, dtype=torch.bfloat16, device=d)
    with pytest.raises(api.CpError):        # H = 6 not divisible by cp = 4
        api.cp_a2a_exchange([x], [h], None, 4, api.A2A_SEQ_TO_HEAD)
    bad = torch.full((16,), 99, dtype=torch.int32, device=d)
    h2 = torch.zeros(2, 16, 3, 64, dtype=torch.bfloat16, device=d)
    api.cp_a2a_exchange([x], [h2], bad, 2, api.A2A_SEQ_TO_HEAD)   # out-of-range rows: skipped
    torch.cuda.synchronize()
    assert api.cp_device_status(reset=True) == -1
    assert api.cp_device_status() == 0


A2A_CASES = {
    "three_docs_d128": lambda: inputs.custom([176, 272, 64], cp=4, H=4, D=128, seed=81),
    "padded_d64": lambda: inputs.custom([100, 7, 250, 33], padded=[112, 16, 256, 48], cp=4, H=8,
                                        D=64, seed=82),
    "one_doc_cp8": lambda: inputs.custom([1024], cp=8, H=8, D=128, seed=83),
}


@pytest.mark.parametrize("strategy", [pipeline.DCS, pipeline.NLB], ids=["dcs", "nlb"])
@pytest.mark.parametrize("name", list(A2A_CASES))
def test_a2a_attention_matches_oracle(name, strategy):
    """Rank r's shard of O, dQ, dK, dV after the a2a round trip equals the
    oracle's full-sequence result at the rank's rows (a2a attention is the
    cp_size = 1 computation per head slice)."""
    d = dev()
    wl = A2A_CASES[name]()
    t = wl.tensors()
    pad = wl.pad_between_seqs
    o, lse = oracle.attn_fwd(t["q"], t["k"], t["v"], wl.cu, wl.cup, pad)
    dq, dk, dv = oracle.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], wl.cu, wl.cup, pad)
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, strategy, pad, wl.H, wl.D, d)
    att = pipeline.CPA2AAttention(plan)
    g = {k: v.to(d) for k, v in t.items()}
    att.step(g["q"], g["k"], g["v"], g["do"])
    torch.cuda.synchronize()
    assert api.cp_device_status() == 0
    hc = wl.H // wl.cp
    for r in range(wl.cp):
        rows = oracle.partition_index(wl.cup, wl.cp, r, strategy)
        assert_close(to_np(plan.local(att.oc, r)), o[rows], f"O rank {r}")
        assert_close(to_np(plan.local(att.dqc, r)), dq[rows], f"dQ rank {r}")
        assert_close(to_np(plan.local(att.dkc, r)), dk[rows], f"dK rank {r}")
        assert_close(to_np(plan.local(att.dvc, r)), dv[rows], f"dV rank {r}")
        # rank r's LSE covers every token of its head slice
        got = att.lse_h[r].cpu().numpy()
        want = lse[r * hc:(r + 1) * hc]
        fin = np.isfinite(want)
        assert np.array_equal(np.isfinite(got), fin)
        assert np.max(np.abs(got[fin] - want[fin])) < 1e-3


def test_a2a_forward_bitwise_matches_all_gather_forward():
    """Per (row, head) the forward takes the same key blocks in the same order
    under both comm types, so O agrees bitwise between a2a and all-gather CP."""
    d = dev()
    wl = inputs.custom([300, 212], cp=2, H=4, D=64, seed=84)
    t = {k: v.to(d) for k, v in wl.tensors().items()}
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, pipeline.NLB, 0, wl.H, wl.D, d)
    ag = pipeline.CPAttention(plan)
    ag.step(t["q"], t["k"], t["v"])
    plan2 = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, pipeline.NLB, 0, wl.H, wl.D, d)
    a2a = pipeline.CPA2AAttention(plan2)
    a2a.step(t["q"], t["k"], t["v"])
    torch.cuda.synchronize()
    assert torch.equal(ag.oc.view(torch.int16), a2a.oc.view(torch.int16))


@pytest.mark.parametrize("strategy", [pipeline.DCS, pipeline.NLB], ids=["dcs", "nlb"])
def test_a2a_bshd_and_sbhd_batches(strategy):
    """A bshd batch is THD with B equal documents (no copy); an sbhd batch is
    the same tokens in [S, B] order, carried to THD and back by one gather each
    way.  Both give the oracle's result, and bitwise the same as each other."""
    d = dev()
    B, S, H, D, cp = 3, 256, 8, 64, 4
    g = torch.Generator().manual_seed(91)
    bshd = {k: torch.randn(B, S, H, D, generator=g).bfloat16() for k in ("q", "k", "v", "do")}
    cu = pipeline.bshd_seqlens(B, S)
    t = {k: v.reshape(B * S, H, D) for k, v in bshd.items()}          # THD view of bshd
    o, lse = oracle.attn_fwd(t["q"], t["k"], t["v"], cu, cu, 0)
    dq, dk, dv = oracle.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], cu, cu, 0)

    def run(thd):
        plan = pipeline.CPPlan(cu, cu, cp, strategy, 0, H, D, d)
        att = pipeline.CPA2AAttention(plan)
        att.step(thd["q"], thd["k"], thd["v"], thd["do"])
        torch.cuda.synchronize()
        assert api.cp_device_status() == 0
        # back to original token order: rank-concatenated rows -> global rows
        G = torch.cat([plan.ranks[r].idx.long() for r in range(cp)])
        out = {}
        for name, buf in (("o", att.oc), ("dq", att.dqc), ("dk", att.dkc), ("dv", att.dvc)):
            x = torch.empty_like(buf)
            x[G] = buf
            out[name] = x
        return out

    got_b = run({k: v.to(d) for k, v in t.items()})
    for name, want in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert_close(to_np(got_b[name]), want, f"bshd {name}")
    # sbhd: the same tokens stored [S, B, H, D]
    rows = pipeline.sbhd_rows(B, S, d)
    sbhd = [bshd[k].transpose(0, 1).contiguous().to(d) for k in ("q", "k", "v", "do")]
    thd = dict(zip(("q", "k", "v", "do"), pipeline.sbhd_to_thd(sbhd, rows)))
    for k in thd:
        assert torch.equal(thd[k].cpu().view(torch.int16), t[k].view(torch.int16))
    got_s = run(thd)
    back = pipeline.thd_to_sbhd([got_s["o"], got_s["dq"]], rows, S, B)
    for name, x in zip(("o", "dq"), back):
        assert torch.equal(x.transpose(0, 1).contiguous().view(torch.int16),
                           got_b[name].view(B, S, H, D).view(torch.int16))
    for name in ("dk", "dv"):
        assert torch.equal(got_s[name].view(torch.int16), got_b[name].view(torch.int16))
