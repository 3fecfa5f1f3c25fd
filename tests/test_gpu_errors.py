"""Rules only the device checks, exercised with inputs made on the host.

* "[PyTorch] Add no-load-balance THD all-gather CP", §What changed: the
  backward uses the forward's strategy.  Here the strategy and the rank are
  explicit arguments of every attention call and the kernels compare them with
  the header of the metadata they are given: metadata of the other strategy,
  or of another rank, makes the call write nothing and report CP_ERR_METADATA.
* Every mbarrier wait of the attention kernels is bounded.  The failure-
  detection hook leaves one K tile of CTA 0 unloaded (a barrier nothing
  completes); the wait for it runs out, the CTA drains its copies and frees its
  tensor memory, the status word reads CP_ERR_TIMEOUT, and the context stays
  usable: the next ordinary call is correct.  No fault, trap or endless wait is
  involved.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from context_packed_sequence_thd_gb300 import api, inputs, pipeline
from gpu_util import assert_close, dev, to_np

pytestmark = pytest.mark.gpu

CP_ERR_METADATA = -7
CP_ERR_TIMEOUT = -8


def _setup(strategy):
    d = dev()
    wl = inputs.custom([256, 128, 384, 256], cp=2, H=2, D=128, seed=77, pad_between_seqs=0)
    t = wl.tensors()
    g = {k: v.to(d) for k, v in t.items()}
    plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, strategy, 0, wl.H, wl.D, d)
    att = pipeline.CPAttention(plan)
    att.step(g["q"], g["k"], g["v"], g["do"])
    torch.cuda.synchronize()
    assert api.cp_device_status() == 0
    return d, wl, t, g, plan, att


@pytest.mark.parametrize("strategy", [pipeline.DCS, pipeline.NLB])
@pytest.mark.parametrize("wrong", ["strategy", "rank"])
def test_attention_refuses_metadata_of_another_strategy_or_rank(strategy, wrong):
    d, wl, t, g, plan, att = _setup(strategy)
    p = plan
    r = 0
    k_full = att.k_full if strategy == pipeline.DCS else att.kc
    v_full = att.v_full if strategy == pipeline.DCS else att.vc
    if wrong == "strategy":
        other = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, 1 - strategy, 0, wl.H, wl.D, d)
        meta, call_rank, call_strategy = other.ranks[r].meta, r, strategy
    else:
        meta, call_rank, call_strategy = p.ranks[1].meta, r, strategy
    torch.cuda.synchronize()
    sentinel = 3.0
    o = torch.full((p.s_local, wl.H, wl.D), sentinel, dtype=torch.bfloat16, device=d)
    lse = torch.full((wl.H, p.s_local), sentinel, device=d)
    api.cp_attn_fwd(p.local(att.qc, r), k_full, v_full, o, lse, meta, p.T, p.cp, call_rank,
                    call_strategy, p.scale)
    torch.cuda.synchronize()
    assert api.cp_device_status(reset=True) == CP_ERR_METADATA
    assert torch.all(o == sentinel) and torch.all(lse == sentinel)
    dq = torch.full((p.s_local, wl.H, wl.D), sentinel, dtype=torch.bfloat16, device=d)
    dk = torch.full((p.T, wl.H, wl.D), sentinel, device=d)
    dv = torch.full((p.T, wl.H, wl.D), sentinel, device=d)
    for mode in (api.BWD_ACCUMULATE, api.BWD_STORE):
        api.cp_attn_bwd(p.local(att.qc, r), k_full, v_full, p.local(att.oc, r), att.lse[r],
                        p.local(att.doc, r), dq, dk, dv, meta, p.T, p.cp, call_rank,
                        call_strategy, p.scale, att.ws, mode=mode)
        torch.cuda.synchronize()
        assert api.cp_device_status(reset=True) == CP_ERR_METADATA
        assert torch.all(dq == sentinel) and torch.all(dk == sentinel) and torch.all(dv == sentinel)
    # the matching metadata is accepted by the same calls
    api.cp_attn_fwd(p.local(att.qc, r), k_full, v_full, o, lse, p.ranks[r].meta, p.T, p.cp, r,
                    strategy, p.scale)
    torch.cuda.synchronize()
    assert api.cp_device_status() == 0
    assert torch.equal(o, p.local(att.oc, r))


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    d, wl, t, g, plan, att = _setup(pipeline.DCS)
    p = plan
    r = 0
    o = torch.zeros(p.s_local, wl.H, wl.D, dtype=torch.bfloat16, device=d)
    lse = torch.zeros(wl.H, p.s_local, device=d)
    L = api.lib()
    fn = L.cpthd_test_attn_fwd_timeout
    fn.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_size_t, ctypes.c_int64] + \
        [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_int, ctypes.c_uint64, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    limit_ns = 50_000_000   # 50 ms
    st = fn(api._dev(p.local(att.qc, r), "q"), api._dev(att.k_full, "k"),
            api._dev(att.v_full, "v"), api._dev(o, "o"), api._dev(lse, "lse"),
            api._dev(p.ranks[r].meta, "meta"), p.ranks[r].meta.numel(), p.T, wl.H, wl.D, p.cp, r,
            p.strategy, p.scale, api._operand_dtype(att.qc), limit_ns, api._stream())
    assert st == 0
    torch.cuda.synchronize()
    assert api.cp_device_status(reset=True) == CP_ERR_TIMEOUT
    assert api.cp_device_status() == 0
    # the same call without the hook, right after, is correct
    api.cp_attn_fwd(p.local(att.qc, r), att.k_full, att.v_full, o, lse, p.ranks[r].meta, p.T, p.cp,
                    r, p.strategy, p.scale)
    torch.cuda.synchronize()
    assert api.cp_device_status() == 0
    o_ref, _ = oracle.attn_fwd(t["q"], t["k"], t["v"], wl.cu, wl.cup, 0)
    rows = p.ranks[r].idx.cpu().numpy()
    assert_close(to_np(o), o_ref[rows], "O after the timed-out call")
