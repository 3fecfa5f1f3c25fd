"""GPU parity of the integer and bandwidth kernels against the oracle, all
bit-exact: the partition index (per-rank rows, restore index, valid end),
THD row gather/scatter, the fp32->bf16 reduce-scatter epilogue and the gated
tail-zeroing."""
import numpy as np
import pytest
import torch

import oracle
from context_packed_sequence_thd_gb300 import api, inputs, pipeline
from gpu_util import check_block_lists, dev

pytestmark = pytest.mark.gpu

WORKLOADS = [inputs.tiny, inputs.cfg2, inputs.cfg3, inputs.cfg4, inputs.cfg5,
             lambda: inputs.cfg5(tail=False), lambda: inputs.cfg5(value_equal=True),
             lambda: inputs.custom([7, 33, 1, 90], cp=4, padded=[8, 40, 8, 96]),
             lambda: inputs.custom([0, 6, 0, 10], padded=[4, 8, 0, 12], cp=2),
             lambda: inputs.custom([3, 5], padded=[4, 12], cp=1)]


def _hdr(meta: torch.Tensor) -> np.ndarray:
    return meta[:64].cpu().numpy().view(np.int32)


@pytest.mark.parametrize("make", WORKLOADS)
def test_partition_index_bit_exact(make):
    d = dev()
    wl = make()
    pad = wl.pad_between_seqs
    valid = oracle.valid_mask(wl.cu, wl.cup, pad)
    for s in wl.strategies:
        plan = pipeline.CPPlan(wl.cu, wl.cup, wl.cp, s, pad, 1, 64, d)
        torch.cuda.synchronize()
        assert api.cp_device_status() == 0
        for r in range(wl.cp):
            want = oracle.partition_index(wl.cup, wl.cp, r, s)
            np.testing.assert_array_equal(plan.ranks[r].idx.cpu().numpy(), want)
            h = _hdr(plan.ranks[r].meta)
            assert h[0] == 0x43505448 and h[1] == 0            # magic, status
            assert h[6] == wl.s_local and h[8] == oracle.valid_end(valid[want])
            # row tables: keys [row_lo, row_hi] of every local row
            nd = wl.n_docs
            rows_off = 64 + 32 * (2 * nd + 2)
            tabs = plan.ranks[r].meta[rows_off:rows_off + 8 * wl.s_local].cpu().numpy().view(np.int32)
            lo, hi = tabs[:wl.s_local], tabs[wl.s_local:]
            start = np.repeat(wl.cup[:-1], np.diff(wl.cup))
            np.testing.assert_array_equal(hi, np.where(valid[want], want, -1))
            np.testing.assert_array_equal(lo, np.where(valid[want], start[want], 0))
            check_block_lists(plan.ranks[r].meta, h, lo, hi, wl.total_tokens)
        np.testing.assert_array_equal(plan.restore.cpu().numpy(),
                                      oracle.restore_index(wl.cup, wl.cp, s))


def test_partition_rejects_bad_metadata_on_device():
    d = dev()
    cup = torch.tensor([0, 10, 24], dtype=torch.int32, device=d)   # 10 % 4 != 0 for DCS, cp=2
    idx = torch.full((12,), -5, dtype=torch.int32, device=d)
    meta = torch.zeros(api.cp_meta_bytes(2, 24, 2), dtype=torch.uint8, device=d)
    api.cp_partition_index(None, cup, 24, 2, 0, pipeline.DCS, 0, idx, None, meta)
    torch.cuda.synchronize()
    assert _hdr(meta)[1] == -2
    assert api.cp_device_status(reset=True) == -2
    assert torch.all(idx == -5)                     # nothing written
    assert api.cp_device_status() == 0
    # inconsistent cu_seqlens (L_0 > P_0) with padding
    cu = torch.tensor([0, 12, 20], dtype=torch.int32, device=d)
    api.cp_partition_index(cu, cup, 24, 2, 0, pipeline.NLB, 1, idx, None, meta)
    torch.cuda.synchronize()
    assert _hdr(meta)[1] == -7
    assert api.cp_device_status(reset=True) == -7
    # attention refuses metadata with a bad status (writes nothing)
    q = torch.randn(12, 1, 64, device=d).bfloat16()
    kv = torch.randn(24, 1, 64, device=d).bfloat16()
    o = torch.full((12, 1, 64), 7.0, device=d).bfloat16()
    lse = torch.zeros(1, 12, device=d)
    api.cp_attn_fwd(q, kv, kv, o, lse, meta, 24, 2, 0, pipeline.NLB, 0.125)
    torch.cuda.synchronize()
    assert torch.all(o == 7.0)
    assert api.cp_device_status(reset=True) == -7


@pytest.mark.parametrize("shape", [(129, 2, 64), (4096, 16, 128), (1000, 40, 128)])
def test_gather_scatter_bitwise(shape):
    d = dev()
    g = torch.Generator().manual_seed(5)
    n_src = shape[0]
    srcs = [torch.randn(*shape, generator=g).bfloat16() for _ in range(3)]
    idx = torch.randperm(n_src, generator=g)[: n_src - 7].to(torch.int32)
    want = [oracle.gather_rows(s.view(torch.int16).numpy(), idx.numpy()) for s in srcs]
    ds = [s.to(d) for s in srcs]
    out = [torch.empty(len(idx), *shape[1:], dtype=torch.bfloat16, device=d) for _ in range(3)]
    api.cp_thd_gather(ds, out, idx.to(d))
    for o, w in zip(out, want):
        np.testing.assert_array_equal(o.cpu().view(torch.int16).numpy(), w)
    back = [torch.zeros_like(s) for s in ds]
    api.cp_thd_scatter(out, back, idx.to(d))
    for b, s in zip(back, srcs):
        ref = oracle.scatter_rows(np.zeros_like(s.view(torch.int16).numpy()), idx.numpy(),
                                  oracle.gather_rows(s.view(torch.int16).numpy(), idx.numpy()))
        np.testing.assert_array_equal(b.cpu().view(torch.int16).numpy(), ref)
    # an out-of-range index is skipped and reported, never dereferenced
    bad = idx.clone()
    bad[3] = n_src + 100
    api.cp_thd_gather(ds[:1], out[:1], bad.to(d))
    torch.cuda.synchronize()
    assert api.cp_device_status(reset=True) == -1


def test_reduce_scatter_emul_bit_exact():
    d = dev()
    g = torch.Generator().manual_seed(9)
    T, H, D = 300, 4, 64
    acc = [torch.randn(T, H, D, generator=g) * 3 for _ in range(2)]
    idx = torch.randperm(T, generator=g)[:100].to(torch.int32)
    out = [torch.empty(100, H, D, dtype=torch.bfloat16, device=d) for _ in range(2)]
    api.cp_reduce_scatter_emul([a.to(d) for a in acc], out, idx.to(d), 0, 100)
    for o, a in zip(out, acc):
        want = oracle.bf16_round(oracle.gather_rows(a.numpy(), idx.numpy()))
        np.testing.assert_array_equal(o.cpu().view(torch.int16).numpy().view(np.uint16), want)
    # contiguous form (no index): rows row0 .. row0+n
    api.cp_reduce_scatter_emul([a.to(d) for a in acc], out, None, 150, 100)
    for o, a in zip(out, acc):
        want = oracle.bf16_round(a.numpy()[150:250])
        np.testing.assert_array_equal(o.cpu().view(torch.int16).numpy().view(np.uint16), want)


def test_zero_tail_gate_and_device_form():
    d = dev()
    x = torch.ones(50, 2, 64, dtype=torch.bfloat16, device=d)
    y = torch.ones(50, 2, 64, dtype=torch.bfloat16, device=d)
    assert api.cp_zero_tail([x, y], 50) is False            # no tail: no launch
    assert torch.all(x == 1) and torch.all(y == 1)
    assert api.cp_zero_tail([x, y], 37) is True
    assert torch.all(x[:37] == 1) and torch.all(x[37:] == 0) and torch.all(y[37:] == 0)
    z = torch.ones(50, 2, 64, dtype=torch.bfloat16, device=d)
    ve = torch.tensor([45], dtype=torch.int32, device=d)
    assert api.cp_zero_tail([z], -1, ve) is True             # graph-safe form always launches
    assert torch.all(z[:45] == 1) and torch.all(z[45:] == 0)
    ve.fill_(50)
    w = torch.ones_like(z)
    api.cp_zero_tail([w], -1, ve)
    assert torch.all(w == 1)                                 # read on device: no tail, no writes


@pytest.mark.parametrize("make", [inputs.tiny, inputs.cfg2, inputs.cfg5,
                                  lambda: inputs.custom([0, 6, 0, 10], padded=[4, 8, 0, 12], cp=2),
                                  lambda: inputs.custom([3, 5], padded=[4, 12], cp=1)],
                         ids=["tiny", "cfg2", "cfg5", "empty_docs", "cp1"])
def test_partition_index_all_ranks_one_launch_bytewise(make):
    """cp_partition_index_all (one CTA per rank) writes byte for byte what the
    cp single-rank calls write: indices, restore index and metadata."""
    d = dev()
    wl = make()
    pad = wl.pad_between_seqs
    d_cu = torch.from_numpy(np.asarray(wl.cu, dtype=np.int32)).to(d)
    d_cup = torch.from_numpy(np.asarray(wl.cup, dtype=np.int32)).to(d)
    T, cp, S = wl.total_tokens, wl.cp, wl.s_local
    nbytes = api.cp_meta_bytes(wl.n_docs, T, cp)
    stride = (nbytes + 15) // 16 * 16 + 32          # room between ranks stays untouched
    for s in wl.strategies:
        idx1 = torch.full((T,), -5, dtype=torch.int32, device=d)
        res1 = torch.full((T,), -5, dtype=torch.int32, device=d)
        meta1 = torch.full((cp * stride,), 0x5A, dtype=torch.uint8, device=d)
        for r in range(cp):
            api.cp_partition_index(d_cu if pad else None, d_cup, T, cp, r, s, pad,
                                   idx1[r * S:(r + 1) * S], res1,
                                   meta1[r * stride:r * stride + nbytes])
        idx2 = torch.full_like(idx1, -5)
        res2 = torch.full_like(res1, -5)
        meta2 = torch.full_like(meta1, 0x5A)
        api.cp_partition_index_all(d_cu if pad else None, d_cup, T, cp, s, pad, idx2, res2, meta2,
                                   stride)
        torch.cuda.synchronize()
        assert api.cp_device_status() == 0
        assert torch.equal(idx1, idx2) and torch.equal(res1, res2)
        assert torch.equal(meta1, meta2)


def test_gather_f16_conversion_and_range():
    """cp_thd_gather_f16: each element is the bf16 source value rounded to the
    nearest fp16 (numpy's float32 -> float16 conversion of the same values,
    ties to even), with and without an index; a finite value beyond 65504
    becomes +-65504 and reports CP_ERR_RANGE; infinities and NaN stay."""
    d = dev()
    g = torch.Generator().manual_seed(91)
    T, H, D = 300, 2, 64
    src = (torch.randn(T, H, D, generator=g) * torch.exp2(torch.randint(-20, 15, (T, H, D), generator=g)
                                                           .float())).bfloat16()
    src[0, 0, :4] = torch.tensor([65504.0, 65520.0, -1e6, 2.0 ** -20]).bfloat16()
    x = src.float().numpy()
    small = np.abs(x) <= 65504
    assert small.mean() > 0.9
    dst = torch.empty(T, H, D, dtype=torch.float16, device=d)
    # only in-range values first: exact agreement, no status
    ok = src.clone()
    ok[torch.from_numpy(~small)] = 1.0
    api.cp_thd_gather_f16([ok.to(d)], [dst], None)
    torch.cuda.synchronize()
    assert api.cp_device_status() == 0
    want = ok.float().numpy().astype(np.float16)
    np.testing.assert_array_equal(dst.cpu().numpy().view(np.uint16), want.view(np.uint16))
    # through an index
    idx = torch.randperm(T, generator=g)[:128].to(torch.int32)
    dst2 = torch.empty(128, H, D, dtype=torch.float16, device=d)
    api.cp_thd_gather_f16([ok.to(d)], [dst2], idx.to(d))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(dst2.cpu().numpy().view(np.uint16),
                                  want[idx.long().numpy()].view(np.uint16))
    # out of range: clamped and reported; inf and nan pass through
    bad = ok.clone()
    bad[1, 1, :4] = torch.tensor([1e6, -7e4, float("inf"), float("nan")]).bfloat16()
    api.cp_thd_gather_f16([bad.to(d)], [dst], None)
    torch.cuda.synchronize()
    assert api.cp_device_status(reset=True) == -9          # CP_ERR_RANGE
    got = dst[1, 1, :4].cpu().float().numpy()
    assert got[0] == 65504 and got[1] == -65504 and np.isposinf(got[2]) and np.isnan(got[3])
