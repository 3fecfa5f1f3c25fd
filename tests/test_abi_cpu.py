"""CPU-only checks of the C ABI: the library builds and loads without a GPU,
exports every function include/cpthd.h declares, and its host-side logic
(value-based pad detection, metadata validation, valid ends, the tail-zero
gate, argument validation) behaves as documented.  No compute call reaches
the GPU here: every call below returns before its first CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from context_packed_sequence_thd_gb300 import api, inputs, pipeline

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return api.lib()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "cpthd.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(cp_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(api.EXPORTED)


def test_version_and_status_strings(lib):
    assert api.lib().cp_version() == 200
    assert api.status_string(0) == "CP_OK"
    assert api.status_string(-2) == "CP_ERR_DIVISIBILITY"
    assert api.status_string(-99) == "CP_ERR_UNKNOWN"


def test_pad_detection_by_values(lib):
    cu = np.array([0, 4096], dtype=np.int32)
    assert api.cp_detect_pad_between_seqs(cu, cu.copy()) == 0
    assert api.cp_detect_pad_between_seqs(cu, None) == 0
    for wl in (inputs.cfg5(), inputs.cfg5(value_equal=True), inputs.cfg2(), inputs.tiny()):
        assert api.cp_detect_pad_between_seqs(wl.cu, wl.cup) == oracle.pad_between_seqs(wl.cu, wl.cup)


def test_validate_seqlens(lib):
    ok = np.array([0, 8, 24], dtype=np.int32)
    assert api.cp_validate_seqlens(ok, ok, 24, 2, pipeline.DCS, 0) == 0
    assert api.cp_validate_seqlens(ok, ok, 24, 4, pipeline.DCS, 0) == 0
    assert api.cp_validate_seqlens(ok, ok, 24, 3, pipeline.DCS, 0) == -2     # 8 % 6 != 0
    bad = np.array([0, 10, 24], dtype=np.int32)
    assert api.cp_validate_seqlens(bad, bad, 24, 2, pipeline.DCS, 0) == -2
    assert api.cp_validate_seqlens(bad, bad, 24, 2, pipeline.NLB, 0) == 0
    assert api.cp_validate_seqlens(bad, bad, 24, 5, pipeline.NLB, 0) == -2
    assert api.cp_validate_seqlens(bad, bad, 25, 2, pipeline.NLB, 0) == -7   # cup[n] != T
    cu_long = np.array([0, 12, 20], dtype=np.int32)                          # L_0 > P_0
    assert api.cp_validate_seqlens(cu_long, bad, 24, 2, pipeline.NLB, 1) == -7
    assert api.cp_validate_seqlens(cu_long, bad, 24, 2, pipeline.NLB, 0) == 0  # cu unread


@pytest.mark.parametrize("wl", [inputs.tiny(), inputs.cfg2(), inputs.cfg4(), inputs.cfg5(),
                                inputs.cfg5(tail=False),
                                inputs.custom([7, 33, 1, 90], cp=4, padded=[8, 40, 8, 96]),
                                inputs.custom([5, 9], padded=[8, 16], cp=2)],
                         ids=lambda w: w.name)
def test_valid_end_and_pairs_match_oracle(lib, wl):
    pad = wl.pad_between_seqs
    valid = oracle.valid_mask(wl.cu, wl.cup, pad)
    assert api.cp_valid_end(wl.cu, wl.cup, wl.cp, -1, 0, pad) == oracle.valid_end(valid)
    for s in wl.strategies:
        for r in range(wl.cp):
            idx = oracle.partition_index(wl.cup, wl.cp, r, s)
            assert api.cp_valid_end(wl.cu, wl.cup, wl.cp, r, s, pad) == oracle.valid_end(valid[idx])
            assert pipeline.rank_pairs(wl.cu, wl.cup, wl.cp, r, s, pad) == \
                oracle.causal_pairs(wl.cu, wl.cup, pad, idx)


def test_meta_and_workspace_sizes(lib):
    # header + segments (2n+2) + row tables + one 64-byte list per 128-row
    # query tile and per 128-key block
    # header, segments, row tables, then per tile a 64-byte block list and an 8-byte order entry
    assert api.cp_meta_bytes(3, 128, 2) == 64 + 32 * 8 + 8 * 64 + (64 + 8) * (1 + 1)
    assert api.cp_meta_bytes(3, 1000, 4) == (64 + 32 * 8 + 8 * 250 + 15) // 16 * 16 + (64 + 8) * (2 + 8)
    assert api.cp_meta_bytes(-1, 64, 1) == 0
    assert api.cp_meta_bytes(3, 65, 2) == 0
    assert api.cp_attn_bwd_workspace_bytes(8192, 16) == 8192 * 16 * 4
    # grouped backward: every rank's Delta, then the key blocks' totals (16-aligned) and order
    assert api.cp_attn_bwd_grouped_workspace_bytes(8192, 16, 4, 32768) == \
        4 * 8192 * 16 * 4 + 256 * 4 + 256 * 8
    assert api.cp_attn_bwd_grouped_workspace_bytes(100, 3, 3, 300) == \
        (3 * 100 * 3 * 4 + 15) // 16 * 16 + (3 * 4 + 15) // 16 * 16 + 3 * 8
    assert api.cp_attn_bwd_grouped_workspace_bytes(-1, 3, 3, 300) == 0


FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced below


def _arr(*vals):
    a = (ctypes.c_void_p * len(vals))()
    for i, v in enumerate(vals):
        a[i] = v
    return a


def test_zero_tail_gate_launches_nothing_without_a_tail(lib):
    """[P2P issue] the tail-zeroing must be skipped when the valid end equals
    the tensor end; with a host-known valid end no kernel is launched."""
    L = api.lib()
    launched = ctypes.c_int(7)
    st = L.cp_zero_tail(_arr(FAKE, FAKE + 4096), 2, 100, 256, 100, None, None, ctypes.byref(launched))
    assert st == 0 and launched.value == 0
    # a tail beyond the tensor end is an argument error, caught before any launch
    st = L.cp_zero_tail(_arr(FAKE), 1, 100, 256, 101, None, None, ctypes.byref(launched))
    assert st == -1 and launched.value == 0
    st = L.cp_zero_tail(_arr(FAKE), 1, 100, 250, 50, None, None, ctypes.byref(launched))
    assert st == -4  # row bytes not a multiple of 16


def test_argument_validation_before_launch(lib):
    L = api.lib()
    # partition: rank out of range, NLB total not divisible, meta too small
    assert L.cp_partition_index(None, FAKE, 2, 24, 2, 2, 0, 0, FAKE, None, FAKE, 10 ** 6, None) == -1
    assert L.cp_partition_index(None, FAKE, 2, 25, 2, 0, 1, 0, FAKE, None, FAKE, 10 ** 6, None) == -2
    assert L.cp_partition_index(None, FAKE, 2, 24, 2, 0, 1, 0, FAKE, None, FAKE, 16, None) == -6
    assert L.cp_partition_index(None, FAKE, 2, 24, 2, 0, 1, 1, FAKE, None, FAKE, 10 ** 6, None) == -1
    # every rank in one launch: stride not a multiple of 16, stride too small
    step = api.cp_meta_bytes(2, 24, 2)
    assert L.cp_partition_index_all(None, FAKE, 2, 24, 2, 0, 0, FAKE, None, FAKE,
                                    (step + 15) // 16 * 16 + 8, None) == -4
    assert L.cp_partition_index_all(None, FAKE, 2, 24, 2, 0, 0, FAKE, None, FAKE, 16, None) == -6
    assert L.cp_partition_index_all(None, FAKE, 2, 25, 2, 1, 0, FAKE, None, FAKE, 4096, None) == -2
    # gather: misaligned pointer, bad row size, too many tensors
    assert L.cp_thd_gather(_arr(FAKE + 8), _arr(FAKE), 1, FAKE, 4, 4, 256, None) == -4
    assert L.cp_thd_gather(_arr(FAKE), _arr(FAKE), 1, FAKE, 4, 4, 255, None) == -4
    assert L.cp_thd_gather(_arr(*[FAKE] * 5), _arr(*[FAKE] * 5), 5, FAKE, 4, 4, 256, None) == -1
    # attention: unsupported head dim, bad rank, bad scale, missing workspace
    f = ctypes.c_float
    assert L.cp_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, 128, 2, 96, 2, 0, 0, f(0.1), 0, None) == -3
    assert L.cp_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, 128, 2, 64, 2, 2, 0, f(0.1), 0, None) == -1
    assert L.cp_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, 128, 2, 64, 2, 0, 0, f(-1.0), 0, None) == -1
    assert L.cp_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, 127, 2, 64, 2, 0, 0, f(0.1), 0, None) == -2
    # a misaligned O residual (the optional second output) is refused like any other pointer
    assert L.cp_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE + 8, FAKE, FAKE, 4096, 128, 2, 64, 2, 0, 0,
                         f(0.1), 0, None) == -4
    # an unknown tensor-core operand type
    assert L.cp_attn_fwd(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 4096, 128, 2, 64, 2, 0, 0,
                         f(0.1), 2, None) == -1
    # fused-gather forward: no index, misaligned index, empty source
    assert L.cp_attn_fwd_gather(FAKE, 4096, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, 4096, 2, 64,
                                2, 0, 0, f(0.1), 0, None) == -1
    assert L.cp_attn_fwd_gather(FAKE, 4096, FAKE + 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, 4096, 2,
                                64, 2, 0, 0, f(0.1), 0, None) == -4
    assert L.cp_attn_fwd_gather(FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, 4096, 2, 64,
                                2, 0, 0, f(0.1), 0, None) == -1
    assert L.cp_attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, 128, 2, 64,
                         2, 0, 0, f(0.1), 1, FAKE, 8, None) == -6
    assert L.cp_attn_bwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, 128, 2,
                            64, 2, 0, 0, f(0.1), 0, 7, FAKE, 1 << 20, None) == -1    # unknown mode
    assert L.cp_attn_bwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, 128, 2,
                            64, 2, 0, 0, f(0.1), 1, 1, FAKE, 8, None) == -6           # store mode, small workspace
    assert L.cp_attn_bwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, 128, 2,
                            64, 2, 0, 0, f(0.1), 0, 6, FAKE, 1 << 20, None) == -1    # both dQ modes
    assert L.cp_attn_bwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, 128, 2,
                            64, 2, 0, 0, f(0.1), 5, 0, FAKE, 1 << 20, None) == -1    # unknown operand type
    # grouped backward: stride not a multiple of 16, small workspace, unknown operand type
    assert L.cp_attn_bwd_grouped(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4104,
                                 4096, 2, 64, 2, 0, f(0.1), 0, FAKE, 1 << 24, None) == -4
    assert L.cp_attn_bwd_grouped(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4096,
                                 4096, 2, 64, 2, 0, f(0.1), 0, FAKE, 8, None) == -6
    assert L.cp_attn_bwd_grouped(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4096,
                                 4096, 2, 64, 2, 0, f(0.1), 3, FAKE, 1 << 24, None) == -1
    # grouped backward with the reduce-scatter fused: DUAL_CHUNK_SWAP needs the
    # restore index, which must be int-aligned; outputs required and 16-aligned;
    # then the grouped call's own checks (stride, workspace)
    rs = L.cp_attn_bwd_grouped_rs
    assert rs(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 4096,
              4096, 2, 64, 2, 0, f(0.1), 0, FAKE, 1 << 24, None) == -1
    assert rs(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 2, FAKE, 4096,
              4096, 2, 64, 2, 0, f(0.1), 0, FAKE, 1 << 24, None) == -4
    assert rs(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, 4096,
              4096, 2, 64, 2, 0, f(0.1), 0, FAKE, 1 << 24, None) == -1
    assert rs(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 8, FAKE, None, FAKE, 4096,
              4096, 2, 64, 2, 1, f(0.1), 0, FAKE, 1 << 24, None) == -4
    assert rs(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 4104,
              4096, 2, 64, 2, 1, f(0.1), 0, FAKE, 1 << 24, None) == -4
    assert rs(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4096,
              4096, 2, 64, 2, 0, f(0.1), 0, FAKE, 8, None) == -6
    # the fp16 gather: index optional, but then the source must cover the rows
    assert L.cp_thd_gather_f16(_arr(FAKE), _arr(FAKE), 1, None, 8, 4, 256, None) == -1
    assert L.cp_thd_gather_f16(_arr(FAKE), _arr(FAKE), 1, None, 0, 4, 250, None) == -4
    assert L.cp_reduce_scatter_emul(_arr(FAKE), _arr(FAKE), 1, None, 0, 10, 5, 2, 64, None) == -1


def test_p2p_sizes_and_argument_validation(lib):
    """Ring metadata: one cp_size = 1 block (header, segments, row tables of
    s_local rows, lists and order entries of s_local/128 query tiles and as
    many key blocks) per step, rounded to 16 bytes; arguments checked before
    any launch."""
    L = api.lib()
    lists_off = (64 + 32 * 8 + 8 * 250 + 15) // 16 * 16
    assert api.cp_p2p_meta_bytes(3, 1000, 4) == lists_off + (64 + 8) * (2 + 2)
    assert api.cp_p2p_meta_bytes(3, 1001, 4) == 0
    step = api.cp_p2p_meta_bytes(2, 24, 2)
    # rank out of range, total not divisible, metadata for one step only,
    # padding flag without cu, misaligned metadata
    assert L.cp_p2p_index(None, FAKE, 2, 24, 2, 2, 0, 0, FAKE, 2 * step, None) == -1
    assert L.cp_p2p_index(None, FAKE, 2, 25, 2, 0, 1, 0, FAKE, 2 * step, None) == -2
    assert L.cp_p2p_index(None, FAKE, 2, 24, 2, 0, 1, 0, FAKE, step, None) == -6
    assert L.cp_p2p_index(None, FAKE, 2, 24, 2, 0, 1, 1, FAKE, 2 * step, None) == -1
    assert L.cp_p2p_index(None, FAKE, 2, 24, 2, 0, 1, 0, FAKE + 8, 2 * step, None) == -4
    # merge: no steps, unsupported head dim, misaligned output
    assert L.cp_p2p_merge(FAKE, None, FAKE, 0, 100, 2, 64, FAKE, None, FAKE, None) == -1
    assert L.cp_p2p_merge(FAKE, None, FAKE, 2, 100, 2, 96, FAKE, None, FAKE, None) == -3
    assert L.cp_p2p_merge(FAKE, None, FAKE, 2, 100, 2, 64, FAKE + 4, None, FAKE, None) == -4
    assert L.cp_p2p_merge(FAKE, FAKE + 8, FAKE, 2, 100, 2, 64, FAKE, None, FAKE, None) == -4
    assert L.cp_p2p_merge(FAKE, None, FAKE, 2, 0, 2, 64, FAKE, None, FAKE, None) == 0  # nothing to do
    # one-pass ring backward with bf16 dK/dV out: outputs required and aligned,
    # s_local a multiple of 32
    f = ctypes.c_float
    rs = L.cp_attn_bwd_ring_rs
    assert rs(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, None, FAKE, FAKE, 64, 128, 64, 2, 64,
              2, 0, f(0.1), 0, FAKE, 1 << 24, None) == -1
    assert rs(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE + 8, FAKE, FAKE, 64, 128, 64, 2,
              64, 2, 0, f(0.1), 0, FAKE, 1 << 24, None) == -4
    assert rs(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 128, 48, 2, 64,
              2, 0, f(0.1), 0, FAKE, 1 << 24, None) == -3


def test_product_path_has_no_oracle_or_cpu_fallback():
    """The package never imports the oracle, and the binding refuses to run
    without the compiled library."""
    pkg = os.path.join(ROOT, "context_packed_sequence_thd_gb300")
    for f in os.listdir(pkg):
        if f.endswith(".py"):
            txt = open(os.path.join(pkg, f)).read()
            assert "import oracle" not in txt and "from oracle" not in txt, f
    for f in os.listdir(os.path.join(pkg, "csrc")):
        assert "oracle" not in open(os.path.join(pkg, "csrc", f)).read().lower(), f
