"""Pins for the oracle's integer parts (partition, restore, gather, pad flag,
valid end).  Each test checks the oracle against something other than itself:
hand-derived examples, closed forms, or invariants the pages fix."""
import json
import os

import numpy as np
import pytest

import oracle
from context_packed_sequence_thd_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "partition_examples.json")


def _ranges_to_rows(ranges):
    return np.concatenate([np.arange(a, b) for a, b in ranges]) if ranges else np.zeros(0)


def _examples():
    with open(GOLDEN) as f:
        return json.load(f)["examples"]


@pytest.mark.parametrize("ex", _examples(), ids=lambda e: e["name"])
def test_hand_derived_partitions(ex):
    cp = ex["cp"]
    for key, strat in (("dual_chunk_swap", oracle.DCS), ("no_load_balance", oracle.NLB)):
        for r in range(cp):
            want = _ranges_to_rows(ex[key][str(r)])
            got = oracle.partition_index(ex["cu_seqlens_padded"], cp, r, strat)
            np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("ex", _examples(), ids=lambda e: e["name"])
def test_hand_derived_valid_end(ex):
    cp = ex["cp"]
    valid = oracle.valid_mask(ex["cu_seqlens"], ex["cu_seqlens_padded"], ex["pad_between_seqs"])
    assert oracle.valid_end(valid) == ex["valid_end_global"]
    for key, strat in (("dual_chunk_swap", oracle.DCS), ("no_load_balance", oracle.NLB)):
        for r in range(cp):
            idx = oracle.partition_index(ex["cu_seqlens_padded"], cp, r, strat)
            assert oracle.valid_end(valid[idx]) == ex["valid_end_local"][key][r]


def _workloads():
    return [inputs.tiny(), inputs.cfg2(), inputs.cfg3(8192), inputs.cfg4(), inputs.cfg5(),
            inputs.custom([7, 33, 1, 90], cp=4, padded=[8, 40, 8, 96])]


@pytest.mark.parametrize("wl", _workloads(), ids=lambda w: w.name)
def test_ranks_tile_the_buffer(wl):
    """The rank partitions are disjoint, each holds s_local rows, and together
    they cover [0, T) exactly."""
    T = wl.total_tokens
    for strat in wl.strategies:
        G = []
        for r in range(wl.cp):
            idx = oracle.partition_index(wl.cup, wl.cp, r, strat)
            assert len(idx) == T // wl.cp
            G.append(idx)
        G = np.concatenate(G)
        np.testing.assert_array_equal(np.sort(G), np.arange(T))


@pytest.mark.parametrize("wl", _workloads(), ids=lambda w: w.name)
def test_restore_inverts_partition(wl):
    T = wl.total_tokens
    rows = np.arange(T, dtype=np.int64) * 7 + 3       # stand-in row payloads
    for strat in wl.strategies:
        concat = np.concatenate([oracle.gather_rows(rows, oracle.partition_index(wl.cup, wl.cp, r, strat))
                                 for r in range(wl.cp)])
        R = oracle.restore_index(wl.cup, wl.cp, strat)
        np.testing.assert_array_equal(oracle.gather_rows(concat, R), rows)
        if strat == oracle.NLB:
            np.testing.assert_array_equal(R, np.arange(T))


def test_dcs_balanced_pairs_closed_form():
    """Without padding, every DUAL_CHUNK_SWAP rank gets the same causal work:
    per document of 2*cp*c tokens, rank r's pairs are
    sum_u (r*c+u+1) + sum_u ((2cp-1-r)*c+u+1) = c^2 (2cp-1) + c(c+1)."""
    wl = inputs.cfg2()
    lens = oracle.doc_lengths(wl.cup)
    for r in range(wl.cp):
        idx = oracle.partition_index(wl.cup, wl.cp, r, oracle.DCS)
        got = oracle.causal_pairs(wl.cu, wl.cup, 0, idx)
        want = sum((P // (2 * wl.cp)) ** 2 * (2 * wl.cp - 1) + (P // (2 * wl.cp)) * (P // (2 * wl.cp) + 1)
                   for P in lens)
        assert got == want
    # and the ranks together do the cp=1 work: sum_i L_i (L_i+1)/2
    assert oracle.causal_pairs(wl.cu, wl.cup, 0) == sum(int(L) * (int(L) + 1) // 2 for L in lens)


def test_nlb_single_sequence_pairs_closed_form():
    """One sequence of s tokens, contiguous shards: rank r's pairs are
    sum_{g=r*m}^{(r+1)m-1} (g+1) = m^2 r + m(m+1)/2 with m = s/cp."""
    wl = inputs.cfg3(32768)
    m = wl.s_local
    for r in range(wl.cp):
        idx = oracle.partition_index(wl.cup, wl.cp, r, oracle.NLB)
        assert oracle.causal_pairs(wl.cu, wl.cup, 0, idx) == m * m * r + m * (m + 1) // 2


def test_strategy_constraints():
    with pytest.raises(ValueError):
        oracle.partition_index([0, 10, 30], 2, 0, oracle.DCS)   # 10 % 4 != 0
    with pytest.raises(ValueError):
        oracle.partition_index([0, 10, 31], 2, 0, oracle.NLB)   # 31 % 2 != 0
    # NO_LOAD_BALANCE drops per-document divisibility entirely
    assert len(oracle.partition_index([0, 9, 30], 2, 1, oracle.NLB)) == 15


def test_pad_flag_is_decided_by_values():
    """The reproduction of the P2P issue: cu_seqlens = [0, s] and a clone of
    it must mean 'no padding between sequences'."""
    import torch
    cu = torch.tensor([0, 4096], dtype=torch.int32)
    cup = cu.clone()
    assert cup is not cu and torch.equal(cup, cu)
    assert oracle.pad_between_seqs(cu.numpy(), cup.numpy()) == 0
    assert oracle.pad_between_seqs([0, 5, 14], [0, 8, 24]) == 1
    assert oracle.pad_between_seqs([0, 5, 14], None) == 0
    # a difference in the last entry alone is padding too
    assert oracle.pad_between_seqs([0, 8, 20], [0, 8, 24]) == 1


def test_gather_scatter_bitwise():
    rng = np.random.default_rng(0)
    src = rng.integers(0, 2 ** 16, size=(50, 3, 8), dtype=np.uint16)
    idx = rng.permutation(50)
    g = oracle.gather_rows(src, idx)
    assert g.dtype == np.uint16
    np.testing.assert_array_equal(g[5], src[idx[5]])
    back = oracle.scatter_rows(np.zeros_like(src), idx, g)
    np.testing.assert_array_equal(back, src)


def test_workload_recipes():
    wl = inputs.cfg2()
    lens = oracle.doc_lengths(wl.cu)
    assert wl.total_tokens == 32768 and len(lens) == 16
    assert np.all(lens % 16 == 0) and lens.min() >= 256 and lens.max() <= 4096
    wl4 = inputs.cfg4()
    l4 = oracle.doc_lengths(wl4.cu)
    assert wl4.total_tokens == 75600 and np.all(l4 % 16 != 0) and l4.min() >= 17
    wl5 = inputs.cfg5()
    L, P = oracle.doc_lengths(wl5.cu), oracle.doc_lengths(wl5.cup)
    assert wl5.total_tokens == 65536 and len(P) == 24
    assert np.all(P % 8 == 0) and np.all(L <= P) and np.all(P - L < 8) and P[-1] - L[-1] == 3
    assert oracle.pad_between_seqs(wl5.cu, wl5.cup) == 1
    eq = inputs.cfg5(value_equal=True)
    assert eq.cu is not eq.cup and oracle.pad_between_seqs(eq.cu, eq.cup) == 0


def test_bf16_round_nearest_even():
    """The oracle's fp32->bf16 rounding, pinned to torch's CPU conversion and
    to hand-made ties (1 + 2^-8 is a tie that rounds to even = 1.0;
    1 + 3*2^-8 rounds up to 1 + 2^-6)."""
    import torch
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(10000).astype(np.float32) * 10,
                        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 0.0, -0.0],
                                 dtype=np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.bf16_round(x), want)
    assert oracle.bf16_round(np.float32(1 + 2 ** -8)) == 0x3F80
    assert oracle.bf16_round(np.float32(1 + 3 * 2 ** -8)) == 0x3F82


# ---------------------------------------------------------------------------
# a2a exchange ("[PyTorch] Extend no-load-balance CP to the a2a comm type")
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("strategy", [0, 1])
def test_a2a_exchange_restores_sequence_and_splits_heads(strategy):
    """After the seq->head exchange of the ranks' shards, rank r holds the
    original sequence with heads [r*H/cp, (r+1)*H/cp); the reverse exchange
    gives the shards back (round trip = identity)."""
    rng = np.random.default_rng(5)
    cup = [0, 16, 48, 64]
    cp, H = 2, 6
    x = rng.integers(0, 2 ** 16, size=(64, H, 4), dtype=np.uint16)   # original order
    G = np.concatenate([oracle.partition_index(cup, cp, r, strategy) for r in range(cp)])
    seq = x[G]                                                       # rank-concatenated shards
    perm = oracle.restore_index(cup, cp, strategy) if strategy == 0 else None
    head = oracle.a2a_seq_to_head(seq, cp, perm)
    assert head.shape == (cp, 64, H // cp, 4)
    for r in range(cp):
        np.testing.assert_array_equal(head[r], x[:, r * 3:(r + 1) * 3])
    np.testing.assert_array_equal(oracle.a2a_head_to_seq(head, perm), seq)


def test_a2a_flat_needs_no_reorder():
    """Flat sharding: the rank-concatenated order is the original order, so the
    exchange with no permutation equals the one with the identity restore."""
    rng = np.random.default_rng(6)
    cup = [0, 10, 40, 64]
    x = rng.integers(0, 2 ** 16, size=(64, 4, 2), dtype=np.uint16)
    R = oracle.restore_index(cup, 4, 1)
    np.testing.assert_array_equal(R, np.arange(64))
    np.testing.assert_array_equal(oracle.a2a_seq_to_head(x, 4, None), oracle.a2a_seq_to_head(x, 4, R))
