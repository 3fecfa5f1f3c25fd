"""Pins for the oracle's attention forward and backward.

The oracle is checked against references that do not share its code path:
torch's fp64 scaled_dot_product_attention with an explicit block-diagonal
causal mask (and its autograd for the gradients), torch.logsumexp of the
masked score matrix, finite differences, and closed forms."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from context_packed_sequence_thd_gb300 import inputs


def _mask(cu, cup, pad):
    """bool [T, T]: query g may attend key j (document-bounded causal)."""
    cup = np.asarray(cup)
    cu = np.asarray(cu)
    T = int(cup[-1])
    m = np.zeros((T, T), dtype=bool)
    for i in range(len(cup) - 1):
        L = (cu[i + 1] - cu[i]) if pad else (cup[i + 1] - cup[i])
        a = int(cup[i])
        for g in range(a, a + int(L)):
            m[g, a:g + 1] = True
    return m


def _sdpa_ref(q, k, v, do, cu, cup, pad, scale):
    """fp64 SDPA over the valid query rows, with autograd gradients."""
    m = _mask(cu, cup, pad)
    valid = np.nonzero(m.any(1))[0]
    qv = q.double()[valid].permute(1, 0, 2).clone().requires_grad_(True)   # [H, Nq, D]
    kk = k.double().permute(1, 0, 2).clone().requires_grad_(True)          # [H, T, D]
    vv = v.double().permute(1, 0, 2).clone().requires_grad_(True)
    am = torch.from_numpy(m[valid])[None]
    out = F.scaled_dot_product_attention(qv, kk, vv, attn_mask=am, scale=scale)
    scores = (qv @ kk.transpose(1, 2)) * scale
    lse = torch.logsumexp(scores.masked_fill(~am, float("-inf")), dim=-1)  # [H, Nq]
    loss = (out * do.double()[valid].permute(1, 0, 2)).sum()
    loss.backward()
    return (valid, out.detach().permute(1, 0, 2).numpy(), lse.detach().numpy(),
            qv.grad.permute(1, 0, 2).numpy(), kk.grad.permute(1, 0, 2).numpy(),
            vv.grad.permute(1, 0, 2).numpy())


CASES = [
    ("tiny", inputs.tiny()),
    ("padded", inputs.custom([5, 9], padded=[8, 16], cp=2, H=2, D=16, seed=11)),
    ("mixed", inputs.custom([7, 33, 1, 20], padded=[8, 40, 8, 24], cp=4, H=3, D=8, seed=12)),
    ("empty_docs", inputs.custom([0, 6, 0, 10], padded=[4, 8, 0, 12], cp=2, H=1, D=8, seed=13)),
]


@pytest.mark.parametrize("name,wl", CASES, ids=[c[0] for c in CASES])
def test_fwd_bwd_match_sdpa_autograd(name, wl):
    t = wl.tensors()
    scale = 1.0 / np.sqrt(wl.D)
    pad = wl.pad_between_seqs
    valid, o_ref, lse_ref, dq_ref, dk_ref, dv_ref = _sdpa_ref(t["q"], t["k"], t["v"], t["do"],
                                                              wl.cu, wl.cup, pad, scale)
    o, lse = oracle.attn_fwd(t["q"], t["k"], t["v"], wl.cu, wl.cup, pad)
    np.testing.assert_allclose(o[valid], o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[:, valid], lse_ref, rtol=0, atol=1e-12)
    dq, dk, dv = oracle.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], wl.cu, wl.cup, pad)
    np.testing.assert_allclose(dq[valid], dq_ref, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, dk_ref, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, dv_ref, rtol=0, atol=1e-11)
    # padding rows: O = 0, LSE = -inf, dQ = 0; no query attends a padding key
    inval = np.setdiff1d(np.arange(wl.total_tokens), valid)
    assert np.all(o[inval] == 0) and np.all(np.isneginf(lse[:, inval]))
    assert np.all(dq[inval] == 0) and np.all(dk[inval] == 0) and np.all(dv[inval] == 0)


def test_bwd_finite_differences():
    """Central differences of loss = sum(dO * O) on one 8-token document."""
    rng = np.random.default_rng(5)
    T, H, D = 8, 1, 4
    q, k, v, do = (rng.standard_normal((T, H, D)) for _ in range(4))
    cu = [0, T]
    o, lse = oracle.attn_fwd(q, k, v, cu, cu, 0)
    dq, dk, dv = oracle.attn_bwd(q, k, v, o, lse, do, cu, cu, 0)
    eps = 1e-6

    def loss(qq, kk, vv):
        oo, _ = oracle.attn_fwd(qq, kk, vv, cu, cu, 0)
        return float(np.sum(oo * do))

    for grad, which in ((dq, 0), (dk, 1), (dv, 2)):
        for flat in range(T * H * D):
            args = [q.copy(), k.copy(), v.copy()]
            args[which].reshape(-1)[flat] += eps
            lp = loss(*args)
            args[which].reshape(-1)[flat] -= 2 * eps
            lm = loss(*args)
            assert abs((lp - lm) / (2 * eps) - grad.reshape(-1)[flat]) < 1e-7


def test_length_one_document_closed_form():
    """A one-token document attends only itself: O = v, LSE = scale * q.k."""
    rng = np.random.default_rng(3)
    q, k, v = (rng.standard_normal((5, 2, 8)) for _ in range(3))
    cu = [0, 1, 5]
    o, lse = oracle.attn_fwd(q, k, v, cu, cu, 0)
    np.testing.assert_array_equal(o[0], v[0])
    np.testing.assert_allclose(lse[:, 0], np.sum(q[0] * k[0], axis=-1) / np.sqrt(8), atol=1e-15)


def test_equal_keys_running_mean():
    """With all keys equal the softmax is uniform: O_g is the running mean of V
    over [doc start, g] and LSE_g = s + ln(g - start + 1)."""
    rng = np.random.default_rng(4)
    T, H, D = 12, 1, 4
    q = rng.standard_normal((T, H, D))
    k = np.tile(rng.standard_normal((1, H, D)), (T, 1, 1))
    v = rng.standard_normal((T, H, D))
    cu = [0, 5, 12]
    o, lse = oracle.attn_fwd(q, k, v, cu, cu, 0)
    for a, b in ((0, 5), (5, 12)):
        for g in range(a, b):
            np.testing.assert_allclose(o[g], v[a:g + 1].mean(0), atol=1e-14)
            s = np.sum(q[g, 0] * k[0, 0]) / np.sqrt(D)
            np.testing.assert_allclose(lse[0, g], s + np.log(g - a + 1), atol=1e-13)


def test_document_isolation():
    """Changing other documents' K/V leaves a document's outputs unchanged."""
    wl = inputs.custom([9, 14, 6], cp=1, H=2, D=8, seed=21)
    t = wl.tensors()
    o1, l1 = oracle.attn_fwd(t["q"], t["k"], t["v"], wl.cu, wl.cup, 0)
    k2, v2 = t["k"].clone(), t["v"].clone()
    k2[:9] = -k2[:9]
    v2[23:] *= 3
    o2, l2 = oracle.attn_fwd(t["q"], k2, v2, wl.cu, wl.cup, 0)
    np.testing.assert_array_equal(o1[9:23], o2[9:23])
    np.testing.assert_array_equal(l1[:, 9:23], l2[:, 9:23])


@pytest.mark.parametrize("strategy", [oracle.DCS, oracle.NLB])
def test_rank_partials_sum_to_cp1(strategy):
    """Per-rank outputs (rows idx_r of the cp=1 result) equal a run restricted
    to rank r's queries, and the ranks' partial dK/dV sum to the cp=1 dK/dV."""
    wl = inputs.custom([7, 33, 1, 20], padded=[8, 40, 8, 24], cp=4, H=2, D=8, seed=31)
    t = wl.tensors()
    pad = wl.pad_between_seqs
    o, lse = oracle.attn_fwd(t["q"], t["k"], t["v"], wl.cu, wl.cup, pad)
    dq, dk, dv = oracle.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], wl.cu, wl.cup, pad)
    sk, sv = np.zeros_like(dk), np.zeros_like(dv)
    for r in range(wl.cp):
        idx = oracle.partition_index(wl.cup, wl.cp, r, strategy)
        qm = np.zeros(wl.total_tokens, dtype=bool)
        qm[idx] = True
        o_r, l_r = oracle.attn_fwd(t["q"], t["k"], t["v"], wl.cu, wl.cup, pad, qmask=qm)
        np.testing.assert_array_equal(o_r[idx], o[idx])
        np.testing.assert_array_equal(l_r[:, idx], lse[:, idx])
        dq_r, dk_r, dv_r = oracle.attn_bwd(t["q"], t["k"], t["v"], o, lse, t["do"], wl.cu, wl.cup,
                                           pad, qmask=qm)
        np.testing.assert_array_equal(dq_r[idx], dq[idx])
        sk += dk_r
        sv += dv_r
    np.testing.assert_allclose(sk, dk, atol=1e-12)
    np.testing.assert_allclose(sv, dv, atol=1e-12)


def test_value_equal_metadata_is_no_padding():
    """cu_seqlens_padded a value-equal clone: pad_between_seqs=1 and =0 give
    identical results, and the detector says 0."""
    wl = inputs.custom([16, 24, 8], cp=2, H=2, D=8, seed=41)
    cup = wl.cu.copy()
    assert oracle.pad_between_seqs(wl.cu, cup) == 0
    t = wl.tensors()
    a = oracle.attn_fwd(t["q"], t["k"], t["v"], wl.cu, cup, 1)
    b = oracle.attn_fwd(t["q"], t["k"], t["v"], wl.cu, cup, 0)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_head_subset_matches_all_heads():
    wl = inputs.custom([20, 12], cp=2, H=4, D=8, seed=51)
    t = wl.tensors()
    o, lse = oracle.attn_fwd(t["q"], t["k"], t["v"], wl.cu, wl.cup, 0)
    o2, lse2 = oracle.attn_fwd(t["q"], t["k"], t["v"], wl.cu, wl.cup, 0, heads=[1, 3])
    np.testing.assert_array_equal(o2[:, [1, 3]], o[:, [1, 3]])
    assert np.all(np.isnan(o2[:, [0, 2]]))


# ---------------------------------------------------------------------------
# P2P ring ("THD P2P context-parallel regression ..."; the ring comm type)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("strategy", [0, 1])
def test_p2p_ring_visits_every_shard_once(strategy):
    for cp in (1, 2, 4):
        for r in range(cp):
            assert sorted(oracle.p2p_schedule(cp, r)) == list(range(cp))
            assert oracle.p2p_schedule(cp, r)[0] == r          # step 0: the rank's own K/V


@pytest.mark.parametrize("strategy", [0, 1])
@pytest.mark.parametrize("cu,cup,pad,cp", [
    ([0, 32, 48, 96, 128], [0, 32, 48, 96, 128], 0, 2),
    # padded: 4, 5 and 3 padding rows at the ends of the documents (a padding
    # query sees no key; no query sees a padding key)
    ([0, 20, 23, 36], [0, 24, 32, 48], 1, 2),
    ([0, 13, 13, 33], [0, 16, 24, 48], 1, 2),
], ids=["unpadded", "padded", "padded_empty_doc"])
def test_p2p_step_keys_cover_the_causal_range(strategy, cu, cup, pad, cp):
    """Over the ring's steps a query row's visible key ranges, mapped back to
    global rows, are disjoint and together exactly [document start, row] for a
    real token, and empty for a padding row."""
    valid = oracle.valid_mask(cu, cup, pad)
    start = np.repeat(np.asarray(cup[:-1]), np.diff(cup))
    for r in range(cp):
        G_r = oracle.partition_index(cup, cp, r, strategy)
        seen = [[] for _ in G_r]
        for j in oracle.p2p_schedule(cp, r):
            G_j = oracle.partition_index(cup, cp, j, strategy)
            lo, hi = oracle.p2p_step_rows(cu, cup, cp, r, j, strategy, pad)
            for t in range(len(G_r)):
                seen[t].extend(G_j[lo[t]:hi[t] + 1].tolist())
        for t, g in enumerate(G_r):
            want = list(range(start[g], g + 1)) if valid[g] else []
            assert sorted(seen[t]) == want
            assert all(valid[x] for x in seen[t])


@pytest.mark.parametrize("strategy", [0, 1])
def test_p2p_merge_equals_full_attention(strategy):
    """Merging the ring's per-step partial softmaxes by their LSE gives the
    full causal attention (the ring only reorders the sum)."""
    rng = np.random.default_rng(17)
    cu = [0, 20, 23, 36]
    cup = [0, 24, 32, 48]
    T, H, D = 48, 2, 8
    q, k, v = (rng.standard_normal((T, H, D)) for _ in range(3))
    o, lse = oracle.attn_fwd(q, k, v, cu, cup, 1)
    o2, lse2 = oracle.p2p_attn_fwd(q, k, v, cu, cup, 1, 2, strategy)
    valid = oracle.valid_mask(cu, cup, 1)
    np.testing.assert_allclose(o2[valid], o[valid], atol=1e-12)
    np.testing.assert_allclose(lse2[:, valid], lse[:, valid], atol=1e-12)
    assert np.all(np.isneginf(lse2[:, ~valid]))


def test_lse_merge_of_a_key_split_is_the_full_softmax():
    """Softmax over a key set split into disjoint parts: each part's
    normalised output and log-sum-exp, merged, give the softmax over all keys
    (brute force on a tiny case); one part is returned unchanged; parts that
    saw no key (LSE = -inf) carry no weight; a row no part saw is 0 / -inf."""
    rng = np.random.default_rng(23)
    rows, H, D, nk = 5, 3, 4, 11
    s = rng.standard_normal((rows, H, nk)) * 3.0
    vals = rng.standard_normal((nk, H, D))
    split = [[0, 4, 7], [1, 2, 9, 10], [], [3, 5, 6, 8]]
    o_parts, l_parts = [], []
    for keys in split:
        o_i = np.zeros((rows, H, D))
        l_i = np.full((H, rows), -np.inf)
        if keys:
            sk = s[:, :, keys]
            l_i = np.log(np.exp(sk).sum(axis=2)).T
            p = np.exp(sk) / np.exp(sk).sum(axis=2, keepdims=True)
            o_i = np.einsum("rhk,khd->rhd", p, vals[keys])
        o_parts.append(o_i)
        l_parts.append(l_i)
    o, lse = oracle.lse_merge(np.stack(o_parts), np.stack(l_parts))
    p_all = np.exp(s) / np.exp(s).sum(axis=2, keepdims=True)
    np.testing.assert_allclose(o, np.einsum("rhk,khd->rhd", p_all, vals), atol=1e-12)
    np.testing.assert_allclose(lse, np.log(np.exp(s).sum(axis=2)).T, atol=1e-12)
    o1, l1 = oracle.lse_merge(np.stack(o_parts[:1]), np.stack(l_parts[:1]))
    np.testing.assert_allclose(o1, o_parts[0], atol=1e-15)
    np.testing.assert_allclose(l1, l_parts[0], atol=1e-15)
    o0, l0 = oracle.lse_merge(np.stack([o_parts[2]] * 2), np.stack([l_parts[2]] * 2))
    assert np.all(o0 == 0) and np.all(np.isneginf(l0))


@pytest.mark.parametrize("strategy", [0, 1])
def test_ring_backward_schedule(strategy):
    """The emulated ring's backward calls: each rank walks the oracle's ring
    order (all cp steps under DUAL_CHUNK_SWAP, steps 0..r under
    NO_LOAD_BALANCE, whose later shards hold only later tokens -- the oracle's
    brute force finds no visible key there); the first call touching a K/V
    shard stores its dK/dV partial and later ones add; a rank's first step
    stores its fp32 dQ and later ones add."""
    from context_packed_sequence_thd_gb300 import api, pipeline
    cu = cup = [0, 32, 48, 96, 128]
    for cp in (1, 2, 4):
        steps = pipeline.ring_steps(cp, strategy)
        seen = set()
        for r in range(cp):
            mine = [(i, j, m) for rr, i, j, m in steps if rr == r]
            ring = oracle.p2p_schedule(cp, r)
            assert [j for _, j, _ in mine] == ring[:len(mine)]
            assert [i for i, _, _ in mine] == list(range(len(mine)))
            for i, j, m in mine:
                assert (m & (api.BWD_DQ_F32_STORE | api.BWD_DQ_F32_ACCUMULATE)) == \
                    (api.BWD_DQ_F32_STORE if i == 0 else api.BWD_DQ_F32_ACCUMULATE)
            # the skipped steps have no visible key at all
            for j in ring[len(mine):]:
                _, hi = oracle.p2p_step_rows(cu, cup, cp, r, j, strategy, 0)
                assert np.all(hi < 0)
        for r, i, j, m in steps:
            seen.add(j)
        assert seen == set(range(cp))
        # Replay the calls in order on buffers that start as garbage (NaN):
        # a store overwrites, an add adds.  Every dK/dV shard buffer must end
        # as the sum of every partial aimed at that shard, and every rank's dQ
        # buffer as the sum of its steps' partials -- a wrong store/add rule
        # either keeps the garbage or drops / doubles a term.
        rng = np.random.default_rng(cp)
        dkv = np.full(cp, np.nan)
        dq = np.full(cp, np.nan)
        want_kv, want_q = np.zeros(cp), np.zeros(cp)
        for r, i, j, m in steps:
            p_kv, p_q = float(rng.integers(1, 1000)), float(rng.integers(1, 1000))
            want_kv[j] += p_kv
            want_q[r] += p_q
            dkv[j] = p_kv if m & api.BWD_STORE else dkv[j] + p_kv
            if m & api.BWD_DQ_F32_STORE:
                dq[r] = p_q
            else:
                assert m & api.BWD_DQ_F32_ACCUMULATE
                dq[r] += p_q
        np.testing.assert_array_equal(dkv, want_kv)
        np.testing.assert_array_equal(dq, want_q)
