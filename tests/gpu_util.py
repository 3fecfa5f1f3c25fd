"""Helpers shared by the GPU parity tests (comparison and tolerance only)."""
import numpy as np
import torch

# BF16 outputs and gradients vs the fp64 oracle: max-abs 2e-2, mean-abs 2e-3.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def dev():
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def assert_close(got, ref, what: str, max_abs: float = MAX_ABS, mean_abs: float = MEAN_ABS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    mx, mn = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= max_abs and mn <= mean_abs, \
        f"{what}: max-abs {mx:.3e} (limit {max_abs}), mean-abs {mn:.3e} (limit {mean_abs}), " \
        f"max |ref| {float(np.abs(ref).max()) if ref.size else 0:.3f}"
    return mx, mn


def assert_lse_close(got, ref, what: str, tol: float = 1e-3):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    inf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf_ref), f"{what}: -inf pattern differs"
    err = np.abs(got[~inf_ref] - ref[~inf_ref])
    assert err.size == 0 or err.max() <= tol, f"{what}: LSE max-abs {err.max():.3e}"


def check_block_lists(meta, h, lo, hi, T, cap=7):
    """Block lists of the metadata against brute force over the row tables:
    the key blocks of every 128-row query tile, the query tiles of every
    128-key block, and the heaviest-first order of each family."""
    s_local, lists_off = int(h[6]), int(h[14])
    n_qt, n_kb = -(-s_local // 128), -(-T // 128)
    raw = meta[lists_off:lists_off + 64 * (n_qt + n_kb)].cpu().numpy().view(np.int32)
    raw = raw.reshape(n_qt + n_kb, 16)
    ord_off = lists_off + 64 * (n_qt + n_kb)
    orders = meta[ord_off:ord_off + 8 * (n_qt + n_kb)].cpu().numpy().view(np.int32).reshape(-1, 2)
    want_q = [set() for _ in range(n_qt)]
    want_k = [set() for _ in range(n_kb)]
    for t in range(s_local):
        if hi[t] >= 0:
            for b in range(lo[t] // 128, hi[t] // 128 + 1):
                want_q[t // 128].add(b)
                want_k[b].add(t // 128)
    for fam, want, order in ((raw[:n_qt], want_q, orders[:n_qt]), (raw[n_qt:], want_k, orders[n_qt:])):
        counts = []
        for q, l in enumerate(fam):
            n = min(int(l[0]), cap)
            got = set()
            for i in range(n):
                assert l[2 + 2 * i] <= l[3 + 2 * i]
                got.update(range(int(l[2 + 2 * i]), int(l[3 + 2 * i]) + 1))
            if int(l[0]) < cap:
                assert got == want[q]
            else:                      # over capacity the last interval widens
                assert want[q] <= got
            counts.append(len(got))
            assert l[1] == len(got)        # header: {count, blocks covered}
        tiles = order[:, 0]
        assert sorted(tiles.tolist()) == list(range(len(fam)))
        assert [counts[t] for t in tiles] == order[:, 1].tolist()
        keys = [(-counts[t], t) for t in tiles]
        assert keys == sorted(keys)    # heaviest first, ties by index
