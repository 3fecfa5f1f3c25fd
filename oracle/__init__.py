"""fp64 CPU oracle for context-parallel causal attention over THD-packed documents.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library never calls it, and it never calls the product
library: the two share no code.

Contents, each the plain definition of what the pages describe:

* ``partition_index``   per-rank token partition (DUAL_CHUNK_SWAP /
  NO_LOAD_BALANCE), "[PyTorch] Add no-load-balance THD all-gather CP", §Why and
  §What changed; "[PyTorch] Extend no-load-balance CP to the a2a comm type",
  first paragraph (flat sharding = contiguous range [r*s_local,(r+1)*s_local)).
* ``restore_index``     inverse of the rank-concatenated partition, the order
  restore of the all-gathered K/V (same page, §Sequence Diagram).
* ``gather_rows`` / ``scatter_rows``  THD row index_select and its inverse.
* ``pad_between_seqs``  decided from values, "THD P2P context-parallel
  regression when padded cu_seqlens are value-equal but not object-identical",
  §Expected behavior.
* ``valid_end``         one past the last valid row of a layout (the tail the
  gradient tail-zeroing clears, same issue, §Describe the bug).
* ``attn_fwd`` / ``attn_bwd``  causal varlen attention, fp64, in
  ``cpthd_oracle.c`` (see its header for the formulas).
* ``a2a_seq_to_head`` / ``a2a_head_to_seq``  the all-to-all exchange of the
  a2a comm type, "[PyTorch] Extend no-load-balance CP to the a2a comm type",
  first two paragraphs and §Diagram.
* ``p2p_schedule`` / ``p2p_step_rows`` / ``p2p_attn_fwd`` / ``lse_merge``  the
  ring (P2P) comm type of "THD P2P context-parallel regression when padded
  cu_seqlens are value-equal but not object-identical", §Describe the bug.
  The page names the comm type, not its arithmetic; these follow the usual
  ring schedule (step i: the K/V shard of rank (r - i) mod cp) and the
  log-sum-exp combination of partial softmaxes.

Every function here is pinned by a ``-m "not gpu"`` test against something
other than itself (hand-derived partitions, closed forms, torch's fp64 SDPA
with an explicit mask and its autograd, finite differences, a brute-force
softmax over a split key set).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import List, Optional, Sequence, Tuple

import numpy as np

DCS = 0
NLB = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libcpthd_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc, -O2, OpenMP) in place; returns the .so path."""
    src = os.path.join(_HERE, "cpthd_oracle.c")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                           src, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        lib.oracle_attn_fwd.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        P, P, ctypes.c_int, ctypes.c_double, P, P, P, P, P,
                                        ctypes.c_int, P, P]
        lib.oracle_attn_fwd.restype = None
        lib.oracle_attn_bwd.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        P, P, ctypes.c_int, ctypes.c_double, P, P, P, P, P, P,
                                        P, P, ctypes.c_int, P, P, P]
        lib.oracle_attn_bwd.restype = None
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# ----------------------------------------------------------------------------
# integer parts
# ----------------------------------------------------------------------------

def doc_lengths(cu: np.ndarray) -> np.ndarray:
    cu = np.asarray(cu, dtype=np.int64)
    return cu[1:] - cu[:-1]


def partition_index(cup: Sequence[int], cp: int, rank: int, strategy: int) -> np.ndarray:
    """Global rows held by CP rank ``rank``, in the rank's local order.

    DUAL_CHUNK_SWAP: every document's padded range is cut into 2*cp equal
    chunks; the rank takes chunk ``rank`` and chunk ``2*cp-1-rank`` of every
    document, documents in order, the early chunk first.
    NO_LOAD_BALANCE: the rank takes the contiguous physical range
    [rank*s_local, (rank+1)*s_local) of the packed buffer, s_local = T/cp.
    """
    cup = np.asarray(cup, dtype=np.int64)
    T = int(cup[-1])
    if strategy == NLB:
        if T % cp:
            raise ValueError("NO_LOAD_BALANCE needs the packed total divisible by cp")
        s_local = T // cp
        return np.arange(rank * s_local, (rank + 1) * s_local, dtype=np.int64)
    if strategy != DCS:
        raise ValueError("unknown strategy")
    parts = []
    for i in range(len(cup) - 1):
        P = int(cup[i + 1] - cup[i])
        if P % (2 * cp):
            raise ValueError("DUAL_CHUNK_SWAP needs every padded length divisible by 2*cp")
        c = P // (2 * cp)
        for chunk in (rank, 2 * cp - 1 - rank):
            start = int(cup[i]) + chunk * c
            parts.append(np.arange(start, start + c, dtype=np.int64))
    return np.concatenate(parts) if parts else np.zeros(0, dtype=np.int64)


def restore_index(cup: Sequence[int], cp: int, strategy: int) -> np.ndarray:
    """R with R[g] = position of global row g in concat_r(partition_index(r)).

    Gathering the rank-concatenated (all-gathered) buffer with R puts the rows
    back in original order."""
    G = np.concatenate([partition_index(cup, cp, r, strategy) for r in range(cp)])
    R = np.empty_like(G)
    R[G] = np.arange(len(G), dtype=np.int64)
    return R


def gather_rows(src: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """dst[i] = src[idx[i]] on whole rows (any dtype, compared bitwise)."""
    return src[np.asarray(idx, dtype=np.int64)]


def scatter_rows(dst: np.ndarray, idx: np.ndarray, src: np.ndarray) -> np.ndarray:
    """dst[idx[i]] = src[i]; returns a new array."""
    out = dst.copy()
    out[np.asarray(idx, dtype=np.int64)] = src
    return out


def a2a_seq_to_head(seq: np.ndarray, cp: int, perm=None) -> np.ndarray:
    """All-to-all before attention ("[PyTorch] Extend no-load-balance CP to the
    a2a comm type", ¶2 and §Diagram): from the rank-concatenated token shards
    [T, H, D] to cp head slices [cp, T, H/cp, D], rank r holding every token in
    original order with heads [r*H/cp, (r+1)*H/cp).  Original token g sits at
    sequence-side row perm[g] (the restore index for DUAL_CHUNK_SWAP; identity
    for flat sharding when perm is None)."""
    T, H = seq.shape[0], seq.shape[1]
    rows = np.arange(T) if perm is None else np.asarray(perm, dtype=np.int64)
    ordered = seq[rows]                        # [T, H, ...] in original order
    hc = H // cp
    return np.stack([ordered[:, r * hc:(r + 1) * hc] for r in range(cp)])


def a2a_head_to_seq(head: np.ndarray, perm=None) -> np.ndarray:
    """The reverse exchange after attention: head slices [cp, T, H/cp, D] back
    to the rank-concatenated token shards [T, H, D]."""
    cp, T = head.shape[0], head.shape[1]
    ordered = np.concatenate([head[r] for r in range(cp)], axis=1)   # [T, H, ...]
    rows = np.arange(T) if perm is None else np.asarray(perm, dtype=np.int64)
    out = np.empty_like(ordered)
    out[rows] = ordered
    return out


def p2p_schedule(cp: int, rank: int) -> List[int]:
    """Ring order of the P2P comm type: at step i rank ``rank`` holds the K/V
    shard that started on rank (rank - i) mod cp (each step passes K/V one rank
    along the ring)."""
    return [(rank - i) % cp for i in range(cp)]


def p2p_step_rows(cu, cup, cp: int, rank: int, kv_rank: int, strategy: int, pad: int):
    """Keys each local query row of ``rank`` sees in ``kv_rank``'s K/V shard,
    as inclusive ranges [lo, hi] of that shard's local rows (lo = 0, hi = -1
    when none): brute force over the two partition indices -- key global row
    in [document start, query row], query a real token.  Asserts that every
    row's keys form one contiguous range of the shard."""
    G_r = partition_index(cup, cp, rank, strategy)
    G_j = partition_index(cup, cp, kv_rank, strategy)
    valid = valid_mask(cu, cup, pad)
    cup_ = np.asarray(cup, dtype=np.int64)
    start = np.repeat(cup_[:-1], np.diff(cup_))
    lo = np.zeros(len(G_r), dtype=np.int32)
    hi = np.full(len(G_r), -1, dtype=np.int32)
    for t0 in range(0, len(G_r), 512):           # 512 query rows at a time
        g = G_r[t0:t0 + 512]
        vis = (G_j[None, :] >= start[g][:, None]) & (G_j[None, :] <= g[:, None])
        vis &= valid[g][:, None]
        n = vis.sum(axis=1)
        first = np.argmax(vis, axis=1)
        last = len(G_j) - 1 - np.argmax(vis[:, ::-1], axis=1)
        some = n > 0
        assert np.all(last[some] - first[some] + 1 == n[some]), "keys of a row are not contiguous"
        lo[t0:t0 + 512] = np.where(some, first, 0)
        hi[t0:t0 + 512] = np.where(some, last, -1)
    return lo, hi


def p2p_attn_fwd(q, k, v, cu, cup, pad: int, cp: int, strategy: int, scale=None):
    """The P2P ring's forward, step by step in fp64: at every step each rank's
    queries attend the visible keys of the K/V shard it holds (dense softmax
    over those keys), giving a partial (O_i, LSE_i); the partials merge as
    LSE = log sum_i exp(LSE_i), O = sum_i exp(LSE_i - LSE) O_i.  Returns O, LSE
    in original row order (equal to attn_fwd: the ring only reorders the sum)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, D = q.shape
    sc = 1.0 / np.sqrt(D) if scale is None else float(scale)
    o = np.zeros((T, H, D))
    lse = np.full((H, T), -np.inf)
    for r in range(cp):
        G_r = partition_index(cup, cp, r, strategy)
        parts = []
        for j in p2p_schedule(cp, r):
            G_j = partition_index(cup, cp, j, strategy)
            lo, hi = p2p_step_rows(cu, cup, cp, r, j, strategy, pad)
            o_i = np.zeros((len(G_r), H, D))
            l_i = np.full((H, len(G_r)), -np.inf)
            for t in range(len(G_r)):
                if hi[t] < lo[t]:
                    continue
                keys = G_j[lo[t]:hi[t] + 1]
                s = np.einsum("hd,khd->hk", q[G_r[t]], k[keys]) * sc
                m = s.max(axis=1, keepdims=True)
                e = np.exp(s - m)
                l_i[:, t] = (m[:, 0] + np.log(e.sum(axis=1)))
                o_i[t] = np.einsum("hk,khd->hd", e / e.sum(axis=1, keepdims=True), v[keys])
            parts.append((o_i, l_i))
        o_r, l_r = lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        o[G_r] = o_r
        lse[:, G_r] = l_r
    return o, lse


def lse_merge(o_parts, lse_parts):
    """Softmax-weighted combination of partial attention results of the same
    queries over disjoint key sets, in fp64: o_parts [n, rows, H, D] (each
    normalised over its own keys), lse_parts [n, H, rows] (-inf: no key).
    LSE = log sum_i exp(LSE_i); O = sum_i exp(LSE_i - LSE) O_i; rows without
    any key get O = 0, LSE = -inf."""
    o_parts, L = _f64(o_parts), _f64(lse_parts)
    Lm = L.max(axis=0)
    fin = np.isfinite(Lm)
    with np.errstate(divide="ignore"):            # log(0) of rows no part saw, discarded
        Ltot = np.where(fin, Lm + np.log(np.exp(L - np.where(fin, Lm, 0)).sum(axis=0)), -np.inf)
    w = np.where(fin, np.exp(L - np.where(fin, Ltot, 0)), 0.0)   # [n, H, rows]
    o = np.einsum("nhr,nrhd->rhd", w, o_parts)
    return o, Ltot


def pad_between_seqs(cu: Sequence[int], cup: Optional[Sequence[int]]) -> int:
    """1 when any entry of the padded offsets differs from the actual offsets."""
    if cup is None:
        return 0
    a = np.asarray(cu, dtype=np.int64)
    b = np.asarray(cup, dtype=np.int64)
    if a.shape != b.shape:
        return 1
    return int(np.any(a != b))


def valid_mask(cu: Sequence[int], cup: Sequence[int], pad: int) -> np.ndarray:
    """bool [T]: row g is a real token (not padding)."""
    cu = np.asarray(cu, dtype=np.int64)
    cup = np.asarray(cup, dtype=np.int64)
    T = int(cup[-1])
    m = np.zeros(T, dtype=bool)
    for i in range(len(cup) - 1):
        L = (cu[i + 1] - cu[i]) if pad else (cup[i + 1] - cup[i])
        m[cup[i]:cup[i] + L] = True
    return m


def valid_end(rows_valid: np.ndarray) -> int:
    """One past the last valid row of a layout (0 when none is valid)."""
    nz = np.nonzero(np.asarray(rows_valid))[0]
    return int(nz[-1]) + 1 if len(nz) else 0


def causal_pairs(cu, cup, pad: int, rows: Optional[np.ndarray] = None) -> int:
    """Number of (query, key) pairs attended by the given global query rows."""
    cu = np.asarray(cu, dtype=np.int64)
    cup = np.asarray(cup, dtype=np.int64)
    T = int(cup[-1])
    valid = valid_mask(cu, cup, pad)
    start = np.zeros(T, dtype=np.int64)
    for i in range(len(cup) - 1):
        start[cup[i]:cup[i + 1]] = cup[i]
    g = np.arange(T, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    return int(np.sum(np.where(valid[g], g - start[g] + 1, 0)))


# ----------------------------------------------------------------------------
# attention (fp64, C)
# ----------------------------------------------------------------------------

def _f64(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to(torch.float64).cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _heads(H: int, heads) -> np.ndarray:
    return _i32(np.arange(H) if heads is None else heads)


def attn_fwd(q, k, v, cu, cup, pad: int, scale: Optional[float] = None, heads=None,
             qmask=None) -> Tuple[np.ndarray, np.ndarray]:
    """fp64 O [T,H,D] and LSE [H,T] (natural log; -inf on padding rows).

    Rows/heads outside ``qmask`` / ``heads`` are left as NaN."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, H, D = q.shape
    cu_, cup_ = _i32(cu), _i32(cup)
    sc = 1.0 / np.sqrt(D) if scale is None else float(scale)
    hs = _heads(H, heads)
    o = np.full((T, H, D), np.nan)
    lse = np.full((H, T), np.nan)
    qm = None if qmask is None else np.ascontiguousarray(np.asarray(qmask, dtype=np.uint8))
    lib = _load()
    lib.oracle_attn_fwd(T, H, D, len(cup_) - 1, cu_.ctypes.data, cup_.ctypes.data, int(pad), sc,
                        q.ctypes.data, k.ctypes.data, v.ctypes.data,
                        None if qm is None else qm.ctypes.data, hs.ctypes.data, len(hs),
                        o.ctypes.data, lse.ctypes.data)
    return o, lse


def attn_bwd(q, k, v, o, lse, dout, cu, cup, pad: int, scale: Optional[float] = None,
             heads=None, qmask=None) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """fp64 dQ, dK, dV [T,H,D].  With ``qmask`` only the masked-in queries
    contribute (one rank's partial dK/dV) and only their dQ rows are written."""
    q, k, v, o, dout = _f64(q), _f64(k), _f64(v), _f64(o), _f64(dout)
    lse = _f64(lse)
    T, H, D = q.shape
    cu_, cup_ = _i32(cu), _i32(cup)
    sc = 1.0 / np.sqrt(D) if scale is None else float(scale)
    hs = _heads(H, heads)
    dq = np.full((T, H, D), np.nan)
    dk = np.full((T, H, D), np.nan)
    dv = np.full((T, H, D), np.nan)
    qm = None if qmask is None else np.ascontiguousarray(np.asarray(qmask, dtype=np.uint8))
    lib = _load()
    lib.oracle_attn_bwd(T, H, D, len(cup_) - 1, cu_.ctypes.data, cup_.ctypes.data, int(pad), sc,
                        q.ctypes.data, k.ctypes.data, v.ctypes.data, o.ctypes.data,
                        lse.ctypes.data, dout.ctypes.data,
                        None if qm is None else qm.ctypes.data, hs.ctypes.data, len(hs),
                        dq.ctypes.data, dk.ctypes.data, dv.ctypes.data)
    return dq, dk, dv


def bf16_round(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 round-to-nearest-even, returned as the bf16 bit patterns
    (uint16).  Plain integer arithmetic on the fp32 bit pattern: add 0x7FFF
    plus the lowest kept bit, then drop the low 16 bits (NaN is not handled;
    the inputs here are finite)."""
    b = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    return ((b + 0x7FFF + lsb) >> 16).astype(np.uint16)
