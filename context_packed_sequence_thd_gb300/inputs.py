"""Seeded synthetic inputs for the five THD workloads.

This module only *draws* inputs: document lengths, the cumulative offsets
built from them, and bf16 ~N(0,1) Q/K/V/dO tensors.  It holds none of the
method's arithmetic (no partitioning, no attention) so that the CUDA path
and the CPU oracle can both be fed from it without sharing any code.

Workloads (the sizes follow the shapes the TransformerEngine pages use:
the tiny CP2 THD check of "[PyTorch] Add no-load-balance THD all-gather CP"
§Validation, and the cp=8, h=40, d=128, s in {8192, 32768, 75600} exchange
of "[PyTorch] Extend no-load-balance CP to the a2a comm type"):

  tiny  3 docs {40,24,64}, cp=2, H=2, D=64, cu_seqlens_padded a value-equal clone
  cfg2  32768 packed tokens, 16 docs with lengths multiple of 16 in [256,4096],
        cp=4, H=16, D=128
  cfg3  one sequence of 32768 tokens, cp=8, H=40, D=128 (plus 8192 / 75600
        for the gather sweep)
  cfg4  75600 packed tokens, lognormal lengths (median 2048, sigma 1) none
        divisible by 2*cp=16, cp=8, H=40, D=128, no-load-balance only
  cfg5  65536 padded tokens, 24 lognormal docs (median 1656, sigma 1) each padded
        up to a multiple of 2*cp=8, cp=4, H=32, D=128; the last document keeps a
        3-row tail unless ``tail=False``

Seeds: workload k uses seed 1000+k for both the numpy length draws and the
torch tensor draws (drawn in the order Q, K, V, dO).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np
import torch

DCS = 0  # dual-chunk-swap strategy code (matches the C enum)
NLB = 1  # no-load-balance strategy code


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    cu: np.ndarray          # int32 [n+1], actual document offsets
    cup: np.ndarray         # int32 [n+1], padded (physical) offsets; a separate array
    cp: int
    H: int
    D: int
    strategies: tuple
    pad_between_seqs: int   # the flag the workload is run with
    bwd: bool

    @property
    def total_tokens(self) -> int:
        return int(self.cup[-1])

    @property
    def n_docs(self) -> int:
        return len(self.cup) - 1

    @property
    def s_local(self) -> int:
        return self.total_tokens // self.cp

    def tensors(self, with_grad: bool = True, device: str = "cpu") -> Dict[str, torch.Tensor]:
        return draw_qkv(self.total_tokens, self.H, self.D, self.seed, with_grad, device)


def draw_qkv(T: int, H: int, D: int, seed: int, with_grad: bool = True,
             device: str = "cpu") -> Dict[str, torch.Tensor]:
    """bf16 ~N(0,1) tensors [T, H, D], drawn on the CPU in the order q, k, v, do."""
    g = torch.Generator().manual_seed(seed)
    names = ["q", "k", "v"] + (["do"] if with_grad else [])
    out = {}
    for n in names:
        t = torch.randn(T, H, D, generator=g, dtype=torch.float32).to(torch.bfloat16)
        out[n] = t.to(device) if device != "cpu" else t
    return out


def _offsets(lengths: List[int]) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(lengths, dtype=np.int64))]).astype(np.int32)


def tiny() -> Workload:
    cu = _offsets([40, 24, 64])
    return Workload("tiny", 1001, cu, cu.copy(), cp=2, H=2, D=64,
                    strategies=(DCS, NLB), pad_between_seqs=0, bwd=False)


def cfg2_lengths(seed: int = 1002) -> List[int]:
    rng = np.random.default_rng(seed)
    choices = np.arange(256, 4096 + 1, 16)
    while True:
        first = [int(x) for x in rng.choice(choices, size=15)]
        last = 32768 - sum(first)
        if 256 <= last <= 4096:
            return first + [last]


def cfg2() -> Workload:
    cu = _offsets(cfg2_lengths())
    return Workload("cfg2", 1002, cu, cu.copy(), cp=4, H=16, D=128,
                    strategies=(DCS, NLB), pad_between_seqs=0, bwd=True)


def cfg3(s: int = 32768) -> Workload:
    cu = _offsets([s])
    return Workload(f"cfg3_s{s}", 1003, cu, cu.copy(), cp=8, H=40, D=128,
                    strategies=(DCS, NLB), pad_between_seqs=0, bwd=False)


def cfg4_lengths(seed: int = 1004, total: int = 75600, div: int = 16) -> List[int]:
    rng = np.random.default_rng(seed)
    lengths: List[int] = []
    while sum(lengths) < total:
        L = int(round(math.exp(math.log(2048.0) + 1.0 * rng.standard_normal())))
        L = min(max(L, 17), 32768)
        if L % div == 0:
            L += 1
        lengths.append(L)
    lengths[-1] = total - sum(lengths[:-1])
    if lengths[-1] < 17 or lengths[-1] % div == 0:
        rem = lengths.pop()
        lengths[-1] += rem
    # keep every length off a multiple of `div`, moving single tokens backwards
    i = len(lengths) - 1
    while i > 0 and lengths[i] % div == 0:
        lengths[i] -= 1
        lengths[i - 1] += 1
        i -= 1
    assert sum(lengths) == total
    return lengths


def cfg4() -> Workload:
    cu = _offsets(cfg4_lengths())
    return Workload("cfg4", 1004, cu, cu.copy(), cp=8, H=40, D=128,
                    strategies=(NLB,), pad_between_seqs=0, bwd=True)


def cfg5_lengths(seed: int = 1005, total: int = 65536, n: int = 24, mult: int = 8,
                 tail: bool = True):
    """Actual lengths L and padded lengths P (P_i = L_i rounded up to `mult`)."""
    rng = np.random.default_rng(seed)
    raw = np.exp(math.log(1656.0) + 1.0 * rng.standard_normal(n))
    f = (total - n * mult) / raw.sum()
    while True:
        L = [max(1, int(round(x * f))) for x in raw[:-1]]
        P = [((x + mult - 1) // mult) * mult for x in L]
        p_last = total - sum(P)
        if p_last >= 2 * mult:
            break
        f *= 0.99
    P.append(p_last)
    L.append(p_last - 3 if tail else p_last)
    return L, P


def cfg5(tail: bool = True, value_equal: bool = False) -> Workload:
    """Padded workload.  value_equal=True gives arm B: cu_seqlens := a clone of
    cu_seqlens_padded (the pad tokens become real tokens at each doc's end)."""
    L, P = cfg5_lengths(tail=tail)
    cup = _offsets(P)
    cu = cup.copy() if value_equal else _offsets(L)
    return Workload("cfg5" + ("" if tail else "_notail") + ("_eq" if value_equal else ""),
                    1005, cu, cup, cp=4, H=32, D=128, strategies=(DCS, NLB),
                    pad_between_seqs=0 if value_equal else 1, bwd=True)


def custom(lengths: List[int], padded: Optional[List[int]] = None, cp: int = 2, H: int = 2,
           D: int = 64, seed: int = 7, pad_between_seqs: Optional[int] = None) -> Workload:
    cu = _offsets(lengths)
    cup = _offsets(padded) if padded is not None else cu.copy()
    pad = int(padded is not None) if pad_between_seqs is None else pad_between_seqs
    return Workload("custom", seed, cu, cup, cp=cp, H=H, D=D, strategies=(DCS, NLB),
                    pad_between_seqs=pad, bwd=True)


ALL = {"tiny": tiny, "cfg2": cfg2, "cfg3": cfg3, "cfg4": cfg4, "cfg5": cfg5}
