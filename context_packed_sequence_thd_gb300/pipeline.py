"""Host orchestration of the emulated context-parallel attention step.

Every CP rank of one all-gather CP group runs on one GPU, one after another
on one stream.  The data movement the pages describe maps onto the library
as follows ("[PyTorch] Add no-load-balance THD all-gather CP", §Sequence
Diagram; "[PyTorch] Extend no-load-balance CP to the a2a comm type"):

  get_batch_on_this_cp_rank   cp_partition_index_all (every rank, one
                              launch) + cp_thd_gather_f16 (Q/K/V/dO of every
                              rank in one launch, converted to the fp16
                              tensor-core operands); with bf16 operands and
                              NO_LOAD_BALANCE a rank's shard is a contiguous
                              slice, so no copy is made at all
  all-gather K/V              the ranks' local shards live side by side in one
                              [cp*s_local, H, D] buffer, which *is* the
                              all-gathered, rank-concatenated tensor
  restore K/V order           cp_thd_gather with the restore index
                              (DUAL_CHUNK_SWAP); a no-op for NO_LOAD_BALANCE,
                              whose rank-concatenated order is the original
                              order (the reorder the a2a page removes)
  attention fwd / bwd         cp_attn_fwd per rank; the backward of every
                              rank in one call (cp_attn_bwd_grouped_rs)
  unrestore + reduce-scatter  by default inside that call: the dK/dV kernel
                              sums the ranks' partials per key block and
                              writes each rank's rows, in bf16, through the
                              restore index; otherwise fp32 sums in original
                              order (grouped, or rank by rank), then
                              cp_reduce_scatter_emul (gather by the rank's
                              index + bf16 cast)
  dQ/dK/dV tail-zeroing       cp_zero_tail, gated by the host-known valid end

Only argument marshalling and buffer management happen here; every step is
a kernel of libcpthd.
"""
from __future__ import annotations

import contextlib
import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from . import api

DCS = api.DUAL_CHUNK_SWAP
NLB = api.NO_LOAD_BALANCE
STRATEGY_NAMES = {DCS: "dual_chunk_swap", NLB: "no_load_balance"}


def rank_pairs(cu, cup, cp: int, rank: int, strategy: int, pad: int) -> int:
    """(query, key) pairs attended by rank `rank`'s real-token queries, summed
    per segment in closed form: a run of v real queries at global rows
    gs..gs+v-1 of a document starting at a attends
    v*(gs-a+1) + v*(v-1)/2 keys."""
    cu = np.asarray(cu, dtype=np.int64)
    cup = np.asarray(cup, dtype=np.int64)
    T = int(cup[-1])
    total = 0

    def run(gs, v, a):
        return v * (gs - a + 1) + v * (v - 1) // 2 if v > 0 else 0

    for i in range(len(cup) - 1):
        a, P = int(cup[i]), int(cup[i + 1] - cup[i])
        L = int(cu[i + 1] - cu[i]) if pad else P
        if strategy == DCS:
            c = P // (2 * cp)
            for ch in (rank, 2 * cp - 1 - rank):
                gs = a + ch * c
                v = min(max(L - ch * c, 0), c)
                total += run(gs, v, a)
        else:
            s_local = T // cp
            lo, hi = max(a, rank * s_local), min(a + P, (rank + 1) * s_local)
            if hi > lo:
                v = min(max(a + L - lo, 0), hi - lo)
                total += run(lo, v, a)
    return total


@dataclass
class RankMeta:
    idx: torch.Tensor          # int32 [s_local]
    meta: torch.Tensor         # uint8 [meta_bytes]
    valid_end: int             # host-known local valid end (gates the tail-zero)
    pairs: int


@dataclass
class CPPlan:
    """Partition metadata of all ranks for one (cu, cup, cp, strategy)."""
    cu: np.ndarray
    cup: np.ndarray
    cp: int
    strategy: int
    pad: int
    H: int
    D: int
    device: torch.device
    d_cu: torch.Tensor = field(init=False)
    d_cup: torch.Tensor = field(init=False)
    idx_all: torch.Tensor = field(init=False)
    restore: torch.Tensor = field(init=False)
    ranks: List[RankMeta] = field(init=False)

    def __post_init__(self):
        self.cu = np.asarray(self.cu, dtype=np.int32)
        self.cup = np.asarray(self.cup, dtype=np.int32)
        st = api.cp_validate_seqlens(self.cu, self.cup, self.T, self.cp, self.strategy, self.pad)
        if st != 0:
            raise api.CpError("cp_validate_seqlens", st)
        self.d_cu = torch.from_numpy(self.cu).to(self.device)
        self.d_cup = torch.from_numpy(self.cup).to(self.device)
        self.restore = torch.empty(self.T, dtype=torch.int32, device=self.device)
        # the ranks' partition indices side by side: rank r's is rows
        # [r*s_local, (r+1)*s_local), so idx_all indexes the rank-concatenated buffers
        self.idx_all = torch.empty(self.T, dtype=torch.int32, device=self.device)
        nbytes = api.cp_meta_bytes(self.n_docs, self.T, self.cp)
        # the ranks' metadata side by side, 16-byte aligned: built in one launch
        self.meta_stride = (nbytes + 15) // 16 * 16
        self.meta_all = torch.empty(self.cp * self.meta_stride, dtype=torch.uint8,
                                    device=self.device)
        self.ranks = []
        for r in range(self.cp):
            self.ranks.append(RankMeta(
                idx=self.local(self.idx_all, r),
                meta=self.meta_all[r * self.meta_stride:r * self.meta_stride + nbytes],
                valid_end=api.cp_valid_end(self.cu, self.cup, self.cp, r, self.strategy, self.pad),
                pairs=rank_pairs(self.cu, self.cup, self.cp, r, self.strategy, self.pad)))
        self.build_index()

    @property
    def T(self) -> int:
        return int(self.cup[-1])

    @property
    def n_docs(self) -> int:
        return len(self.cup) - 1

    @property
    def s_local(self) -> int:
        return self.T // self.cp

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def build_index(self, stream=None) -> int:
        """Every rank's partition index, metadata and restore entries in one
        launch (one CTA per rank)."""
        api.cp_partition_index_all(self.d_cu if self.pad else None, self.d_cup, self.T, self.cp,
                                   self.strategy, self.pad, self.idx_all, self.restore,
                                   self.meta_all, self.meta_stride, stream)
        return 1

    def local(self, buf: torch.Tensor, r: int) -> torch.Tensor:
        return buf[r * self.s_local:(r + 1) * self.s_local]


class CPAttention:
    """Buffers and the full emulated CP forward/backward for one plan."""

    def __init__(self, plan: CPPlan, fuse_q_gather: bool = False,
                 operand_dtype: Optional[torch.dtype] = None, grouped_bwd: bool = True,
                 fused_rs: bool = True):
        self.plan = plan
        p = plan
        # backward of all ranks in one call (cp_attn_bwd_grouped: dK/dV summed
        # over the ranks inside one dK/dV launch) or rank by rank (cp_attn_bwd)
        self.grouped_bwd = grouped_bwd
        # with the grouped backward, the reduce-scatter's scatter and bf16 cast
        # in the dK/dV kernel's epilogue (cp_attn_bwd_grouped_rs): no fp32 sums
        self.fused_rs = grouped_bwd and fused_rs
        # forward-only steps under DUAL_CHUNK_SWAP: the attention loads query
        # rows through the partition index (cp_attn_fwd_gather), no Q shard copy
        self.fuse_q_gather = fuse_q_gather
        self.q_src: Optional[torch.Tensor] = None
        # tensor-core operand type of Q/K/V/dO: fp16 (the shard gathers convert
        # the bf16 inputs; 11 significant bits, one product per term) unless
        # the queries are read straight from the bf16 batch (fused gather)
        if operand_dtype is None:
            operand_dtype = torch.bfloat16 if fuse_q_gather else torch.float16
        if operand_dtype not in (torch.bfloat16, torch.float16):
            raise ValueError("operand_dtype must be torch.bfloat16 or torch.float16")
        if fuse_q_gather and operand_dtype != torch.bfloat16:
            raise ValueError("the fused query gather reads the bf16 batch: bf16 operands")
        self.operand_dtype = operand_dtype
        self.f16 = operand_dtype == torch.float16
        dev, T, H, D = p.device, p.T, p.H, p.D
        bf = dict(dtype=torch.bfloat16, device=dev)
        op = dict(dtype=operand_dtype, device=dev)
        # rank-concatenated buffers: rank r's shard is rows [r*s_local, (r+1)*s_local);
        # bf16 NO_LOAD_BALANCE shards are views of the inputs, so nothing is
        # allocated; fp16 ones are converted copies
        own = p.strategy == DCS or self.f16
        self.qc = torch.empty(T, H, D, **op) if own else None
        self.kc = torch.empty(T, H, D, **op) if own else None
        self.vc = torch.empty(T, H, D, **op) if own else None
        self.doc = torch.empty(T, H, D, **op) if own else None
        self.oc = torch.empty(T, H, D, **bf)
        # O's bf16 rounding remainder: the backward's Delta = rowsum(dO * O) reads O + it
        self.oc_resid = torch.empty(T, H, D, **bf)
        self.lse = torch.empty(p.cp, H, p.s_local, dtype=torch.float32, device=dev)
        self.k_full = torch.empty(T, H, D, **op) if p.strategy == DCS else None
        self.v_full = torch.empty(T, H, D, **op) if p.strategy == DCS else None
        self.dqc = torch.empty(T, H, D, **bf)
        self.dkc = torch.empty(T, H, D, **bf)
        self.dvc = torch.empty(T, H, D, **bf)
        acc = None if self.fused_rs else dict(dtype=torch.float32, device=dev)
        self.dk_acc = torch.empty(T, H, D, **acc) if acc else None
        self.dv_acc = torch.empty(T, H, D, **acc) if acc else None
        ws = api.cp_attn_bwd_workspace_bytes(p.s_local, H)
        self.ws = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        wsg = api.cp_attn_bwd_grouped_workspace_bytes(p.s_local, H, p.cp, T) if grouped_bwd else 0
        self.ws_grouped = torch.empty(max(wsg, 16), dtype=torch.uint8, device=dev)
        self.launches = 0
        # optional per-call CUDA-event timing: category -> [(start, end), ...]
        self.events: Optional[Dict[str, list]] = None

    @contextlib.contextmanager
    def _timed(self, category: str, stream=None):
        if self.events is None:
            yield
            return
        s = torch.cuda.current_stream() if stream is None else stream
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s)
        yield
        e1.record(s)
        self.events.setdefault(category, []).append((e0, e1))

    def event_ms(self) -> Dict[str, List[float]]:
        """Per-call durations (ms) recorded since events were enabled."""
        return {k: [a.elapsed_time(b) for a, b in v] for k, v in (self.events or {}).items()}

    # -- data movement ------------------------------------------------------
    def shard_inputs(self, q, k, v, do=None, stream=None):
        """get_batch_on_this_cp_rank for every rank (plus dO for the backward)."""
        p = self.plan
        if p.strategy == NLB and not self.f16:
            # contiguous shards: the rank-concatenated buffer is the input itself
            self.qc, self.kc, self.vc = q, k, v
            if do is not None:
                self.doc = do
            return
        # every rank's shard in one gather: the rank-concatenated buffer is the
        # input gathered by the ranks' indices side by side (NO_LOAD_BALANCE:
        # the identity), converted to fp16 operands on the way.  A forward-only
        # step with the fused gather leaves Q where it is.
        self.q_src = q if (self.fuse_q_gather and do is None) else None
        srcs = ([q] if self.q_src is None else []) + [k, v] + ([do] if do is not None else [])
        dsts = ([self.qc] if self.q_src is None else []) + [self.kc, self.vc] + \
            ([self.doc] if do is not None else [])
        idx = p.idx_all if p.strategy == DCS else None
        with self._timed("partition_gather", stream):
            if self.f16:
                api.cp_thd_gather_f16(srcs, dsts, idx, stream)
            else:
                api.cp_thd_gather(srcs, dsts, idx, stream)
        self.launches += 1

    def restore_kv(self, stream=None):
        """All-gather (free: shards are side by side) + restore to original order."""
        p = self.plan
        if p.strategy == NLB:
            return self.kc, self.vc
        with self._timed("restore_gather", stream):
            api.cp_thd_gather([self.kc, self.vc], [self.k_full, self.v_full], p.restore, stream)
        self.launches += 1
        return self.k_full, self.v_full

    # -- attention ------------------------------------------------------------
    def forward(self, stream=None):
        p = self.plan
        k_full, v_full = self.restore_kv(stream)
        fused = self.q_src is not None and p.strategy == DCS
        for r in range(p.cp):
            with self._timed("attn_fwd", stream):
                if fused:
                    api.cp_attn_fwd_gather(self.q_src, p.ranks[r].idx, k_full, v_full,
                                           p.local(self.oc, r), self.lse[r], p.ranks[r].meta, p.T,
                                           p.cp, r, p.strategy, p.scale, stream,
                                           o_resid=p.local(self.oc_resid, r))
                else:
                    api.cp_attn_fwd(p.local(self.qc, r), k_full, v_full, p.local(self.oc, r),
                                    self.lse[r], p.ranks[r].meta, p.T, p.cp, r, p.strategy,
                                    p.scale, stream, o_resid=p.local(self.oc_resid, r))
            self.launches += 1
        return k_full, v_full

    def backward(self, k_full, v_full, stream=None):
        """Every rank's backward and the emulated reduce-scatter's sum of the
        partial dK/dV: by default one grouped call whose dK/dV kernel sums the
        ranks' terms per key block and stores them; rank by rank otherwise
        (rank 0 stores its partial into the fp32 accumulators, the others add
        theirs in rank order)."""
        p = self.plan
        if self.fused_rs:
            # the whole reduce-scatter inside the dK/dV kernel: each rank's
            # rows of dK/dV (its partition order) written once, in bf16
            with self._timed("attn_bwd", stream):
                api.cp_attn_bwd_grouped_rs(self.qc, k_full, v_full, self.oc, self.lse, self.doc,
                                           self.dqc, self.dkc, self.dvc,
                                           p.restore if p.strategy == DCS else None, p.meta_all,
                                           p.meta_stride, p.T, p.cp, p.strategy, p.scale,
                                           self.ws_grouped, stream, o_resid_all=self.oc_resid)
            self.launches += 2 * p.cp + 2
        elif self.grouped_bwd:
            with self._timed("attn_bwd", stream):
                api.cp_attn_bwd_grouped(self.qc, k_full, v_full, self.oc, self.lse, self.doc,
                                        self.dqc, self.dk_acc, self.dv_acc, p.meta_all,
                                        p.meta_stride, p.T, p.cp, p.strategy, p.scale,
                                        self.ws_grouped, stream, o_resid_all=self.oc_resid)
            self.launches += 2 * p.cp + 2
        else:
            for r in range(p.cp):
                with self._timed("attn_bwd", stream):
                    api.cp_attn_bwd(p.local(self.qc, r), k_full, v_full, p.local(self.oc, r),
                                    self.lse[r], p.local(self.doc, r), p.local(self.dqc, r),
                                    self.dk_acc, self.dv_acc, p.ranks[r].meta, p.T, p.cp, r,
                                    p.strategy, p.scale, self.ws, stream,
                                    mode=api.BWD_STORE if r == 0 else api.BWD_ACCUMULATE,
                                    o_resid=p.local(self.oc_resid, r))
                self.launches += 3
        if not self.fused_rs:
            # the scatter half of the reduce-scatter for every rank in one launch:
            # rank r's rows of the rank-concatenated dK/dV are the summed
            # accumulators at its partition index (NO_LOAD_BALANCE: contiguous)
            with self._timed("reduce_scatter_emul", stream):
                api.cp_reduce_scatter_emul([self.dk_acc, self.dv_acc], [self.dkc, self.dvc],
                                           p.idx_all if p.strategy == DCS else None, 0, p.T,
                                           stream)
            self.launches += 1
        for r, rm in enumerate(p.ranks):
            if api.cp_zero_tail([p.local(self.dqc, r), p.local(self.dkc, r), p.local(self.dvc, r)],
                                rm.valid_end, stream=stream):
                self.launches += 1

    def step(self, q, k, v, do=None, stream=None, rebuild_index: bool = True):
        """One pass of the whole hot path: partition, shard, restore, fwd (+bwd)."""
        if rebuild_index:
            self.launches += self.plan.build_index(stream)
        self.shard_inputs(q, k, v, do, stream)
        k_full, v_full = self.forward(stream)
        if do is not None:
            self.backward(k_full, v_full, stream)

    # -- results in original order (for checks) ------------------------------
    def rank_rows(self, r: int) -> torch.Tensor:
        return self.plan.ranks[r].idx.long()

    def flops(self, bwd: bool) -> Dict[str, float]:
        p = self.plan
        pairs = sum(rm.pairs for rm in p.ranks)
        f = {"fwd": 4.0 * p.D * p.H * pairs}
        if bwd:
            f["bwd"] = 10.0 * p.D * p.H * pairs
        return f


class CPA2AAttention(CPAttention):
    """The a2a comm type with every rank on one GPU ("[PyTorch] Extend
    no-load-balance CP to the a2a comm type", ¶1-2, §Diagram).

    Token shards come from the plan's partition (gathered under
    DUAL_CHUNK_SWAP, views under NO_LOAD_BALANCE).  The seq->head exchange gives
    rank r the whole sequence with heads [r*H/cp, (r+1)*H/cp) -- under
    DUAL_CHUNK_SWAP the restore reorder is folded into that pass, under flat
    sharding there is none -- so every rank's attention uses cp_size = 1
    metadata for the whole packed sequence, and owns the full dQ/dK/dV of its
    heads (no reduction).  The head->seq exchange brings outputs and gradients
    back to token shards.
    """

    def __init__(self, plan: CPPlan, operand_dtype: Optional[torch.dtype] = None):
        super().__init__(plan, operand_dtype=operand_dtype, fused_rs=False)
        p = plan
        if p.H % p.cp:
            raise ValueError("the a2a comm type needs H divisible by cp_size")
        dev, T, D = p.device, p.T, p.D
        self.Hc = p.H // p.cp
        # cp = 1 metadata of the whole packed sequence, for every rank's head slice
        self.full = CPPlan(p.cu, p.cup, 1, NLB, p.pad, self.Hc, D, dev)
        bf = dict(dtype=torch.bfloat16, device=dev)
        op = dict(dtype=self.operand_dtype, device=dev)
        shape = (p.cp, T, self.Hc, D)
        self.qh, self.kh, self.vh, self.doh = (torch.empty(shape, **op) for _ in range(4))
        self.oh, self.dqh, self.dkh, self.dvh = (torch.empty(shape, **bf) for _ in range(4))
        self.oh_resid = torch.empty(shape, **bf)
        self.lse_h = torch.empty(p.cp, self.Hc, T, dtype=torch.float32, device=dev)
        self.acc_k = torch.empty(T, self.Hc, D, dtype=torch.float32, device=dev)
        self.acc_v = torch.empty(T, self.Hc, D, dtype=torch.float32, device=dev)
        ws = api.cp_attn_bwd_workspace_bytes(T, self.Hc)
        self.ws_h = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)

    def _perm(self):
        return self.plan.restore if self.plan.strategy == DCS else None

    def forward(self, stream=None):
        p = self.plan
        with self._timed("a2a_exchange", stream):
            api.cp_a2a_exchange([self.qc, self.kc, self.vc], [self.qh, self.kh, self.vh],
                                self._perm(), p.cp, api.A2A_SEQ_TO_HEAD, stream)
        self.launches += 1
        for r in range(p.cp):
            with self._timed("attn_fwd", stream):
                api.cp_attn_fwd(self.qh[r], self.kh[r], self.vh[r], self.oh[r], self.lse_h[r],
                                self.full.ranks[0].meta, p.T, 1, 0, NLB, p.scale, stream,
                                o_resid=self.oh_resid[r])
            self.launches += 1
        with self._timed("a2a_exchange", stream):
            api.cp_a2a_exchange([self.oh], [self.oc], self._perm(), p.cp, api.A2A_HEAD_TO_SEQ,
                                stream)
        self.launches += 1
        return None, None

    def backward(self, k_full=None, v_full=None, stream=None):
        p = self.plan
        with self._timed("a2a_exchange", stream):
            api.cp_a2a_exchange([self.doc], [self.doh], self._perm(), p.cp, api.A2A_SEQ_TO_HEAD,
                                stream)
        self.launches += 1
        for r in range(p.cp):
            with self._timed("attn_bwd", stream):
                api.cp_attn_bwd(self.qh[r], self.kh[r], self.vh[r], self.oh[r], self.lse_h[r],
                                self.doh[r], self.dqh[r], self.acc_k, self.acc_v,
                                self.full.ranks[0].meta, p.T, 1, 0, NLB, p.scale, self.ws_h,
                                stream, mode=api.BWD_STORE, o_resid=self.oh_resid[r])
            self.launches += 3
            with self._timed("grad_cast", stream):
                api.cp_reduce_scatter_emul([self.acc_k, self.acc_v], [self.dkh[r], self.dvh[r]],
                                           None, 0, p.T, stream)
            self.launches += 1
        with self._timed("a2a_exchange", stream):
            api.cp_a2a_exchange([self.dqh, self.dkh, self.dvh], [self.dqc, self.dkc, self.dvc],
                                self._perm(), p.cp, api.A2A_HEAD_TO_SEQ, stream)
        self.launches += 1
        for r, rm in enumerate(p.ranks):
            if api.cp_zero_tail([p.local(self.dqc, r), p.local(self.dkc, r), p.local(self.dvc, r)],
                                rm.valid_end, stream=stream):
                self.launches += 1

    def step(self, q, k, v, do=None, stream=None, rebuild_index: bool = True):
        if rebuild_index:
            self.launches += self.plan.build_index(stream) + self.full.build_index(stream)
        self.shard_inputs(q, k, v, do, stream)
        self.forward(stream)
        if do is not None:
            self.backward(stream=stream)


def ring_steps(cp: int, strategy: int) -> List[tuple]:
    """The emulated ring's backward calls in execution order: (rank r, step i,
    K/V owner j = (r - i) mod cp, cp_bwd_mode bits).  Under NO_LOAD_BALANCE
    rank r runs steps 0..r only (the shards of later ranks hold later tokens).
    The first call that touches shard j stores its dK/dV partial, later ones
    add; a rank's first step stores its fp32 dQ, later steps add."""
    out, written = [], set()
    for r in range(cp):
        for i in range(cp if strategy == DCS else r + 1):
            j = (r - i) % cp
            mode = api.BWD_ACCUMULATE if j in written else api.BWD_STORE
            mode |= api.BWD_DQ_F32_STORE if i == 0 else api.BWD_DQ_F32_ACCUMULATE
            written.add(j)
            out.append((r, i, j, mode))
    return out


class CPP2PAttention(CPAttention):
    """The P2P (ring) comm type with every rank on one GPU ("THD P2P
    context-parallel regression when padded cu_seqlens are value-equal but not
    object-identical", §Describe the bug: the P2P context-parallel path).

    Rank r keeps its token shard (partition of the plan's strategy) and at
    ring step i attends it to the K/V shard of rank j = (r - i) mod cp.  The
    ranks' shards lie side by side in the rank-concatenated buffers, so the
    ring's send/receive of K/V is a pointer offset here.  Every step is a
    cp_size = 1 attention call with per-step metadata; all steps of a rank get
    their metadata from one cp_p2p_index launch (instead of the per-step
    get_cu_seqlens_on_cp_rank helper calls).  Under NO_LOAD_BALANCE the shards
    of later ranks hold only later tokens, so rank r runs steps 0..r only.

    Forward: by default one cp_attn_fwd_ring pass per rank, which walks the
    held shards in ring order within one online softmax (the merge is its
    rescaling, so no partial outputs are written); fused_ring=False runs the
    per-step partials (O_i, LSE_i) and combines them with cp_p2p_merge.
    Backward: by default one cp_attn_bwd_ring call (s_local a multiple of 32):
    per rank one dQ pass over its ring steps, one dK/dV pass over every
    shard's key blocks walking the ranks that hold the shard, every sum formed
    inside the kernels.  Otherwise per step with the merged O / LSE; dQ is
    summed over the rank's steps in an fp32 buffer (first step stores, later
    steps add), dK/dV of shard j are summed in fp32 over the ranks that
    attended it (the partial dK/dV that travel back along the ring to their
    owner), the first contribution to each shard stored; one launch casts all
    three to bf16.
    """

    def __init__(self, plan: CPPlan, operand_dtype: Optional[torch.dtype] = None,
                 fused_ring: bool = True):
        super().__init__(plan, operand_dtype=operand_dtype, fused_rs=False)
        p = plan
        dev, T, H, D, S = p.device, p.T, p.H, p.D, p.s_local
        self.k_full = self.v_full = None   # no restore: attention reads the shards
        self.fused_ring = fused_ring
        self.ws_ring = torch.empty(max(api.cp_attn_fwd_ring_workspace_bytes(S), 16),
                                   dtype=torch.uint8, device=dev)
        self.step_bytes = api.cp_p2p_meta_bytes(p.n_docs, T, p.cp)
        # every rank's step metadata in one buffer, rank r at r * rank_stride
        # (the one-pass ring backward reads all of them in one launch)
        self.rank_stride = p.cp * self.step_bytes
        self.p2p_meta_all = torch.empty(p.cp * self.rank_stride, dtype=torch.uint8, device=dev)
        self.p2p_meta = [self.p2p_meta_all[r * self.rank_stride:(r + 1) * self.rank_stride]
                         for r in range(p.cp)]
        wsb = api.cp_attn_bwd_ring_workspace_bytes(S, H, p.cp) if S % 32 == 0 else 0
        self.ws_ring_bwd = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
        self.o_steps = torch.empty(p.cp, S, H, D, dtype=torch.bfloat16, device=dev)
        self.o_steps_resid = torch.empty(p.cp, S, H, D, dtype=torch.bfloat16, device=dev)
        self.lse_steps = torch.empty(p.cp, H, S, dtype=torch.float32, device=dev)
        self.dq_acc = torch.empty(T, H, D, dtype=torch.float32, device=dev)
        self.build_p2p_index()

    def n_steps(self, r: int) -> int:
        return sum(1 for rr, _, _, _ in ring_steps(self.plan.cp, self.plan.strategy) if rr == r)

    def step_meta(self, r: int, i: int) -> torch.Tensor:
        return self.p2p_meta[r][i * self.step_bytes:(i + 1) * self.step_bytes]

    def build_p2p_index(self, stream=None) -> int:
        """One cp_p2p_index launch per rank (every ring step's metadata)."""
        p = self.plan
        for r in range(p.cp):
            api.cp_p2p_index(p.d_cu if p.pad else None, p.d_cup, p.T, p.cp, r, p.strategy,
                             p.pad, self.p2p_meta[r], stream)
        return p.cp

    def forward(self, stream=None):
        p = self.plan
        S = p.s_local
        for r in range(p.cp):
            n = self.n_steps(r)
            if self.fused_ring:
                with self._timed("attn_fwd", stream):
                    api.cp_attn_fwd_ring(p.local(self.qc, r), self.kc, self.vc, p.local(self.oc, r),
                                         self.lse[r], self.p2p_meta[r], self.step_bytes, n, p.cp, r,
                                         p.strategy, p.scale, self.ws_ring, stream,
                                         o_resid=p.local(self.oc_resid, r))
                self.launches += 2
                continue
            for i in range(n):
                j = (r - i) % p.cp
                with self._timed("attn_fwd", stream):
                    api.cp_attn_fwd(p.local(self.qc, r), p.local(self.kc, j), p.local(self.vc, j),
                                    self.o_steps[i], self.lse_steps[i], self.step_meta(r, i), S,
                                    1, 0, p.strategy, p.scale, stream,
                                    o_resid=self.o_steps_resid[i])
                self.launches += 1
            with self._timed("p2p_merge", stream):
                api.cp_p2p_merge(self.o_steps[:n], self.lse_steps[:n], p.local(self.oc, r),
                                 self.lse[r], stream, o_steps_resid=self.o_steps_resid[:n],
                                 out_resid=p.local(self.oc_resid, r))
            self.launches += 1
        return None, None

    def backward(self, k_full=None, v_full=None, stream=None):
        p = self.plan
        S = p.s_local
        if self.fused_ring and S % 32 == 0:
            # every rank's ring steps in one pass per gradient: dQ stored as bf16,
            # dK/dV of every shard summed over the ranks inside the kernel and
            # written as bf16 by its epilogue (the reduce-scatter's cast fused)
            with self._timed("attn_bwd", stream):
                api.cp_attn_bwd_ring_rs(self.qc, self.kc, self.vc, self.oc, self.lse, self.doc,
                                        self.dqc, self.dkc, self.dvc, self.p2p_meta_all,
                                        self.step_bytes, self.rank_stride, p.cp, p.strategy,
                                        p.scale, self.ws_ring_bwd, stream,
                                        o_resid_all=self.oc_resid)
            self.launches += 3 * p.cp + 2
            for r, rm in enumerate(p.ranks):
                if api.cp_zero_tail([p.local(self.dqc, r), p.local(self.dkc, r),
                                     p.local(self.dvc, r)], rm.valid_end, stream=stream):
                    self.launches += 1
            return
        for r, i, j, mode in ring_steps(p.cp, p.strategy):
            with self._timed("attn_bwd", stream):
                api.cp_attn_bwd(p.local(self.qc, r), p.local(self.kc, j), p.local(self.vc, j),
                                p.local(self.oc, r), self.lse[r], p.local(self.doc, r),
                                p.local(self.dq_acc, r), p.local(self.dk_acc, j),
                                p.local(self.dv_acc, j), self.step_meta(r, i), S, 1, 0,
                                p.strategy, p.scale, self.ws, stream, mode=mode,
                                o_resid=p.local(self.oc_resid, r))
            self.launches += 3
        with self._timed("grad_cast", stream):
            api.cp_reduce_scatter_emul([self.dq_acc, self.dk_acc, self.dv_acc],
                                       [self.dqc, self.dkc, self.dvc], None, 0, p.T, stream)
        self.launches += 1
        for r, rm in enumerate(p.ranks):
            if api.cp_zero_tail([p.local(self.dqc, r), p.local(self.dkc, r), p.local(self.dvc, r)],
                                rm.valid_end, stream=stream):
                self.launches += 1

    def step(self, q, k, v, do=None, stream=None, rebuild_index: bool = True):
        if rebuild_index:
            self.launches += self.plan.build_index(stream) + self.build_p2p_index(stream)
        self.shard_inputs(q, k, v, do, stream)
        self.forward(stream)
        if do is not None:
            self.backward(stream=stream)


# ---------------------------------------------------------------------------
# bshd / sbhd batches ("[PyTorch] Extend no-load-balance CP to the a2a comm
# type", §Tests: flat a2a over bshd, sbhd and THD)
# ---------------------------------------------------------------------------

def bshd_seqlens(B: int, S: int) -> np.ndarray:
    """cu_seqlens of a bshd batch [B, S, H, D] seen as THD: B documents of S
    tokens, token (b, s) at row b*S + s -- the same memory, no copy."""
    return (np.arange(B + 1, dtype=np.int64) * S).astype(np.int32)


def sbhd_rows(B: int, S: int, device) -> Dict[str, torch.Tensor]:
    """Row maps between an sbhd batch [S, B, H, D] (token (s, b) at row s*B + b)
    and its THD form (row b*S + s): ``to_thd`` gathers sbhd -> THD,
    ``to_sbhd`` gathers THD -> sbhd."""
    b = np.arange(B)[:, None]
    s = np.arange(S)[None, :]
    to_thd = (s * B + b).reshape(-1)                 # THD row b*S+s reads sbhd row s*B+b
    to_sbhd = np.empty_like(to_thd)
    to_sbhd[to_thd] = np.arange(B * S)
    return {k: torch.from_numpy(v.astype(np.int32)).to(device)
            for k, v in (("to_thd", to_thd), ("to_sbhd", to_sbhd))}


def sbhd_to_thd(xs: Sequence[torch.Tensor], rows: Dict[str, torch.Tensor], stream=None):
    """[S, B, H, D] tensors -> THD [B*S, H, D] copies (one gather launch)."""
    S, B = xs[0].shape[:2]
    flat = [x.view(S * B, *x.shape[2:]) for x in xs]
    out = [torch.empty_like(f) for f in flat]
    api.cp_thd_gather(flat, out, rows["to_thd"], stream)
    return out


def thd_to_sbhd(xs: Sequence[torch.Tensor], rows: Dict[str, torch.Tensor], S: int, B: int,
                stream=None):
    """THD [B*S, H, D] tensors -> sbhd [S, B, H, D] copies (one gather launch)."""
    out = [torch.empty_like(x) for x in xs]
    api.cp_thd_gather(list(xs), out, rows["to_sbhd"], stream)
    return [o.view(S, B, *o.shape[1:]) for o in out]
