"""Thin ctypes binding of libcpthd.so (declared in include/cpthd.h).

Argument marshalling only: every function here validates Python-side types,
turns torch tensors into raw pointers and the current CUDA stream into a
cudaStream_t, calls the C entry point of the same name and raises CpError on
a non-zero status.  All computation runs in the library's CUDA kernels; there
is no fallback -- importing this module on a machine without the built
library raises immediately when a function is first called.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

DUAL_CHUNK_SWAP = 0
NO_LOAD_BALANCE = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcpthd.so")
_lib = None

_c_i32p = ctypes.POINTER(ctypes.c_int32)
_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t

_SIGNATURES = {
    "cp_status_string": ([_I], ctypes.c_char_p),
    "cp_version": ([], _I),
    "cp_detect_pad_between_seqs": ([_P, _P, _I, ctypes.POINTER(_I)], _I),
    "cp_validate_seqlens": ([_P, _P, _I, _I64, _I, _I, _I], _I),
    "cp_valid_end": ([_P, _P, _I, _I, _I, _I, _I, ctypes.POINTER(_I64)], _I),
    "cp_meta_bytes": ([_I, _I64, _I], _SZ),
    "cp_partition_index": ([_P, _P, _I, _I64, _I, _I, _I, _I, _P, _P, _P, _SZ, _P], _I),
    "cp_partition_index_all": ([_P, _P, _I, _I64, _I, _I, _I, _P, _P, _P, _SZ, _P], _I),
    "cp_thd_gather": ([_P, _P, _I, _P, _I64, _I64, _I64, _P], _I),
    "cp_thd_scatter": ([_P, _P, _I, _P, _I64, _I64, _I64, _P], _I),
    "cp_thd_gather_f16": ([_P, _P, _I, _P, _I64, _I64, _I64, _P], _I),
    "cp_reduce_scatter_emul": ([_P, _P, _I, _P, _I64, _I64, _I64, _I, _I, _P], _I),
    "cp_a2a_exchange": ([_P, _P, _I, _P, _I64, _I, _I, _I, _I, _P], _I),
    "cp_zero_tail": ([_P, _I, _I64, _I64, _I64, _P, _P, ctypes.POINTER(_I)], _I),
    "cp_attn_fwd": ([_P, _P, _P, _P, _P, _P, _P, _SZ, _I64, _I, _I, _I, _I, _I, ctypes.c_float,
                     _I, _P], _I),
    "cp_attn_fwd_gather": ([_P, _I64, _P, _P, _P, _P, _P, _P, _P, _SZ, _I64, _I, _I, _I, _I, _I,
                           ctypes.c_float, _I, _P], _I),
    "cp_attn_bwd_workspace_bytes": ([_I64, _I], _SZ),
    "cp_attn_bwd": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I64, _I, _I, _I, _I, _I,
                     ctypes.c_float, _I, _P, _SZ, _P], _I),
    "cp_attn_bwd_ex": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I64, _I, _I, _I, _I,
                        _I, ctypes.c_float, _I, _I, _P, _SZ, _P], _I),
    "cp_attn_bwd_noalloc": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I64, _I, _I, _I,
                             _I, _I, ctypes.c_float, _I, _P], _I),
    "cp_attn_bwd_grouped_workspace_bytes": ([_I64, _I, _I, _I64], _SZ),
    "cp_attn_bwd_grouped": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I64, _I, _I, _I,
                             _I, ctypes.c_float, _I, _P, _SZ, _P], _I),
    "cp_attn_bwd_grouped_rs": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I64, _I,
                                _I, _I, _I, ctypes.c_float, _I, _P, _SZ, _P], _I),
    "cp_p2p_meta_bytes": ([_I, _I64, _I], _SZ),
    "cp_p2p_index": ([_P, _P, _I, _I64, _I, _I, _I, _I, _P, _SZ, _P], _I),
    "cp_p2p_merge": ([_P, _P, _P, _I, _I64, _I, _I, _P, _P, _P, _P], _I),
    "cp_device_status": ([ctypes.POINTER(_I), _I], _I),
    "cp_attn_fwd_ring_workspace_bytes": ([_I64], _SZ),
    "cp_attn_bwd_ring_workspace_bytes": ([_I64, _I, _I], _SZ),
    "cp_attn_bwd_ring": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _SZ, _I64, _I, _I, _I,
                          _I, ctypes.c_float, _I, _P, _SZ, _P], _I),
    "cp_attn_bwd_ring_rs": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _SZ, _I64, _I, _I,
                             _I, _I, ctypes.c_float, _I, _P, _SZ, _P], _I),
    "cp_attn_fwd_ring": ([_P, _P, _P, _P, _P, _P, _P, _SZ, _I, _I64, _I, _I, _I, _I, _I,
                          ctypes.c_float, _I, _P, _SZ, _P], _I),
}

EXPORTED = tuple(_SIGNATURES)


class CpError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")
        self.status = status


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libcpthd.so is not built ({LIB_PATH}); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().cp_status_string(int(status)).decode()


def _check(fn: str, st: int):
    if st != 0:
        raise CpError(fn, st)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _dev(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return _ptr(t)


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _host_i32(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr_array(ts: Sequence[torch.Tensor], name: str):
    arr = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = _dev(t, name).value
    return arr


# ---------------------------------------------------------------------------
# host metadata helpers
# ---------------------------------------------------------------------------

def cp_detect_pad_between_seqs(cu, cup) -> int:
    a = _host_i32(cu)
    b = None if cup is None else _host_i32(cup)
    out = _I(0)
    st = lib().cp_detect_pad_between_seqs(a.ctypes.data, None if b is None else b.ctypes.data,
                                          len(a) - 1, ctypes.byref(out))
    _check("cp_detect_pad_between_seqs", st)
    return int(out.value)


def cp_validate_seqlens(cu, cup, total_tokens: int, cp_size: int, strategy: int,
                        pad_between_seqs: int) -> int:
    """Returns the status code (0 = valid) without raising."""
    a, b = _host_i32(cu), _host_i32(cup)
    return int(lib().cp_validate_seqlens(a.ctypes.data, b.ctypes.data, len(b) - 1, total_tokens,
                                         cp_size, strategy, pad_between_seqs))


def cp_valid_end(cu, cup, cp_size: int, rank: int, strategy: int, pad_between_seqs: int) -> int:
    a, b = _host_i32(cu), _host_i32(cup)
    out = _I64(0)
    st = lib().cp_valid_end(a.ctypes.data, b.ctypes.data, len(b) - 1, cp_size, rank, strategy,
                            pad_between_seqs, ctypes.byref(out))
    _check("cp_valid_end", st)
    return int(out.value)


def cp_meta_bytes(n_docs: int, total_tokens: int, cp_size: int) -> int:
    return int(lib().cp_meta_bytes(n_docs, total_tokens, cp_size))


def cp_attn_bwd_workspace_bytes(s_local: int, H: int) -> int:
    return int(lib().cp_attn_bwd_workspace_bytes(s_local, H))


# ---------------------------------------------------------------------------
# device entry points
# ---------------------------------------------------------------------------

def cp_partition_index(d_cu: Optional[torch.Tensor], d_cup: torch.Tensor, total_tokens: int,
                       cp_size: int, rank: int, strategy: int, pad_between_seqs: int,
                       d_idx: torch.Tensor, d_restore: Optional[torch.Tensor],
                       d_meta: torch.Tensor, stream=None) -> None:
    n_docs = d_cup.numel() - 1
    st = lib().cp_partition_index(None if d_cu is None else _dev(d_cu, "cu"), _dev(d_cup, "cup"),
                                  n_docs, total_tokens, cp_size, rank, strategy,
                                  pad_between_seqs, _dev(d_idx, "idx"),
                                  None if d_restore is None else _dev(d_restore, "restore"),
                                  _dev(d_meta, "meta"), d_meta.numel() * d_meta.element_size(),
                                  _stream(stream))
    _check("cp_partition_index", st)


def cp_partition_index_all(d_cu: Optional[torch.Tensor], d_cup: torch.Tensor, total_tokens: int,
                           cp_size: int, strategy: int, pad_between_seqs: int,
                           d_idx_all: torch.Tensor, d_restore: Optional[torch.Tensor],
                           d_meta: torch.Tensor, meta_stride: int, stream=None) -> None:
    """Every rank's partition index and metadata in one launch (rank r's
    metadata at byte r * meta_stride of d_meta)."""
    if d_meta.numel() * d_meta.element_size() < cp_size * meta_stride:
        raise ValueError("metadata buffer smaller than cp_size * meta_stride")
    st = lib().cp_partition_index_all(None if d_cu is None else _dev(d_cu, "cu"),
                                      _dev(d_cup, "cup"), d_cup.numel() - 1, total_tokens,
                                      cp_size, strategy, pad_between_seqs,
                                      _dev(d_idx_all, "idx_all"),
                                      None if d_restore is None else _dev(d_restore, "restore"),
                                      _dev(d_meta, "meta"), meta_stride, _stream(stream))
    _check("cp_partition_index_all", st)


def _row_bytes(t: torch.Tensor) -> int:
    return t[0].numel() * t.element_size() if t.shape[0] > 0 else t.numel() * t.element_size()


def cp_thd_gather(srcs: Sequence[torch.Tensor], dsts: Sequence[torch.Tensor],
                  d_idx: torch.Tensor, stream=None) -> None:
    n_rows = d_idx.numel()
    src_rows = srcs[0].shape[0]
    st = lib().cp_thd_gather(_ptr_array(srcs, "src"), _ptr_array(dsts, "dst"), len(srcs),
                             _dev(d_idx, "idx"), n_rows, src_rows, _row_bytes(srcs[0]),
                             _stream(stream))
    _check("cp_thd_gather", st)


def cp_thd_gather_f16(srcs: Sequence[torch.Tensor], dsts: Sequence[torch.Tensor],
                      d_idx: Optional[torch.Tensor], stream=None) -> None:
    """dst[k][i] = fp16(src[k][idx[i]]) for bf16 sources (idx None: row i)."""
    n_rows = dsts[0].shape[0] if d_idx is None else d_idx.numel()
    src_rows = srcs[0].shape[0]
    st = lib().cp_thd_gather_f16(_ptr_array(srcs, "src"), _ptr_array(dsts, "dst"), len(srcs),
                                 None if d_idx is None else _dev(d_idx, "idx"), n_rows, src_rows,
                                 _row_bytes(srcs[0]), _stream(stream))
    _check("cp_thd_gather_f16", st)


def cp_thd_scatter(srcs: Sequence[torch.Tensor], dsts: Sequence[torch.Tensor],
                   d_idx: torch.Tensor, stream=None) -> None:
    n_rows = d_idx.numel()
    dst_rows = dsts[0].shape[0]
    st = lib().cp_thd_scatter(_ptr_array(srcs, "src"), _ptr_array(dsts, "dst"), len(srcs),
                              _dev(d_idx, "idx"), n_rows, dst_rows, _row_bytes(srcs[0]),
                              _stream(stream))
    _check("cp_thd_scatter", st)


A2A_SEQ_TO_HEAD, A2A_HEAD_TO_SEQ = 0, 1


def cp_a2a_exchange(srcs: Sequence[torch.Tensor], dsts: Sequence[torch.Tensor],
                    d_perm: Optional[torch.Tensor], cp_size: int, direction: int,
                    stream=None) -> None:
    """Sequence side [T, H, D] <-> head side [cp, T, H/cp, D] (see cp_a2a_exchange)."""
    seq = srcs[0] if direction == A2A_SEQ_TO_HEAD else dsts[0]
    T, H, D = seq.shape
    st = lib().cp_a2a_exchange(_ptr_array(srcs, "src"), _ptr_array(dsts, "dst"), len(srcs),
                               _dev(d_perm, "perm") if d_perm is not None else None, T, cp_size,
                               H, D, int(direction), _stream(stream))
    _check("cp_a2a_exchange", st)


def cp_reduce_scatter_emul(accums: Sequence[torch.Tensor], dsts: Sequence[torch.Tensor],
                           d_idx: Optional[torch.Tensor], row0: int, n_rows: int,
                           stream=None) -> None:
    T, H, D = accums[0].shape
    st = lib().cp_reduce_scatter_emul(_ptr_array(accums, "accum"), _ptr_array(dsts, "dst"),
                                      len(accums), None if d_idx is None else _dev(d_idx, "idx"),
                                      row0, n_rows, T, H, D, _stream(stream))
    _check("cp_reduce_scatter_emul", st)


def cp_zero_tail(tensors: Sequence[torch.Tensor], valid_end: int,
                 d_valid_end: Optional[torch.Tensor] = None, stream=None) -> bool:
    """Returns True when a kernel was launched."""
    rows = tensors[0].shape[0]
    launched = _I(0)
    st = lib().cp_zero_tail(_ptr_array(tensors, "rows"), len(tensors), rows,
                            _row_bytes(tensors[0]), valid_end,
                            None if d_valid_end is None else _dev(d_valid_end, "valid_end"),
                            _stream(stream), ctypes.byref(launched))
    _check("cp_zero_tail", st)
    return bool(launched.value)


def _opt(t, name):
    return None if t is None else _dev(t, name)


OPERAND_BF16, OPERAND_F16 = 0, 1


def _operand_dtype(*ts) -> int:
    """The tensor-core operand type of Q/K/V(/dO): all bf16 or all fp16."""
    kinds = {t.dtype for t in ts}
    if kinds == {torch.bfloat16}:
        return OPERAND_BF16
    if kinds == {torch.float16}:
        return OPERAND_F16
    raise ValueError(f"attention operands must be all bf16 or all fp16, got {kinds}")


def cp_attn_fwd(q_local, k_full, v_full, o_local, lse_local, d_meta, total_tokens: int,
                cp_size: int, rank: int, strategy: int, softmax_scale: float,
                stream=None, o_resid=None) -> None:
    """o_resid (optional, bf16 like o_local) receives O's bf16 rounding remainder,
    which the backward's Delta uses."""
    _, H, D = k_full.shape
    dt = _operand_dtype(q_local, k_full, v_full)
    st = lib().cp_attn_fwd(_dev(q_local, "q"), _dev(k_full, "k"), _dev(v_full, "v"),
                           _dev(o_local, "o"), _opt(o_resid, "o_resid"), _dev(lse_local, "lse"),
                           _dev(d_meta, "meta"),
                           d_meta.numel() * d_meta.element_size(), total_tokens, H, D, cp_size,
                           rank, strategy, float(softmax_scale), dt, _stream(stream))
    _check("cp_attn_fwd", st)


def cp_attn_fwd_gather(q_src, d_idx, k_full, v_full, o_local, lse_local, d_meta,
                       total_tokens: int, cp_size: int, rank: int, strategy: int,
                       softmax_scale: float, stream=None, o_resid=None) -> None:
    """cp_attn_fwd reading query row t from q_src[d_idx[t]] (no q_local copy)."""
    _, H, D = k_full.shape
    dt = _operand_dtype(q_src, k_full, v_full)
    st = lib().cp_attn_fwd_gather(_dev(q_src, "q_src"), q_src.shape[0], _dev(d_idx, "idx"),
                                  _dev(k_full, "k"), _dev(v_full, "v"), _dev(o_local, "o"),
                                  _opt(o_resid, "o_resid"), _dev(lse_local, "lse"),
                                  _dev(d_meta, "meta"), d_meta.numel() * d_meta.element_size(),
                                  total_tokens, H, D, cp_size, rank, strategy,
                                  float(softmax_scale), dt, _stream(stream))
    _check("cp_attn_fwd_gather", st)


BWD_ACCUMULATE, BWD_STORE, BWD_DQ_F32_STORE, BWD_DQ_F32_ACCUMULATE = 0, 1, 2, 4


def cp_attn_bwd(q_local, k_full, v_full, o_local, lse_local, do_local, dq_local, dk_accum,
                dv_accum, d_meta, total_tokens: int, cp_size: int, rank: int, strategy: int,
                softmax_scale: float, d_workspace, stream=None, mode: int = BWD_ACCUMULATE,
                o_resid=None) -> None:
    """cp_attn_bwd (mode BWD_ACCUMULATE) or cp_attn_bwd_ex with the given mode;
    o_resid: the forward's O rounding remainder (optional)."""
    _, H, D = k_full.shape
    dt = _operand_dtype(q_local, k_full, v_full, do_local)
    args = (_dev(q_local, "q"), _dev(k_full, "k"), _dev(v_full, "v"),
            _dev(o_local, "o"), _opt(o_resid, "o_resid"), _dev(lse_local, "lse"),
            _dev(do_local, "do"),
            _dev(dq_local, "dq"), _dev(dk_accum, "dk"), _dev(dv_accum, "dv"),
            _dev(d_meta, "meta"), d_meta.numel() * d_meta.element_size(),
            total_tokens, H, D, cp_size, rank, strategy, float(softmax_scale), dt)
    tail = (_dev(d_workspace, "workspace"), d_workspace.numel() * d_workspace.element_size(),
            _stream(stream))
    if mode == BWD_ACCUMULATE:
        _check("cp_attn_bwd", lib().cp_attn_bwd(*args, *tail))
    else:
        _check("cp_attn_bwd_ex", lib().cp_attn_bwd_ex(*args, int(mode), *tail))


def cp_attn_bwd_grouped_workspace_bytes(s_local: int, H: int, cp_size: int,
                                        total_tokens: int) -> int:
    return int(lib().cp_attn_bwd_grouped_workspace_bytes(s_local, H, cp_size, total_tokens))


def cp_attn_bwd_grouped(q_all, k_full, v_full, o_all, lse_all, do_all, dq_all, dk_accum,
                        dv_accum, d_meta_all, meta_stride: int, total_tokens: int, cp_size: int,
                        strategy: int, softmax_scale: float, d_workspace, stream=None,
                        o_resid_all=None) -> None:
    """cp_attn_bwd_grouped: every rank's backward, dK/dV summed over the ranks
    inside one dK/dV launch and stored.  *_all are the ranks' tensors side by
    side ([cp*s_local, H, D]; lse_all [cp, H, s_local]); d_meta_all holds the
    ranks' metadata meta_stride bytes apart."""
    _, H, D = k_full.shape
    dt = _operand_dtype(q_all, k_full, v_full, do_all)
    _check("cp_attn_bwd_grouped", lib().cp_attn_bwd_grouped(
        _dev(q_all, "q"), _dev(k_full, "k"), _dev(v_full, "v"), _dev(o_all, "o"),
        _opt(o_resid_all, "o_resid"), _dev(lse_all, "lse"), _dev(do_all, "do"),
        _dev(dq_all, "dq"), _dev(dk_accum, "dk"), _dev(dv_accum, "dv"),
        _dev(d_meta_all, "meta"), int(meta_stride), total_tokens, H, D, cp_size, strategy,
        float(softmax_scale), dt, _dev(d_workspace, "workspace"),
        d_workspace.numel() * d_workspace.element_size(), _stream(stream)))


def cp_attn_bwd_grouped_rs(q_all, k_full, v_full, o_all, lse_all, do_all, dq_all, dk_all, dv_all,
                           d_restore, d_meta_all, meta_stride: int, total_tokens: int,
                           cp_size: int, strategy: int, softmax_scale: float, d_workspace,
                           stream=None, o_resid_all=None) -> None:
    """cp_attn_bwd_grouped_rs: cp_attn_bwd_grouped with the reduce-scatter fused
    into the dK/dV kernel: dk_all / dv_all are the rank-concatenated bf16
    outputs (rank r's rows at r*s_local in its partition order), written
    through d_restore (None under NO_LOAD_BALANCE)."""
    _, H, D = k_full.shape
    dt = _operand_dtype(q_all, k_full, v_full, do_all)
    _check("cp_attn_bwd_grouped_rs", lib().cp_attn_bwd_grouped_rs(
        _dev(q_all, "q"), _dev(k_full, "k"), _dev(v_full, "v"), _dev(o_all, "o"),
        _opt(o_resid_all, "o_resid"), _dev(lse_all, "lse"), _dev(do_all, "do"),
        _dev(dq_all, "dq"), _dev(dk_all, "dk"), _dev(dv_all, "dv"), _opt(d_restore, "restore"),
        _dev(d_meta_all, "meta"), int(meta_stride), total_tokens, H, D, cp_size, strategy,
        float(softmax_scale), dt, _dev(d_workspace, "workspace"),
        d_workspace.numel() * d_workspace.element_size(), _stream(stream)))


def cp_attn_fwd_ring_workspace_bytes(s_local: int) -> int:
    return int(lib().cp_attn_fwd_ring_workspace_bytes(s_local))


def cp_attn_fwd_ring(q_local, k_shards, v_shards, o_local, lse_local, d_step_meta, step_bytes: int,
                     n_steps: int, cp_size: int, rank: int, strategy: int, softmax_scale: float,
                     d_workspace, stream=None, o_resid=None) -> None:
    """cp_attn_fwd_ring: every ring step of a rank in one pass (no partial outputs,
    no merge); k_shards / v_shards are the ranks' shards side by side."""
    s_local, H, D = q_local.shape
    dt = _operand_dtype(q_local, k_shards, v_shards)
    _check("cp_attn_fwd_ring", lib().cp_attn_fwd_ring(
        _dev(q_local, "q"), _dev(k_shards, "k"), _dev(v_shards, "v"), _dev(o_local, "o"),
        _opt(o_resid, "o_resid"), _dev(lse_local, "lse"), _dev(d_step_meta, "meta"),
        int(step_bytes), int(n_steps), s_local, H, D, cp_size, rank, strategy,
        float(softmax_scale), dt, _dev(d_workspace, "workspace"),
        d_workspace.numel() * d_workspace.element_size(), _stream(stream)))


def cp_attn_bwd_ring_workspace_bytes(s_local: int, H: int, cp_size: int) -> int:
    return int(lib().cp_attn_bwd_ring_workspace_bytes(s_local, H, cp_size))


def cp_attn_bwd_ring(q_all, k_shards, v_shards, o_all, lse_all, do_all, dq_all, dk_accum,
                     dv_accum, d_ring_meta, step_bytes: int, rank_stride: int, cp_size: int,
                     strategy: int, softmax_scale: float, d_workspace, stream=None,
                     o_resid_all=None) -> None:
    """cp_attn_bwd_ring: the ring backward of every rank in one pass per gradient
    (dq_all bf16, dk_accum / dv_accum fp32 rank-concatenated, all stored)."""
    rows, H, D = q_all.shape
    s_local = rows // cp_size
    dt = _operand_dtype(q_all, k_shards, v_shards, do_all)
    _check("cp_attn_bwd_ring", lib().cp_attn_bwd_ring(
        _dev(q_all, "q"), _dev(k_shards, "k"), _dev(v_shards, "v"), _dev(o_all, "o"),
        _opt(o_resid_all, "o_resid"), _dev(lse_all, "lse"), _dev(do_all, "do"),
        _dev(dq_all, "dq"), _dev(dk_accum, "dk"), _dev(dv_accum, "dv"), _dev(d_ring_meta, "meta"),
        int(step_bytes), int(rank_stride), s_local, H, D, cp_size, strategy, float(softmax_scale),
        dt, _dev(d_workspace, "workspace"), d_workspace.numel() * d_workspace.element_size(),
        _stream(stream)))


def cp_attn_bwd_ring_rs(q_all, k_shards, v_shards, o_all, lse_all, do_all, dq_all, dk_all,
                        dv_all, d_ring_meta, step_bytes: int, rank_stride: int, cp_size: int,
                        strategy: int, softmax_scale: float, d_workspace, stream=None,
                        o_resid_all=None) -> None:
    """cp_attn_bwd_ring_rs: cp_attn_bwd_ring with dK/dV written as bf16
    rank-concatenated shards by the dK/dV kernel itself (no fp32 sums, no cast
    pass)."""
    rows, H, D = q_all.shape
    s_local = rows // cp_size
    dt = _operand_dtype(q_all, k_shards, v_shards, do_all)
    _check("cp_attn_bwd_ring_rs", lib().cp_attn_bwd_ring_rs(
        _dev(q_all, "q"), _dev(k_shards, "k"), _dev(v_shards, "v"), _dev(o_all, "o"),
        _opt(o_resid_all, "o_resid"), _dev(lse_all, "lse"), _dev(do_all, "do"),
        _dev(dq_all, "dq"), _dev(dk_all, "dk"), _dev(dv_all, "dv"), _dev(d_ring_meta, "meta"),
        int(step_bytes), int(rank_stride), s_local, H, D, cp_size, strategy, float(softmax_scale),
        dt, _dev(d_workspace, "workspace"), d_workspace.numel() * d_workspace.element_size(),
        _stream(stream)))


NOALLOC_MAX_SCRATCH_FLOATS = 1048576  # CP_NOALLOC_MAX_SCRATCH_FLOATS in cpthd.h


def cp_attn_bwd_noalloc(q_local, k_full, v_full, o_local, lse_local, do_local, dq_local,
                        dk_accum, dv_accum, d_meta, total_tokens: int, cp_size: int, rank: int,
                        strategy: int, softmax_scale: float, stream=None, o_resid=None) -> None:
    """cp_attn_bwd for callers that cannot allocate device memory: the Delta
    scratch is a fixed array inside the library (s_local*H <= 1,048,576
    floats).  Calls that overlap on the GPU share that array and race."""
    _, H, D = k_full.shape
    dt = _operand_dtype(q_local, k_full, v_full, do_local)
    st = lib().cp_attn_bwd_noalloc(_dev(q_local, "q"), _dev(k_full, "k"), _dev(v_full, "v"),
                                   _dev(o_local, "o"), _opt(o_resid, "o_resid"),
                                   _dev(lse_local, "lse"),
                                   _dev(do_local, "do"), _dev(dq_local, "dq"),
                                   _dev(dk_accum, "dk"), _dev(dv_accum, "dv"),
                                   _dev(d_meta, "meta"), d_meta.numel() * d_meta.element_size(),
                                   total_tokens, H, D, cp_size, rank, strategy,
                                   float(softmax_scale), dt, _stream(stream))
    _check("cp_attn_bwd_noalloc", st)


def cp_p2p_meta_bytes(n_docs: int, total_tokens: int, cp_size: int) -> int:
    return int(lib().cp_p2p_meta_bytes(n_docs, total_tokens, cp_size))


def cp_p2p_index(d_cu: Optional[torch.Tensor], d_cup: torch.Tensor, total_tokens: int,
                 cp_size: int, rank: int, strategy: int, pad_between_seqs: int,
                 d_meta: torch.Tensor, stream=None) -> None:
    """Metadata of all cp_size ring steps of `rank` (step i at i * cp_p2p_meta_bytes)."""
    st = lib().cp_p2p_index(None if d_cu is None else _dev(d_cu, "cu"), _dev(d_cup, "cup"),
                            d_cup.numel() - 1, total_tokens, cp_size, rank, strategy,
                            pad_between_seqs, _dev(d_meta, "meta"),
                            d_meta.numel() * d_meta.element_size(), _stream(stream))
    _check("cp_p2p_index", st)


def cp_p2p_merge(o_steps: torch.Tensor, lse_steps: torch.Tensor, out: torch.Tensor,
                 lse: torch.Tensor, stream=None, o_steps_resid=None, out_resid=None) -> None:
    """o_steps [n, s_local, H, D] bf16, lse_steps [n, H, s_local] -> out, lse;
    optionally the steps' O rounding remainders in and the output's out."""
    n, s_local, H, D = o_steps.shape
    st = lib().cp_p2p_merge(_dev(o_steps, "o_steps"), _opt(o_steps_resid, "o_steps_resid"),
                            _dev(lse_steps, "lse_steps"), n, s_local, H, D, _dev(out, "out"),
                            _opt(out_resid, "out_resid"), _dev(lse, "lse"), _stream(stream))
    _check("cp_p2p_merge", st)


def cp_device_status(reset: bool = True) -> int:
    out = _I(0)
    _check("cp_device_status", lib().cp_device_status(ctypes.byref(out), int(reset)))
    return int(out.value)
