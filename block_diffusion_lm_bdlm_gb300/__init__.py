"""GB300-native BDLM attention: Python binding of libbdlm.

Argument marshalling only. Every step of the computation runs in the CUDA
kernels of libbdlm.so (built in-tree from csrc/ for sm_103a); there is no
Python or CPU fallback, and a missing library raises. PyTorch supplies device
memory and the current stream.

The C functions are declared in include/bdlm.h; the Python names are the same:
  bdlm_attn_fwd(q, k, v, block, ...) -> (o, lse)
  bdlm_attn_bwd(q, k, v, o, lse, dO, block, ...) -> (dq, dk, dv)
  bdlm_lse_merge(partials, lses) -> (o, lse)
  bdlm_attn_fwd_tasks(q, k, v, block, tasks, n_slots) -> (o [S,L,H,d], lse [S,H,L])
                                    a token-level task list in one launch
  bdlm_attn_bwd_tasks(q, k, v, o, lse, dO, block, tasks, n_slots) -> (dq, dk [S,L,Hk,d], dv)
  bdlm_attn_fwd_noalloc(...)        forward without a caller workspace
  bdlm_selftest_timeout(workspace)  device wait-timeout self-test
Restrictions of a call (see Partial):
  Partial.window(lo, hi)                     keys at positions [lo, hi) (a clean shard)
  Partial.window(lo, hi, accumulate=True)    merge into a running (out, lse)
  Partial.window(lo, hi, q_lo=a, q_hi=b)     only the query rows [a, b)
  Partial.group(blocks)                      the corrupted rows of a block list
Packed documents: cu_seqlens (device int32 offsets); ragged last blocks are
allowed wherever the block size does not divide a half's length.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

from .build import LIB

__all__ = [
    "BDLMError", "Partial", "Task", "bdlm_attn_fwd", "bdlm_attn_fwd_tasks", "bdlm_attn_fwd_tasks_workspace_bytes",
    "bdlm_attn_bwd_tasks", "bdlm_attn_bwd_tasks_workspace_bytes", "bdlm_attn_fwd_noalloc", "bdlm_attn_bwd", "bdlm_lse_merge", "bdlm_read_error",
    "bdlm_attn_fwd_workspace_bytes", "bdlm_attn_bwd_workspace_bytes", "bdlm_last_launch_count",
    "bdlm_selftest_timeout", "load_library", "EXPORTED_SYMBOLS",
]

BDLM_OK = 0
BDLM_BF16, BDLM_F32 = 0, 1
PART_NONE, PART_KEY_WINDOW, PART_BLOCK_GROUP = 0, 1, 2
PART_ACCUMULATE = 1

EXPORTED_SYMBOLS = (
    "bdlm_attn_fwd_workspace_bytes", "bdlm_attn_bwd_workspace_bytes", "bdlm_attn_fwd", "bdlm_attn_bwd",
    "bdlm_lse_merge", "bdlm_read_error", "bdlm_status_string", "bdlm_last_launch_count",
    "bdlm_attn_fwd_noalloc",
    "bdlm_attn_fwd_tasks_workspace_bytes", "bdlm_attn_fwd_tasks",
    "bdlm_attn_bwd_tasks_workspace_bytes", "bdlm_attn_bwd_tasks",
    "bdlm_selftest_timeout",
)


class BDLMError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


class _CPartial(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("n_q_blocks", ctypes.c_int32), ("key_lo", ctypes.c_int64),
                ("key_hi", ctypes.c_int64), ("q_blocks", ctypes.c_void_p), ("flags", ctypes.c_int32),
                ("o_dtype", ctypes.c_int32), ("q_lo", ctypes.c_int64), ("q_hi", ctypes.c_int64)]


@dataclass
class Partial:
    """Restriction of a call (see bdlm_partial in include/bdlm.h).

    Partial.window(lo, hi): k/v hold the keys at positions [lo, hi).
    Partial.window(lo, hi, accumulate=True): forward only; `out` and `lse`
        hold the merged result of earlier windows and this call merges in.
    Partial.window(lo, hi, q_lo=a, q_hi=b): q (o, lse, dO, dq) hold only the
        rows at positions [a, b); pass L = 2n to the call.
    Partial.group(blocks): q holds the corrupted rows of `blocks` (device int32).
    The element type of a partial forward's o follows the `out` tensor (bf16
    or fp32).
    """
    kind: int
    key_lo: int = 0
    key_hi: int = 0
    q_blocks: Optional[torch.Tensor] = None
    accumulate: bool = False
    q_lo: int = 0
    q_hi: int = 0

    @staticmethod
    def window(lo: int, hi: int, accumulate: bool = False, q_lo: int = 0, q_hi: int = 0) -> "Partial":
        return Partial(PART_KEY_WINDOW, key_lo=int(lo), key_hi=int(hi), accumulate=bool(accumulate),
                       q_lo=int(q_lo), q_hi=int(q_hi))

    @property
    def row_range(self) -> bool:
        return self.q_hi != 0 or self.q_lo != 0

    @staticmethod
    def group(blocks: torch.Tensor) -> "Partial":
        return Partial(PART_BLOCK_GROUP, q_blocks=blocks)

    def c(self, o_dtype: int = 0) -> _CPartial:
        nb, ptr = 0, None
        if self.kind == PART_BLOCK_GROUP:
            b = self.q_blocks
            if b is None or b.dtype != torch.int32 or not b.is_cuda or not b.is_contiguous():
                raise ValueError("q_blocks must be a contiguous int32 CUDA tensor")
            nb, ptr = b.numel(), b.data_ptr()
        flags = PART_ACCUMULATE if self.accumulate else 0
        return _CPartial(self.kind, nb, self.key_lo, self.key_hi, ptr, flags, o_dtype, self.q_lo, self.q_hi)


class _CTask(ctypes.Structure):
    _fields_ = [("seq_start", ctypes.c_int64), ("n", ctypes.c_int64), ("q_lo", ctypes.c_int64),
                ("q_hi", ctypes.c_int64), ("key_lo", ctypes.c_int64), ("key_hi", ctypes.c_int64),
                ("slot", ctypes.c_int32), ("reserved", ctypes.c_int32)]


@dataclass(frozen=True)
class Task:
    """One token-level task: the query positions [q_lo, q_hi) of the sequence
    at rows [seq_start, seq_start + 2n) against its key positions
    [key_lo, key_hi), written to output slot `slot`."""
    seq_start: int
    n: int
    q_lo: int
    q_hi: int
    key_lo: int
    key_hi: int
    slot: int = 0


def _task_array(tasks: Sequence[Task]):
    arr = (_CTask * len(tasks))()
    for i, t in enumerate(tasks):
        arr[i] = _CTask(t.seq_start, t.n, t.q_lo, t.q_hi, t.key_lo, t.key_hi, t.slot, 0)
    return arr


_lib = None


def load_library() -> ctypes.CDLL:
    """Load libbdlm.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB):
        raise RuntimeError(f"{LIB} is missing: build it with `python -m block_diffusion_lm_bdlm_gb300.build`")
    lib = ctypes.CDLL(LIB)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.bdlm_attn_fwd_workspace_bytes.argtypes = [i64, i32, i32, i32]
    lib.bdlm_attn_fwd_workspace_bytes.restype = sz
    lib.bdlm_attn_bwd_workspace_bytes.argtypes = [i64, i32, i32, i32]
    lib.bdlm_attn_bwd_workspace_bytes.restype = sz
    lib.bdlm_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, vp, i32, f32,
                                  ctypes.POINTER(_CPartial), vp, sz, vp]
    lib.bdlm_attn_fwd.restype = ctypes.c_int
    lib.bdlm_attn_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, vp, i32, f32,
                                          ctypes.POINTER(_CPartial), vp]
    lib.bdlm_attn_fwd_noalloc.restype = ctypes.c_int
    lib.bdlm_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, vp, i32, f32,
                                  ctypes.POINTER(_CPartial), vp, sz, vp]
    lib.bdlm_attn_bwd.restype = ctypes.c_int
    lib.bdlm_lse_merge.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(vp), i32, i32, i64, i32, i32, vp, vp, vp]
    lib.bdlm_lse_merge.restype = ctypes.c_int
    lib.bdlm_read_error.argtypes = [vp, vp]
    lib.bdlm_read_error.restype = ctypes.c_int
    lib.bdlm_status_string.argtypes = [ctypes.c_int]
    lib.bdlm_status_string.restype = ctypes.c_char_p
    lib.bdlm_last_launch_count.argtypes = []
    lib.bdlm_last_launch_count.restype = ctypes.c_int
    lib.bdlm_attn_fwd_tasks_workspace_bytes.argtypes = [ctypes.POINTER(_CTask), i32]
    lib.bdlm_attn_fwd_tasks_workspace_bytes.restype = sz
    lib.bdlm_attn_fwd_tasks.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, f32,
                                        ctypes.POINTER(_CTask), i32, i32, i32, vp, sz, vp]
    lib.bdlm_attn_fwd_tasks.restype = ctypes.c_int
    lib.bdlm_attn_bwd_tasks_workspace_bytes.argtypes = [ctypes.POINTER(_CTask), i32, i64, i32, i32]
    lib.bdlm_attn_bwd_tasks_workspace_bytes.restype = sz
    lib.bdlm_attn_bwd_tasks.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i32, f32,
                                        ctypes.POINTER(_CTask), i32, i32, vp, sz, vp]
    lib.bdlm_attn_bwd_tasks.restype = ctypes.c_int
    lib.bdlm_selftest_timeout.argtypes = [vp, sz, ctypes.c_uint32, vp]
    lib.bdlm_selftest_timeout.restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().bdlm_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != BDLM_OK:
        raise BDLMError(status, where)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _bf16_cuda(name, t):
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")


def _shape(name, t, shape):
    """The library reads and writes exactly the rows the call describes, so a
    tensor of another shape would be read or written out of bounds."""
    if tuple(t.shape) != tuple(int(v) for v in shape):
        raise ValueError(f"{name} must be shaped {tuple(int(v) for v in shape)}, got {tuple(t.shape)}")


def _call_rows(L: int, part: Optional[Partial], block: int):
    """(rows of q, rows of k) that a call with total rows L and restriction
    `part` reads, as include/bdlm.h defines them."""
    if part is None or part.kind == PART_NONE:
        return L, L
    if part.kind == PART_KEY_WINDOW:
        return (part.q_hi - part.q_lo if part.row_range else L), part.key_hi - part.key_lo
    if part.q_blocks is None:
        raise ValueError("a block group needs its q_blocks")
    nq = part.q_blocks.numel() * block
    return nq, L // 2 + nq


def _check_qkv(q, k, v, L, part, block):
    Lq, Lk = _call_rows(L, part, block)
    d = q.shape[2]
    _shape("q", q, (Lq, q.shape[1], d))
    _shape("k", k, (Lk, k.shape[1], d))
    _shape("v", v, k.shape)
    return Lq, Lk


def _cu(cu_seqlens):
    if cu_seqlens is None:
        return None, 1
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be a contiguous int32 CUDA tensor")
    return cu_seqlens.data_ptr(), cu_seqlens.numel() - 1


def bdlm_attn_fwd_workspace_bytes(L: int, heads: int, head_dim: int, n_docs: int = 1) -> int:
    return int(load_library().bdlm_attn_fwd_workspace_bytes(L, heads, head_dim, n_docs))


def bdlm_attn_bwd_workspace_bytes(L: int, heads: int, head_dim: int, n_docs: int = 1) -> int:
    return int(load_library().bdlm_attn_bwd_workspace_bytes(L, heads, head_dim, n_docs))


def bdlm_last_launch_count() -> int:
    return int(load_library().bdlm_last_launch_count())


def _total_rows(q, L, part):
    """L of the call: q's rows by default; a block group or a window over a
    row range must name the sequence's 2n."""
    if L is not None:
        return int(L)
    if part is not None and (part.kind == PART_BLOCK_GROUP or part.row_range):
        raise ValueError("pass L = 2n: q holds only some rows of the sequence")
    return q.shape[0]


def _fwd_outputs(q, part, out, lse):
    """Allocate or check the forward's o and lse; returns (out, lse, o_dtype)."""
    Lq, H, d = q.shape
    if part is not None and part.accumulate and (out is None or lse is None):
        raise ValueError("an accumulating window needs the running `out` and `lse`")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((H, Lq), dtype=torch.float32, device=q.device)
    if out.dtype not in (torch.bfloat16, torch.float32) or tuple(out.shape) != (Lq, H, d) or not out.is_cuda \
            or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 or fp32 CUDA tensor shaped like q")
    if out.dtype == torch.float32 and part is None:
        raise ValueError("fp32 o is for partial calls; full attention writes bf16")
    if tuple(lse.shape) != (H, Lq) or lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 CUDA tensor [H, Lq]")
    return out, lse, (BDLM_F32 if out.dtype == torch.float32 else BDLM_BF16)


def bdlm_attn_fwd(q, k, v, block: int, *, L: Optional[int] = None, cu_seqlens=None, softmax_scale: float = 0.0,
                  part: Optional[Partial] = None, out=None, lse=None, workspace=None, stream=None):
    """BDLM attention forward. q [Lq,H,d], k/v [Lk,Hk,d] bf16 CUDA tensors.
    L defaults to q's rows (full attention, key window) and must be given as
    2n for a block group. Returns (o [Lq,H,d], lse [H,Lq] fp32); o is bf16
    unless a partial call is given an fp32 `out`."""
    lib = load_library()
    for nm, t in (("q", q), ("k", k), ("v", v)):
        _bf16_cuda(nm, t)
    Lq, H, d = q.shape
    Hk = k.shape[1]
    L = _total_rows(q, L, part)
    _check_qkv(q, k, v, L, part, block)
    cu_ptr, n_docs = _cu(cu_seqlens)
    out, lse, o_dtype = _fwd_outputs(q, part, out, lse)
    ws_bytes = lib.bdlm_attn_fwd_workspace_bytes(L, H, d, n_docs)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    cpart = ctypes.byref(part.c(o_dtype)) if part is not None else None
    st = lib.bdlm_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), L, block, H,
                           Hk, d, cu_ptr, n_docs, softmax_scale, cpart, workspace.data_ptr(),
                           workspace.numel(), _stream(stream))
    _check(st, "bdlm_attn_fwd")
    return out, lse


def bdlm_attn_fwd_tasks_workspace_bytes(tasks: Sequence[Task]) -> int:
    return int(load_library().bdlm_attn_fwd_tasks_workspace_bytes(_task_array(tasks), len(tasks)))


def bdlm_attn_fwd_tasks(q, k, v, block: int, tasks: Sequence[Task], n_slots: int, *, softmax_scale: float = 0.0,
                        out=None, lse=None, workspace=None, stream=None):
    """Every task's partial forward in one launch. q [L,H,d], k/v [L,Hk,d]
    hold every row. Returns (o [n_slots,L,H,d], lse [n_slots,H,L]): task t
    fills slot t.slot at its rows; rows no task of a slot covers keep what
    `out` / `lse` held (fresh outputs start as o = 0, lse = -inf, so merging
    the slots with bdlm_lse_merge combines tasks that split a row's keys).
    `out` may be fp32 to keep the partials unrounded."""
    lib = load_library()
    for nm, t in (("q", q), ("k", k), ("v", v)):
        _bf16_cuda(nm, t)
    L, H, d = q.shape
    Hk = k.shape[1]
    _shape("k", k, (L, Hk, d))
    _shape("v", v, k.shape)
    if out is None:
        out = torch.zeros((n_slots, L, H, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.full((n_slots, H, L), float("-inf"), dtype=torch.float32, device=q.device)
    if out.dtype not in (torch.bfloat16, torch.float32) or tuple(out.shape) != (n_slots, L, H, d) \
            or not out.is_cuda or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 or fp32 CUDA tensor [n_slots, L, H, d]")
    if tuple(lse.shape) != (n_slots, H, L) or lse.dtype != torch.float32 or not lse.is_cuda \
            or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 CUDA tensor [n_slots, H, L]")
    arr = _task_array(tasks)
    ws_bytes = lib.bdlm_attn_fwd_tasks_workspace_bytes(arr, len(tasks))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    o_dtype = BDLM_F32 if out.dtype == torch.float32 else BDLM_BF16
    st = lib.bdlm_attn_fwd_tasks(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), L, block,
                                 H, Hk, d, softmax_scale, arr, len(tasks), n_slots, o_dtype, workspace.data_ptr(),
                                 workspace.numel(), _stream(stream))
    _check(st, "bdlm_attn_fwd_tasks")
    return out, lse


def bdlm_attn_bwd_tasks_workspace_bytes(tasks: Sequence[Task], L: int, heads: int, head_dim: int) -> int:
    return int(load_library().bdlm_attn_bwd_tasks_workspace_bytes(_task_array(tasks), len(tasks), L, heads,
                                                                  head_dim))


def bdlm_attn_bwd_tasks(q, k, v, o, lse, dO, block: int, tasks: Sequence[Task], n_slots: int, *,
                        softmax_scale: float = 0.0, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Every task's backward in one launch, each with the full softmax of its
    rows (o, lse: the merged forward results). Returns (dq [L,H,d]: the sum of
    the tasks' dq shares; dk, dv [n_slots,L,Hk,d]: task t's window keys in
    slot t.slot; keys no task of a slot covers keep what `dk` / `dv` held,
    zeros for fresh outputs)."""
    lib = load_library()
    for nm, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dO", dO)):
        _bf16_cuda(nm, t)
    L, H, d = q.shape
    Hk = k.shape[1]
    _shape("k", k, (L, Hk, d))
    _shape("v", v, k.shape)
    _shape("o", o, q.shape)
    _shape("dO", dO, q.shape)
    if dq is None:
        dq = torch.empty_like(q)
    if dk is None:
        dk = torch.zeros((n_slots, L, Hk, d), dtype=torch.bfloat16, device=q.device)
    if dv is None:
        dv = torch.zeros((n_slots, L, Hk, d), dtype=torch.bfloat16, device=q.device)
    _bf16_cuda("dq", dq)
    _shape("dq", dq, q.shape)
    for nm, t in (("dk", dk), ("dv", dv)):
        _bf16_cuda(nm, t)
        if tuple(t.shape) != (n_slots, L, Hk, d):
            raise ValueError(f"{nm} must be [n_slots, L, Hk, d]")
    if tuple(lse.shape) != (H, L) or lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 CUDA tensor [H, L]")
    arr = _task_array(tasks)
    if workspace is None:
        ws_bytes = lib.bdlm_attn_bwd_tasks_workspace_bytes(arr, len(tasks), L, H, d)
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    st = lib.bdlm_attn_bwd_tasks(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dO.data_ptr(),
                                 dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), L, block, H, Hk, d, softmax_scale, arr,
                                 len(tasks), n_slots, workspace.data_ptr(), workspace.numel(), _stream(stream))
    _check(st, "bdlm_attn_bwd_tasks")
    return dq, dk, dv


def bdlm_attn_fwd_noalloc(q, k, v, block: int, *, L: Optional[int] = None, cu_seqlens=None,
                          softmax_scale: float = 0.0, part: Optional[Partial] = None, out=None, lse=None,
                          stream=None, check: bool = False):
    """The forward without a workspace (see bdlm_attn_fwd_noalloc in
    include/bdlm.h): the library uses its own fixed scratch, so the call
    allocates nothing on the device beyond the outputs (pass `out` and `lse`
    to allocate nothing at all). Problems found on the device (a malformed
    cu_seqlens or block list) leave o and lse unwritten and are reported by
    bdlm_read_error(None); check=True synchronises the stream after the call
    and raises BDLMError for them."""
    lib = load_library()
    for nm, t in (("q", q), ("k", k), ("v", v)):
        _bf16_cuda(nm, t)
    Lq, H, d = q.shape
    Hk = k.shape[1]
    L = _total_rows(q, L, part)
    _check_qkv(q, k, v, L, part, block)
    cu_ptr, n_docs = _cu(cu_seqlens)
    out, lse, o_dtype = _fwd_outputs(q, part, out, lse)
    cpart = ctypes.byref(part.c(o_dtype)) if part is not None else None
    st = lib.bdlm_attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), L,
                                   block, H, Hk, d, cu_ptr, n_docs, softmax_scale, cpart, _stream(stream))
    _check(st, "bdlm_attn_fwd_noalloc")
    if check:
        _check(bdlm_read_error(None, stream), "bdlm_attn_fwd_noalloc (device)")
    return out, lse


def bdlm_attn_bwd(q, k, v, o, lse, dO, block: int, *, L: Optional[int] = None, cu_seqlens=None,
                  softmax_scale: float = 0.0, part: Optional[Partial] = None, dq=None, dk=None, dv=None,
                  workspace=None, stream=None):
    """BDLM attention backward. q/o/dO [Lq,H,d], k/v [Lk,Hk,d] bf16 CUDA
    tensors, lse [H,Lq] fp32. L defaults to q's rows and must be given as 2n
    for a block group. With Partial.window, o and lse are the merged full
    forward's and dq is the window's share. Returns (dq, dk, dv) bf16."""
    lib = load_library()
    for nm, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dO", dO)):
        _bf16_cuda(nm, t)
    Lq, H, d = q.shape
    Hk = k.shape[1]
    L = _total_rows(q, L, part)
    _check_qkv(q, k, v, L, part, block)
    cu_ptr, n_docs = _cu(cu_seqlens)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for nm, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _bf16_cuda(nm, t)
    for nm, t, ref in (("o", o, q), ("dO", dO, q), ("dq", dq, q), ("dk", dk, k), ("dv", dv, k)):
        _shape(nm, t, ref.shape)
    _shape("lse", lse, (H, Lq))
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 CUDA tensor")
    ws_bytes = lib.bdlm_attn_bwd_workspace_bytes(L, H, d, n_docs)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    cpart = ctypes.byref(part.c()) if part is not None else None
    st = lib.bdlm_attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dO.data_ptr(),
                           dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), L, block, H, Hk, d, cu_ptr, n_docs,
                           softmax_scale, cpart, workspace.data_ptr(), workspace.numel(), _stream(stream))
    _check(st, "bdlm_attn_bwd")
    return dq, dk, dv


def bdlm_lse_merge(partials: Sequence[torch.Tensor], lses: Sequence[torch.Tensor], *, out=None, lse=None,
                   stream=None):
    """Merge partials [rows,H,d] (bf16 or fp32) with their lse [H,rows]."""
    lib = load_library()
    P = len(partials)
    if P == 0 or P != len(lses):
        raise ValueError("need as many lse tensors as partials (at least one)")
    rows, H, d = partials[0].shape
    dt = partials[0].dtype
    if dt not in (torch.bfloat16, torch.float32):
        raise ValueError("partials must be bf16 or fp32")
    for p, l in zip(partials, lses):
        if p.shape != partials[0].shape or p.dtype != dt or not p.is_cuda or not p.is_contiguous():
            raise ValueError("partials must share one shape and dtype and be contiguous CUDA tensors")
        if l.shape != (H, rows) or l.dtype != torch.float32 or not l.is_cuda or not l.is_contiguous():
            raise ValueError("each lse must be a contiguous fp32 CUDA tensor [H, rows]")
    if out is None:
        out = torch.empty((rows, H, d), dtype=torch.bfloat16, device=partials[0].device)
    if lse is None:
        lse = torch.empty((H, rows), dtype=torch.float32, device=partials[0].device)
    _bf16_cuda("out", out)
    _shape("out", out, (rows, H, d))
    _shape("lse", lse, (H, rows))
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 CUDA tensor")
    pp = (ctypes.c_void_p * P)(*[p.data_ptr() for p in partials])
    lp = (ctypes.c_void_p * P)(*[l.data_ptr() for l in lses])
    st = lib.bdlm_lse_merge(pp, lp, P, BDLM_F32 if dt == torch.float32 else BDLM_BF16, rows, H, d,
                            out.data_ptr(), lse.data_ptr(), _stream(stream))
    _check(st, "bdlm_lse_merge")
    return out, lse


def bdlm_selftest_timeout(workspace: torch.Tensor, wait_ns: int = 100_000_000, stream=None) -> None:
    """Run the device failure-path self-test: a wait that nothing completes
    gives up after wait_ns and records BDLM_ERR_TIMEOUT in `workspace` (read it
    with bdlm_read_error)."""
    st = load_library().bdlm_selftest_timeout(workspace.data_ptr(), workspace.numel(), int(wait_ns), _stream(stream))
    _check(st, "bdlm_selftest_timeout")


def bdlm_read_error(workspace: Optional[torch.Tensor], stream=None) -> int:
    """Synchronise the stream and return the device error word of the last call
    that used `workspace` (0 = none). workspace=None reads the fixed scratch of
    bdlm_attn_fwd_noalloc on the current device."""
    ptr = None if workspace is None else workspace.data_ptr()
    return int(load_library().bdlm_read_error(ptr, _stream(stream)))
