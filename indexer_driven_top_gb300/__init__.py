"""Indexer-driven Top-K sparse attention on GB300: Python binding of libsi.

This module only marshals arguments: torch tensors (device memory) become the
plain pointers and sizes of the C ABI in ``include/si.h``, and every step of
the path runs in the CUDA kernels of ``libsi.so``.  There is no CPU or
PyTorch fallback: if the library is missing, importing this package raises.

Entry points (same names as the C ABI, minus the ``si_`` prefix):
  indexer_scores, topk, sparse_attn, fused_decode, fused_decode_noalloc,
  workspace_size, workspace_min, workspace_status.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

from . import _build

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = _build.LIB

F32, BF16, E4M3, E2M1, MXE4M3 = 0, 1, 2, 3, 4
DTYPES = {"f32": F32, "bf16": BF16, "e4m3": E4M3, "e2m1": E2M1, "mxe4m3": MXE4M3}
OP_INDEXER, OP_TOPK, OP_ATTN, OP_FUSED, OP_SELECT = 0, 1, 2, 3, 4
DEVFLAG_BAD_BLOCK, DEVFLAG_BAD_INDEX, DEVFLAG_TIMEOUT, DEVFLAG_RANGE = 1, 2, 4, 8


class SIError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"libsi status {status}: {detail}")
        self.status = status


class c_batch(ctypes.Structure):
    _fields_ = [("block_table", ctypes.c_void_p), ("ctx_len", ctypes.c_void_p),
                ("q_seq", ctypes.c_void_p), ("q_pos", ctypes.c_void_p),
                ("n_seq", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("n_q", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("max_ctx", ctypes.c_int32), ("n_blocks", ctypes.c_int32),
                ("host_q_seq", ctypes.c_void_p)]


class c_paged(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("dtype", ctypes.c_int),
                ("row_dim", ctypes.c_int32), ("row_stride", ctypes.c_int64),
                ("scale_tile", ctypes.c_int32)]


class c_indexer(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("q_dtype", ctypes.c_int), ("q_scale", ctypes.c_void_p),
                ("w", ctypes.c_void_p), ("n_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("k", c_paged)]


class c_attention(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("q_dtype", ctypes.c_int), ("n_heads", ctypes.c_int32),
                ("d_qk", ctypes.c_int32), ("d_v", ctypes.c_int32), ("k", c_paged),
                ("v", c_paged), ("softmax_scale", ctypes.c_float)]


_lib = None


def load() -> ctypes.CDLL:
    """Load libsi.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libsi.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    B, IX, AT = ctypes.POINTER(c_batch), ctypes.POINTER(c_indexer), ctypes.POINTER(c_attention)
    sig = {
        "si_workspace_size": (SZ, [ctypes.c_int, B, IX, AT, I32]),
        "si_workspace_min": (SZ, [ctypes.c_int, B, IX, AT, I32]),
        "si_indexer_scores": (ctypes.c_int, [B, IX, P, I64, P, SZ, P]),
        "si_topk": (ctypes.c_int, [B, P, I64, I32, P, P, SZ, P]),
        "si_sparse_attn": (ctypes.c_int, [B, AT, P, I32, P, ctypes.c_int, P, P, SZ, P]),
        "si_fused_decode": (ctypes.c_int, [B, IX, AT, I32, P, P, ctypes.c_int, P, P, SZ, P]),
        "si_fused_decode_noalloc": (ctypes.c_int, [B, IX, AT, I32, P, P, ctypes.c_int, P,
                                                   ctypes.POINTER(ctypes.c_void_p), P]),
        "si_workspace_size_cand": (SZ, [B, IX, I32]),
        "si_indexer_topk_cand": (ctypes.c_int, [B, IX, P, I32, I64, I32, P, P, I64, P, SZ, P]),
        "si_workspace_status": (ctypes.c_int, [P, ctypes.POINTER(ctypes.c_uint32), P]),
        "si_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "si_last_error": (ctypes.c_char_p, []),
        "si_version": (I32, []),
        "si_launch_count": (ctypes.c_uint64, []),
        "si_quant_mxfp8": (ctypes.c_int, [P, ctypes.c_int, I64, I32, P, P, P]),
        "si_indexer_topk": (ctypes.c_int, [B, IX, I32, P, P, SZ, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    _lib = lib
    return lib


# Loading is eager so that a missing library fails at import time.
load()

EXPORTED = ("si_workspace_size", "si_workspace_min", "si_indexer_scores", "si_topk",
            "si_sparse_attn", "si_fused_decode", "si_fused_decode_noalloc",
            "si_workspace_size_cand", "si_indexer_topk_cand", "si_workspace_status",
            "si_status_string",
            "si_last_error", "si_version", "si_launch_count", "si_quant_mxfp8",
            "si_indexer_topk")


def _check(status: int):
    if status != 0:
        raise SIError(status, load().si_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libsi must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ------------------------------------------------------------------ operands

@dataclasses.dataclass
class Batch:
    """Ragged batch over paged sequences (device int32 tensors)."""
    block_table: torch.Tensor   # [n_seq, max_blocks]
    ctx_len: torch.Tensor       # [n_seq]
    q_seq: torch.Tensor         # [n_q]
    q_pos: torch.Tensor         # [n_q]
    page_size: int
    max_ctx: int                # host-known bound of q_pos + 1
    n_blocks: int
    host_q_seq: Optional[object] = None  # host int32 copy of q_seq (numpy), lets prefill
                                         # chunks of a mixed batch take the prefill kernel

    def c(self) -> c_batch:
        hq = None
        if self.host_q_seq is not None:
            import numpy as np
            self._host_q_seq = np.ascontiguousarray(self.host_q_seq, dtype=np.int32)
            if self._host_q_seq.shape[0] != self.q_pos.shape[0]:
                raise ValueError("host_q_seq must have one entry per query row")
            hq = self._host_q_seq.ctypes.data
        return c_batch(_ptr(self.block_table), _ptr(self.ctx_len), _ptr(self.q_seq),
                       _ptr(self.q_pos), self.ctx_len.shape[0], self.block_table.shape[1],
                       self.q_pos.shape[0], self.page_size, self.max_ctx, self.n_blocks, hq)


@dataclasses.dataclass
class Paged:
    """Paged cache [n_blocks, page_size, row_stride] with optional scales: one
    per row, or one per `scale_tile` consecutive entries of a row."""
    data: torch.Tensor
    dtype: str                  # "f32" | "bf16" | "e4m3" | "e2m1" (two per byte) | "mxe4m3"
    row_dim: int
    scale: Optional[torch.Tensor] = None
    scale_tile: int = 0

    def c(self) -> c_paged:
        stride = self.data.shape[-1] * (2 if self.dtype == "e2m1" else 1)  # in elements
        # MXFP8 rows take one E8M0 byte per 32 entries
        tile = 32 if self.dtype == "mxe4m3" else self.scale_tile
        return c_paged(_ptr(self.data), _ptr(self.scale), DTYPES[self.dtype], self.row_dim,
                       stride, tile)


@dataclasses.dataclass
class Indexer:
    q: torch.Tensor             # [n_q, n_heads, head_dim]
    q_dtype: str
    w: torch.Tensor             # [n_q, n_heads] float32
    k: Paged
    q_scale: Optional[torch.Tensor] = None   # [n_q, n_heads] float32 for an e4m3 query,
                                             # [n_q, n_heads, head_dim / 32] uint8 for mxe4m3

    def c(self) -> c_indexer:
        return c_indexer(_ptr(self.q), DTYPES[self.q_dtype], _ptr(self.q_scale), _ptr(self.w),
                         self.q.shape[1], self.q.shape[2], self.k.c())


@dataclasses.dataclass
class Attention:
    q: torch.Tensor             # [n_q, n_heads, d_qk]
    q_dtype: str
    k: Paged
    v: Paged
    d_v: int
    softmax_scale: float

    def c(self) -> c_attention:
        return c_attention(_ptr(self.q), DTYPES[self.q_dtype], self.q.shape[1], self.q.shape[2],
                           self.d_v, self.k.c(), self.v.c(), self.softmax_scale)


def _ref(x):
    return None if x is None else ctypes.byref(x)


# ------------------------------------------------------------------ calls

def workspace_size(op: int, b: Batch, ix: Optional[Indexer] = None,
                   at: Optional[Attention] = None, k_top: int = 0) -> int:
    cb, ci, ca = b.c(), ix.c() if ix else None, at.c() if at else None
    return int(load().si_workspace_size(op, ctypes.byref(cb), _ref(ci), _ref(ca), k_top))


def workspace_min(op: int, b: Batch, ix: Optional[Indexer] = None,
                  at: Optional[Attention] = None, k_top: int = 0) -> int:
    cb, ci, ca = b.c(), ix.c() if ix else None, at.c() if at else None
    return int(load().si_workspace_min(op, ctypes.byref(cb), _ref(ci), _ref(ca), k_top))


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Zeroed workspace (the status word must start at 0); 256-byte aligned
    because the CUDA caching allocator aligns every block to at least 512."""
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)


def indexer_scores(b: Batch, ix: Indexer, scores: torch.Tensor, ws: torch.Tensor, stream=None):
    cb, ci = b.c(), ix.c()
    _check(load().si_indexer_scores(ctypes.byref(cb), ctypes.byref(ci), _ptr(scores),
                                    scores.shape[-1], _ptr(ws), ws.numel(), _stream(stream)))


def topk(b: Batch, scores: torch.Tensor, k_top: int, idx: torch.Tensor, ws: torch.Tensor,
         stream=None):
    cb = b.c()
    _check(load().si_topk(ctypes.byref(cb), _ptr(scores), scores.shape[-1], k_top, _ptr(idx),
                          _ptr(ws), ws.numel(), _stream(stream)))


def workspace_size_cand(b: Batch, ix: Indexer, n_cand: int) -> int:
    cb, ci = b.c(), ix.c()
    return int(load().si_workspace_size_cand(ctypes.byref(cb), ctypes.byref(ci), n_cand))


def indexer_topk_cand(b: Batch, ix: Indexer, cand: torch.Tensor, k_top: int, idx: torch.Tensor,
                      ws: torch.Tensor, scores: Optional[torch.Tensor] = None, stream=None):
    """Candidate-restricted selection: cand [n_q, n_cand] int32 positions per
    row (candidates first, strictly ascending; -1 or past the row after them)."""
    cb, ci = b.c(), ix.c()
    ld_s = scores.shape[-1] if scores is not None else 0
    _check(load().si_indexer_topk_cand(ctypes.byref(cb), ctypes.byref(ci), _ptr(cand),
                                       cand.shape[-1], cand.shape[-1], k_top, _ptr(idx),
                                       _ptr(scores), ld_s, _ptr(ws), ws.numel(),
                                       _stream(stream)))


def _out_dtype(out: torch.Tensor) -> int:
    if out.dtype == torch.float32:
        return F32
    if out.dtype == torch.bfloat16:
        return BF16
    raise ValueError(f"output dtype {out.dtype} not supported")


def sparse_attn(b: Batch, at: Attention, idx: torch.Tensor, k_top: int, out: torch.Tensor,
                ws: torch.Tensor, lse: Optional[torch.Tensor] = None, stream=None):
    cb, ca = b.c(), at.c()
    _check(load().si_sparse_attn(ctypes.byref(cb), ctypes.byref(ca), _ptr(idx), k_top, _ptr(out),
                                 _out_dtype(out), _ptr(lse), _ptr(ws), ws.numel(),
                                 _stream(stream)))


def indexer_topk(b: Batch, ix: Indexer, k_top: int, idx: torch.Tensor, ws: torch.Tensor,
                 stream=None):
    """Section 4.1's fused indexer operator: scores and Top-K in one call, the
    scores kept in the workspace (si_indexer_topk)."""
    _check(load().si_indexer_topk(ctypes.byref(b.c()), ctypes.byref(ix.c()), k_top, _ptr(idx),
                                  _ptr(ws), ws.numel(), _stream(stream)))


def fused_decode(b: Batch, ix: Indexer, at: Attention, k_top: int, idx: torch.Tensor,
                 out: torch.Tensor, ws: torch.Tensor, lse: Optional[torch.Tensor] = None,
                 stream=None):
    cb, ci, ca = b.c(), ix.c(), at.c()
    _check(load().si_fused_decode(ctypes.byref(cb), ctypes.byref(ci), ctypes.byref(ca), k_top,
                                  _ptr(idx), _ptr(out), _out_dtype(out), _ptr(lse), _ptr(ws),
                                  ws.numel(), _stream(stream)))


def fused_decode_noalloc(b: Batch, ix: Indexer, at: Attention, k_top: int, idx: torch.Tensor,
                         out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                         stream=None) -> int:
    """si_fused_decode_noalloc: the fused path on the library's static scratch
    (nothing is allocated).  Returns the scratch's device address, which
    ``workspace_status_at`` reads.  Overlapping calls on one device race."""
    cb, ci, ca = b.c(), ix.c(), at.c()
    scratch = ctypes.c_void_p(0)
    _check(load().si_fused_decode_noalloc(ctypes.byref(cb), ctypes.byref(ci), ctypes.byref(ca),
                                          k_top, _ptr(idx), _ptr(out), _out_dtype(out),
                                          _ptr(lse), ctypes.byref(scratch), _stream(stream)))
    return int(scratch.value or 0)


def quant_mxfp8(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, stream=None):
    """MXFP8 conversion of the rows of x ([..., dim], float32 or bfloat16, dim
    a multiple of 32) into codes (uint8, x's shape) and E8M0 scale bytes
    (uint8 [..., dim / 32]): si_quant_mxfp8."""
    dt = {torch.float32: F32, torch.bfloat16: BF16}.get(x.dtype)
    if dt is None:
        raise ValueError("x must be float32 or bfloat16")
    dim = x.shape[-1]
    n = x.numel() // dim if dim else 0
    if codes.dtype != torch.uint8 or scales.dtype != torch.uint8:
        raise ValueError("codes and scales are uint8")
    if codes.numel() != x.numel() or scales.numel() * 32 != x.numel():
        raise ValueError("codes / scales do not match x")
    _check(load().si_quant_mxfp8(_ptr(x), dt, n, dim, _ptr(codes), _ptr(scales),
                                 _stream(stream)))


def workspace_status_at(addr: int, stream=None) -> int:
    """Synchronise and return the device flags of the status word at `addr`."""
    flags = ctypes.c_uint32(0)
    st = load().si_workspace_status(addr, ctypes.byref(flags), _stream(stream))
    if st not in (0, 5):
        _check(st)
    return int(flags.value)


def launch_count() -> int:
    """Kernels launched by libsi in this process so far."""
    return int(load().si_launch_count())


def workspace_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronise and return the sticky device flags of a workspace."""
    flags = ctypes.c_uint32(0)
    st = load().si_workspace_status(_ptr(ws), ctypes.byref(flags), _stream(stream))
    if st not in (0, 5):
        _check(st)
    return int(flags.value)


# ---------------------------------------------------------- host -> device

@dataclasses.dataclass
class DeviceWorkload:
    """Device copies of a workload's arrays plus the ABI operand objects."""
    batch: Batch
    indexer: Indexer
    attention: Attention
    k_top: int
    n_q: int
    tensors: dict


def _dev(a, device, dtype=None):
    t = torch.from_numpy(a)
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device, non_blocking=False).contiguous()


def upload(wl, device="cuda") -> DeviceWorkload:
    """Copy the numpy arrays of a workload description (attributes as in the
    synthetic-input generator: block_table, ctx_len, q_seq, q_pos, q_idx, w,
    k_idx, k_scale, q, k, v, dtypes and sizes) to the device."""
    bf = torch.bfloat16
    ten = {}
    ten["block_table"] = _dev(wl.block_table, device)
    ten["ctx_len"] = _dev(wl.ctx_len, device)
    ten["q_seq"] = _dev(wl.q_seq, device)
    ten["q_pos"] = _dev(wl.q_pos, device)
    ten["q_idx"] = _dev(wl.q_idx, device, bf if wl.q_idx_dtype == "bf16" else None)
    q_scale = getattr(wl, "q_scale", None)
    ten["q_scale"] = None if q_scale is None else _dev(q_scale, device)
    ten["w"] = _dev(wl.w, device)
    ten["k_idx"] = _dev(wl.k_idx, device)
    ten["k_scale"] = None if wl.k_scale is None else _dev(wl.k_scale, device)
    kvt = bf if wl.kv_dtype == "bf16" else None
    qt = getattr(wl, "attn_q_dtype", "") or wl.kv_dtype
    ten["q"] = _dev(wl.q, device, bf if qt == "bf16" else None)
    ten["k"] = _dev(wl.k, device, kvt)
    ten["v"] = None if wl.v is None else _dev(wl.v, device, kvt)
    kv_scale = getattr(wl, "kv_scale", None)
    ten["kv_scale"] = None if kv_scale is None else _dev(kv_scale, device)
    tile = getattr(wl, "kv_scale_tile", 0) if kv_scale is not None else 0
    b = Batch(ten["block_table"], ten["ctx_len"], ten["q_seq"], ten["q_pos"], wl.page,
              wl.max_ctx, wl.n_blocks, host_q_seq=wl.q_seq)
    ix = Indexer(ten["q_idx"], wl.q_idx_dtype, ten["w"],
                 Paged(ten["k_idx"], wl.k_idx_dtype, wl.Di, ten["k_scale"]), ten["q_scale"])
    kp = Paged(ten["k"], wl.kv_dtype, wl.Dqk, ten["kv_scale"], tile)
    vp = kp if ten["v"] is None else Paged(ten["v"], wl.kv_dtype, wl.Dv)
    at = Attention(ten["q"], qt, kp, Paged(vp.data, vp.dtype, wl.Dv, vp.scale, vp.scale_tile),
                   wl.Dv, wl.scale)
    return DeviceWorkload(b, ix, at, wl.K, wl.n_q, ten)
