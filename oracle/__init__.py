"""CPU oracle for the indexer -> Top-K -> sparse-attention path.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``indexer_driven_top_gb300``) never imports it, and the two share no code.

The arithmetic lives in ``si_oracle.c`` (plain C, double precision, loops in
the order of the definitions); this module compiles it with gcc and wraps it
with ctypes over numpy arrays.  Each function follows the page "Day0 Inference
Support and Performance Optimization for New Architecture LLMs", section 2.2
(indexer scoring, head weighting, Top-K, sparse attention core) and section 4
(4.1 fused indexer over the paged K-cache, 4.2 index-based reading).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "si_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None
_lock = threading.Lock()

TYPE_CODE = {"f32": 0, "bf16": 1, "e4m3": 2, "e2m1": 3, "mxe4m3": 4}


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, -O2, no fast-math, no FMA contraction so that
    results are identical on x86-64 and aarch64 hosts)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Batch(ctypes.Structure):
    _fields_ = [("n_seq", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("page", ctypes.c_int32), ("n_q", ctypes.c_int32),
                ("block_table", ctypes.c_void_p), ("ctx_len", ctypes.c_void_p),
                ("q_seq", ctypes.c_void_p), ("q_pos", ctypes.c_void_p)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P, I32, I64, D = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.oracle_indexer_scores.argtypes = [P, P, I32, I32, I32, P, ctypes.c_int, P, P, P,
                                                  ctypes.c_int, P, I64, P, I64, ctypes.c_int]
            lib.oracle_topk.argtypes = [P, P, I32, P, I64, I32, P, P, ctypes.c_int]
            lib.oracle_topk_cand.argtypes = [P, P, I32, I32, I32, P, ctypes.c_int, P, P, P,
                                             ctypes.c_int, P, I64, P, I64, I32, I32, P, P, P,
                                             ctypes.c_int]
            lib.oracle_sparse_attn.argtypes = [P, P, I32, I32, I32, I32, P, ctypes.c_int, P, P,
                                               ctypes.c_int, I64, I64, P, P, I32, I32, I32, P,
                                               I32, D, P, P, ctypes.c_int]
            lib.oracle_indexer_scores_mx.argtypes = [P, P, I32, I32, I32, P, ctypes.c_int, P, P,
                                                     P, P, I64, P, I64, ctypes.c_int]
            lib.oracle_mx_quantize.argtypes = [P, ctypes.c_int, I64, I32, P, P]
            lib.orc_mx_group.argtypes = [P, P]
            lib.orc_mx_group.restype = ctypes.c_uint8
            lib.orc_f64_to_e4m3_sat.argtypes = [D]
            lib.orc_f64_to_e4m3_sat.restype = ctypes.c_uint8
            lib.orc_e8m0_to_f64.argtypes = [ctypes.c_uint8]
            lib.orc_e8m0_to_f64.restype = D
            lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_f64.restype = D
            lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_to_f64.restype = D
            lib.orc_e2m1_to_f64.argtypes = [ctypes.c_uint8]
            lib.orc_e2m1_to_f64.restype = D
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _c(a, dtype=None):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype) if dtype else np.ascontiguousarray(a)


class Batch:
    """Keeps the int32 arrays alive while the C structure points at them."""

    def __init__(self, block_table, ctx_len, q_seq, q_pos, page):
        self.block_table = _c(block_table, np.int32)
        self.ctx_len = _c(ctx_len, np.int32)
        self.q_seq = _c(q_seq, np.int32)
        self.q_pos = _c(q_pos, np.int32)
        self.s = _Batch(self.ctx_len.shape[0], self.block_table.shape[1], page,
                        self.q_pos.shape[0], _ptr(self.block_table), _ptr(self.ctx_len),
                        _ptr(self.q_seq), _ptr(self.q_pos))

    @classmethod
    def of(cls, wl) -> "Batch":
        return cls(wl.block_table, wl.ctx_len, wl.q_seq, wl.q_pos, wl.page)


def _rows(rows, n_q):
    if rows is None:
        return None, n_q
    r = _c(rows, np.int32)
    return r, int(r.shape[0])


def e4m3_to_f64(code: int) -> float:
    return _load().orc_e4m3_to_f64(code)


def e2m1_to_f64(code: int) -> float:
    return _load().orc_e2m1_to_f64(code)


def e8m0_to_f64(code: int) -> float:
    return _load().orc_e8m0_to_f64(code)


def f64_to_e4m3(x: float) -> int:
    """Nearest e4m3 code (ties to the even code, clamped to +-448, sign kept)."""
    return _load().orc_f64_to_e4m3_sat(float(x))


def mx_group(values):
    """One MXFP8 group of 32 values: (codes uint8 [32], scale byte)."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    assert v.shape == (32,)
    codes = np.empty(32, dtype=np.uint8)
    sb = _load().orc_mx_group(_ptr(v), _ptr(codes))
    return codes, int(sb)


def mx_quantize(x, x_type: str):
    """Rows of float32 values or bf16 bit patterns [..., dim] (dim a multiple
    of 32) to MXFP8: (codes uint8 [..., dim], scale bytes uint8 [..., dim / 32])."""
    x = _c(x)
    dim = int(x.shape[-1])
    n = int(x.size // dim) if dim else 0
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty(x.shape[:-1] + (dim // 32,), dtype=np.uint8)
    _load().oracle_mx_quantize(_ptr(x), TYPE_CODE[x_type], n, dim, _ptr(codes), _ptr(scales))
    return codes, scales


def _elem_stride(a, type_: str) -> int:
    """Row stride in elements of a cache array (e2m1 packs two per byte)."""
    return a.shape[-1] * (2 if type_ == "e2m1" else 1)


def bf16_to_f64(bits: int) -> float:
    return _load().orc_bf16_to_f64(bits)


def indexer_scores(b: Batch, q_idx, q_type: str, w, k, k_type: str, k_scale, Hi: int, Di: int,
                   ld: int, rows: Optional[Sequence[int]] = None, threads: Optional[int] = None,
                   q_scale=None):
    """score[i, s] = sum_h w[r,h] * ReLU(q_idx[r,h,:] . k[s,:]) for s <= pos(r),
    -inf beyond; r = rows[i].  Keys are dequantised as code * k_scale[row];
    with ``q_scale`` [n_q, Hi] the query too, as code * q_scale[r, h].
    MXFP8 keys (k_type "mxe4m3", k_scale the E8M0 bytes [..., Di / 32]) take
    an MXFP8 query (q_scale its bytes [n_q, Hi, Di / 32]) or a float32 / bf16
    one, converted per group of 32 first."""
    lib = _load()
    rr, n = _rows(rows, b.s.n_q)
    if k_type == "mxe4m3":
        q_idx, w, k = _c(q_idx), _c(w, np.float32), _c(k, np.uint8)
        k_mx = _c(k_scale, np.uint8)
        q_mx = None if q_type != "mxe4m3" else _c(q_scale, np.uint8)
        out = np.empty((n, ld), dtype=np.float64)
        lib.oracle_indexer_scores_mx(ctypes.byref(b.s), _ptr(rr), n, Hi, Di, _ptr(q_idx),
                                     TYPE_CODE[q_type], _ptr(q_mx), _ptr(w), _ptr(k), _ptr(k_mx),
                                     k.shape[-1], _ptr(out), ld, threads or default_threads())
        return out
    q_idx, w, k, k_scale = _c(q_idx), _c(w, np.float32), _c(k), _c(k_scale, np.float32)
    q_scale = None if q_scale is None else _c(q_scale, np.float32)
    out = np.empty((n, ld), dtype=np.float64)
    lib.oracle_indexer_scores(ctypes.byref(b.s), _ptr(rr), n, Hi, Di, _ptr(q_idx),
                              TYPE_CODE[q_type], _ptr(q_scale), _ptr(w), _ptr(k),
                              TYPE_CODE[k_type],
                              _ptr(k_scale), k.shape[-1], _ptr(out), ld,
                              threads or default_threads())
    return out


def topk(b: Batch, scores, K: int, rows: Optional[Sequence[int]] = None,
         threads: Optional[int] = None, return_kth: bool = False):
    """Indices of the K best scores per row (ties -> lower position), sorted
    ascending and padded with -1; all positions 0..pos when pos + 1 <= K.
    ``scores`` rows correspond to ``rows`` (or to all query rows)."""
    lib = _load()
    rr, n = _rows(rows, b.s.n_q)
    sc = _c(scores, np.float64)
    idx = np.empty((n, K), dtype=np.int32)
    kth = np.empty((n, 2), dtype=np.float64)
    lib.oracle_topk(ctypes.byref(b.s), _ptr(rr), n, _ptr(sc), sc.shape[1], K, _ptr(idx),
                    _ptr(kth), threads or default_threads())
    return (idx, kth) if return_kth else idx


def topk_cand(b: Batch, q_idx, q_type: str, w, k, k_type: str, k_scale, Hi: int, Di: int,
              cand, K: int, rows: Optional[Sequence[int]] = None, threads: Optional[int] = None,
              q_scale=None):
    """Candidate-restricted selection (the vLLM article on DeepSeek-V4.1,
    "Kernels": indexer logits over a fixed candidate set per query).  Row r's
    candidates are the entries s of cand[r] with 0 <= s <= pos(r); each is
    scored as in indexer_scores and the K best (ties -> lower position) are
    returned ascending, -1 padded.  Returns (idx [n, K], scores [n, n_cand]
    with -inf for list entries that are not candidates, kth [n, 2])."""
    lib = _load()
    rr, n = _rows(rows, b.s.n_q)
    q_idx, w, k, k_scale = _c(q_idx), _c(w, np.float32), _c(k), _c(k_scale, np.float32)
    q_scale = None if q_scale is None else _c(q_scale, np.float32)
    cd = _c(cand, np.int32)
    n_cand = int(cd.shape[1])
    idx = np.empty((n, K), dtype=np.int32)
    sc = np.empty((n, n_cand), dtype=np.float64)
    kth = np.empty((n, 2), dtype=np.float64)
    lib.oracle_topk_cand(ctypes.byref(b.s), _ptr(rr), n, Hi, Di, _ptr(q_idx), TYPE_CODE[q_type],
                         _ptr(q_scale), _ptr(w), _ptr(k), TYPE_CODE[k_type], _ptr(k_scale),
                         k.shape[-1], _ptr(cd), n_cand, n_cand, K, _ptr(idx), _ptr(sc), _ptr(kth),
                         threads or default_threads())
    return idx, sc, kth


def sparse_attn(b: Batch, q, q_type: str, k, v, kv_type: str, idx, K: int, Hq: int, Dqk: int,
                Dv: int, scale: float, rows: Optional[Sequence[int]] = None,
                threads: Optional[int] = None, q_dtype: Optional[str] = None, kv_scale=None,
                scale_tile: int = 0):
    """out[i, h] = softmax over the selected rows of scale * q . k, applied to
    the values; returns (out [n, Hq, Dv], lse [n, Hq]) in float64.  ``v=None``
    means the value row is the first Dv entries of the key row.  ``q_type`` is
    the storage type of q and of the caches, unless ``q_dtype`` gives q's own
    (FP8 caches with a bf16 query).  ``kv_scale`` [n_blocks, page, n_tiles]
    dequantises the key rows (and the value rows cut from them) per tile of
    ``scale_tile`` entries."""
    lib = _load()
    rr, n = _rows(rows, b.s.n_q)
    q, k = _c(q), _c(k)
    v = k if v is None else _c(v)
    ix = _c(idx, np.int32)
    ks = None if kv_scale is None else _c(kv_scale, np.float32)
    nsc = 0 if ks is None else int(ks.shape[-1]) if scale_tile > 0 else 1
    out = np.empty((n, Hq, Dv), dtype=np.float64)
    lse = np.empty((n, Hq), dtype=np.float64)
    lib.oracle_sparse_attn(ctypes.byref(b.s), _ptr(rr), n, Hq, Dqk, Dv, _ptr(q),
                           TYPE_CODE[q_dtype or q_type], _ptr(k), _ptr(v), TYPE_CODE[kv_type],
                           _elem_stride(k, kv_type), _elem_stride(v, kv_type), _ptr(ks), _ptr(ks),
                           scale_tile, nsc, nsc,
                           _ptr(ix), K, scale, _ptr(out), _ptr(lse), threads or default_threads())
    return out, lse


def attn_kv_args(wl) -> dict:
    """Keyword arguments of sparse_attn for a workload's KV storage: an FP8
    cache carries per-tile scales and a query of its own type."""
    if getattr(wl, "kv_scale", None) is None:
        return {}
    return {"q_dtype": wl.attn_q_dtype, "kv_scale": wl.kv_scale, "scale_tile": wl.kv_scale_tile}


def run(wl, rows: Optional[Sequence[int]] = None, threads: Optional[int] = None):
    """Whole path on a synthetic workload: (scores, idx, kth, out, lse) for the
    given query rows (default all)."""
    b = Batch.of(wl)
    ld = wl.max_ctx
    sc = indexer_scores(b, wl.q_idx, wl.q_idx_dtype, wl.w, wl.k_idx, wl.k_idx_dtype, wl.k_scale,
                        wl.Hi, wl.Di, ld, rows=rows, threads=threads,
                        q_scale=getattr(wl, "q_scale", None))
    idx, kth = topk(b, sc, wl.K, rows=rows, threads=threads, return_kth=True)
    out, lse = sparse_attn(b, wl.q, wl.kv_dtype, wl.k, wl.v, wl.kv_dtype, idx, wl.K, wl.Hq,
                           wl.Dqk, wl.Dv, wl.scale, rows=rows, threads=threads,
                           **attn_kv_args(wl))
    return sc, idx, kth, out, lse
