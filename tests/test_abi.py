"""The C-ABI library loads, exports every symbol include/si.h declares, and
rejects bad arguments on the host before touching the GPU."""
import ctypes
import os
import re

import pytest

import __graft_entry__

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def si():
    __graft_entry__.build()
    import indexer_driven_top_gb300 as si
    return si


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(si_[a-z0-9_]+)\s*\(", txt))
    return names


def test_every_declared_symbol_is_exported(si):
    names = _declared()
    assert {"si_indexer_scores", "si_topk", "si_sparse_attn", "si_fused_decode"} <= names
    lib = si.load()
    for n in names:
        assert hasattr(lib, n), n
    assert set(si.EXPORTED) <= names


def test_version_and_status_strings(si):
    lib = si.load()
    assert lib.si_version() == 5
    assert lib.si_status_string(0) == b"ok"
    assert lib.si_status_string(3) == b"workspace error"


def _batch(si, **kw):
    b = si.c_batch(1 << 20, 2 << 20, 3 << 20, 4 << 20, 1, 4, 2, 64, 256, 4)
    for k, v in kw.items():
        setattr(b, k, v)
    return b


def test_host_validation_rejects_bad_arguments(si):
    lib = si.load()
    P = ctypes.c_void_p
    fake = 1 << 20
    ws = 256 << 20   # 256-aligned fake device address, never dereferenced
    # NULL batch
    assert lib.si_topk(None, P(fake), 256, 8, P(fake), P(ws), 4096, None) == 1
    # k_top out of range
    assert lib.si_topk(ctypes.byref(_batch(si)), P(fake), 256, 0, P(fake), P(ws), 4096, None) == 1
    # ld_scores below max_ctx
    assert lib.si_topk(ctypes.byref(_batch(si)), P(fake), 100, 8, P(fake), P(ws), 4096, None) == 1
    assert b"ld_scores" in lib.si_last_error()
    # max_ctx beyond the block table
    assert lib.si_topk(ctypes.byref(_batch(si, max_ctx=999)), P(fake), 1024, 8, P(fake), P(ws),
                       4096, None) == 1
    # workspace: NULL, misaligned, too small
    b = ctypes.byref(_batch(si))
    assert lib.si_topk(b, P(fake), 256, 8, P(fake), None, 4096, None) == 3
    assert lib.si_topk(b, P(fake), 256, 8, P(fake), P(ws + 16), 4096, None) == 3
    assert lib.si_topk(b, P(fake), 256, 8, P(fake), P(ws), 16, None) == 3
    # attention: dtype mismatch, FP8 caches without scales, bad dims
    kp = si.c_paged(fake, None, si.F32, 64, 64)
    at = si.c_attention(fake, si.BF16, 4, 64, 64, kp, kp, 0.125)
    assert lib.si_sparse_attn(b, ctypes.byref(at), P(fake), 8, P(fake), si.F32, None, P(ws),
                              4096, None) == 2
    kp = si.c_paged(fake, None, si.E4M3, 64, 64)
    at = si.c_attention(fake, si.BF16, 4, 64, 64, kp, kp, 0.125)
    assert lib.si_sparse_attn(b, ctypes.byref(at), P(fake), 8, P(fake), si.F32, None, P(ws),
                              4096, None) == 1
    assert b"need scales" in lib.si_last_error()
    kp = si.c_paged(fake, None, si.E4M3, 64, 64, 32)      # tiles of 32 entries without scales
    at = si.c_attention(fake, si.BF16, 4, 64, 64, kp, kp, 0.125)
    assert lib.si_sparse_attn(b, ctypes.byref(at), P(fake), 8, P(fake), si.F32, None, P(ws),
                              4096, None) == 1
    kp = si.c_paged(fake, None, si.BF16, 64, 64)
    at = si.c_attention(fake, si.BF16, 4, 2000, 64, kp, kp, 0.125)
    assert lib.si_sparse_attn(b, ctypes.byref(at), P(fake), 8, P(fake), si.F32, None, P(ws),
                              4096, None) == 1
    # indexer: misaligned key cache, bad head count
    kp8 = si.c_paged(fake, None, si.E4M3, 128, 128)
    ix = si.c_indexer(fake, si.BF16, None, fake, 64, 128,
                      si.c_paged(fake + 3, None, si.E4M3, 128, 128))
    assert lib.si_indexer_scores(b, ctypes.byref(ix), P(fake), 256, P(ws), 4096, None) == 1
    # an FP8 query without its scale
    ix = si.c_indexer(fake, si.E4M3, None, fake, 64, 128, kp8)
    assert lib.si_indexer_scores(b, ctypes.byref(ix), P(fake), 256, P(ws), 4096, None) == 1
    assert b"q_scale" in lib.si_last_error()
    ix = si.c_indexer(fake, si.BF16, None, fake, 0, 128, si.c_paged(fake, None, si.E4M3, 128, 128))
    assert lib.si_indexer_scores(b, ctypes.byref(ix), P(fake), 256, P(ws), 4096, None) == 1
    # empty batch is a no-op that succeeds without touching anything
    assert lib.si_topk(ctypes.byref(_batch(si, n_q=0)), None, 0, 8, None, None, 0, None) == 0


def test_workspace_sizes(si):
    lib = si.load()
    b = _batch(si)
    fused = lib.si_workspace_size(3, ctypes.byref(b), None, None, 8)
    mn = lib.si_workspace_min(3, ctypes.byref(b), None, None, 8)
    assert fused >= mn >= 256 + 256 * 4
    assert lib.si_workspace_size(1, None, None, None, 8) == 0


def test_candidate_selection_host_validation_and_sizes(si):
    """si_indexer_topk_cand rejects bad lists, strides and workspaces on the
    host; its workspace holds the gathered rows, scales and scores."""
    lib = si.load()
    P = ctypes.c_void_p
    fake = 1 << 20
    ws = 256 << 20
    b = ctypes.byref(_batch(si))
    ix = si.c_indexer(fake, si.BF16, None, fake, 64, 128, si.c_paged(fake, None, si.E4M3, 128, 128))
    need = lib.si_workspace_size_cand(b, ctypes.byref(ix), 300)
    # 64 x 128 FP8 keys: the tensor-core indexer gathers the candidates itself,
    # the workspace holds the status word and 2 rows x 320 scores (2560 bytes,
    # a multiple of the 256-byte region alignment)
    assert need == 256 + 2 * 320 * 4
    # other shapes gather them into the workspace first: 2 rows x 384 slots x
    # (128-byte f32 key row + 4-byte scale) besides the scores
    ixf = si.c_indexer(fake, si.F32, None, fake, 4, 32, si.c_paged(fake, None, si.F32, 32, 32))
    assert lib.si_workspace_size_cand(b, ctypes.byref(ixf), 300) >= 256 + 2 * 384 * (128 + 4) + 2 * 320 * 4
    assert lib.si_workspace_size_cand(b, ctypes.byref(ix), 0) == 0
    args = lambda **kw: dict(dict(cand=P(fake), n_cand=300, ld_cand=300, k_top=8, idx=P(fake),
                                  scores=None, ld_scores=0, ws=P(ws), ws_bytes=need), **kw)

    def call(**kw):
        a = args(**kw)
        return lib.si_indexer_topk_cand(b, ctypes.byref(ix), a["cand"], a["n_cand"], a["ld_cand"],
                                        a["k_top"], a["idx"], a["scores"], a["ld_scores"],
                                        a["ws"], a["ws_bytes"], None)
    assert call(cand=None) == 1
    assert call(n_cand=0) == 1
    assert call(ld_cand=299) == 1 and b"ld_cand" in lib.si_last_error()
    assert call(scores=P(fake), ld_scores=100) == 1 and b"ld_scores" in lib.si_last_error()
    assert call(k_top=0) == 1
    assert call(ws_bytes=need - 1) == 3
    assert call(ws=P(ws + 16)) == 3
    assert lib.si_indexer_topk_cand(ctypes.byref(_batch(si, n_q=0)), ctypes.byref(ix), None, 0, 0,
                                    8, None, None, 0, None, 0, None) == 0


def test_fp4_cache_host_validation(si):
    """SI_E2M1 (FP4 codes, two per byte) is accepted for attention caches with
    per-tile scales and an even row stride, and refused elsewhere."""
    lib = si.load()
    P = ctypes.c_void_p
    fake = 1 << 20
    ws = 256 << 20
    b = ctypes.byref(_batch(si))
    E2M1 = 3
    # no per-tile scales
    kp = si.c_paged(fake, None, E2M1, 64, 64)
    at = si.c_attention(fake, si.BF16, 4, 64, 64, kp, kp, 0.125)
    assert lib.si_sparse_attn(b, ctypes.byref(at), P(fake), 8, P(fake), si.F32, None, P(ws),
                              4096, None) == 1
    assert b"e2m1" in lib.si_last_error()
    # odd row stride
    kp = si.c_paged(fake, fake, E2M1, 63, 63, 16)
    at = si.c_attention(fake, si.BF16, 4, 63, 63, kp, kp, 0.125)
    assert lib.si_sparse_attn(b, ctypes.byref(at), P(fake), 8, P(fake), si.F32, None, P(ws),
                              4096, None) == 1
    # FP4 indexer keys are not supported
    ix = si.c_indexer(fake, si.BF16, None, fake, 4, 32, si.c_paged(fake, fake, E2M1, 32, 32, 16))
    assert lib.si_indexer_scores(b, ctypes.byref(ix), P(fake), 256, P(ws), 4096, None) in (1, 2)
    # FP4 keys and bf16 values do not mix
    kp = si.c_paged(fake, fake, E2M1, 64, 64, 16)
    vp = si.c_paged(fake, None, si.BF16, 64, 64)
    at = si.c_attention(fake, si.BF16, 4, 64, 64, kp, vp, 0.125)
    assert lib.si_sparse_attn(b, ctypes.byref(at), P(fake), 8, P(fake), si.F32, None, P(ws),
                              4096, None) == 2


def test_mxfp8_host_validation(si):
    """SI_MXE4M3 (section 5.1's MXFP8 indexer format): keys need E8M0 scales
    with scale_tile 32, head_dim a multiple of 32, and an mxe4m3, bf16 or f32
    query; an mxe4m3 query needs MXFP8 keys; candidate lists refuse MXFP8
    keys; attention caches refuse it.  si_quant_mxfp8 validates its shape,
    dtype and alignment before any launch."""
    lib = si.load()
    P = ctypes.c_void_p
    fake = 1 << 20
    ws = 256 << 20
    b = ctypes.byref(_batch(si))
    MX = si.MXE4M3
    good_k = si.c_paged(fake, fake, MX, 128, 128, 32)
    # scales missing, wrong tile, ragged stride
    for kp in (si.c_paged(fake, None, MX, 128, 128, 32), si.c_paged(fake, fake, MX, 128, 128, 0),
               si.c_paged(fake, fake, MX, 100, 100, 32)):
        ix = si.c_indexer(fake, si.BF16, None, fake, 64, 128, kp)
        assert lib.si_indexer_scores(b, ctypes.byref(ix), P(fake), 256, P(ws), 4096, None) == 1
        assert b"MXFP8" in lib.si_last_error()
    # head_dim not a multiple of 32
    ix = si.c_indexer(fake, si.BF16, None, fake, 4, 48, si.c_paged(fake, fake, MX, 64, 64, 32))
    assert lib.si_indexer_scores(b, ctypes.byref(ix), P(fake), 256, P(ws), 4096, None) == 1
    # an e4m3 (per-head scale) query with MXFP8 keys; an MX query with FP8 keys
    ix = si.c_indexer(fake, si.E4M3, fake, fake, 64, 128, good_k)
    assert lib.si_indexer_scores(b, ctypes.byref(ix), P(fake), 256, P(ws), 4096, None) == 2
    ix = si.c_indexer(fake, MX, fake, fake, 64, 128, si.c_paged(fake, fake, si.E4M3, 128, 128))
    assert lib.si_indexer_scores(b, ctypes.byref(ix), P(fake), 256, P(ws), 4096, None) == 2
    # an MX query without its scale bytes
    ix = si.c_indexer(fake, MX, None, fake, 64, 128, good_k)
    assert lib.si_indexer_scores(b, ctypes.byref(ix), P(fake), 256, P(ws), 4096, None) == 1
    # candidate lists
    ix = si.c_indexer(fake, si.BF16, None, fake, 64, 128, good_k)
    assert lib.si_workspace_size_cand(b, ctypes.byref(ix), 300) == 0
    assert lib.si_indexer_topk_cand(b, ctypes.byref(ix), P(fake), 300, 300, 8, P(fake), None, 0,
                                    P(ws), 1 << 20, None) == 2
    # attention caches
    at = si.c_attention(fake, si.BF16, 4, 64, 64, si.c_paged(fake, fake, MX, 64, 64, 32),
                        si.c_paged(fake, fake, MX, 64, 64, 32), 0.125)
    assert lib.si_sparse_attn(b, ctypes.byref(at), P(fake), 8, P(fake), si.F32, None, P(ws),
                              4096, None) == 2
    # si_quant_mxfp8
    q = lib.si_quant_mxfp8
    assert q(P(fake), si.BF16, 4, 48, P(fake), P(fake), None) == 1          # dim % 32
    assert q(P(fake), si.BF16, 4, 0, P(fake), P(fake), None) == 1
    assert q(P(fake), si.E4M3, 4, 64, P(fake), P(fake), None) == 1          # dtype
    assert q(P(fake + 8), si.BF16, 4, 64, P(fake), P(fake), None) == 1      # alignment
    assert q(None, si.BF16, 4, 64, P(fake), P(fake), None) == 1
    assert q(P(fake), si.BF16, -1, 64, P(fake), P(fake), None) == 1
    assert q(None, si.BF16, 0, 64, None, None, None) == 0                    # empty: no-op


def test_binding_refuses_to_import_without_the_library(tmp_path):
    """No fallback: the Python binding, copied without libsi.so, raises at
    import instead of running anything on the CPU."""
    import shutil
    import subprocess
    import sys
    pkg = tmp_path / "indexer_driven_top_gb300"
    pkg.mkdir()
    for fn in ("__init__.py", "_build.py"):
        shutil.copy(os.path.join(ROOT, "indexer_driven_top_gb300", fn), pkg / fn)
    code = ("import sys; sys.path.insert(0, sys.argv[1]); "
            "import indexer_driven_top_gb300")
    r = subprocess.run([sys.executable, "-c", code, str(tmp_path)], capture_output=True,
                       text=True, timeout=600)
    assert r.returncode != 0
    assert "libsi.so is not built" in r.stderr
