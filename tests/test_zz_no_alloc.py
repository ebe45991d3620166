"""si_fused_decode_noalloc: the fused path on the library's static scratch.

It must agree with si_fused_decode (which takes a caller workspace) within the
parity tolerance, call after call, and refuse requests whose score strip does
not fit the scratch before touching the GPU.  This file sorts last so that its
GPU tests also run after every other test has used the library in the same
process.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from _parity import ATOL_BF16, ATOL_F32, max_abs

SCRATCH = 8 << 20  # SI_NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module")
def si():
    import __graft_entry__
    __graft_entry__.build()
    import indexer_driven_top_gb300 as si
    return si


def test_oversize_request_is_refused_on_the_host(si):
    """max_ctx beyond what one score row of the scratch holds: SI_ERR_WORKSPACE,
    decided by host arithmetic alone (the pointers are never dereferenced)."""
    lib = si.load()
    fake = 1 << 20
    max_ctx = (SCRATCH - 256) // 4 + 64       # one 64-position step past the limit
    page = 64
    blocks = (max_ctx + page - 1) // page
    b = si.c_batch(fake, fake, fake, fake, 1, blocks, 1, page, max_ctx, blocks)
    kp = si.c_paged(fake, None, si.E4M3, 128, 128)
    ix = si.c_indexer(fake, si.BF16, None, fake, 64, 128, kp)
    ap = si.c_paged(fake, None, si.BF16, 576, 576)
    at = si.c_attention(fake, si.BF16, 128, 576, 512, ap, ap, 0.04)
    scratch = ctypes.c_void_p(123)
    st = lib.si_fused_decode_noalloc(ctypes.byref(b), ctypes.byref(ix), ctypes.byref(at), 2048,
                                     ctypes.c_void_p(fake), ctypes.c_void_p(fake), si.F32, None,
                                     ctypes.byref(scratch), None)
    assert st == 3
    assert b"static scratch" in lib.si_last_error()
    assert not scratch.value
    # invalid arguments are reported as si_fused_decode reports them
    b.max_ctx = 256
    st = lib.si_fused_decode_noalloc(ctypes.byref(b), ctypes.byref(ix), ctypes.byref(at), 0,
                                     ctypes.c_void_p(fake), ctypes.c_void_p(fake), si.F32, None,
                                     None, None)
    assert st == 1


def _fused_ws(si, dw, out_dtype):
    ws = si.alloc_workspace(si.workspace_size(si.OP_FUSED, dw.batch, dw.indexer, dw.attention,
                                              dw.k_top))
    idx = torch.empty((dw.n_q, dw.k_top), dtype=torch.int32, device="cuda")
    out = torch.empty((dw.n_q, dw.attention.q.shape[1], dw.attention.d_v), dtype=out_dtype,
                      device="cuda")
    si.fused_decode(dw.batch, dw.indexer, dw.attention, dw.k_top, idx, out, ws)
    assert si.workspace_status(ws) == 0
    return idx.cpu().numpy(), out.float().cpu().numpy()


def _noalloc(si, dw, out_dtype):
    idx = torch.full((dw.n_q, dw.k_top), 7, dtype=torch.int32, device="cuda")
    out = torch.full((dw.n_q, dw.attention.q.shape[1], dw.attention.d_v), 3.0, dtype=out_dtype,
                     device="cuda")
    addr = si.fused_decode_noalloc(dw.batch, dw.indexer, dw.attention, dw.k_top, idx, out)
    assert addr != 0 and addr % 256 == 0
    assert si.workspace_status_at(addr) == 0
    return idx.cpu().numpy(), out.float().cpu().numpy(), addr


def _compare_twice(si, wl, out_dtype, atol):
    dw = si.upload(wl)
    r_idx, r_out = _fused_ws(si, dw, out_dtype)
    addrs = []
    for _ in range(2):
        n_idx, n_out, addr = _noalloc(si, dw, out_dtype)
        addrs.append(addr)
        assert np.array_equal(n_idx, r_idx)
        assert max_abs(n_out, r_out) <= atol
    assert addrs[0] == addrs[1]   # one scratch per device, looked up once


@pytest.mark.gpu
def test_noalloc_matches_fused_decode_tensor_core_path(si):
    """Decode rows on the tensor-core kernels (64 x 128 indexer, 128 x 576 attention)."""
    wl = synth.make("c1", batch=3, ctx_list=[3001, 2048, 130], K=2048)
    _compare_twice(si, wl, torch.float32, ATOL_BF16)


@pytest.mark.gpu
def test_noalloc_matches_fused_decode_strips(si):
    """Contexts long enough that the scratch holds fewer score rows (6) than
    the batch has (8): the fused call walks the rows in two strips."""
    wl = synth.make("c1", ctx_list=[300000, 1000, 5000, 70000, 299999, 12, 64, 200000],
                    K=256, Hi=4, Di=32, Hq=4, Dqk=64, Dv=32)
    assert (SCRATCH - 256) // (4 * ((wl.max_ctx + 63) // 64 * 64)) < wl.n_q
    _compare_twice(si, wl, torch.float32, ATOL_BF16)


@pytest.mark.gpu
def test_noalloc_matches_fused_decode_fp32_prefill(si):
    wl = synth.make("c0")
    _compare_twice(si, wl, torch.float32, ATOL_F32)
