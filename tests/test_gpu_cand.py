"""Candidate-restricted selection on the GPU (si_indexer_topk_cand through the
C ABI) against the oracle, on seeded synthetic inputs.

The rule: row r's candidates are its list entries 0 <= s <= pos(r); the K
with the largest score win (ties -> lower position), written ascending and
-1 padded.  Top-K indices must equal the oracle's except inside the tie band
(1e-5 relative of the K-th candidate score, only when the K-th and (K+1)-th
lie within it); scores within 1e-5 of the row's largest."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import TOPK_REL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def si():
    import __graft_entry__
    __graft_entry__.build()
    import indexer_driven_top_gb300 as si
    return si


def _oracle(wl, cand, rows=None):
    return oracle.topk_cand(oracle.Batch.of(wl), wl.q_idx, wl.q_idx_dtype, wl.w, wl.k_idx,
                            wl.k_idx_dtype, wl.k_scale, wl.Hi, wl.Di, cand, wl.K, rows=rows,
                            q_scale=getattr(wl, "q_scale", None))


def _gpu(si, dw, wl, cand, scores=True, extra_cols=3):
    c = torch.from_numpy(np.ascontiguousarray(cand)).cuda()
    ws = si.alloc_workspace(si.workspace_size_cand(dw.batch, dw.indexer, cand.shape[1]))
    idx = torch.empty((wl.n_q, wl.K), dtype=torch.int32, device="cuda")
    sc = (torch.empty((wl.n_q, cand.shape[1] + extra_cols), dtype=torch.float32, device="cuda")
          if scores else None)
    si.indexer_topk_cand(dw.batch, dw.indexer, c, wl.K, idx, ws, scores=sc)
    flags = si.workspace_status(ws)
    return idx.cpu().numpy(), (sc.cpu().numpy() if scores else None), flags


def _check_row(g, o, cand_row, o_sc, pos, K):
    """Tie-aware comparison of one row's selection; returns the swaps."""
    valid = [(int(s), float(v)) for s, v in zip(cand_row, o_sc) if 0 <= s <= pos]
    n = min(K, len(valid))
    g = np.asarray(g)
    assert (g[n:] == -1).all(), "padding must be -1"
    gs = g[:n]
    by_pos = dict(valid)
    assert all(int(s) in by_pos for s in gs), "selected a position that is not a candidate"
    assert (np.diff(gs) > 0).all(), "positions must be strictly ascending"
    os_ = np.asarray(o)[:n]
    if np.array_equal(gs, os_):
        return 0
    srt = sorted((v for _, v in valid), reverse=True)
    th_k, th_k1 = srt[K - 1], srt[K]
    band = TOPK_REL * abs(th_k)
    assert th_k - th_k1 < band, f"differs although the K-th/K+1-th gap {th_k - th_k1} >= {band}"
    diff = np.setxor1d(gs, os_)
    assert all(abs(by_pos[int(s)] - th_k) <= band for s in diff), "swap outside the tie band"
    return len(diff) // 2


def _check(wl, cand, g_idx, g_sc, o_idx, o_sc, rows=None):
    rows = list(range(wl.n_q)) if rows is None else rows
    nc = cand.shape[1]
    for i, r in enumerate(rows):
        fin = np.isfinite(o_sc[i])
        if g_sc is not None:
            assert np.array_equal(np.isfinite(g_sc[r, :nc]), fin)
            assert np.isneginf(g_sc[r, :nc][~fin]).all() and np.isneginf(g_sc[r, nc:]).all()
            if fin.any():
                scale = np.abs(o_sc[i][fin]).max() + 1e-30
                assert np.abs(g_sc[r, :nc][fin] - o_sc[i][fin]).max() <= 1e-5 * scale
        _check_row(g_idx[r], o_idx[i], cand[r], o_sc[i], int(wl.q_pos[r]), wl.K)


def test_candidates_tensor_core_ragged_decode(si):
    """64 x 128 FP8-key indexer on the tensor cores: rows with more and fewer
    candidates than K, a list length that is not a multiple of the 128-slot
    page, and entries past each row's position."""
    wl = synth.make("c1", batch=4, ctx_list=[3001, 2048, 130, 40], K=256)
    cand = synth.candidates(wl, 700, seed=11, pad_beyond=5)
    dw = si.upload(wl)
    g_idx, g_sc, flags = _gpu(si, dw, wl, cand)
    assert flags == 0
    o_idx, o_sc, _ = _oracle(wl, cand)
    _check(wl, cand, g_idx, g_sc, o_idx, o_sc)


def test_candidates_fp8_query(si):
    wl = synth.make("c1", batch=3, ctx_list=[5000, 1500, 300], K=128, q_idx_fp8=True)
    cand = synth.candidates(wl, 1000, seed=4)
    dw = si.upload(wl)
    g_idx, g_sc, flags = _gpu(si, dw, wl, cand)
    assert flags == 0
    o_idx, o_sc, _ = _oracle(wl, cand)
    _check(wl, cand, g_idx, g_sc, o_idx, o_sc)


def test_candidates_cuda_core_indexer_fp32(si):
    """Shapes the tensor-core indexer does not take (fp32, 4 heads x 32): the
    CUDA-core indexer, whose empty slots are masked to -inf; many rows have
    fewer candidates than K; no score buffer passed."""
    wl = synth.make("c0")
    cand = synth.candidates(wl, 100, seed=2, pad_beyond=4)
    dw = si.upload(wl)
    g_idx, _, flags = _gpu(si, dw, wl, cand, scores=False)
    assert flags == 0
    o_idx, o_sc, _ = _oracle(wl, cand)
    _check(wl, cand, g_idx, None, o_idx, o_sc)
    g_idx2, g_sc, _ = _gpu(si, dw, wl, cand)
    assert np.array_equal(g_idx2, g_idx)
    _check(wl, cand, g_idx2, g_sc, o_idx, o_sc)


def test_all_positions_as_candidates_equal_unrestricted_selection(si):
    """Listing every position reproduces the full-context path bit for bit
    (the same kernels score the same key bytes)."""
    wl = synth.make("c1", batch=3, ctx_list=[3001, 2048, 130], K=512)
    dw = si.upload(wl)
    ld = wl.max_ctx
    ws = si.alloc_workspace(si.workspace_size(si.OP_FUSED, dw.batch, dw.indexer, dw.attention,
                                              wl.K))
    scores = torch.empty((wl.n_q, ld), dtype=torch.float32, device="cuda")
    idx = torch.empty((wl.n_q, wl.K), dtype=torch.int32, device="cuda")
    si.indexer_scores(dw.batch, dw.indexer, scores, ws)
    si.topk(dw.batch, scores, wl.K, idx, ws)
    cand = np.tile(np.arange(ld, dtype=np.int32), (wl.n_q, 1))
    g_idx, g_sc, flags = _gpu(si, dw, wl, cand, extra_cols=0)
    assert flags == 0
    assert np.array_equal(g_idx, idx.cpu().numpy())
    assert np.array_equal(g_sc, scores.cpu().numpy())


def test_single_candidate_and_empty_lists(si):
    """A list of one entry; rows whose only entry is -1 or past the row."""
    wl = synth.make("c1", batch=3, ctx_list=[900, 500, 200], K=8)
    cand = np.array([[450], [-1], [199 + 5]], dtype=np.int32)
    dw = si.upload(wl)
    g_idx, g_sc, flags = _gpu(si, dw, wl, cand)
    assert flags == 0
    assert g_idx[0].tolist() == [450] + [-1] * 7
    assert (g_idx[1:] == -1).all()
    assert np.isfinite(g_sc[0, 0]) and np.isneginf(g_sc[1:, 0]).all()
    o_idx, o_sc, _ = _oracle(wl, cand)
    _check(wl, cand, g_idx, g_sc, o_idx, o_sc)


def test_candidates_out_of_order_raise_flag(si):
    """A list whose candidates are not strictly ascending is reported in the
    status word (host-made error; nothing faults)."""
    wl = synth.make("c1", batch=2, ctx_list=[900, 500], K=8)
    cand = synth.candidates(wl, 40, seed=9)
    cand[1, [3, 4]] = cand[1, [4, 3]]
    dw = si.upload(wl)
    _, _, flags = _gpu(si, dw, wl, cand)
    assert flags & si.DEVFLAG_BAD_INDEX


def test_candidates_long_context_full_size(si):
    """Decode batch 16 x context 131072 with 1 % planted keys, 16384
    candidates per row (the fixed candidate-set size of the vLLM article's
    measurement), K = 2048: every row against the oracle."""
    wl = synth.make("c3")
    cand = synth.candidates(wl, 16384, seed=31)
    dw = si.upload(wl)
    g_idx, g_sc, flags = _gpu(si, dw, wl, cand)
    assert flags == 0
    o_idx, o_sc, _ = _oracle(wl, cand)
    _check(wl, cand, g_idx, g_sc, o_idx, o_sc)


def test_long_candidate_lists_take_cluster_top_k(si):
    """40000 candidates per row on two rows: the Top-K over the candidate
    slots runs as a cluster of three CTAs per row."""
    wl = synth.make("c3", batch=2, ctx=60000, K=2048, Hq=1, Dqk=16, Dv=8)
    cand = synth.candidates(wl, 40000, seed=13)
    dw = si.upload(wl)
    g_idx, g_sc, flags = _gpu(si, dw, wl, cand)
    assert flags == 0
    o_idx, o_sc, _ = _oracle(wl, cand)
    _check(wl, cand, g_idx, g_sc, o_idx, o_sc)


def test_many_long_candidate_lists_take_one_cta_per_row(si):
    """160 rows with 17000 candidates each: too many rows for a cluster of
    several CTAs per row, so each row's slots take one CTA that caches 32
    keys per thread in shared memory.  Indexer shapes of 4 heads x 32 take the
    gather kernel and the CUDA-core indexer.  Eight sampled rows are checked
    against the oracle."""
    wl = synth.make("c1", batch=160, ctx=17500, K=512, Hi=4, Di=32, Hq=1, Dqk=16, Dv=8)
    cand = synth.candidates(wl, 17000, seed=17)
    dw = si.upload(wl)
    g_idx, g_sc, flags = _gpu(si, dw, wl, cand)
    assert flags == 0
    rows = [0, 1, 37, 80, 81, 120, 158, 159]
    o_idx, o_sc, _ = _oracle(wl, cand, rows=rows)
    _check(wl, cand, g_idx, g_sc, o_idx, o_sc, rows=rows)
