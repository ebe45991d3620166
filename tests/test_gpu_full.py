"""Parity at full size: the decode workload the benchmark times (batch 64 x
context 8192, indexer 64 x 128 FP8, Top-K 2048, 128 heads over 576-dim latent
rows), run through exactly the calls the benchmark makes, checked against the
oracle on every query row.  The long-context decode (16 x 131072) is checked on
every row too; the causal prefill of 16384 on 256+ rows spread over the zigzag
pairs of row blocks the prefill indexer deals out, and the mixed batch on all
of its decode rows plus 64 rows of each prefill chunk.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import ATOL_BF16, check_topk, max_abs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def si():
    import __graft_entry__
    __graft_entry__.build()
    import indexer_driven_top_gb300 as si
    return si


def _separate(si, dw):
    """The benchmark's timed step: scores, Top-K, attention as three calls."""
    b = dw.batch
    ws = si.alloc_workspace(si.workspace_size(si.OP_FUSED, b, dw.indexer, dw.attention, dw.k_top))
    scores = torch.empty((dw.n_q, b.max_ctx), dtype=torch.float32, device="cuda")
    idx = torch.empty((dw.n_q, dw.k_top), dtype=torch.int32, device="cuda")
    out = torch.empty((dw.n_q, dw.attention.q.shape[1], dw.attention.d_v), dtype=torch.float32,
                      device="cuda")
    si.indexer_scores(b, dw.indexer, scores, ws)
    si.topk(b, scores, dw.k_top, idx, ws)
    si.sparse_attn(b, dw.attention, idx, dw.k_top, out, ws)
    assert si.workspace_status(ws) == 0
    return scores, idx, out


def _fused(si, dw):
    """The end-to-end call: si_fused_decode with a workspace."""
    b = dw.batch
    ws = si.alloc_workspace(si.workspace_size(si.OP_FUSED, b, dw.indexer, dw.attention, dw.k_top))
    idx = torch.empty((dw.n_q, dw.k_top), dtype=torch.int32, device="cuda")
    out = torch.empty((dw.n_q, dw.attention.q.shape[1], dw.attention.d_v), dtype=torch.float32,
                      device="cuda")
    si.fused_decode(b, dw.indexer, dw.attention, dw.k_top, idx, out, ws)
    assert si.workspace_status(ws) == 0
    return idx, out


def _check_rows(wl, rows, g_scores, g_idx, g_out):
    """Oracle on the sampled rows only; scores, Top-K and attention."""
    o_sc, o_idx, _, _, _ = oracle.run(wl, rows=rows)
    for i, r in enumerate(rows):
        o = o_sc[i]
        fin = np.isfinite(o)
        g = g_scores[r][: len(o)]
        assert np.array_equal(np.isfinite(g), fin)
        assert np.abs(g[fin] - o[fin]).max() <= 1e-5 * (np.abs(o[fin]).max() + 1e-30)
    check_topk(g_idx[rows], o_idx, o_sc, wl.q_pos, wl.K, rows=rows)
    # row i of the index list belongs to rows[i]
    ref, _ = oracle.sparse_attn(oracle.Batch.of(wl), wl.q, wl.kv_dtype, wl.k, wl.v, wl.kv_dtype,
                                g_idx[rows], wl.K, wl.Hq, wl.Dqk, wl.Dv, wl.scale, rows=rows,
                                **oracle.attn_kv_args(wl))
    assert max_abs(g_out[rows], ref) <= ATOL_BF16


def _run(si, wl, rows):
    dw = si.upload(wl)
    scores, idx, out = _separate(si, dw)
    g_scores, g_idx, g_out = scores.cpu().numpy(), idx.cpu().numpy(), out.cpu().numpy()
    _check_rows(wl, rows, g_scores, g_idx, g_out)
    f_idx, f_out = _fused(si, dw)
    assert np.array_equal(f_idx.cpu().numpy(), g_idx)
    assert max_abs(f_out.cpu().numpy(), g_out) <= ATOL_BF16
    return dw


def test_benchmark_workload_full_size_all_rows(si):
    wl = synth.make("c1")
    assert wl.n_q == 64 and wl.max_ctx == 8192 and wl.K == 2048
    _run(si, wl, rows=list(range(wl.n_q)))


def _bf16_step(x):
    """Spacing of bfloat16 numbers (8 significant bits) around |x|."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def test_benchmark_workload_bf16_output(si):
    """The benchmarked decode step writes its output in bf16, the activation
    type the output projection consumes.  Bound: the fp32-output tolerance
    plus half a bf16 step of the exact value (the final rounding)."""
    wl = synth.make("c1")
    dw = si.upload(wl)
    b = dw.batch
    ws = si.alloc_workspace(si.workspace_size(si.OP_FUSED, b, dw.indexer, dw.attention, dw.k_top))
    scores = torch.empty((dw.n_q, b.max_ctx), dtype=torch.float32, device="cuda")
    idx = torch.empty((dw.n_q, dw.k_top), dtype=torch.int32, device="cuda")
    out = torch.empty((dw.n_q, wl.Hq, wl.Dv), dtype=torch.bfloat16, device="cuda")
    si.indexer_scores(b, dw.indexer, scores, ws)
    si.topk(b, scores, dw.k_top, idx, ws)
    si.sparse_attn(b, dw.attention, idx, dw.k_top, out, ws)
    assert si.workspace_status(ws) == 0
    rows = list(range(wl.n_q))
    g_idx = idx.cpu().numpy()
    g_out = out.float().cpu().numpy()
    ref, _ = oracle.sparse_attn(oracle.Batch.of(wl), wl.q, wl.kv_dtype, wl.k, wl.v, wl.kv_dtype,
                                g_idx[rows], wl.K, wl.Hq, wl.Dqk, wl.Dv, wl.scale, rows=rows,
                                **oracle.attn_kv_args(wl))
    err = np.abs(g_out[rows] - ref)
    assert (err <= ATOL_BF16 + 0.5 * _bf16_step(ref)).all(), float(err.max())
    # the fused call writes the same bf16 values
    f_idx = torch.empty_like(idx)
    f_out = torch.empty_like(out)
    si.fused_decode(b, dw.indexer, dw.attention, dw.k_top, f_idx, f_out, ws)
    assert si.workspace_status(ws) == 0
    assert torch.equal(f_idx, idx) and torch.equal(f_out, out)


def test_long_context_planted_full_size(si):
    """Batch 16 x context 131072 with 1 % planted keys, every row; Top-K over
    131072 scores takes the cluster path, attention the split one."""
    wl = synth.make("c3")
    assert wl.n_q == 16 and wl.max_ctx == 131072
    _run(si, wl, rows=list(range(wl.n_q)))


def _spread(lo, hi, n):
    """n distinct rows spread over [lo, hi], both ends included."""
    return sorted(set(int(x) for x in np.linspace(lo, hi, n).round()))


def test_mixed_batch_full_size(si):
    """32 requests with log-uniform contexts in [1024, 65536]: all 28 decode
    rows and 64 rows of each of the 4 prefill chunks of 2048 rows (first and
    last rows included)."""
    wl = synth.make("c4")
    assert wl.n_q == 28 + 4 * 2048
    rows = list(range(28))
    for c in range(4):
        rows += _spread(28 + 2048 * c, 28 + 2048 * c + 2047, 64)
    _run(si, wl, rows=rows)


def _prefill_rows(n_q, rows_per_block, k_top, n_pairs=128):
    """Rows spread over the zigzag pairing of row blocks (block b goes with
    block nb - 1 - b): the first row of block b and the last row of its
    partner for n_pairs blocks b spread over the first half, plus the rows on
    both sides of pos = K - 1 (where rows start to select) and the ends."""
    nb = n_q // rows_per_block
    rows = set()
    for b in _spread(0, nb // 2 - 1, n_pairs):
        rows.add(b * rows_per_block)
        rows.add((nb - 1 - b) * rows_per_block + rows_per_block - 1)
    rows.update(range(k_top - 3, k_top + 3))
    rows.update((0, 1, n_q - 2, n_q - 1))
    return sorted(rows)


def test_causal_prefill_full_size(si):
    """Causal prefill of 16384 rows: rows below K = 2048 keep every position,
    later rows select.  The bf16 query takes blocks of four rows."""
    wl = synth.make("c2")
    assert wl.n_q == 16384
    rows = _prefill_rows(wl.n_q, 4, wl.K)
    assert len(rows) >= 256
    _run(si, wl, rows=rows)


def test_causal_prefill_full_size_fp8_query(si):
    """The same prefill with the indexer query stored in FP8 (per-(row, head)
    scale): the four-row prefill blocks at full size."""
    wl = synth.make("c2", q_idx_fp8=True)
    rows = _prefill_rows(wl.n_q, 4, wl.K)
    assert len(rows) >= 256
    _run(si, wl, rows=rows)


def test_benchmark_workload_fp8_kv_cache(si):
    """The benchmarked decode step over an FP8 latent cache (one scale per row
    and 128-entry tile) on the tensor-core attention kernel."""
    wl = synth.make("c1", kv_fp8=True)
    _run(si, wl, rows=list(range(wl.n_q)))


def test_benchmark_workload_fp4_kv_cache(si):
    """The benchmarked decode step over an FP4 e2m1 latent cache (one scale
    per row and 16-entry block)."""
    wl = synth.make("c1", kv_fp4=True)
    _run(si, wl, rows=list(range(wl.n_q)))


def test_long_context_fp8_kv_cache_split(si):
    """Long-context decode over an FP8 cache: few rows, so each row's key
    tiles are split over clusters and merged."""
    wl = synth.make("c3", batch=4, ctx=40000, kv_fp8=True)
    _run(si, wl, rows=list(range(wl.n_q)))


def test_benchmark_workload_mxfp8_indexer(si):
    """The benchmarked decode step with the MXFP8 indexer of section 5.1:
    keys in groups of 32 with E8M0 scales, the bf16 query converted on the
    device; every row."""
    wl = synth.make("c1", idx_mx=True)
    _run(si, wl, rows=list(range(wl.n_q)))


def test_long_context_mxfp8_indexer(si):
    wl = synth.make("c3", idx_mx=True)
    _run(si, wl, rows=list(range(wl.n_q)))


def test_causal_prefill_full_size_mxfp8(si):
    """The 16384-row prefill with the MXFP8 indexer: blocks of three rows."""
    wl = synth.make("c2", idx_mx=True)
    rows = _prefill_rows(wl.n_q, 3, wl.K)
    assert len(rows) >= 256
    _run(si, wl, rows=rows)
