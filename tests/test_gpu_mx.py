"""MXFP8 indexer (section 5.1's format: query and keys in groups of 32
entries with E8M0 scales) on the GPU against the oracle, through the C ABI:
the conversion entry point bit for bit, the conversion of a bf16 query inside
the indexer kernels against it, and the decode, prefill and CUDA-core
indexers on small ragged cases (scores, Top-K and the attention after them).
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


# ------------------------------------------------------------ conversion

def _quant_inputs(rng, n_rows, dim):
    """Rows mixing magnitudes from 2^-140 to 2^100 per group, plus the edge
    groups of the conversion rule."""
    x = rng.standard_normal((n_rows, dim)) * 2.0 ** rng.integers(-60, 60, (n_rows, dim // 32)
                                                               ).repeat(32, axis=1)
    g = x.reshape(n_rows, dim // 32, 32)
    if n_rows >= 8:
        g[0, 0] = 0.0                                            # all-zero group -> byte 0
        g[1, 0] = rng.standard_normal(32) * 2.0 ** -132          # bf16 subnormals only
        g[2, 0, :] = 2.0 ** -30
        g[2, 0, 0] = 3.0                                         # the rest rounds to +-0
        g[2, 0, 1::2] *= -1
        g[3, 0, 0] = 511 / 256 * 2.0 ** 7                        # clamps to 448 * X
        g[3, 0, 1] = -2.0 ** 7
        # exact midpoints between neighbouring e4m3 codes: the group's
        # largest entry 256 gives E = 0, so they stay midpoints after scaling
        mids = [(oracle.e4m3_to_f64(c) + oracle.e4m3_to_f64(c + 1)) / 2 for c in range(0, 120, 4)]
        g[4, 0, 0] = 256.0
        g[4, 0, 1:1 + len(mids)] = mids
        g[5, 0] = 2.0 ** 100 * rng.standard_normal(32)
    return x


@pytest.mark.parametrize("dtype,n_rows,dim", [("bf16", 300, 128), ("f32", 300, 128),
                                              ("bf16", 5, 32), ("bf16", 8192, 512)])
def test_quant_mxfp8_bit_exact(si, dtype, n_rows, dim):
    """si_quant_mxfp8 against the oracle's conversion: codes and scale bytes
    identical (the last case spans several grid-stride trips, the 5 x 32
    one a partial warp)."""
    rng = np.random.default_rng(n_rows + dim)
    x = _quant_inputs(rng, n_rows, dim).astype(np.float32)
    if dtype == "bf16":
        host = synth.f32_to_bf16_bits(x)
        dev = torch.from_numpy(host.view(np.int16)).view(torch.bfloat16).cuda()
    else:
        host = x
        dev = torch.from_numpy(x).cuda()
    codes = torch.empty((n_rows, dim), dtype=torch.uint8, device="cuda")
    scales = torch.empty((n_rows, dim // 32), dtype=torch.uint8, device="cuda")
    si.quant_mxfp8(dev, codes, scales)
    torch.cuda.synchronize()
    oc, os_ = oracle.mx_quantize(host, dtype)
    assert np.array_equal(scales.cpu().numpy(), os_)
    assert np.array_equal(codes.cpu().numpy(), oc)


# ---------------------------------------------------------------- indexer

def _scores(si, dw, ld=None):
    b = dw.batch
    ld = ld or b.max_ctx
    ws = si.alloc_workspace(4096)
    sc = torch.empty((dw.n_q, ld), dtype=torch.float32, device="cuda")
    si.indexer_scores(b, dw.indexer, sc, ws)
    flags = si.workspace_status(ws)
    return sc.cpu().numpy(), flags


def _check(si, wl, rows=None):
    """Scores within 1e-5 of the oracle's largest, Top-K by the tie-band rule,
    attention on the GPU's selection; the fused call gives the same result."""
    dw = si.upload(wl)
    b = dw.batch
    ws = si.alloc_workspace(si.workspace_size(si.OP_FUSED, b, dw.indexer, dw.attention, dw.k_top))
    sc = torch.empty((dw.n_q, b.max_ctx), dtype=torch.float32, device="cuda")
    idx = torch.empty((dw.n_q, dw.k_top), dtype=torch.int32, device="cuda")
    out = torch.empty((dw.n_q, wl.Hq, wl.Dv), dtype=torch.float32, device="cuda")
    si.indexer_scores(b, dw.indexer, sc, ws)
    si.topk(b, sc, dw.k_top, idx, ws)
    si.sparse_attn(b, dw.attention, idx, dw.k_top, out, ws)
    assert si.workspace_status(ws) == 0
    g_sc, g_idx, g_out = sc.cpu().numpy(), idx.cpu().numpy(), out.cpu().numpy()
    rows = list(range(wl.n_q)) if rows is None else rows
    o_sc, o_idx, _, _, _ = oracle.run(wl, rows=rows)
    for i, r in enumerate(rows):
        o, g = o_sc[i], g_sc[r]
        fin = np.isfinite(o)
        assert np.array_equal(np.isfinite(g), fin)
        assert np.abs(g[fin] - o[fin]).max() <= 1e-5 * (np.abs(o[fin]).max() + 1e-30)
    check_topk(g_idx[rows], o_idx, o_sc, wl.q_pos, wl.K, rows=rows)
    ref, _ = oracle.sparse_attn(oracle.Batch.of(wl), wl.q, wl.kv_dtype, wl.k, wl.v, wl.kv_dtype,
                                g_idx[rows], wl.K, wl.Hq, wl.Dqk, wl.Dv, wl.scale, rows=rows,
                                **oracle.attn_kv_args(wl))
    assert max_abs(g_out[rows], ref) <= ATOL_BF16
    f_idx = torch.empty_like(idx)
    f_out = torch.empty_like(out)
    si.fused_decode(b, dw.indexer, dw.attention, dw.k_top, f_idx, f_out, ws)
    assert si.workspace_status(ws) == 0
    assert torch.equal(f_idx, idx) and torch.equal(f_out, out)
    return dw, g_sc


@pytest.mark.parametrize("q_mx", [False, True])
def test_decode_tensor_core_mx(si, q_mx):
    """64 x 128 MXFP8 indexer on the decode kernel (bf16 query converted in
    the kernel, or stored MXFP8), ragged contexts over several tiles."""
    wl = synth.make("c1", batch=3, ctx_list=[3001, 2048, 130], K=2048, idx_mx=True, q_idx_mx=q_mx)
    _check(si, wl)


@pytest.mark.parametrize("q_mx", [False, True])
def test_prefill_tensor_core_mx_ragged_block(si, q_mx):
    """Causal prefill of 701 rows: blocks of three rows (the last holds two),
    MXFP8 block-scaled UMMA 192 wide."""
    wl = synth.make("c2", L=701, K=64, idx_mx=True, q_idx_mx=q_mx)
    _check(si, wl)


@pytest.mark.parametrize("q_mx", [False, True])
def test_mixed_batch_mx(si, q_mx):
    """Decode rows and prefill chunks in one batch: both tensor-core kernels."""
    wl = synth.make("c4", n_req=6, n_prefill=2, chunk=200, ctx_lo=300, ctx_hi=2500, K=256,
                    idx_mx=True, q_idx_mx=q_mx)
    _check(si, wl)


@pytest.mark.parametrize("q_mx", [False, True])
def test_generic_shapes_mx(si, q_mx):
    """Indexer shapes the tensor-core kernels do not take (4 heads x 64):
    the CUDA-core kernel dequantises each group, converting a bf16 query
    first."""
    wl = synth.make("c4", n_req=5, n_prefill=1, chunk=40, ctx_lo=100, ctx_hi=1500, K=128,
                    Hi=4, Di=64, idx_mx=True, q_idx_mx=q_mx)
    _check(si, wl)


@pytest.mark.parametrize("page", [16, 256])
def test_decode_mx_page_sizes(si, page):
    wl = synth.make("c1", batch=3, ctx_list=[1000, 300, 77], K=64, page=page, idx_mx=True)
    dw = si.upload(wl)
    g, flags = _scores(si, dw)
    assert flags == 0
    o = oracle.indexer_scores(oracle.Batch.of(wl), wl.q_idx, wl.q_idx_dtype, wl.w, wl.k_idx,
                              wl.k_idx_dtype, wl.k_scale, wl.Hi, wl.Di, wl.max_ctx)
    fin = np.isfinite(o)
    assert np.array_equal(np.isfinite(g), fin)
    assert np.abs(g[fin] - o[fin]).max() <= 1e-5 * np.abs(o[fin]).max()


def _as_mx_query(si, wl, dw):
    """The workload's bf16 query converted by si_quant_mxfp8, as an MXFP8
    indexer operand."""
    q = dw.indexer.q
    codes = torch.empty(q.shape, dtype=torch.uint8, device="cuda")
    scales = torch.empty(q.shape[:-1] + (q.shape[-1] // 32,), dtype=torch.uint8, device="cuda")
    si.quant_mxfp8(q, codes, scales)
    return si.Indexer(codes, "mxe4m3", dw.indexer.w, dw.indexer.k, scales)


@pytest.mark.parametrize("name,over", [
    ("c1", dict(batch=3, ctx_list=[3001, 2048, 130], K=64)),        # decode kernel
    ("c2", dict(L=400, K=64)),                                       # prefill kernel
    ("c1", dict(batch=2, ctx_list=[500, 90], K=64, Hi=4, Di=64)),    # CUDA-core kernel
])
def test_kernel_query_conversion_equals_quant_entry(si, name, over):
    """A bf16 query converted inside each indexer kernel scores exactly like
    the same query converted by si_quant_mxfp8 and passed as MXFP8 (same
    codes and scales reach the same arithmetic)."""
    wl = synth.make(name, idx_mx=True, **over)
    dw = si.upload(wl)
    g_bf16, f1 = _scores(si, dw)
    dw.indexer = _as_mx_query(si, wl, dw)
    g_mx, f2 = _scores(si, dw)
    assert f1 == 0 and f2 == 0
    assert np.array_equal(g_bf16, g_mx)


def test_decode_mx_bad_block(si):
    """An invalid page of one row: the flag, -inf over that page, the rest
    unaffected."""
    wl = synth.make("c1", batch=2, ctx=300, K=64, idx_mx=True)
    bt = wl.block_table.copy()
    bt[1, 2] = 1 << 20
    wl2 = synth.Workload(**{**wl.__dict__, "block_table": bt})
    g, flags = _scores(si, si.upload(wl2))
    assert flags & si.DEVFLAG_BAD_BLOCK
    assert np.isneginf(g[1, 128:192]).all()
    o = oracle.indexer_scores(oracle.Batch.of(wl), wl.q_idx, wl.q_idx_dtype, wl.w, wl.k_idx,
                              wl.k_idx_dtype, wl.k_scale, wl.Hi, wl.Di, wl.max_ctx)
    ok = np.isfinite(o)
    ok[1, 128:192] = False
    assert np.abs(g[ok] - o[ok]).max() <= 1e-5 * np.abs(o[ok]).max()
