"""CUDA path vs the CPU oracle on seeded synthetic inputs (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _parity import ATOL_BF16, ATOL_F32, check_topk, max_abs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def si():
    import __graft_entry__
    __graft_entry__.build()
    import indexer_driven_top_gb300 as si
    return si


def _run_separate(si, dw, out_dtype=torch.float32):
    b = dw.batch
    ld = b.max_ctx
    ws = si.alloc_workspace(si.workspace_size(si.OP_FUSED, b, dw.indexer, dw.attention, dw.k_top))
    scores = torch.empty((dw.n_q, ld), dtype=torch.float32, device="cuda")
    idx = torch.empty((dw.n_q, dw.k_top), dtype=torch.int32, device="cuda")
    out = torch.empty((dw.n_q, dw.attention.q.shape[1], dw.attention.d_v), dtype=out_dtype,
                      device="cuda")
    lse = torch.empty((dw.n_q, dw.attention.q.shape[1]), dtype=torch.float32, device="cuda")
    si.indexer_scores(b, dw.indexer, scores, ws)
    si.topk(b, scores, dw.k_top, idx, ws)
    si.sparse_attn(b, dw.attention, idx, dw.k_top, out, ws, lse=lse)
    assert si.workspace_status(ws) == 0
    return scores.cpu().numpy(), idx.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy()


def _run_fused(si, dw, out_dtype=torch.float32, ws_bytes=None):
    b = dw.batch
    n = ws_bytes or si.workspace_size(si.OP_FUSED, b, dw.indexer, dw.attention, dw.k_top)
    ws = si.alloc_workspace(n)
    idx = torch.empty((dw.n_q, dw.k_top), dtype=torch.int32, device="cuda")
    out = torch.empty((dw.n_q, dw.attention.q.shape[1], dw.attention.d_v), dtype=out_dtype,
                      device="cuda")
    lse = torch.empty((dw.n_q, dw.attention.q.shape[1]), dtype=torch.float32, device="cuda")
    si.fused_decode(b, dw.indexer, dw.attention, dw.k_top, idx, out, ws, lse=lse)
    assert si.workspace_status(ws) == 0
    return idx.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy()


def _attn_ref(wl, g_idx, rows=None):
    return oracle.sparse_attn(oracle.Batch.of(wl), wl.q, wl.kv_dtype, wl.k, wl.v, wl.kv_dtype,
                              g_idx, wl.K, wl.Hq, wl.Dqk, wl.Dv, wl.scale, rows=rows,
                              **oracle.attn_kv_args(wl))


def _full_check(si, wl, atol):
    dw = si.upload(wl)
    g_sc, g_idx, g_out, g_lse = _run_separate(si, dw)
    o_sc, o_idx, _, _, _ = oracle.run(wl)
    # indexer scores: fp32 accumulation vs fp64
    fin = np.isfinite(o_sc)
    assert np.array_equal(np.isfinite(g_sc), fin)
    scale = np.abs(o_sc[fin]).max() + 1e-30
    assert np.abs(g_sc[fin] - o_sc[fin]).max() <= 1e-5 * scale
    check_topk(g_idx, o_idx, o_sc, wl.q_pos, wl.K)
    ref, ref_lse = _attn_ref(wl, g_idx)
    assert max_abs(g_out, ref) <= atol
    assert max_abs(g_lse, ref_lse) <= atol
    f_idx, f_out, f_lse = _run_fused(si, dw)
    assert np.array_equal(f_idx, g_idx)
    assert np.array_equal(f_out, g_out)
    return g_idx, o_idx


def test_c0_tiny_prefill_fp32(si):
    wl = synth.make("c0")
    g_idx, o_idx = _full_check(si, wl, ATOL_F32)
    assert np.array_equal(g_idx, o_idx)


def test_decode_ragged_bf16_fp8(si):
    wl = synth.make("c1", batch=3, ctx_list=[3001, 2048, 130], K=2048)
    _full_check(si, wl, ATOL_BF16)


def test_planted_long_decode(si):
    wl = synth.make("c3", batch=2, ctx=9000, K=256)
    g_idx, _ = _full_check(si, wl, ATOL_BF16)
    for i in range(2):       # every planted key is selected (they beat the rest by ~3 sigma)
        assert np.isin(wl.planted[i], g_idx[i]).mean() > 0.95


def test_prefill_chunk_small(si):
    wl = synth.make("c2", L=300, K=64)
    _full_check(si, wl, ATOL_BF16)


def test_fp8_query_decode_tensor_core(si):
    """FP8 indexer query with a per-(row, head) scale on the 64 x 128
    tensor-core decode indexer."""
    wl = synth.make("c1", batch=3, ctx_list=[3001, 2048, 130], K=2048, q_idx_fp8=True)
    _full_check(si, wl, ATOL_BF16)


def test_fp8_query_prefill_ragged_block(si):
    """Prefill indexer with an FP8 query: blocks of four rows, the last one
    holding a single row."""
    wl = synth.make("c2", L=701, K=64, q_idx_fp8=True)
    _full_check(si, wl, ATOL_BF16)


def test_fp8_query_generic_shapes(si):
    """FP8 query on indexer shapes the tensor-core kernels do not take."""
    wl = synth.make("c4", n_req=5, n_prefill=1, chunk=40, ctx_lo=100, ctx_hi=1500, K=128,
                    Hi=4, Di=32, q_idx_fp8=True)
    _full_check(si, wl, ATOL_BF16)


def test_fp8_kv_cache(si):
    """Latent KV rows stored as e4m3 with one scale per 128-entry tile
    (section 5.2): the whole path against the oracle on the dequantised rows."""
    wl = synth.make("c1", batch=3, ctx_list=[3001, 2048, 130], K=512, kv_fp8=True)
    _full_check(si, wl, ATOL_BF16)


def test_fp4_kv_cache(si):
    """Latent KV rows stored as FP4 e2m1 codes with one scale per block of 16
    entries (the NVFP4 block): the whole path against the oracle on the
    dequantised rows, through the CUDA-core attention kernel."""
    wl = synth.make("c1", batch=3, ctx_list=[3001, 2048, 130], K=512, kv_fp4=True)
    _full_check(si, wl, ATOL_BF16)


def test_bf16_query_prefill_ragged_block(si):
    """Prefill indexer with a bf16 query: blocks of two rows, the last one
    holding a single row."""
    wl = synth.make("c2", L=301, K=64)
    _full_check(si, wl, ATOL_BF16)


def test_mixed_ragged_batch(si):
    wl = synth.make("c4", n_req=5, n_prefill=1, chunk=40, ctx_lo=100, ctx_hi=1500, K=128)
    _full_check(si, wl, ATOL_BF16)


def test_mixed_batch_prefill_chunks_take_prefill_kernel(si):
    """Decode rows followed by two prefill chunks of 100 rows: with the host
    copy of q_seq the indexer sends each chunk to the prefill kernel (one
    launch per chunk plus one for the decode rows); the scores match the
    unplanned single launch and the oracle."""
    wl = synth.make("c4", n_req=6, n_prefill=2, chunk=100, ctx_lo=200, ctx_hi=3000, K=128)
    _full_check(si, wl, ATOL_BF16)
    dw = si.upload(wl)
    ws = si.alloc_workspace(4096)
    planned = torch.empty((wl.n_q, wl.max_ctx), dtype=torch.float32, device="cuda")
    c0 = si.launch_count()
    si.indexer_scores(dw.batch, dw.indexer, planned, ws)
    torch.cuda.synchronize()
    assert si.launch_count() - c0 == 3
    import dataclasses
    plain_b = dataclasses.replace(dw.batch, host_q_seq=None)
    plain = torch.empty_like(planned)
    c0 = si.launch_count()
    si.indexer_scores(plain_b, dw.indexer, plain, ws)
    torch.cuda.synchronize()
    assert si.launch_count() - c0 == 1
    assert si.workspace_status(ws) == 0
    a, b_ = planned.cpu().numpy(), plain.cpu().numpy()
    fin = np.isfinite(b_)
    assert np.array_equal(np.isfinite(a), fin)
    assert np.abs(a[fin] - b_[fin]).max() <= 1e-6 * np.abs(b_[fin]).max()


def test_attention_split_matches_unsplit(si):
    """A few decode rows: with a full workspace each row's key tiles are
    split over several clusters and merged by the combine kernel (two
    launches); with the minimal workspace one cluster takes the whole row
    (one launch).  Both match the oracle, and each other."""
    wl = synth.make("c1", batch=3, ctx_list=[9000, 3001, 300], K=2048)
    dw = si.upload(wl)
    b = dw.batch
    ws = si.alloc_workspace(si.workspace_size(si.OP_FUSED, b, dw.indexer, dw.attention, wl.K))
    sc = torch.empty((wl.n_q, b.max_ctx), dtype=torch.float32, device="cuda")
    idx = torch.empty((wl.n_q, wl.K), dtype=torch.int32, device="cuda")
    si.indexer_scores(b, dw.indexer, sc, ws)
    si.topk(b, sc, wl.K, idx, ws)
    outs, lses, launches = [], [], []
    for nbytes in (si.workspace_size(si.OP_ATTN, b, None, dw.attention, wl.K),
                   si.workspace_min(si.OP_ATTN, b, None, dw.attention, wl.K)):
        w = si.alloc_workspace(nbytes)
        out = torch.empty((wl.n_q, 128, 512), dtype=torch.float32, device="cuda")
        lse = torch.empty((wl.n_q, 128), dtype=torch.float32, device="cuda")
        c0 = si.launch_count()
        si.sparse_attn(b, dw.attention, idx, wl.K, out, w, lse=lse)
        torch.cuda.synchronize()
        launches.append(si.launch_count() - c0)
        assert si.workspace_status(w) == 0
        outs.append(out.cpu().numpy())
        lses.append(lse.cpu().numpy())
    assert launches == [2, 1]
    ref, ref_lse = _attn_ref(wl, idx.cpu().numpy())
    for o, l in zip(outs, lses):
        assert max_abs(o, ref) <= ATOL_BF16 and max_abs(l, ref_lse) <= ATOL_BF16
    assert max_abs(outs[0], outs[1]) <= 1e-3


def test_fused_small_workspace_uses_strips(si):
    wl = synth.make("c4", n_req=4, n_prefill=1, chunk=30, ctx_lo=100, ctx_hi=900, K=64)
    dw = si.upload(wl)
    a_idx, a_out, _ = _run_fused(si, dw)
    mn = si.workspace_min(si.OP_FUSED, dw.batch, dw.indexer, dw.attention, wl.K)
    b_idx, b_out, _ = _run_fused(si, dw, ws_bytes=mn + 3 * 4 * wl.max_ctx)
    assert np.array_equal(a_idx, b_idx) and np.array_equal(a_out, b_out)


def test_topk_exact_on_identical_scores(si):
    """si_topk and the oracle's Top-K on the same float32 scores agree bit
    for bit, including heavy ties (integer scores) and -0/+0."""
    rng = np.random.default_rng(3)
    n_q, ld = 40, 5000
    pos = np.concatenate([rng.integers(0, ld, n_q - 4), [0, 9, 10, ld - 1]]).astype(np.int32)
    sc = rng.integers(-20, 20, size=(n_q, ld)).astype(np.float32)
    sc[1::3] = rng.standard_normal((len(sc[1::3]), ld)).astype(np.float32)
    sc[2, :100] = -0.0
    import indexer_driven_top_gb300 as si_
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    b = si_.Batch(dev(np.zeros((1, 100), np.int32)), dev(np.array([ld], np.int32)),
                  dev(np.zeros(n_q, np.int32)), dev(pos), 64, ld, 100)
    ws = si_.alloc_workspace(256)
    for K in (1, 10, 64, 2048):
        idx = torch.empty((n_q, K), dtype=torch.int32, device="cuda")
        si_.topk(b, dev(sc), K, idx, ws)
        ob = oracle.Batch(np.zeros((1, 100), np.int32), [ld], np.zeros(n_q, np.int32), pos, 64)
        want = oracle.topk(ob, sc.astype(np.float64), K)
        assert np.array_equal(idx.cpu().numpy(), want), K


@pytest.mark.parametrize("ld", [3000, 12000, 16384])
def test_topk_exact_many_rows_shared_memory(si, ld):
    """A batch of more rows than the GPU has SMs: rows of up to 8192 keep
    the register-cached kernel (3000), longer rows that fit one CTA (a late
    prefill strip) take one CTA per row with its keys in shared memory, two
    CTAs per SM (12000, 16384).  Bit-exact against the oracle with heavy
    ties, -0/+0, rows that select everything and rows ending at the last
    position."""
    rng = np.random.default_rng(ld + 7)
    n_q = 400
    edges = np.minimum([0, 100, 2047, 2048, 2049, 8191, 8192, 16383], ld - 1)
    pos = np.concatenate([rng.integers(0, ld, n_q - len(edges) - 1), edges, [ld - 1]]).astype(np.int32)
    sc = rng.integers(-30, 30, size=(n_q, ld)).astype(np.float32)   # many equal keys
    sc[1::3] = rng.standard_normal((len(sc[1::3]), ld)).astype(np.float32)
    sc[2, :1000] = -0.0
    sc[5, :] = 0.0
    sc[5, ::2] = -0.0
    import indexer_driven_top_gb300 as si_
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    nb = (ld + 63) // 64
    b = si_.Batch(dev(np.zeros((1, nb), np.int32)), dev(np.array([ld], np.int32)),
                  dev(np.zeros(n_q, np.int32)), dev(pos), 64, ld, nb)
    ws = si_.alloc_workspace(256)
    ob = oracle.Batch(np.zeros((1, nb), np.int32), [ld], np.zeros(n_q, np.int32), pos, 64)
    for K in (1, 77, 2048):
        idx = torch.empty((n_q, K), dtype=torch.int32, device="cuda")
        si_.topk(b, dev(sc), K, idx, ws)
        want = oracle.topk(ob, sc.astype(np.float64), K)
        assert np.array_equal(idx.cpu().numpy(), want), K


@pytest.mark.parametrize("ld,n_q", [(16385, 12), (40000, 12), (131072, 12), (131072, 40)])
def test_topk_exact_long_rows_cluster(si, ld, n_q):
    """Rows longer than one CTA's register cache (16384) take a cluster of
    CTAs, each caching a 32768-position segment in shared memory (16385: one
    CTA; 40000: two; 131072: four, with 12 and with 40 rows).  Bit-exact
    against the oracle with heavy ties spread over segments, rows that select
    everything, rows inside one segment, and rows ending at and one past a
    segment boundary."""
    rng = np.random.default_rng(ld + n_q)
    edges = np.minimum([0, 100, 16383, 16384, 32767, 32768], ld - 1)
    pos = np.concatenate([rng.integers(0, ld, n_q - 7), edges, [ld - 1]]).astype(np.int32)
    sc = rng.integers(-30, 30, size=(n_q, ld)).astype(np.float32)   # many equal keys
    sc[1::3] = rng.standard_normal((len(sc[1::3]), ld)).astype(np.float32)
    sc[2, :5000] = -0.0
    import indexer_driven_top_gb300 as si_
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    nb = (ld + 63) // 64
    b = si_.Batch(dev(np.zeros((1, nb), np.int32)), dev(np.array([ld], np.int32)),
                  dev(np.zeros(n_q, np.int32)), dev(pos), 64, ld, nb)
    ws = si_.alloc_workspace(256)
    ob = oracle.Batch(np.zeros((1, nb), np.int32), [ld], np.zeros(n_q, np.int32), pos, 64)
    for K in (1, 77, 2048):
        idx = torch.empty((n_q, K), dtype=torch.int32, device="cuda")
        si_.topk(b, dev(sc), K, idx, ws)
        want = oracle.topk(ob, sc.astype(np.float64), K)
        assert np.array_equal(idx.cpu().numpy(), want), K


def test_bad_block_and_bad_index_raise_flags(si):
    wl = synth.make("c1", batch=2, ctx=200, Hi=4, Di=32, Hq=4, Dqk=64, Dv=32, K=16)
    bt = wl.block_table.copy()
    bt[1, 1] = 10_000                       # outside the cache
    wl2 = synth.Workload(**{**wl.__dict__, "block_table": bt})
    dw = si.upload(wl2)
    ws = si.alloc_workspace(si.workspace_size(si.OP_FUSED, dw.batch, dw.indexer, dw.attention, 16))
    sc = torch.empty((2, wl.max_ctx), dtype=torch.float32, device="cuda")
    si.indexer_scores(dw.batch, dw.indexer, sc, ws)
    assert si.workspace_status(ws) & si.DEVFLAG_BAD_BLOCK
    # row 0 unaffected, row 1's bad page scores -inf (skipped)
    s = sc.cpu().numpy()
    assert np.isfinite(s[0, :200]).all() and np.isneginf(s[1, 64:128]).all()
    dw = si.upload(wl)
    ws = si.alloc_workspace(4096)
    idx = torch.tensor([[0, 5, 199, -1] + [-1] * 12, [3, 250, -7, -1] + [-1] * 12],
                       dtype=torch.int32, device="cuda")
    out = torch.empty((2, 4, 32), dtype=torch.float32, device="cuda")
    si.sparse_attn(dw.batch, dw.attention, idx, 16, out, ws)
    assert si.workspace_status(ws) == si.DEVFLAG_BAD_INDEX
    ref, _ = _attn_ref(wl, np.where(idx.cpu().numpy() > 199, -1, np.maximum(idx.cpu().numpy(), -1)))
    assert max_abs(out.cpu().numpy(), ref) <= ATOL_BF16


def _large_entry(wl, seq, pos, entry, value):
    """The workload with entry `entry` of the latent row at (seq, pos) set to
    `value` (bf16)."""
    k = wl.k.copy()
    row = int(wl.block_table[seq, pos // wl.page]) * wl.page + pos % wl.page
    k.reshape(-1, k.shape[-1])[row, entry] = synth.f32_to_bf16_bits(np.float32([value]))[0]
    return synth.Workload(**{**wl.__dict__, "k": k})


def test_value_beyond_f16_range_raises_flag(si):
    """The tensor-core attention multiplies f16 softmax weights with value
    entries converted bf16 -> f16.  A selected value above 65504 has no f16
    form: the call must finish and raise SI_DEVFLAG_RANGE (no fault, no
    trap); the same inputs without it raise nothing."""
    wl = synth.make("c1", batch=2, ctx=300, K=2048)  # every position is selected
    dw = si.upload(wl)
    idx = torch.empty((2, 2048), dtype=torch.int32, device="cuda")
    out = torch.empty((2, wl.Hq, wl.Dv), dtype=torch.float32, device="cuda")
    ws = si.alloc_workspace(si.workspace_size(si.OP_FUSED, dw.batch, dw.indexer, dw.attention, 2048))
    si.fused_decode(dw.batch, dw.indexer, dw.attention, 2048, idx, out, ws)
    assert si.workspace_status(ws) == 0
    for entry in (3, 511):  # a value entry in each half of the row
        big = si.upload(_large_entry(wl, 0, 5, entry, 1e5))
        ws = si.alloc_workspace(si.workspace_size(si.OP_FUSED, big.batch, big.indexer,
                                                  big.attention, 2048))
        si.fused_decode(big.batch, big.indexer, big.attention, 2048, idx, out, ws)
        assert si.workspace_status(ws) == si.DEVFLAG_RANGE, entry
    # the boundary: 65280 (the largest bf16 below 2^16) has an f16 form,
    # 65536 has none
    for value, flag in ((65280.0, 0), (-65280.0, 0), (65536.0, si.DEVFLAG_RANGE),
                        (-65536.0, si.DEVFLAG_RANGE)):
        edge = si.upload(_large_entry(wl, 1, 7, 100, value))
        ws = si.alloc_workspace(si.workspace_size(si.OP_FUSED, edge.batch, edge.indexer,
                                                  edge.attention, 2048))
        si.fused_decode(edge.batch, edge.indexer, edge.attention, 2048, idx, out, ws)
        assert si.workspace_status(ws) == flag, value


def test_empty_batch_is_noop(si):
    wl = synth.make("c0", L=64)
    dw = si.upload(wl)
    b = dw.batch
    empty = si.Batch(b.block_table, b.ctx_len, b.q_seq[:0], b.q_pos[:0], b.page_size, 1, b.n_blocks)
    ws = si.alloc_workspace(256)
    out = torch.empty((0, 4, 64), device="cuda")
    idx = torch.empty((0, 32), dtype=torch.int32, device="cuda")
    si.fused_decode(empty, dw.indexer, dw.attention, 32, idx, out, ws)
    assert si.workspace_status(ws) == 0


def _scores_check(si, wl, wl_ref=None):
    """GPU scores of ``wl``; oracle scores of ``wl_ref`` (default ``wl``; the
    oracle must only ever see a valid block table)."""
    dw = si.upload(wl)
    ws = si.alloc_workspace(4096)
    sc = torch.empty((wl.n_q, wl.max_ctx), dtype=torch.float32, device="cuda")
    si.indexer_scores(dw.batch, dw.indexer, sc, ws)
    flags = si.workspace_status(ws)
    g = sc.cpu().numpy()
    r = wl_ref or wl
    o = oracle.indexer_scores(oracle.Batch.of(r), r.q_idx, r.q_idx_dtype, r.w, r.k_idx,
                              r.k_idx_dtype, r.k_scale, r.Hi, r.Di, r.max_ctx,
                              q_scale=r.q_scale)
    return g, o, flags


@pytest.mark.parametrize("page", [16, 256])
def test_tensor_core_indexer_page_sizes(si, page):
    wl = synth.make("c1", batch=3, ctx_list=[1000, 300, 77], K=64, page=page)
    g, o, flags = _scores_check(si, wl)
    assert flags == 0
    fin = np.isfinite(o)
    assert np.array_equal(np.isfinite(g), fin)
    assert np.abs(g[fin] - o[fin]).max() <= 1e-5 * np.abs(o[fin]).max()


def test_tensor_core_indexer_bad_block(si):
    wl = synth.make("c1", batch=2, ctx=300, K=64)
    bt = wl.block_table.copy()
    bt[1, 2] = 1 << 20                     # page 2 of row 1 points outside the cache
    wl2 = synth.Workload(**{**wl.__dict__, "block_table": bt})
    g, o, flags = _scores_check(si, wl2, wl_ref=wl)
    assert flags & si.DEVFLAG_BAD_BLOCK
    assert np.isneginf(g[1, 128:192]).all()
    ok = np.ones_like(g, dtype=bool)
    ok[1, 128:192] = False
    fin = np.isfinite(o) & ok
    assert np.abs(g[fin] - o[fin]).max() <= 1e-5 * np.abs(o[fin]).max()


def test_fused_workspace_reused_across_batch_shapes(si):
    """One workspace serves fused calls on batches of other shapes in turn
    (their score strips overlap): every result equals the separate indexer +
    Top-K of the same batch."""
    wls = [synth.make("c1", batch=5, ctx_list=[3000, 130, 2048, 4097, 777], K=512),
           synth.make("c1", batch=9, ctx=1500, K=256, seed=7),
           synth.make("c1", batch=5, ctx_list=[3000, 130, 2048, 4097, 777], K=512)]
    size = max(si.workspace_size(si.OP_FUSED, d.batch, d.indexer, d.attention, d.k_top)
               for d in (si.upload(w) for w in wls))
    ws = si.alloc_workspace(size)
    for wl in wls:
        dw = si.upload(wl)
        b = dw.batch
        ref_sc = torch.empty((dw.n_q, b.max_ctx), dtype=torch.float32, device="cuda")
        ref_idx = torch.empty((dw.n_q, dw.k_top), dtype=torch.int32, device="cuda")
        ws2 = si.alloc_workspace(si.workspace_size(si.OP_FUSED, b, dw.indexer, dw.attention,
                                                   dw.k_top))
        si.indexer_scores(b, dw.indexer, ref_sc, ws2)
        si.topk(b, ref_sc, dw.k_top, ref_idx, ws2)
        idx = torch.empty_like(ref_idx)
        out = torch.empty((dw.n_q, wl.Hq, wl.Dv), dtype=torch.float32, device="cuda")
        for _ in range(2):
            si.fused_decode(b, dw.indexer, dw.attention, dw.k_top, idx, out, ws)
            assert si.workspace_status(ws) == 0
            assert torch.equal(idx, ref_idx)


@pytest.mark.parametrize("name,over", [
    ("c1", dict(batch=5, ctx_list=[3000, 130, 2048, 4097, 777], K=512)),  # select in the indexer
    ("c3", dict(batch=2, ctx=9000, K=256)),                               # rows over 8192
    ("c4", dict(n_req=6, n_prefill=2, chunk=200, ctx_lo=300, ctx_hi=2500, K=256)),  # planned
    ("c0", {}),                                                           # generic kernels
])
def test_indexer_topk_equals_scores_then_topk(si, name, over):
    """si_indexer_topk (section 4.1's fused operator) gives exactly the Top-K
    of si_indexer_scores followed by si_topk, with the minimal and the full
    workspace."""
    wl = synth.make(name, **over)
    dw = si.upload(wl)
    b = dw.batch
    ws = si.alloc_workspace(si.workspace_size(si.OP_FUSED, b, dw.indexer, dw.attention, dw.k_top))
    sc = torch.empty((dw.n_q, b.max_ctx), dtype=torch.float32, device="cuda")
    ref = torch.empty((dw.n_q, dw.k_top), dtype=torch.int32, device="cuda")
    si.indexer_scores(b, dw.indexer, sc, ws)
    si.topk(b, sc, dw.k_top, ref, ws)
    for nbytes in (si.workspace_size(si.OP_SELECT, b, dw.indexer, None, dw.k_top),
                   si.workspace_min(si.OP_SELECT, b, dw.indexer, None, dw.k_top)):
        ws2 = si.alloc_workspace(nbytes)
        idx = torch.empty_like(ref)
        si.indexer_topk(b, dw.indexer, dw.k_top, idx, ws2)
        assert si.workspace_status(ws2) == 0
        assert torch.equal(idx, ref)


@pytest.mark.parametrize("q_fmt", ["bf16", "e4m3", "mx"])
def test_indexer_topk_prefill_in_strips(si, q_fmt):
    """A causal prefill through si_indexer_topk with a workspace of 256 score
    rows: 12 strips on the prefill kernel, each after the first launched to
    overlap the previous strip's Top-K, none writing the -inf tail.  The
    selection equals si_indexer_scores (which writes the tail) followed by
    si_topk, for each indexer query format."""
    over = {"bf16": {}, "e4m3": {"q_idx_fp8": True}, "mx": {"idx_mx": True}}[q_fmt]
    wl = synth.make("c2", L=3000, K=256, Hq=1, Dqk=64, Dv=64, **over)
    dw = si.upload(wl)
    b = dw.batch
    sc = torch.empty((dw.n_q, b.max_ctx), dtype=torch.float32, device="cuda")
    ref = torch.empty((dw.n_q, dw.k_top), dtype=torch.int32, device="cuda")
    ws = si.alloc_workspace(4096)
    si.indexer_scores(b, dw.indexer, sc, ws)
    si.topk(b, sc, dw.k_top, ref, ws)
    assert si.workspace_status(ws) == 0
    assert np.isneginf(sc[0, 1:].cpu().numpy()).all()  # the tail of the separate call
    row_bytes = 4 * ((b.max_ctx + 63) // 64 * 64)
    ws2 = si.alloc_workspace(256 + 256 * row_bytes)
    assert ws2.numel() >= si.workspace_min(si.OP_SELECT, b, dw.indexer, None, dw.k_top)
    idx = torch.full_like(ref, -7)
    si.indexer_topk(b, dw.indexer, dw.k_top, idx, ws2)
    assert si.workspace_status(ws2) == 0
    assert torch.equal(idx, ref)
