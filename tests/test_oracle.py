"""Pins for the CPU oracle: each check ties it to something other than itself
(hand-computed values, library routines, closed forms, invariants)."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------ format decoders

def test_e4m3_decoder_all_codes_match_torch():
    """Every one of the 256 FP8 e4m3 codes decodes like torch's float8_e4m3fn."""
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_f64(c) for c in range(256)])
    nan = np.isnan(ref)
    assert nan.sum() == 2 and np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_decoder_hand_values():
    """Known codes of the OCP e4m3 format: max normal 448, min subnormal 2^-9,
    min normal 2^-6, one, minus two."""
    assert oracle.e4m3_to_f64(0x7E) == 448.0
    assert oracle.e4m3_to_f64(0x01) == 2.0 ** -9
    assert oracle.e4m3_to_f64(0x08) == 2.0 ** -6
    assert oracle.e4m3_to_f64(0x38) == 1.0
    assert oracle.e4m3_to_f64(0xC0) == -2.0
    assert oracle.e4m3_to_f64(0x07) == 7 * 2.0 ** -9
    assert math.isnan(oracle.e4m3_to_f64(0x7F))


def test_bf16_decoder_matches_torch():
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 16, size=4000, dtype=np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]          # finite patterns only
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(int(b)) for b in bits])
    assert np.array_equal(got, ref)


# ------------------------------------------------------ hand-computed fixture

def _golden():
    with open(os.path.join(GOLDEN, "tiny_indexer_topk_attn.json")) as f:
        return json.load(f)


def _golden_batch(g, pos_list):
    page = g["page"]
    bt = np.array(g["block_table"], dtype=np.int32)
    n_blocks = int(bt.max()) + 1
    k = np.full((n_blocks, page, 2), np.nan, dtype=np.float32)
    for s, row in enumerate(g["k_idx_logical"]):
        k[bt[0, s // page], s % page] = row
    b = oracle.Batch(bt, g["ctx_len"], np.zeros(len(pos_list), np.int32), pos_list, page)
    return b, k, bt, n_blocks


def test_golden_scores_and_topk():
    g = _golden()
    rows = g["rows"]
    b, k, _, _ = _golden_batch(g, [r["pos"] for r in rows])
    q_idx = np.array([r["q_idx"] for r in rows], dtype=np.float32)
    w = np.array([r["w"] for r in rows], dtype=np.float32)
    sc = oracle.indexer_scores(b, q_idx, "f32", w, k, "f32", None, 2, 2, ld=5)
    for i, r in enumerate(rows):
        exp = np.array([float(x) for x in r["scores"]])
        assert np.array_equal(sc[i], exp), (i, sc[i], exp)
        for K, want in r["topk"].items():
            K = int(K)
            idx = oracle.topk(b, sc, K)
            assert idx[i].tolist() == want, (i, K, idx[i])


def test_golden_attention():
    g = _golden()
    a = g["attention"]
    b, _, bt, n_blocks = _golden_batch(g, [g["rows"][0]["pos"]])
    page = g["page"]
    kc = np.full((n_blocks, page, 2), np.nan, dtype=np.float32)
    vc = np.full((n_blocks, page, 1), np.nan, dtype=np.float32)
    for s, row in a["k_logical"].items():
        s = int(s)
        kc[bt[0, s // page], s % page] = row
        vc[bt[0, s // page], s % page] = a["v_logical"][str(s)]
    idx = np.array([a["selected"]], dtype=np.int32)
    q = np.array([a["q"]], dtype=np.float32)
    out, lse = oracle.sparse_attn(b, q, "f32", kc, vc, "f32", idx, a["K"], 1, 2, 1, a["scale"])
    assert abs(out[0, 0, 0] - a["out"][0][0]) < 1e-6
    assert abs(lse[0, 0] - a["lse"][0]) < 1e-6


# ------------------------------------------------------------- library pins

def _tiny(seed=0, L=40, Hi=3, Di=5, Hq=2, D=6, K=7, page=4):
    return synth.make("c0", seed=seed, L=L, Hi=Hi, Di=Di, Hq=Hq, Dqk=D, Dv=D, K=K, page=page)


def test_topk_matches_library_sort_with_many_ties():
    """Top-K of integer-valued scores (many ties) equals a lexsort by
    (score descending, position ascending)."""
    rng = np.random.default_rng(1)
    n_q, ld, K = 30, 50, 9
    pos = rng.integers(0, ld, size=n_q).astype(np.int32)
    scores = rng.integers(-3, 4, size=(n_q, ld)).astype(np.float64)
    b = oracle.Batch(np.zeros((1, 1), np.int32), [ld], np.zeros(n_q, np.int32), pos, ld)
    idx = oracle.topk(b, scores, K)
    for r in range(n_q):
        n = pos[r] + 1
        order = np.lexsort((np.arange(n), -scores[r, :n]))
        want = np.sort(order[:min(K, n)])
        got = idx[r]
        assert got[:len(want)].tolist() == want.tolist()
        assert (got[len(want):] == -1).all()


def test_dense_limit_equals_library_causal_attention():
    """With K >= pos + 1 every earlier position is selected, so the path is
    dense causal attention: compare with torch's scaled_dot_product_attention
    (float64, is_causal=True) on the logical (unpaged) tensors."""
    wl = _tiny(seed=3, L=37, K=64)
    b = oracle.Batch.of(wl)
    sc = oracle.indexer_scores(b, wl.q_idx, "f32", wl.w, wl.k_idx, "f32", None, wl.Hi, wl.Di, 37)
    idx = oracle.topk(b, sc, wl.K)
    out, lse = oracle.sparse_attn(b, wl.q, "f32", wl.k, wl.v, "f32", idx, wl.K, wl.Hq, wl.Dqk,
                                  wl.Dv, wl.scale)
    L = 37
    rows_k = np.stack([wl.k[wl.block_table[0, s // wl.page], s % wl.page] for s in range(L)])
    rows_v = np.stack([wl.v[wl.block_table[0, s // wl.page], s % wl.page] for s in range(L)])
    q = torch.from_numpy(wl.q.astype(np.float64)).transpose(0, 1)      # [Hq, L, D]
    kk = torch.from_numpy(rows_k.astype(np.float64))[None].expand(wl.Hq, L, wl.Dqk)
    vv = torch.from_numpy(rows_v.astype(np.float64))[None].expand(wl.Hq, L, wl.Dv)
    ref = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, is_causal=True,
                                                           scale=wl.scale)
    assert np.abs(out - ref.transpose(0, 1).numpy()).max() < 1e-12
    # log-sum-exp against torch.logsumexp over the causal logits
    z = (q @ kk.transpose(1, 2)) * wl.scale
    z = z.masked_fill(torch.ones(L, L, dtype=torch.bool).triu(1), float("-inf"))
    assert np.abs(lse - torch.logsumexp(z, -1).transpose(0, 1).numpy()).max() < 1e-12


def test_sparse_attention_equals_masked_library_attention():
    """Attention over a Top-K set equals dense attention with every other
    position masked out (torch SDPA with a boolean mask)."""
    wl = _tiny(seed=4, L=33, K=5)
    b = oracle.Batch.of(wl)
    sc = oracle.indexer_scores(b, wl.q_idx, "f32", wl.w, wl.k_idx, "f32", None, wl.Hi, wl.Di, 33)
    idx = oracle.topk(b, sc, wl.K)
    out, _ = oracle.sparse_attn(b, wl.q, "f32", wl.k, wl.v, "f32", idx, wl.K, wl.Hq, wl.Dqk,
                                wl.Dv, wl.scale)
    L = 33
    mask = torch.zeros(L, L, dtype=torch.bool)
    for r in range(L):
        for s in idx[r]:
            if s >= 0:
                mask[r, s] = True
    rows_k = np.stack([wl.k[wl.block_table[0, s // wl.page], s % wl.page] for s in range(L)])
    rows_v = np.stack([wl.v[wl.block_table[0, s // wl.page], s % wl.page] for s in range(L)])
    q = torch.from_numpy(wl.q.astype(np.float64)).transpose(0, 1)
    kk = torch.from_numpy(rows_k.astype(np.float64))[None].expand(wl.Hq, L, wl.Dqk)
    vv = torch.from_numpy(rows_v.astype(np.float64))[None].expand(wl.Hq, L, wl.Dv)
    ref = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=mask,
                                                           scale=wl.scale)
    assert np.abs(out - ref.transpose(0, 1).numpy()).max() < 1e-12


def test_single_head_unit_weight_is_argtopk_of_dot_products():
    """H=1, w=1 and all dot products positive: the score is the dot product
    itself, so the selection is numpy's arg-top-K of q.k (ties excluded)."""
    rng = np.random.default_rng(7)
    L, D, K, page = 50, 4, 8, 8
    keys = rng.uniform(0.5, 1.5, size=(L, D)).astype(np.float32)
    qi = rng.uniform(0.5, 1.5, size=(L, 1, D)).astype(np.float32)
    bt = np.arange((L + page - 1) // page, dtype=np.int32)[::-1].copy()[None]
    kc = np.full((bt.size, page, D), np.nan, dtype=np.float32)
    for s in range(L):
        kc[bt[0, s // page], s % page] = keys[s]
    b = oracle.Batch(bt, [L], np.zeros(L, np.int32), np.arange(L), page)
    sc = oracle.indexer_scores(b, qi, "f32", np.ones((L, 1), np.float32), kc, "f32", None, 1, D, L)
    idx = oracle.topk(b, sc, K)
    for r in range(K, L):
        dots = keys[: r + 1].astype(np.float64) @ qi[r, 0].astype(np.float64)
        want = np.sort(np.argsort(-dots, kind="stable")[:K])
        assert idx[r].tolist() == want.tolist()


# -------------------------------------------------------------- closed forms

def test_first_position_returns_its_value_row():
    """t = 0 selects only position 0, so the output is v[0] exactly."""
    wl = _tiny(seed=5)
    b = oracle.Batch.of(wl)
    idx = np.full((wl.n_q, wl.K), -1, np.int32)
    idx[:, 0] = 0
    out, lse = oracle.sparse_attn(b, wl.q, "f32", wl.k, wl.v, "f32", idx, wl.K, wl.Hq, wl.Dqk,
                                  wl.Dv, wl.scale)
    v0 = wl.v[wl.block_table[0, 0], 0].astype(np.float64)
    assert np.array_equal(out, np.broadcast_to(v0, out.shape))


def test_identical_keys_give_mean_of_values():
    """All selected key rows equal -> uniform softmax -> mean of the values."""
    wl = _tiny(seed=6, L=20, K=6)
    kc = wl.k.copy()
    kc[:] = kc[wl.block_table[0, 0], 0]
    b = oracle.Batch.of(wl)
    idx = np.tile(np.array([1, 3, 4, 9, 10, 11], np.int32), (wl.n_q, 1))
    out, lse = oracle.sparse_attn(b, wl.q, "f32", kc, wl.v, "f32", idx, 6, wl.Hq, wl.Dqk,
                                  wl.Dv, wl.scale)
    vs = np.stack([wl.v[wl.block_table[0, s // wl.page], s % wl.page] for s in idx[0]])
    assert np.abs(out - vs.astype(np.float64).mean(0)).max() < 1e-13


def test_zero_weights_select_lowest_positions():
    """w = 0 makes every score 0: all ties, so the K lowest positions win."""
    wl = _tiny(seed=8, L=30, K=4)
    b = oracle.Batch.of(wl)
    sc = oracle.indexer_scores(b, wl.q_idx, "f32", np.zeros_like(wl.w), wl.k_idx, "f32", None,
                               wl.Hi, wl.Di, 30)
    for r in range(30):
        assert (sc[r, : r + 1] == 0).all() and np.isneginf(sc[r, r + 1:]).all()
    idx = oracle.topk(b, sc, 4)
    for r in range(30):
        n = min(4, r + 1)
        assert idx[r, :n].tolist() == list(range(n))


def test_per_token_scale_and_fp8_dequantisation():
    """FP8 keys with per-token scale c: score equals the fp32 score of the
    dequantised keys code*c (checked against keys decoded by torch)."""
    wl = synth.make("c1", batch=2, ctx=70, Hi=3, Di=16, Hq=2, Dqk=8, Dv=4, K=5)
    b = oracle.Batch.of(wl)
    sc = oracle.indexer_scores(b, wl.q_idx, "bf16", wl.w, wl.k_idx, "e4m3", wl.k_scale, wl.Hi,
                               wl.Di, wl.max_ctx)
    deq = (torch.from_numpy(wl.k_idx).view(torch.float8_e4m3fn).to(torch.float64).numpy()
           * wl.k_scale.astype(np.float64)[..., None])
    sc2 = oracle.indexer_scores(b, wl.q_idx, "bf16", wl.w, deq.astype(np.float32), "f32", None,
                                wl.Hi, wl.Di, wl.max_ctx)
    # dequantised value code*scale is exact in fp64 but rounded in fp32
    assert np.allclose(sc, sc2, rtol=1e-6, atol=1e-9)


def _e4m3_by_definition(codes):
    """OCP e4m3 decode written out from the format: sign, 4 exponent bits
    (bias 7), 3 mantissa bits; exponent field 0 is subnormal (m / 8 * 2^-6)."""
    c = codes.astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e, m = (c >> 3) & 0xF, c & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    return sign * val


def test_fp8_query_with_per_head_scale_brute_force():
    """FP8 query codes with one scale per (row, head) (the query quantisation
    of the indexer prolog): the oracle's score equals the definition evaluated
    by brute force on the dequantised query and keys, both decoded here from
    the format's definition."""
    wl = synth.make("c1", batch=2, ctx_list=[37, 20], Hi=3, Di=16, Hq=2, Dqk=8, Dv=4, K=5,
                    q_idx_fp8=True)
    assert wl.q_idx_dtype == "e4m3" and wl.q_scale.shape == (2, 3)
    b = oracle.Batch.of(wl)
    sc = oracle.indexer_scores(b, wl.q_idx, "e4m3", wl.w, wl.k_idx, "e4m3", wl.k_scale, wl.Hi,
                               wl.Di, wl.max_ctx, q_scale=wl.q_scale)
    q = _e4m3_by_definition(wl.q_idx) * wl.q_scale.astype(np.float64)[..., None]
    kd = _e4m3_by_definition(wl.k_idx) * wl.k_scale.astype(np.float64)[..., None]
    for r in range(wl.n_q):
        seq, pos = wl.q_seq[r], wl.q_pos[r]
        for s_ in range(wl.max_ctx):
            if s_ > pos:
                assert np.isneginf(sc[r, s_])
                continue
            krow = kd[wl.block_table[seq, s_ // wl.page], s_ % wl.page]
            ref = sum(float(wl.w[r, h]) * max(0.0, float(q[r, h] @ krow)) for h in range(wl.Hi))
            assert abs(sc[r, s_] - ref) <= 1e-12 * (abs(ref) + 1e-30)
    # dropping the scale (a plausible slip) changes the scores
    sc_noscale = oracle.indexer_scores(b, wl.q_idx, "e4m3", wl.w, wl.k_idx, "e4m3", wl.k_scale,
                                       wl.Hi, wl.Di, wl.max_ctx)
    fin = np.isfinite(sc)
    assert not np.allclose(sc[fin], sc_noscale[fin])


# ---------------------------------------------------------------- invariants

def test_page_placement_does_not_change_results():
    wl = synth.make("c1", batch=3, ctx=150, Hi=4, Di=16, Hq=2, Dqk=12, Dv=8, K=10)
    wl2 = synth.permute_pages(wl, seed=11)
    assert not np.array_equal(wl.block_table, wl2.block_table)
    r1 = oracle.run(wl)
    r2 = oracle.run(wl2)
    for a, c in zip(r1, r2):
        assert np.array_equal(a, c, equal_nan=True)


def test_selected_index_order_does_not_change_attention():
    wl = _tiny(seed=9, L=25, K=6)
    b = oracle.Batch.of(wl)
    sc = oracle.indexer_scores(b, wl.q_idx, "f32", wl.w, wl.k_idx, "f32", None, wl.Hi, wl.Di, 25)
    idx = oracle.topk(b, sc, wl.K)
    out, lse = oracle.sparse_attn(b, wl.q, "f32", wl.k, wl.v, "f32", idx, wl.K, wl.Hq, wl.Dqk,
                                  wl.Dv, wl.scale)
    rng = np.random.default_rng(0)
    idx2 = np.stack([rng.permutation(r) for r in idx])
    out2, lse2 = oracle.sparse_attn(b, wl.q, "f32", wl.k, wl.v, "f32", idx2, wl.K, wl.Hq, wl.Dqk,
                                    wl.Dv, wl.scale)
    assert np.abs(out - out2).max() < 1e-13 and np.abs(lse - lse2).max() < 1e-13


def test_permuting_key_positions_permutes_selection():
    """Swapping the content of two key positions (indexer key and K/V row)
    swaps them in the selected set for a query that sees both."""
    wl = _tiny(seed=10, L=24, K=5)
    b = oracle.Batch.of(wl)
    r = 23
    sc = oracle.indexer_scores(b, wl.q_idx, "f32", wl.w, wl.k_idx, "f32", None, wl.Hi, wl.Di, 24)
    idx = oracle.topk(b, sc, wl.K)
    a = int(idx[r, 0])
    c = next(s for s in range(24) if s not in idx[r])
    wl2 = synth.make("c0", seed=10, L=24, Hi=3, Di=5, Hq=2, Dqk=6, Dv=6, K=5, page=4)
    for arr in (wl2.k_idx, wl2.k, wl2.v):
        pa = (wl2.block_table[0, a // 4], a % 4)
        pc = (wl2.block_table[0, c // 4], c % 4)
        tmp = arr[pa].copy()
        arr[pa] = arr[pc]
        arr[pc] = tmp
    sc2 = oracle.indexer_scores(b, wl2.q_idx, "f32", wl2.w, wl2.k_idx, "f32", None, 3, 5, 24)
    idx2 = oracle.topk(b, sc2, 5)
    want = sorted(c if s == a else s for s in idx[r])
    assert idx2[r].tolist() == want
    o1, _ = oracle.sparse_attn(b, wl.q, "f32", wl.k, wl.v, "f32", idx[[r]], 5, 2, 6, 6, wl.scale,
                               rows=[r])
    o2, _ = oracle.sparse_attn(b, wl2.q, "f32", wl2.k, wl2.v, "f32", idx2[[r]], 5, 2, 6, 6,
                               wl.scale, rows=[r])
    assert np.abs(o1 - o2).max() < 1e-13


def test_rows_subset_equals_full_run():
    wl = synth.make("c4", n_req=4, n_prefill=1, chunk=40, ctx_lo=60, ctx_hi=300, Hi=4, Di=16,
                    Hq=2, Dqk=12, Dv=8, K=16)
    full = oracle.run(wl)
    rows = [0, 3, wl.n_q - 1, 5]
    part = oracle.run(wl, rows=rows)
    for a, c in zip(full, part):
        assert np.array_equal(a[rows], c, equal_nan=True)


def test_fp8_kv_tiles_brute_force():
    """FP8 KV cache with one scale per row and tile of 128 entries (the last
    tile of a 576-entry row holds 64): the oracle's attention equals dense
    softmax attention over the selected rows, computed here in numpy from
    rows decoded with the format's own definition."""
    wl = synth.make("c1", batch=2, ctx_list=[90, 40], Hi=4, Di=16, Hq=3, K=16, kv_fp8=True)
    assert wl.kv_dtype == "e4m3" and wl.kv_scale.shape[-1] == 5 and wl.kv_scale_tile == 128
    b = oracle.Batch.of(wl)
    rng = np.random.default_rng(5)
    idx = np.full((wl.n_q, wl.K), -1, dtype=np.int32)
    for r in range(wl.n_q):
        sel = np.sort(rng.choice(int(wl.q_pos[r]) + 1, size=wl.K - 3, replace=False))
        idx[r, : len(sel)] = sel
    out, lse = oracle.sparse_attn(b, wl.q, wl.kv_dtype, wl.k, None, wl.kv_dtype, idx, wl.K, wl.Hq,
                                  wl.Dqk, wl.Dv, wl.scale, **oracle.attn_kv_args(wl))
    q = synth._bf16_bits_to_f32(wl.q).astype(np.float64)
    tile_of = np.arange(wl.Dqk) // 128
    deq = _e4m3_by_definition(wl.k) * wl.kv_scale.astype(np.float64)[..., tile_of]
    for r in range(wl.n_q):
        sel = idx[r][idx[r] >= 0]
        rows = np.array([deq[wl.block_table[wl.q_seq[r], s // wl.page], s % wl.page] for s in sel])
        z = wl.scale * q[r] @ rows.T                        # [Hq, n]
        p = np.exp(z - z.max(axis=1, keepdims=True))
        ref = (p @ rows[:, : wl.Dv]) / p.sum(axis=1, keepdims=True)
        assert np.abs(out[r] - ref).max() <= 1e-12 * np.abs(ref).max()
        assert np.abs(lse[r] - (z.max(axis=1) + np.log(p.sum(axis=1)))).max() <= 1e-12
    # a dropped tile scale (plausible slip: scales per row instead of per tile) is caught
    out_row, _ = oracle.sparse_attn(b, wl.q, wl.kv_dtype, wl.k, None, wl.kv_dtype, idx, wl.K,
                                    wl.Hq, wl.Dqk, wl.Dv, wl.scale, q_dtype="bf16",
                                    kv_scale=wl.kv_scale[..., :1].copy(), scale_tile=0)
    assert not np.allclose(out, out_row)


# ---------------------------------------- candidate-restricted selection

def test_golden_candidate_topk():
    """Hand-derived candidate selections on the fixture's keys and queries:
    only listed positions 0..pos compete, ties go to the lower position."""
    g = _golden()
    with open(os.path.join(GOLDEN, "tiny_candidate_topk.json")) as f:
        gc = json.load(f)
    rows = g["rows"]
    b, k, _, _ = _golden_batch(g, [r["pos"] for r in rows])
    q_idx = np.array([r["q_idx"] for r in rows], dtype=np.float32)
    w = np.array([r["w"] for r in rows], dtype=np.float32)
    for case in gc["cases"]:
        r = case["row"]
        n = len(case["cand"])
        cand = np.full((2, n), -1, dtype=np.int32)
        cand[r] = case["cand"]
        for K, want in case["topk"].items():
            idx, sc, _ = oracle.topk_cand(b, q_idx, "f32", w, k, "f32", None, 2, 2, cand, int(K))
            assert idx[r].tolist() == want, (case, K, idx[r])
            assert sc[r].tolist() == [float(x) for x in case["scores"]], (case, sc[r])


def _cand_args(wl):
    return (oracle.Batch.of(wl), wl.q_idx, wl.q_idx_dtype, wl.w, wl.k_idx, wl.k_idx_dtype,
            wl.k_scale, wl.Hi, wl.Di)


@pytest.mark.parametrize("name,over", [("c0", {}),
                                       ("c1", dict(batch=3, ctx=300, K=64, Hq=2, Dqk=16,
                                                   Dv=8))])
def test_all_positions_as_candidates_equal_full_selection(name, over):
    """With every position 0..pos listed, candidate-restricted selection is
    the full selection (the unrestricted path is pinned above)."""
    wl = synth.make(name, **over)
    args = _cand_args(wl)
    sc = oracle.indexer_scores(args[0], *args[1:], ld=wl.max_ctx)
    full = oracle.topk(args[0], sc, wl.K)
    cand = np.tile(np.arange(wl.max_ctx, dtype=np.int32), (wl.n_q, 1))
    idx, csc, _ = oracle.topk_cand(*args, cand, wl.K)
    assert np.array_equal(idx, full)
    assert np.array_equal(csc, sc)


def test_candidate_list_order_and_non_candidates_do_not_matter():
    """Shuffling each row's list, or adding -1 entries and positions past the
    row, leaves the selection unchanged; each score follows its position."""
    wl = synth.make("c1", batch=4, ctx=500, K=32, Hq=2, Dqk=16, Dv=8)
    args = _cand_args(wl)
    cand = synth.candidates(wl, 96, seed=3)
    idx, sc, _ = oracle.topk_cand(*args, cand, wl.K)
    rng = np.random.default_rng(7)
    perm = np.stack([rng.permutation(cand.shape[1]) for _ in range(wl.n_q)])
    shuf = np.take_along_axis(cand, perm, axis=1)
    idx2, sc2, _ = oracle.topk_cand(*args, shuf, wl.K)
    assert np.array_equal(idx2, idx)
    assert np.array_equal(sc2, np.take_along_axis(sc, perm, axis=1))
    extra = np.concatenate([cand, np.full((wl.n_q, 5), -1, np.int32),
                            (wl.q_pos[:, None] + 1 + np.arange(5)).astype(np.int32)], axis=1)
    idx3, sc3, _ = oracle.topk_cand(*args, extra, wl.K)
    assert np.array_equal(idx3, idx)
    assert np.all(np.isneginf(sc3[:, cand.shape[1]:]))


def test_fewer_candidates_than_k_returns_all_of_them():
    wl = synth.make("c1", batch=3, ctx=400, K=64, Hq=2, Dqk=16, Dv=8)
    args = _cand_args(wl)
    cand = synth.candidates(wl, 40, seed=1)
    idx, _, kth = oracle.topk_cand(*args, cand, wl.K)
    for r in range(wl.n_q):
        valid = cand[r][cand[r] >= 0]
        assert idx[r, :len(valid)].tolist() == sorted(valid.tolist())
        assert np.all(idx[r, len(valid):] == -1)
        assert np.isnan(kth[r, 0])


# ---------------------------------------------- NVFP4-style KV cache (e2m1)

E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]   # OCP FP4: codes 0..7, bit 3 = sign


def test_e2m1_decoder_all_codes():
    """All 16 FP4 e2m1 codes against the format's value table (1 sign, 2
    exponent bits with bias 1, 1 mantissa bit; no NaN or infinity)."""
    for c in range(16):
        want = (-1.0 if c & 8 else 1.0) * E2M1_TABLE[c & 7]
        got = oracle.e2m1_to_f64(c)
        assert got == want and (c != 8 or math.copysign(1.0, got) == -1.0), (c, got)


def _e2m1_rows_by_definition(packed):
    """Unpack two codes per byte (even entry in the low nibble) and decode
    them with the value table."""
    lo, hi = packed & 0x0F, packed >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(packed.shape[:-1] + (packed.shape[-1] * 2,))
    table = np.array(E2M1_TABLE)
    return np.where(codes & 8, -1.0, 1.0) * table[codes & 7]


def test_fp4_kv_blocks_brute_force():
    """FP4 e2m1 KV cache with one scale per block of 16 entries: the oracle's
    attention equals dense softmax attention over the selected rows, computed
    here in numpy from rows decoded with the value table."""
    wl = synth.make("c1", batch=2, ctx_list=[90, 40], Hi=4, Di=16, Hq=3, K=16, kv_fp4=True)
    assert wl.kv_dtype == "e2m1" and wl.kv_scale_tile == 16
    assert wl.k.shape[-1] * 2 == wl.Dqk and wl.kv_scale.shape[-1] == wl.Dqk // 16
    b = oracle.Batch.of(wl)
    rng = np.random.default_rng(6)
    idx = np.full((wl.n_q, wl.K), -1, dtype=np.int32)
    for r in range(wl.n_q):
        sel = np.sort(rng.choice(int(wl.q_pos[r]) + 1, size=wl.K - 2, replace=False))
        idx[r, : len(sel)] = sel
    out, lse = oracle.sparse_attn(b, wl.q, wl.kv_dtype, wl.k, None, wl.kv_dtype, idx, wl.K, wl.Hq,
                                  wl.Dqk, wl.Dv, wl.scale, **oracle.attn_kv_args(wl))
    q = synth._bf16_bits_to_f32(wl.q).astype(np.float64)
    blk_of = np.arange(wl.Dqk) // 16
    deq = _e2m1_rows_by_definition(wl.k) * wl.kv_scale.astype(np.float64)[..., blk_of]
    for r in range(wl.n_q):
        sel = idx[r][idx[r] >= 0]
        rows = np.array([deq[wl.block_table[wl.q_seq[r], s // wl.page], s % wl.page] for s in sel])
        z = wl.scale * q[r] @ rows.T
        p = np.exp(z - z.max(axis=1, keepdims=True))
        ref = (p @ rows[:, : wl.Dv]) / p.sum(axis=1, keepdims=True)
        assert np.abs(out[r] - ref).max() <= 1e-12 * np.abs(ref).max()
        assert np.abs(lse[r] - (z.max(axis=1) + np.log(p.sum(axis=1)))).max() <= 1e-12
    # swapped nibble order (a plausible slip) is caught
    swapped = ((wl.k >> 4) | (wl.k << 4)).astype(np.uint8)
    out_sw, _ = oracle.sparse_attn(b, wl.q, wl.kv_dtype, swapped, None, wl.kv_dtype, idx, wl.K,
                                   wl.Hq, wl.Dqk, wl.Dv, wl.scale, **oracle.attn_kv_args(wl))
    assert not np.allclose(out, out_sw)


# ------------------------------------------------------------------- MXFP8

def test_e8m0_decoder_bytes():
    """E8M0 (the MX scale type): byte e is 2^(e - 127), 255 is NaN."""
    for e, v in ((0, 2.0 ** -127), (1, 2.0 ** -126), (126, 0.5), (127, 1.0), (128, 2.0),
                 (254, 2.0 ** 127)):
        assert oracle.e8m0_to_f64(e) == v
    assert math.isnan(oracle.e8m0_to_f64(255))


def test_e4m3_encoder_round_trips_every_finite_code():
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        assert oracle.f64_to_e4m3(oracle.e4m3_to_f64(c)) == c


def test_e4m3_encoder_matches_torch_rounding():
    """Round to nearest even into e4m3, checked against torch's float32 ->
    float8_e4m3fn conversion on float32 inputs inside the finite range
    (subnormals, exact midpoints and negative values that round to zero
    included)."""
    rng = np.random.default_rng(21)
    x = np.concatenate([
        rng.uniform(-448, 448, 4000), rng.standard_normal(4000) * 2.0 ** -7,
        rng.standard_normal(2000) * 2.0 ** -12,
        # midpoints between neighbouring codes
        np.array([(oracle.e4m3_to_f64(c) + oracle.e4m3_to_f64(c + 1)) / 2 for c in range(126)]),
    ]).astype(np.float32)
    x = np.concatenate([x, -x])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.f64_to_e4m3(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_encoder_ties_to_even_and_saturates():
    for c in range(126):
        lo, hi = oracle.e4m3_to_f64(c), oracle.e4m3_to_f64(c + 1)
        mid = (lo + hi) / 2
        assert oracle.f64_to_e4m3(mid) == (c if c % 2 == 0 else c + 1)
        assert oracle.f64_to_e4m3(np.nextafter(mid, 0)) == c
        assert oracle.f64_to_e4m3(np.nextafter(mid, 1000)) == c + 1
    for v in (448.5, 480.0, 1e6, math.inf):
        assert oracle.f64_to_e4m3(v) == 0x7E and oracle.f64_to_e4m3(-v) == 0xFE
    assert oracle.f64_to_e4m3(-1e-30) == 0x80 and oracle.f64_to_e4m3(0.0) == 0x00


def _mx_values(codes, sb):
    """X * P for one group, decoded here from the formats' definitions."""
    return _e4m3_by_definition(np.asarray(codes)) * 2.0 ** (int(sb) - 127)


def test_mx_group_closed_forms():
    """The MX conversion rule: exponent floor(log2 amax) - 8, so the largest
    entry lands in [256, 512) before rounding and clamps to 448 beyond it."""
    codes, sb = oracle.mx_group(np.zeros(32))
    assert sb == 0 and (codes == 0).all()
    for k in (-100, -20, -1, 0, 3, 60, 110):
        v = np.zeros(32)
        v[7] = 2.0 ** k
        v[8] = -(2.0 ** k) / 3
        codes, sb = oracle.mx_group(v)
        assert sb == 127 + k - 8
        assert codes[7] == 0x78                         # 256 = 1.0 * 2^8
        assert codes[8] == 0x80 | oracle.f64_to_e4m3(256 / 3)
    # just below the next power of two: 511/256 * 2^k scales to 511 -> 448
    v = np.full(32, 0.25)
    v[0] = 511 / 256 * 2.0 ** 5
    codes, sb = oracle.mx_group(v)
    assert sb == 127 + 5 - 8 and codes[0] == 0x7E
    # values that are e4m3 numbers times 2^E with amax in [256, 448] come back exactly
    rng = np.random.default_rng(3)
    for _ in range(50):
        E = int(rng.integers(-60, 60))
        c = rng.integers(0, 0x7F, size=32).astype(np.uint8)
        c[rng.integers(32)] = rng.integers(0x78, 0x7F)    # a code in [256, 448]
        c = np.where(rng.random(32) < 0.5, c | 0x80, c).astype(np.uint8)
        v = _e4m3_by_definition(c) * 2.0 ** E
        codes, sb = oracle.mx_group(v)
        assert sb == 127 + E
        assert np.array_equal(_mx_values(codes, sb), v)


def test_mx_group_symmetry_scaling_and_error_bound():
    rng = np.random.default_rng(8)
    for _ in range(200):
        v = rng.standard_normal(32) * 2.0 ** rng.integers(-30, 30)
        codes, sb = oracle.mx_group(v)
        c2, s2 = oracle.mx_group(2 * v)
        assert s2 == sb + 1 and np.array_equal(c2, codes)
        c3, s3 = oracle.mx_group(-v)
        assert s3 == sb and np.array_equal(c3, codes ^ 0x80)
        X = 2.0 ** (sb - 127)
        err = np.abs(_mx_values(codes, sb) - v)
        y = np.abs(v) / X
        normal = (y >= 2.0 ** -6) & (y <= 448)
        # half an e4m3 step: 2^(floor(log2 y) - 4) in scaled units
        assert (err[normal] <= 2.0 ** (np.floor(np.log2(y[normal])) - 4) * X).all()
        assert (err[y < 2.0 ** -6] <= 2.0 ** -10 * X).all()
        clip = y > 448
        assert np.allclose(err[clip], np.abs(v[clip]) - 448 * X)


def test_mx_quantize_rows_group_by_group():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((5, 3, 96)).astype(np.float32)
    codes, scales = oracle.mx_quantize(x, "f32")
    assert codes.shape == x.shape and scales.shape == (5, 3, 3)
    for i in range(5):
        for j in range(3):
            for g in range(3):
                c, s = oracle.mx_group(x[i, j, 32 * g: 32 * g + 32].astype(np.float64))
                assert s == scales[i, j, g] and np.array_equal(c, codes[i, j, 32 * g: 32 * g + 32])
    # bf16 input: the bit patterns decode first
    xb = synth.f32_to_bf16_bits(x)
    cb, sbb = oracle.mx_quantize(xb, "bf16")
    c2, s2 = oracle.mx_quantize((xb.astype(np.uint32) << 16).view(np.float32), "f32")
    assert np.array_equal(cb, c2) and np.array_equal(sbb, s2)


def _mx_workload(q_mx, **over):
    args = dict(batch=2, ctx_list=[70, 45], Hi=3, Di=64, Hq=2, Dqk=8, Dv=4, K=5, idx_mx=True,
                q_idx_mx=q_mx)
    args.update(over)
    return synth.make("c1", **args)


def test_mx_scores_equal_scores_of_the_dequantised_values():
    """MXFP8 keys and query: the scores equal the oracle's float32 path on the
    values X * P decoded here from the definitions (each is exact in float32
    at these magnitudes), and brute force on two rows."""
    wl = _mx_workload(True)
    assert wl.k_scale.dtype == np.uint8 and wl.k_scale.shape[-1] == 2
    b = oracle.Batch.of(wl)
    sc = oracle.indexer_scores(b, wl.q_idx, "mxe4m3", wl.w, wl.k_idx, "mxe4m3", wl.k_scale,
                               wl.Hi, wl.Di, wl.max_ctx, q_scale=wl.q_scale)

    def deq(codes, sbytes):
        """X * P; scale byte 255 (unused slots) is NaN"""
        vals = _e4m3_by_definition(codes).reshape(codes.shape[:-1] + (-1, 32))
        x = np.where(sbytes == 255, np.nan, 2.0 ** (sbytes.astype(np.float64) - 127))
        return (vals * x[..., None]).reshape(codes.shape)

    qd = deq(wl.q_idx, wl.q_scale)
    kd = deq(wl.k_idx, wl.k_scale)
    assert np.array_equal(qd.astype(np.float32).astype(np.float64), qd)
    fin_k = np.isfinite(kd)
    assert np.array_equal(kd[fin_k].astype(np.float32).astype(np.float64), kd[fin_k])
    sc2 = oracle.indexer_scores(b, qd.astype(np.float32), "f32", wl.w, kd.astype(np.float32),
                                "f32", None, wl.Hi, wl.Di, wl.max_ctx)
    assert np.array_equal(np.isfinite(sc), np.isfinite(sc2))
    fin = np.isfinite(sc)
    assert np.allclose(sc[fin], sc2[fin], rtol=1e-12, atol=0)
    for r in range(wl.n_q):
        seq = wl.q_seq[r]
        for s_ in range(0, int(wl.q_pos[r]) + 1, 7):
            krow = kd[wl.block_table[seq, s_ // wl.page], s_ % wl.page]
            ref = sum(float(wl.w[r, h]) * max(0.0, float(qd[r, h] @ krow)) for h in range(wl.Hi))
            assert abs(sc[r, s_] - ref) <= 1e-12 * (abs(ref) + 1e-30)
    # a scale taken from the wrong group (a plausible slip) changes the scores
    bad = wl.k_scale[..., ::-1].copy()
    sc_bad = oracle.indexer_scores(b, wl.q_idx, "mxe4m3", wl.w, wl.k_idx, "mxe4m3", bad,
                                   wl.Hi, wl.Di, wl.max_ctx, q_scale=wl.q_scale)
    assert not np.allclose(sc_bad[fin], sc[fin])


def test_mx_bf16_query_is_converted_per_group_first():
    """A bf16 query with MXFP8 keys is the MX query of the conversion rule."""
    wl = _mx_workload(False)
    assert wl.q_idx_dtype == "bf16"
    b = oracle.Batch.of(wl)
    sc = oracle.indexer_scores(b, wl.q_idx, "bf16", wl.w, wl.k_idx, "mxe4m3", wl.k_scale,
                               wl.Hi, wl.Di, wl.max_ctx)
    qc, qs = oracle.mx_quantize(wl.q_idx, "bf16")
    sc2 = oracle.indexer_scores(b, qc, "mxe4m3", wl.w, wl.k_idx, "mxe4m3", wl.k_scale,
                                wl.Hi, wl.Di, wl.max_ctx, q_scale=qs)
    assert np.array_equal(sc, sc2)
