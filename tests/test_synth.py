"""The input generator's format encoders agree with torch's conversions."""
import numpy as np
import torch

import oracle
import synth


def test_e4m3_encoder_matches_torch_rounding():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(5000) * 0.01,
                        np.array([448.0, -448.0, 0.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -11,
                                  1.0625, 1.1875, 240.0, 232.0])]).astype(np.float32)
    x = np.clip(x, -448, 448)
    got = synth.f32_to_e4m3_bits(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # torch keeps the sign of values that round to zero; the generator writes +0
    zero = (ref & 0x7F) == 0
    assert np.array_equal(got[~zero], ref[~zero])
    assert (got[zero] == 0).all()


def test_bf16_encoder_matches_torch_rounding():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(50000) * 10.0 ** rng.integers(-20, 20, 50000)).astype(np.float32)
    got = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_workload_structure():
    wl = synth.make("c4", n_req=6, n_prefill=2, chunk=50, ctx_lo=64, ctx_hi=400, Hi=2, Di=16,
                    Hq=2, Dqk=8, Dv=4, K=8)
    assert wl.n_q == 4 + 2 * 50
    for i in range(wl.n_seq):
        rows = np.nonzero(wl.q_seq == i)[0]
        assert wl.q_pos[rows].max() == wl.ctx_len[i] - 1
        nb = (wl.ctx_len[i] + wl.page - 1) // wl.page
        assert (wl.block_table[i, :nb] >= 0).all() and (wl.block_table[i, nb:] == -1).all()
    used = wl.block_table[wl.block_table >= 0]
    assert len(np.unique(used)) == len(used)


def test_planted_keys_raise_every_head_by_three_sigma():
    wl = synth.make("c3", batch=2, ctx=2000, K=64)
    from synth import _bf16_bits_to_f32
    for i in range(2):
        pos = wl.planted[i]
        assert len(pos) == 20
        q = _bf16_bits_to_f32(wl.q_idx[i]).astype(np.float64)
        deq = torch.from_numpy(wl.k_idx).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        rows = [wl.block_table[i, p // 64] * 64 + p % 64 for p in pos]
        k = deq.reshape(-1, wl.Di)[rows] * wl.k_scale.reshape(-1)[rows, None]
        z = (k @ q.T) / np.linalg.norm(q, axis=1)      # per-head logit in units of sigma
        assert z.mean() > 2.0                          # 3 sigma shift + N(0,1) noise


def test_fp8_query_quantisation():
    """q_idx_fp8 stores the same query draw as e4m3 codes with scale
    max|q_h| / 448 per (row, head): every head's largest code is 448 and the
    dequantised query is within e4m3's half-step of the bf16 one."""
    a = synth.make("c1", batch=3, ctx=100, Hi=4, Di=32, Hq=2, Dqk=8, Dv=4, K=8)
    b = synth.make("c1", batch=3, ctx=100, Hi=4, Di=32, Hq=2, Dqk=8, Dv=4, K=8, q_idx_fp8=True)
    assert b.q_idx.dtype == np.uint8 and b.q_scale.dtype == np.float32
    codes = torch.from_numpy(b.q_idx).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.all(np.abs(codes).max(axis=-1) == 448.0)
    deq = codes * b.q_scale[..., None]
    qa = synth._bf16_bits_to_f32(a.q_idx).astype(np.float64)
    amax = np.abs(qa).max(axis=-1, keepdims=True)
    assert np.all(np.abs(deq - qa) <= amax / 448 * 16 + amax * 2.0 ** -8)
    # the rest of the workload is unchanged
    assert np.array_equal(a.k_idx, b.k_idx) and np.array_equal(a.q, b.q)


def test_e2m1_quantisation_rounds_to_nearest_even_and_saturates():
    """FP4 e2m1 codes: grid values map to themselves, halfway points go to the
    even code (mantissa bit 0), values above 6 saturate, the sign is bit 3."""
    x = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                  0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 100.0, -1.0, -0.74])
    want = [0, 1, 2, 3, 4, 5, 6, 7,
            0, 2, 2, 4, 4, 6, 6, 7, 7, 8 | 2, 8 | 1]
    assert synth.f32_to_e2m1_codes(x).tolist() == want


def test_nvfp4_blocks_bound_the_error():
    """Each block of 16 gets scale e4m3(amax / 6); the dequantised value is
    within half a grid step (at most 1 * scale, the 4 -> 6 gap) of the input,
    plus the clipping of an e4m3 scale rounded below amax / 6."""
    rng = np.random.default_rng(1)
    rows = rng.standard_normal((50, 64)).astype(np.float32)
    packed, scale = synth.quantize_blocks_nvfp4(rows)
    assert packed.shape == (50, 32) and scale.shape == (50, 4)
    codes = np.stack([packed & 15, packed >> 4], axis=-1).reshape(50, 64)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    deq = np.where(codes & 8, -1.0, 1.0) * grid[codes & 7] * np.repeat(scale, 16, axis=1)
    amax = np.abs(rows.reshape(50, 4, 16)).max(axis=-1)
    assert np.all(scale <= amax / 6 * (1 + 2.0 ** -4)) and np.all(scale >= amax / 6 * (1 - 2.0 ** -4))
    bound = np.repeat(scale, 16, axis=1) * 1.0 + np.abs(rows) * 2.0 ** -3
    assert np.all(np.abs(deq - rows) <= bound)


def test_mx_keys_layout_and_encoder_agrees_with_the_oracle():
    """MXFP8 keys: codes and E8M0 bytes per group of 32; unused slots hold NaN
    codes and byte 255.  The generator's numpy encoder and the oracle's
    conversion (separate code, written from the same rule) agree bit for bit,
    negative values that round to zero included."""
    wl = synth.make("c1", batch=3, ctx_list=[100, 64, 1], Hi=2, Di=128, Hq=2, Dqk=8, Dv=4, K=4,
                    idx_mx=True)
    assert wl.k_idx_dtype == "mxe4m3" and wl.k_scale.shape == wl.k_idx.shape[:2] + (4,)
    used = np.zeros(wl.k_idx.shape[:2], dtype=bool)
    for i, c in enumerate(wl.ctx_len):
        for s in range(int(c)):
            used[wl.block_table[i, s // wl.page], s % wl.page] = True
    assert (wl.k_scale[~used] == 255).all() and (wl.k_idx[~used] == 0x7F).all()
    assert (wl.k_scale[used] < 255).all()
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((64, 128)) * 2.0 ** rng.integers(-40, 40, (64, 1))).astype(np.float32)
    x[0, :32] = 0
    x[1, 3] = -1e-30
    x[2, :32] = np.float32(-2.0 ** -130)
    c1, s1 = synth.quantize_groups_mx(x)
    c2, s2 = oracle.mx_quantize(x, "f32")
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)
