"""Seeded synthetic inputs for the indexer -> Top-K -> sparse-attention path.

This module only *generates* data.  It holds none of the method's arithmetic
(no scoring, selection or attention); both the CPU oracle and the CUDA path
consume the bytes it produces.  Everything is drawn from one numpy PCG64
stream per (config, seed) in a fixed order, so a workload is reproducible
byte-for-byte on any host.

Workload shapes follow the five synthetic configurations of the hot path:

  c0  tiny causal prefill, fp32: 1 sequence of 256 tokens, indexer 4x32,
      Top-K 32, attention 4 heads x 64 with separate K and V caches.
  c1  decode, batch 64, context 8192; indexer 64 heads x 128 with FP8 e4m3
      keys (per-token fp32 scale) and bf16 queries; Top-K 2048; attention
      128 query heads over one shared latent row of 576 bf16 (V = first 512).
  c2  causal prefill of 16384 tokens, shapes as c1.
  c3  decode, batch 16, context 131072, shapes as c1, 1% of key positions
      planted with +3 sigma alignment to every indexer head of the query.
  c4  ragged batch of 32 requests with log-uniform contexts in [1024, 65536]:
      28 single-token decodes and 4 chunks of 2048 prefill rows.

Option ``q_idx_fp8=True`` (any config) stores the indexer query quantised the
way the key cache is: e4m3 codes with one fp32 scale per (row, head), scale =
max|q_h| / 448, drawn from the same q_idx values.

Option ``idx_mx=True`` (bf16 configs) stores the indexer keys in MXFP8: e4m3
codes in groups of 32 entries, each group with one E8M0 scale byte (2^(e -
127)) set by the OCP MX rule, exponent floor(log2 max|group|) - 8, codes
rounded to nearest even and clamped at 448 with the sign kept; unused slots
hold NaN codes and scale byte 255.  With ``q_idx_mx=True`` as well the
indexer query is stored the same way (otherwise it stays bf16).

Option ``kv_fp8=True`` (latent-row configs) stores the attention KV cache as
e4m3 codes with one fp32 scale per row and tile of 128 entries (576 entries:
four full tiles and one of 64), scale = max|tile| / 448, quantised from the
same N(0,1) draws; the attention query stays bf16.

Option ``kv_fp4=True`` (latent-row configs) stores it as OCP FP4 e2m1 codes,
two per byte (even entry in the low nibble), in blocks of 16 entries with the
NVFP4 block scale: e4m3(max|block| / 6) (round to nearest even) times a
tensor scale of 1, kept as one fp32 per block; codes round to nearest even
on the e2m1 grid and saturate at +-6.

Draw order (per config): context lengths (c4 only) -> physical block
permutation -> q_idx -> w -> indexer keys (sequence by sequence, logical
order) -> planted positions and offsets (c3) -> attention q -> K/V rows
(sequence by sequence).  Unused slots of a sequence's last page and the
spare pages of the pool are filled with NaN so that any read outside a
sequence's context poisons the result.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

F32, BF16, E4M3, E2M1, MXE4M3 = "f32", "bf16", "e4m3", "e2m1", "mxe4m3"
MX_GROUP = 32                                    # entries per MXFP8 scale
PAGE = 64
E4M3_MAX = 448.0

# Base configurations (names c0..c4).  Overrides shrink them for tests.
CONFIGS = {
    "c0": dict(kind="prefill", L=256, Hi=4, Di=32, K=32, Hq=4, Dqk=64, Dv=64,
               dtype=F32, split_kv=True, q_idx_std=1 / math.sqrt(32),
               k_idx_std=1 / math.sqrt(32), w_scale=1.0, scale=1 / math.sqrt(64),
               seed=0),
    "c1": dict(kind="decode", batch=64, ctx=8192, Hi=64, Di=128, K=2048, Hq=128,
               Dqk=576, Dv=512, dtype=BF16, split_kv=False,
               q_idx_std=1 / math.sqrt(128), k_idx_std=1.0, w_scale=1 / 64,
               scale=1 / math.sqrt(576), seed=1),
    "c2": dict(kind="prefill", L=16384, Hi=64, Di=128, K=2048, Hq=128, Dqk=576,
               Dv=512, dtype=BF16, split_kv=False, q_idx_std=1 / math.sqrt(128),
               k_idx_std=1.0, w_scale=1 / 64, scale=1 / math.sqrt(576), seed=2),
    "c3": dict(kind="decode", batch=16, ctx=131072, Hi=64, Di=128, K=2048,
               Hq=128, Dqk=576, Dv=512, dtype=BF16, split_kv=False,
               q_idx_std=1 / math.sqrt(128), k_idx_std=1.0, w_scale=1 / 64,
               scale=1 / math.sqrt(576), planted=0.01, seed=3),
    "c4": dict(kind="mixed", n_req=32, n_prefill=4, chunk=2048, ctx_lo=1024,
               ctx_hi=65536, Hi=64, Di=128, K=2048, Hq=128, Dqk=576, Dv=512,
               dtype=BF16, split_kv=False, q_idx_std=1 / math.sqrt(128),
               k_idx_std=1.0, w_scale=1 / 64, scale=1 / math.sqrt(576), seed=4),
}


@dataclasses.dataclass
class Workload:
    """Host-side arrays of one workload (all numpy, C-contiguous).

    Storage conventions (shared by oracle and CUDA path):
      * bf16 tensors are uint16 bit patterns, e4m3 tensors uint8 codes.
      * caches are paged: [n_blocks, page, row] in the physical order given
        by ``block_table`` ([n_seq, max_blocks], int32, -1 = unused).
      * query row r belongs to sequence ``q_seq[r]`` at absolute position
        ``q_pos[r]`` and may look at key positions 0..q_pos[r].
    """
    name: str
    Hi: int
    Di: int
    Hq: int
    Dqk: int
    Dv: int
    K: int
    page: int
    scale: float                 # softmax scale of the attention logits
    block_table: np.ndarray      # int32 [n_seq, max_blocks]
    ctx_len: np.ndarray          # int32 [n_seq]
    q_seq: np.ndarray            # int32 [n_q]
    q_pos: np.ndarray            # int32 [n_q]
    q_idx: np.ndarray            # f32, bf16 bits or e4m3 / MX codes [n_q, Hi, Di]
    q_idx_dtype: str
    w: np.ndarray                # f32 [n_q, Hi]
    k_idx: np.ndarray            # f32 or e4m3 / MX codes [n_blocks, page, Di]
    k_idx_dtype: str
    k_scale: Optional[np.ndarray]  # f32 [n_blocks, page], None (=1), or for MX
                                   # keys the E8M0 bytes uint8 [n_blocks, page, Di / 32]
    q: np.ndarray                # f32 or bf16 bits [n_q, Hq, Dqk]
    kv_dtype: str
    k: np.ndarray                # [n_blocks, page, Dqk] (row stride = last dim)
    v: Optional[np.ndarray]      # [n_blocks, page, Dv]; None = V is the first Dv cols of k
    planted: Optional[list] = None  # c3: per-sequence arrays of planted positions
    q_scale: Optional[np.ndarray] = None  # f32 [n_q, Hi] when q_idx holds e4m3 codes,
                                          # uint8 E8M0 [n_q, Hi, Di / 32] for MX codes
    kv_scale: Optional[np.ndarray] = None  # f32 [n_blocks, page, n_tiles] for an e4m3 KV cache
    kv_scale_tile: int = 0                 # entries per KV scale tile (0: none)
    attn_q_dtype: str = ""                 # attention q storage ("" = kv_dtype)

    @property
    def n_q(self) -> int:
        return int(self.q_pos.shape[0])

    @property
    def n_seq(self) -> int:
        return int(self.ctx_len.shape[0])

    @property
    def max_ctx(self) -> int:
        return int(self.q_pos.max()) + 1 if self.n_q else 0

    @property
    def n_blocks(self) -> int:
        return int(self.k.shape[0])


# ---------------------------------------------------------------- encoders

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); NaN kept."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    fin = np.isfinite(x)
    u = np.where(fin, u, 0)          # finite inputs cannot overflow the add below
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    out = r.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Encode float32 values as OCP FP8 e4m3 codes (nearest, ties to even,
    saturating at 448).  Input generation only.

    Normal range: drop the low 20 of float32's 23 mantissa bits with
    round-half-even, then rebias the exponent from 127 to 7.  Below 2^-6 the
    code is the multiple of 2^-9 nearest to |x| (ties to even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    a = np.abs(x)
    u = a.view(np.uint32)
    norm = ((u + np.uint32(0x7FFFF) + ((u >> np.uint32(20)) & np.uint32(1))) >> np.uint32(20))
    norm = norm.astype(np.int32) - (120 << 3)
    sub = np.rint(a * np.float32(512.0)).astype(np.int32)
    code = np.where(a < np.float32(2.0 ** -6), sub, norm)
    code = np.minimum(code, 0x7E)
    code = np.where((x < 0) & (code != 0), code | 0x80, code)
    return code.astype(np.uint8)


KV_TILE = 128
FP4_BLOCK = 16                                   # entries per NVFP4 block scale
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def f32_to_e2m1_codes(x: np.ndarray) -> np.ndarray:
    """OCP FP4 e2m1 codes (uint8, one per value) of x: round to nearest on
    the grid 0, 0.5, 1, 1.5, 2, 3, 4, 6, ties to the even code (mantissa bit
    0), saturating at 6; the sign is bit 3."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x)
    # count the midpoints below a; at a midpoint, ">" keeps the lower code and
    # ">=" takes the upper, whichever of the two has mantissa bit 0
    code = np.zeros(a.shape, dtype=np.uint8)
    for mid, upper_even in ((0.25, False), (0.75, True), (1.25, False), (1.75, True),
                            (2.5, False), (3.5, True), (5.0, False)):
        code += (a >= mid) if upper_even else (a > mid)
    return np.where(np.signbit(x) & (code != 0), code | 8, code).astype(np.uint8)


def quantize_blocks_nvfp4(rows: np.ndarray, block: int = FP4_BLOCK):
    """NVFP4-style storage along the last axis (a multiple of 2 * block):
    returns (packed codes uint8 [..., D / 2], block scales float32
    [..., D / block]) with scale = e4m3(max|block| / 6)."""
    rows = np.asarray(rows, dtype=np.float32)
    d = rows.shape[-1]
    assert d % block == 0 and block % 2 == 0
    blk = rows.reshape(rows.shape[:-1] + (d // block, block))
    amax = np.abs(blk).max(axis=-1)
    sc_code = f32_to_e4m3_bits(np.maximum(amax / np.float32(6.0), np.float32(2.0 ** -9)))
    scale = _e4m3_bits_to_f32(sc_code)
    codes = f32_to_e2m1_codes(blk / scale[..., None]).reshape(rows.shape)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return packed, scale.astype(np.float32)


def _e4m3_bits_to_f32(c: np.ndarray) -> np.ndarray:
    c = np.asarray(c).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e, m = (c >> 3) & 0xF, c & 0x7
    return (sign * np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7))).astype(
        np.float32)


def quantize_tiles_e4m3(rows: np.ndarray, tile: int = KV_TILE):
    """Per-(row, tile) FP8 storage along the last axis: each run of `tile`
    entries (the last one may be shorter) gets scale = amax/448.  Returns
    (codes uint8 [..., D], scales float32 [..., ceil(D / tile)])."""
    rows = np.asarray(rows, dtype=np.float32)
    d = rows.shape[-1]
    nt = (d + tile - 1) // tile
    codes = np.empty(rows.shape, dtype=np.uint8)
    scales = np.empty(rows.shape[:-1] + (nt,), dtype=np.float32)
    for t in range(nt):
        c, sc = quantize_rows_e4m3(rows[..., t * tile: min(d, (t + 1) * tile)])
        codes[..., t * tile: min(d, (t + 1) * tile)] = c
        scales[..., t] = sc
    return codes, scales


def quantize_rows_e4m3(rows: np.ndarray):
    """Per-row (per-token) FP8 storage: scale = amax(|row|)/448, codes =
    e4m3(row/scale).  Returns (codes uint8, scale float32)."""
    rows = np.asarray(rows, dtype=np.float32)
    amax = np.abs(rows).max(axis=-1)
    scale = (np.maximum(amax, np.float32(1e-30)) / np.float32(E4M3_MAX)).astype(np.float32)
    codes = f32_to_e4m3_bits(rows / scale[..., None])
    return codes, scale


def quantize_groups_mx(x: np.ndarray):
    """MXFP8 storage along the last axis (a multiple of 32): per group of 32,
    exponent E = floor(log2 max|group|) - 8 clamped to [-127, 127] (-127 for
    an all-zero group), codes = e4m3(x / 2^E) with the sign of x kept.
    Returns (codes uint8 [..., D], E8M0 bytes uint8 [..., D / 32])."""
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[-1]
    assert d % MX_GROUP == 0
    g = x.reshape(x.shape[:-1] + (d // MX_GROUP, MX_GROUP)).astype(np.float64)
    amax = np.abs(g).max(axis=-1)
    _, ex = np.frexp(amax)                       # amax = m 2^ex, m in [0.5, 1)
    E = np.where(amax > 0, ex.astype(np.int64) - 1 - 8, -127)
    E = np.clip(E, -127, 127)
    y = np.ldexp(g, -E[..., None]).astype(np.float32)
    mag = f32_to_e4m3_bits(np.abs(y))
    codes = np.where(np.signbit(g), mag | 0x80, mag).astype(np.uint8).reshape(x.shape)
    return codes, (E + 127).astype(np.uint8)


# ---------------------------------------------------------------- layout

def _paged_pool(rng, ctx_len, page, spare=2):
    """Shuffled physical page assignment: logical block j of sequence i lives
    at physical block ``block_table[i, j]``."""
    nb = [(c + page - 1) // page for c in ctx_len]
    total = int(sum(nb)) + spare
    perm = rng.permutation(total).astype(np.int32)
    max_blocks = max(nb) if nb else 1
    bt = np.full((len(ctx_len), max_blocks), -1, dtype=np.int32)
    off = 0
    for i, n in enumerate(nb):
        bt[i, :n] = perm[off:off + n]
        off += n
    return bt, total


def _scatter_rows(pool, bt, seq, rows, page):
    """Write logical rows [0, len(rows)) of sequence ``seq`` into the pool."""
    n = rows.shape[0]
    for j in range((n + page - 1) // page):
        lo, hi = j * page, min(n, (j + 1) * page)
        pool[bt[seq, j], : hi - lo] = rows[lo:hi]


def _normal(rng, shape, std=1.0):
    return (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std))


# ---------------------------------------------------------------- builder

def config(name: str, **over) -> dict:
    cfg = dict(CONFIGS[name])
    cfg.update(over)
    return cfg


def make(name: str, seed: Optional[int] = None, **over) -> Workload:
    """Build workload ``name`` (c0..c4) with optional size overrides, e.g.
    ``make("c1", batch=4, ctx=3000)``.  ``seed`` defaults to the config's."""
    cfg = config(name, **over)
    if seed is None:
        seed = cfg["seed"]
    rng = np.random.Generator(np.random.PCG64(seed))
    page = cfg.get("page", PAGE)
    Hi, Di, Hq, Dqk, Dv = cfg["Hi"], cfg["Di"], cfg["Hq"], cfg["Dqk"], cfg["Dv"]
    kind = cfg["kind"]

    # 1. request structure: (ctx_len per sequence, query rows)
    if kind == "prefill":
        L = cfg["L"]
        ctx_len = np.array([L], dtype=np.int32)
        q_seq = np.zeros(L, dtype=np.int32)
        q_pos = np.arange(L, dtype=np.int32)
    elif kind == "decode":
        B, ctx = cfg["batch"], cfg["ctx"]
        ctxs = cfg.get("ctx_list")
        ctx_len = np.array(ctxs if ctxs is not None else [ctx] * B, dtype=np.int32)
        q_seq = np.arange(len(ctx_len), dtype=np.int32)
        q_pos = ctx_len - 1
    elif kind == "mixed":
        n_req, n_pf, chunk = cfg["n_req"], cfg["n_prefill"], cfg["chunk"]
        lo, hi = math.log(cfg["ctx_lo"]), math.log(cfg["ctx_hi"])
        existing = np.exp(rng.uniform(lo, hi, size=n_req)).astype(np.int64)
        existing = np.clip(existing, cfg["ctx_lo"], cfg["ctx_hi"]).astype(np.int32)
        # the first n_req - n_pf requests decode one token, the rest prefill a chunk
        new_tok = np.array([1] * (n_req - n_pf) + [chunk] * n_pf, dtype=np.int32)
        ctx_len = (existing + new_tok).astype(np.int32)
        q_seq_l, q_pos_l = [], []
        for i in range(n_req):
            q_seq_l.append(np.full(new_tok[i], i, dtype=np.int32))
            q_pos_l.append(np.arange(existing[i], existing[i] + new_tok[i], dtype=np.int32))
        q_seq = np.concatenate(q_seq_l)
        q_pos = np.concatenate(q_pos_l)
    else:
        raise ValueError(kind)
    n_seq = len(ctx_len)
    n_q = len(q_pos)

    # 2. physical page placement (shared by the indexer-key and KV caches)
    bt, n_blocks = _paged_pool(rng, ctx_len.tolist(), page)

    fp32 = cfg["dtype"] == F32

    # 3. indexer queries and head weights; with q_idx_fp8 the query is
    # stored as e4m3 codes with one fp32 scale per (row, head)
    qi = _normal(rng, (n_q, Hi, Di), cfg["q_idx_std"])
    q8 = bool(cfg.get("q_idx_fp8", False))
    mx = bool(cfg.get("idx_mx", False))
    q_mx = bool(cfg.get("q_idx_mx", False))
    if (mx or q_mx) and fp32:
        raise ValueError("idx_mx applies to the bf16 configurations")
    if q_mx and not mx:
        raise ValueError("q_idx_mx needs idx_mx")
    if q_mx and q8:
        raise ValueError("q_idx_mx and q_idx_fp8 exclude each other")
    q_scale = None
    if q_mx:
        q_idx, q_scale = quantize_groups_mx(qi)
        q_idx_dtype = MXE4M3
    elif q8:
        q_idx, q_scale = quantize_rows_e4m3(qi)
        q_idx_dtype = E4M3
    else:
        q_idx = qi if fp32 else f32_to_bf16_bits(qi)
        q_idx_dtype = F32 if fp32 else BF16
    w = (rng.random(size=(n_q, Hi), dtype=np.float32) * np.float32(cfg["w_scale"])).astype(np.float32)

    # 4. indexer keys, logical order, sequence by sequence
    k_idx = np.full((n_blocks, page, Di), np.nan if fp32 else 0, dtype=np.float32 if fp32 else np.uint8)
    if not fp32:
        k_idx[:] = 0x7F                       # e4m3 NaN in unused slots
    if mx:
        k_scale = np.full((n_blocks, page, Di // MX_GROUP), 255, dtype=np.uint8)
    else:
        k_scale = None if fp32 else np.full((n_blocks, page), np.nan, dtype=np.float32)
    planted = None
    raw_keys = []
    for i in range(n_seq):
        raw_keys.append(_normal(rng, (int(ctx_len[i]), Di), cfg["k_idx_std"]))

    # 5. planted structure (c3): 1% of positions aligned with every head of
    # the sequence's query by +3 sigma, sigma = ||q_h|| (std of q_h . k, k ~ N(0, I)).
    if cfg.get("planted"):
        planted = []
        for i in range(n_seq):
            c = int(ctx_len[i])
            n_pl = int(round(cfg["planted"] * c))
            pos = np.sort(rng.choice(c, size=n_pl, replace=False)).astype(np.int32)
            rows = np.nonzero(q_seq == i)[0]
            qmat = (qi[rows[-1]] if (fp32 or q8 or q_mx) else _bf16_bits_to_f32(q_idx[rows[-1]]))
            qmat = qmat.astype(np.float64)
            target = 3.0 * np.linalg.norm(qmat, axis=1)
            delta = qmat.T @ np.linalg.solve(qmat @ qmat.T, target)   # min-norm solution
            raw_keys[i][pos] += delta.astype(np.float32)
            planted.append(pos)

    for i in range(n_seq):
        if fp32:
            _scatter_rows(k_idx, bt, i, raw_keys[i], page)
        else:
            codes, sc = (quantize_groups_mx if mx else quantize_rows_e4m3)(raw_keys[i])
            _scatter_rows(k_idx, bt, i, codes, page)
            _scatter_rows(k_scale, bt, i, sc, page)
    del raw_keys

    # 6. attention queries
    qa = _normal(rng, (n_q, Hq, Dqk))
    q = qa if fp32 else f32_to_bf16_bits(qa)
    del qa

    # 7. K/V rows
    kv_scale = None
    kv_dtype = F32 if fp32 else BF16
    if (cfg.get("kv_fp8") or cfg.get("kv_fp4")) and (cfg["split_kv"] or fp32):
        raise ValueError("kv_fp8 / kv_fp4 apply to the bf16 latent-row configurations")
    if cfg.get("kv_fp8") and cfg.get("kv_fp4"):
        raise ValueError("kv_fp8 and kv_fp4 exclude each other")
    if cfg.get("kv_fp8"):
        kv_dtype = E4M3
    if cfg.get("kv_fp4"):
        kv_dtype = E2M1
    if cfg["split_kv"]:
        k = np.full((n_blocks, page, Dqk), np.nan, dtype=np.float32)
        v = np.full((n_blocks, page, Dv), np.nan, dtype=np.float32)
        for i in range(n_seq):
            c = int(ctx_len[i])
            _scatter_rows(k, bt, i, _normal(rng, (c, Dqk)), page)
            _scatter_rows(v, bt, i, _normal(rng, (c, Dv)), page)
        if not fp32:
            k, v = f32_to_bf16_bits(k), f32_to_bf16_bits(v)
    else:
        kv8 = bool(cfg.get("kv_fp8", False))
        kv4 = bool(cfg.get("kv_fp4", False))
        if kv8:
            k = np.full((n_blocks, page, Dqk), 0x7F, dtype=np.uint8)     # e4m3 NaN when unused
            n_tiles = (Dqk + KV_TILE - 1) // KV_TILE
            kv_scale = np.full((n_blocks, page, n_tiles), np.nan, dtype=np.float32)
        elif kv4:
            # e2m1 has no NaN: unused slots get NaN block scales instead
            k = np.zeros((n_blocks, page, Dqk // 2), dtype=np.uint8)
            kv_scale = np.full((n_blocks, page, Dqk // FP4_BLOCK), np.nan, dtype=np.float32)
        else:
            k = np.full((n_blocks, page, Dqk), np.nan if fp32 else 0x7FC0,
                        dtype=np.float32 if fp32 else np.uint16)
        v = None
        for i in range(n_seq):
            c = int(ctx_len[i])
            # draw in pieces to bound host memory for long contexts
            step = 16384
            for s0 in range(0, c, step):
                s1 = min(c, s0 + step)
                rows = _normal(rng, (s1 - s0, Dqk))
                if kv8:
                    rows, rsc = quantize_tiles_e4m3(rows)
                elif kv4:
                    rows, rsc = quantize_blocks_nvfp4(rows)
                else:
                    rows = rows if fp32 else f32_to_bf16_bits(rows)
                for j in range(s0 // page, (s1 + page - 1) // page):
                    lo, hi = j * page, min(s1, (j + 1) * page)
                    k[bt[i, j], lo - j * page: hi - j * page] = rows[lo - s0: hi - s0]
                    if kv8 or kv4:
                        kv_scale[bt[i, j], lo - j * page: hi - j * page] = rsc[lo - s0: hi - s0]

    return Workload(
        name=name, Hi=Hi, Di=Di, Hq=Hq, Dqk=Dqk, Dv=Dv, K=int(cfg["K"]), page=page,
        scale=float(cfg["scale"]), block_table=bt, ctx_len=ctx_len, q_seq=q_seq,
        q_pos=q_pos, q_idx=q_idx, q_idx_dtype=q_idx_dtype, w=w,
        k_idx=k_idx, k_idx_dtype=F32 if fp32 else (MXE4M3 if mx else E4M3), k_scale=k_scale, q=q,
        kv_dtype=kv_dtype, k=k, v=v, planted=planted, q_scale=q_scale, kv_scale=kv_scale,
        kv_scale_tile=(FP4_BLOCK if kv_dtype == E2M1 else KV_TILE) if kv_scale is not None else 0,
        attn_q_dtype=F32 if fp32 else BF16)


def _bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def permute_pages(wl: Workload, seed: int) -> Workload:
    """Same logical content, different physical page placement."""
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = rng.permutation(wl.n_blocks).astype(np.int32)     # old block b -> new perm[b]
    inv = np.empty_like(perm)
    inv[perm] = np.arange(wl.n_blocks, dtype=np.int32)

    def mv(a):
        return None if a is None else np.ascontiguousarray(a[inv])

    bt = np.where(wl.block_table >= 0, perm[np.maximum(wl.block_table, 0)], -1).astype(np.int32)
    return dataclasses.replace(wl, block_table=bt, k_idx=mv(wl.k_idx), k_scale=mv(wl.k_scale),
                               k=mv(wl.k), v=mv(wl.v), kv_scale=mv(wl.kv_scale))


def candidates(wl: Workload, n_cand: int, seed: int = 0, pad_beyond: int = 0) -> np.ndarray:
    """Candidate position lists [n_q, n_cand] int32 for candidate-restricted
    selection: row r draws min(n_cand, pos + 1) distinct positions uniformly
    from 0..pos (its own PCG64 stream, seeded by `seed`), sorted ascending and
    padded with -1.  With pad_beyond > 0, that many entries after a row's
    draws (where room is left) are set to positions past the row's pos, which
    are not candidates."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = np.full((wl.n_q, n_cand), -1, dtype=np.int32)
    for r in range(wl.n_q):
        pos = int(wl.q_pos[r])
        m = min(n_cand, pos + 1)
        pick = rng.choice(pos + 1, size=m, replace=False) if m < pos + 1 else np.arange(pos + 1)
        out[r, :m] = np.sort(pick).astype(np.int32)
        extra = min(pad_beyond, n_cand - m)
        if extra > 0:
            out[r, m:m + extra] = pos + 1 + np.arange(extra, dtype=np.int32)
    return out
