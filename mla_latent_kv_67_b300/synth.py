"""Seeded synthetic inputs for absorbed-MLA decode workloads.

This module draws random numbers and lays them out in memory; it holds none of
the attention arithmetic. Both the CUDA path (through tests and bench.py) and
the fp64 oracle take their inputs from here, and from nowhere else.

Value recipe (stated once, used everywhere):

* latent cache rows ``[c_kv | k_R]`` and queries ``[q_C | q_R]`` ~ N(0, 1);
* weights ~ N(0, 1/fan_in) (variance 1/fan_in);
* token hidden states ``x`` ~ N(0, 1);
* bf16 workloads round every drawn value to bf16 (round-to-nearest-even) once,
  here, so both sides see exactly the same numbers;
* fp8 workloads store the cache's latent part as E4M3 codes with one float
  scale per row (scale = max |c| / 448, codes = c / scale rounded to the
  nearest E4M3 value, ties to even) and its RoPE part in bf16; everything
  else is bf16. Both sides see the decoded values code * scale;
* context lengths are either fixed or uniform integers in ``[lo, hi]``
  (inclusive);
* the physical page pool is a seeded random permutation of all logical pages
  (the block table), so neighbouring logical pages sit far apart in memory.

Every array is a pure function of ``(workload.seed, stream id, index)``: the
cache is drawn page by page, so any sequence's rows can be regenerated alone
(the oracle checks sampled sequences without rebuilding the whole pool).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np

# Rows of a physical page that no sequence owns are filled with this value.
# It is large enough that a kernel which forgets to mask the ragged tail of a
# sequence produces a visibly wrong result.
PAD_VALUE = 300.0

# Stream ids: one per kind of drawn tensor.
_S_LENS, _S_PERM, _S_CACHE, _S_QUERY, _S_X, _S_W = 1, 2, 3, 4, 5, 6
_W_IDS = {"w_dkv": 1, "w_kr": 2, "w_uk": 3, "w_uv": 4, "w_dq": 5,
          "w_uq": 6, "w_qr": 7, "w_o": 8}


@dataclass(frozen=True)
class Workload:
    """Shape and value recipe of one decode workload.

    ``mode``:
      * ``"attn"``   - queries and the latent cache are drawn directly
                       (absorb_q -> attention -> absorb_out);
      * ``"layer"``  - one new token per sequence: x is drawn, appended to a
                       cache pre-filled with ``ctx - 1`` drawn rows, the query
                       is projected from x, and the output goes through W^O;
      * ``"prefill"``- a single sequence whose whole cache is produced by the
                       append step from drawn x at positions 0..ctx-1; the
                       query is projected from the last token (no W^O).
      * ``"prefill_mha"`` - the same single sequence, but every one of its
                       ctx tokens is a query: causal attention in the MHA form
                       over keys and values expanded from the latent rows.
    """

    name: str
    batch: int
    n_h: int = 128
    d_h: int = 128
    d_r: int = 64
    d_c: int = 512
    d_v: int = 128
    d_model: int = 0
    d_cq: int = 0
    page_size: int = 64
    ctx: int = 4096
    ctx_range: tuple[int, int] | None = None
    dtype: str = "bf16"
    mode: str = "attn"
    rope_base: float = 10000.0
    seed: int = 67000
    shuffle_pages: bool = True
    spare_pages: int = 0
    lens: tuple[int, ...] | None = None   # explicit per-sequence lengths
    q_len: int = 1                        # new tokens decoded per sequence at once
    fused: bool = False                   # full layer with W^UK / W^UV folded into W^UQ / W^O

    @property
    def row_width(self) -> int:
        return self.d_c + self.d_r

    @property
    def scale(self) -> float:
        return float(1.0 / np.sqrt(self.d_h + self.d_r))

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the DeepSeek-V2-shaped decode benchmark.
WORKLOADS: dict[str, Workload] = {
    "tiny_f32_ctx256": Workload(
        name="tiny_f32_ctx256", batch=1, n_h=8, d_h=32, d_r=16, d_c=64,
        d_v=32, d_model=128, d_cq=0, page_size=256, ctx=256, dtype="f32",
        mode="prefill", seed=67001, shuffle_pages=False),
    "dsv2_b32_ctx4k": Workload(
        name="dsv2_b32_ctx4k", batch=32, ctx=4096, seed=67002),
    "dsv2_b4_ctx128k": Workload(
        name="dsv2_b4_ctx128k", batch=4, ctx=131072, seed=67003),
    "dsv2_b128_ragged": Workload(
        name="dsv2_b128_ragged", batch=128, ctx=0, ctx_range=(512, 16384),
        seed=67004),
    "dsv2_layer_b64_ctx32k": Workload(
        name="dsv2_layer_b64_ctx32k", batch=64, d_model=5120, d_cq=1536,
        ctx=32768, mode="layer", seed=67005),
}

# Beyond the five: two new tokens per sequence decoded at once (multi-token
# prediction / a speculative draft), on the batch-32, 4096-token shape.
# The full-layer step again with the absorption folded into the weights
# once (W~^Q, W~^O) instead of applied per head at every step.
EXTRA_WORKLOADS: dict[str, Workload] = {
    "dsv2_b32_ctx4k_mtp2": Workload(name="dsv2_b32_ctx4k_mtp2", batch=32, ctx=4096, q_len=2,
                                    seed=67006),
    # the batch-32, 4096-token decode over an FP8 latent cache
    "dsv2_b32_ctx4k_fp8": Workload(name="dsv2_b32_ctx4k_fp8", batch=32, ctx=4096, dtype="fp8",
                                   seed=67008),
    "dsv2_layer_b64_ctx32k_fused": WORKLOADS["dsv2_layer_b64_ctx32k"].replace(
        name="dsv2_layer_b64_ctx32k_fused", fused=True),
    # a 4096-token prompt prefilled in the MHA form (DeepSeek-V2 shapes)
    "dsv2_prefill_4k": Workload(name="dsv2_prefill_4k", batch=1, ctx=4096, d_model=5120,
                                d_cq=1536, mode="prefill_mha", seed=67007, shuffle_pages=True),
}


def _rng(wl: Workload, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([wl.seed, *key])))


# ---------------------------------------------------------------- bf16 codec
def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    u = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (u >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_bf16(a: np.ndarray) -> np.ndarray:
    """float32 values rounded to the nearest bf16 (returned as float32)."""
    return bf16_to_f32(bf16_bits(a))


def _draw(wl: Workload, g: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    v = g.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    return round_bf16(v) if wl.dtype in ("bf16", "fp8") else v


def storage(wl: Workload, a: np.ndarray) -> np.ndarray:
    """Device storage form of float32 values: uint16 bf16 bits or float32
    (fp8 workloads keep everything but the cache in bf16)."""
    if wl.dtype in ("bf16", "fp8"):
        return bf16_bits(a)
    return np.ascontiguousarray(a, np.float32)


# ------------------------------------------------------------ E4M3 format
def _e4m3_table() -> np.ndarray:
    """Value of every E4M3 code (OCP FP8: 1 sign, 4 exponent bits with bias
    7, 3 mantissa bits; exponent 0 is subnormal; 0x7F / 0xFF are NaN)."""
    out = np.empty(256, np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e, m = (code >> 3) & 0xF, code & 0x7
        if e == 15 and m == 7:
            out[code] = np.nan
        elif e == 0:
            out[code] = sign * (m / 8.0) * 2.0 ** -6
        else:
            out[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


E4M3 = _e4m3_table()
E4M3_MAX = 448.0


def e4m3_codes(x: np.ndarray) -> np.ndarray:
    """float32 -> the nearest finite E4M3 code (ties to the even code),
    magnitudes past 448 clamped to 448."""
    x = np.asarray(x, np.float32)
    a = np.abs(x).astype(np.float64)
    pos = E4M3[:127]                          # codes 0x00 .. 0x7E, ascending
    idx = np.clip(np.searchsorted(pos, a), 1, 126)
    lo, hi = pos[idx - 1], pos[idx]
    up = (a - lo > hi - a) | ((a - lo == hi - a) & (idx % 2 == 0))
    code = np.where(up, idx, idx - 1)
    code = np.where(a >= E4M3_MAX, 126, code).astype(np.uint8)
    return code | np.where(np.signbit(x), np.uint8(0x80), np.uint8(0))


def fp8_row_bytes(d_c: int, d_r: int) -> int:
    return (d_c + 2 * d_r + 4 + 15) // 16 * 16


def fp8_rows(wl: Workload, rows: np.ndarray):
    """float32 cache rows [n][d_c + d_r] -> (the FP8 row bytes [n][row_bytes],
    the values they decode to, float32 [n][d_c + d_r])."""
    rows = np.asarray(rows, np.float32)
    c, k = rows[:, :wl.d_c], rows[:, wl.d_c:]
    amax = np.max(np.abs(c), axis=1)
    s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    codes = e4m3_codes(c / s[:, None])
    dec = np.empty_like(rows)
    dec[:, :wl.d_c] = E4M3[codes].astype(np.float32) * s[:, None]
    kb = bf16_bits(k)
    dec[:, wl.d_c:] = bf16_to_f32(kb)
    rb = fp8_row_bytes(wl.d_c, wl.d_r)
    out = np.zeros((rows.shape[0], rb), np.uint8)
    out[:, :wl.d_c] = codes
    out[:, wl.d_c:wl.d_c + 2 * wl.d_r] = kb.view(np.uint8).reshape(rows.shape[0], -1)
    out[:, wl.d_c + 2 * wl.d_r:wl.d_c + 2 * wl.d_r + 4] = s.view(np.uint8).reshape(-1, 4)
    return out, dec


# ---------------------------------------------------------- lengths / paging
def seq_lens(wl: Workload) -> np.ndarray:
    if wl.lens is not None:
        assert len(wl.lens) == wl.batch
        return np.asarray(wl.lens, dtype=np.int32)
    if wl.ctx_range is None:
        return np.full(wl.batch, wl.ctx, dtype=np.int32)
    lo, hi = wl.ctx_range
    return _rng(wl, _S_LENS).integers(lo, hi + 1, size=wl.batch, dtype=np.int64).astype(np.int32)


def pages_needed(lens: np.ndarray, page_size: int) -> np.ndarray:
    return (np.asarray(lens, np.int64) + page_size - 1) // page_size


def block_table(wl: Workload, lens: np.ndarray) -> tuple[np.ndarray, int]:
    """Block table ``[B][max_pages]`` (int32, -1 past a sequence's pages) and
    the physical pool size. Logical pages are laid out sequence after
    sequence and then, if ``shuffle_pages``, scattered by a seeded
    permutation of the pool. ``spare_pages`` extra pages are never mapped."""
    npg = pages_needed(lens, wl.page_size)
    total = int(npg.sum())
    pool = total + wl.spare_pages
    perm = (_rng(wl, _S_PERM).permutation(pool) if wl.shuffle_pages
            else np.arange(pool))
    max_pages = int(npg.max()) if len(npg) else 0
    bt = np.full((wl.batch, max(max_pages, 1)), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(npg):
        bt[b, :n] = perm[off:off + n]
        off += int(n)
    return bt, pool


def cache_page(wl: Workload, b: int, p: int) -> np.ndarray:
    """Logical page ``p`` of sequence ``b``: float32 ``[page_size][d_c+d_r]``
    (for fp8 workloads the values the stored FP8 rows decode to)."""
    if wl.dtype == "fp8":
        raw = _rng(wl, _S_CACHE, b, p).standard_normal((wl.page_size, wl.row_width),
                                                       dtype=np.float32)
        return fp8_rows(wl, raw)[1]
    return _draw(wl, _rng(wl, _S_CACHE, b, p), (wl.page_size, wl.row_width))


def cache_rows(wl: Workload, b: int, n_rows: int) -> np.ndarray:
    """The first ``n_rows`` drawn cache rows of sequence ``b`` (float32)."""
    if n_rows <= 0:
        return np.zeros((0, wl.row_width), np.float32)
    npg = (n_rows + wl.page_size - 1) // wl.page_size
    rows = np.concatenate([cache_page(wl, b, p) for p in range(npg)], axis=0)
    return rows[:n_rows]


def drawn_rows(wl: Workload, lens: np.ndarray) -> np.ndarray:
    """How many cache rows of each sequence are drawn (not produced by the
    append step)."""
    lens = np.asarray(lens)
    if wl.mode == "attn":
        return lens.copy()
    if wl.mode == "layer":
        return lens - 1
    return np.zeros_like(lens)  # prefill modes: every row comes from the append step


def paged_cache(wl: Workload, lens: np.ndarray, bt: np.ndarray, pool: int) -> np.ndarray:
    """The physical page pool in storage form ``[pool][page_size][d_c+d_r]``.

    Rows a sequence owns hold its drawn rows; rows to be written by the append
    step, rows past a sequence's end and unmapped pages hold ``PAD_VALUE``."""
    P, W = wl.page_size, wl.row_width
    pad = np.float32(PAD_VALUE)
    if wl.dtype == "fp8":
        return _paged_cache_fp8(wl, lens, bt, pool)
    out = np.empty((pool, P, W), dtype=np.uint16 if wl.dtype == "bf16" else np.float32)
    out[...] = storage(wl, np.full((1,), pad, np.float32))[0]
    nd = drawn_rows(wl, lens)
    for b in range(wl.batch):
        n = int(nd[b])
        for p in range((n + P - 1) // P):
            page = cache_page(wl, b, p)
            keep = min(P, n - p * P)
            if keep < P:
                page = page.copy()
                page[keep:] = pad
            out[bt[b, p]] = storage(wl, page)
    return out


def _paged_cache_fp8(wl: Workload, lens, bt, pool) -> np.ndarray:
    """The FP8 page pool ``[pool][page_size][row_bytes]`` (attention-only
    workloads: every owned row drawn; other rows encode PAD_VALUE)."""
    P, W = wl.page_size, wl.row_width
    pad_row = fp8_rows(wl, np.full((1, W), PAD_VALUE, np.float32))[0][0]
    out = np.empty((pool, P, fp8_row_bytes(wl.d_c, wl.d_r)), np.uint8)
    out[...] = pad_row
    nd = drawn_rows(wl, lens)
    for b in range(wl.batch):
        n = int(nd[b])
        for p in range((n + P - 1) // P):
            raw = _rng(wl, _S_CACHE, b, p).standard_normal((P, W), dtype=np.float32)
            enc = fp8_rows(wl, raw)[0]
            keep = min(P, n - p * P)
            page = out[bt[b, p]]
            page[:keep] = enc[:keep]
    return out


# ------------------------------------------------------- queries / weights
def query(wl: Workload) -> np.ndarray:
    """Drawn queries ``[B * q_len][n_h][d_h+d_r]`` (no-PE part first, RoPE
    part last; row ``b * q_len + t`` is new token t of sequence b), treated
    as already rotated."""
    return _draw(wl, _rng(wl, _S_QUERY), (wl.batch * wl.q_len, wl.n_h, wl.d_h + wl.d_r))


def tokens(wl: Workload) -> np.ndarray:
    """Hidden states x: ``[ctx][d_model]`` (prefill modes) or ``[B][d_model]``."""
    n = wl.ctx if wl.mode in ("prefill", "prefill_mha") else wl.batch
    return _draw(wl, _rng(wl, _S_X), (n, wl.d_model))


def weight(wl: Workload, name: str) -> np.ndarray:
    """One weight in the column-vector convention ``W in R^{out x in}``,
    stored row-major ``[out][in]``, drawn N(0, 1/in)."""
    shapes = {
        "w_dkv": (wl.d_c, wl.d_model),
        "w_kr": (wl.d_r, wl.d_model),
        "w_uk": (wl.n_h * wl.d_h, wl.d_c),
        "w_uv": (wl.n_h * wl.d_v, wl.d_c),
        "w_dq": (wl.d_cq, wl.d_model),
        "w_uq": (wl.n_h * wl.d_h, wl.d_cq or wl.d_model),
        "w_qr": (wl.n_h * wl.d_r, wl.d_cq or wl.d_model),
        "w_o": (wl.d_model, wl.n_h * wl.d_v),
    }
    out_dim, in_dim = shapes[name]
    return _draw(wl, _rng(wl, _S_W, _W_IDS[name]), (out_dim, in_dim), std=in_dim ** -0.5)


# ------------------------------------------------- joint (device) layouts
def joint_w_dkv_kr(w_dkv: np.ndarray, w_kr: np.ndarray) -> np.ndarray:
    """``[(d_c+d_r)][d_model]``: rows of W^DKV then rows of W^KR, so one
    product yields a whole cache row ``[c_kv | k_R(before RoPE)]``."""
    return np.ascontiguousarray(np.concatenate([w_dkv, w_kr], axis=0))


def joint_w_uq_qr(w_uq: np.ndarray, w_qr: np.ndarray, n_h: int) -> np.ndarray:
    """``[n_h][(d_h+d_r)][in]``: per head the d_h rows of W^UQ then the d_r
    rows of W^QR, so one product yields ``[q_C | q_R(before RoPE)]`` per
    head."""
    d_in = w_uq.shape[1]
    a = w_uq.reshape(n_h, -1, d_in)
    r = w_qr.reshape(n_h, -1, d_in)
    return np.ascontiguousarray(np.concatenate([a, r], axis=1).reshape(-1, d_in))
