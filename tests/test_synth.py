"""The seeded input generator: determinism, bf16 rounding, paging layout."""
import numpy as np

from mla_latent_kv_67_b300 import synth


def test_bf16_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 3.0e38], np.float32)
    got = synth.round_bf16(x)
    # 1+2^-8 is a tie between 1 and 1+2^-7: even mantissa wins (1.0)
    want = np.array([1.0, 1.0, 1.0 + 2 ** -6, 1.0, -2.5, np.float32(3.0e38)], np.float32)
    assert np.array_equal(got[:5], want[:5])
    assert abs(got[5] / 3.0e38 - 1) < 2 ** -8
    v = np.random.default_rng(0).standard_normal(10000).astype(np.float32)
    r = synth.round_bf16(v)
    assert np.all(np.abs(r - v) <= np.abs(v) * 2 ** -8)
    assert np.array_equal(synth.round_bf16(r), r)


def test_block_table_is_a_permutation_and_deterministic():
    wl = synth.WORKLOADS["dsv2_b128_ragged"].replace(batch=9, spare_pages=3)
    lens = synth.seq_lens(wl)
    assert lens.min() >= 512 and lens.max() <= 16384
    bt, pool = synth.block_table(wl, lens)
    npg = synth.pages_needed(lens, wl.page_size)
    used = np.concatenate([bt[b, :n] for b, n in enumerate(npg)])
    assert pool == npg.sum() + 3 and len(set(used.tolist())) == len(used)
    assert used.min() >= 0 and used.max() < pool
    for b, n in enumerate(npg):
        assert np.all(bt[b, n:] == -1)
    bt2, _ = synth.block_table(wl, synth.seq_lens(wl))
    assert np.array_equal(bt, bt2)


def test_paged_cache_places_logical_pages():
    wl = synth.WORKLOADS["dsv2_b32_ctx4k"].replace(batch=3, ctx=200)
    lens = synth.seq_lens(wl)
    bt, pool = synth.block_table(wl, lens)
    cache = synth.paged_cache(wl, lens, bt, pool)
    for b in range(3):
        rows = synth.cache_rows(wl, b, 200)
        phys = np.concatenate([cache[bt[b, p]] for p in range(4)])
        assert np.array_equal(synth.bf16_to_f32(phys[:200]), rows)
        assert np.all(synth.bf16_to_f32(phys[200:]) == synth.PAD_VALUE)


def test_layer_mode_leaves_append_slot_padded():
    wl = synth.WORKLOADS["dsv2_layer_b64_ctx32k"].replace(batch=2, ctx=130, d_model=64, d_cq=32)
    lens = synth.seq_lens(wl)
    bt, pool = synth.block_table(wl, lens)
    cache = synth.bf16_to_f32(synth.paged_cache(wl, lens, bt, pool))
    for b in range(2):
        p, r = divmod(129, 64)
        assert np.all(cache[bt[b, p], r] == synth.PAD_VALUE)
        assert np.array_equal(cache[bt[b, 0]], synth.cache_page(wl, b, 0))


def test_e4m3_format_and_fp8_rows():
    """The E4M3 codes of the FP8 cache: the format's fixed points (448 the
    largest finite value, 2^-9 the smallest subnormal, 2^-6 the smallest
    normal, 0x7F not a number), every finite value encodes to itself, ties go
    to the even code, magnitudes past 448 clamp; a row decodes to its codes
    times its scale and its bf16 RoPE part."""
    import numpy as np
    from mla_latent_kv_67_b300 import synth
    t = synth.E4M3
    assert t[0x7E] == 448.0 and t[0x01] == 2.0 ** -9 and t[0x08] == 2.0 ** -6 and np.isnan(t[0x7F])
    assert t[0xFE] == -448.0 and t[0x38] == 1.0
    finite = np.array([c for c in range(256) if not np.isnan(t[c]) and c != 0x80], np.uint8)
    assert np.array_equal(synth.e4m3_codes(t[finite].astype(np.float32)), finite)
    # 1.0625 lies halfway between 1.0 (0x38) and 1.125 (0x39): even code 0x38;
    # 1.1875 halfway between 1.125 (0x39) and 1.25 (0x3A): 0x3A
    got = synth.e4m3_codes(np.array([1.0625, 1.1875, 1e9, -1e9], np.float32))
    assert list(got) == [0x38, 0x3A, 0x7E, 0xFE]
    wl = synth.EXTRA_WORKLOADS["dsv2_b32_ctx4k_fp8"]
    rows = np.random.default_rng(3).standard_normal((5, wl.row_width)).astype(np.float32)
    enc, dec = synth.fp8_rows(wl, rows)
    assert enc.shape == (5, synth.fp8_row_bytes(wl.d_c, wl.d_r)) and enc.shape[1] % 16 == 0
    s = enc[:, wl.d_c + 2 * wl.d_r:wl.d_c + 2 * wl.d_r + 4].copy().view(np.float32)[:, 0]
    assert np.array_equal(dec[:, :wl.d_c], t[enc[:, :wl.d_c]].astype(np.float32) * s[:, None])
    assert np.max(np.abs(dec[:, :wl.d_c])) <= 448.0 * s.max()
    assert np.allclose(dec[:, :wl.d_c], rows[:, :wl.d_c], rtol=2.0 ** -4, atol=2.0 ** -9 * s.max())
    assert np.array_equal(dec[:, wl.d_c:], synth.round_bf16(rows[:, wl.d_c:]))
