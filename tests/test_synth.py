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
