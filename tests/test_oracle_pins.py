"""Pins for the fp64 oracle: each oracle function is checked against
something other than itself -- brute force on tiny inputs, a library routine
on a special case that reduces to it, closed forms, invariants and the numbers
the pages print. Each pin is a ``check_*`` function returning an error; the
``planted`` tests show that a plausible mistake planted in (a copy of) the
oracle makes the matching pin fail.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import mla_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(12345)


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ======================================================================= RoPE
def check_rope_2d_closed_form(rope=O.rope):
    """d_R = 2: theta_0 = 1, so RoPE is the plane rotation by ``pos`` rad."""
    err = 0.0
    for pos in (0.0, 1.0, 2.5, 17.0, 1000.0):
        v = rng.standard_normal(2)
        c, s = math.cos(pos), math.sin(pos)
        want = np.array([c * v[0] - s * v[1], s * v[0] + c * v[1]])
        err = max(err, float(np.max(np.abs(rope(v, pos) - want))))
    return err


def check_rope_frequency(rope=O.rope):
    """d_R = 4, base 10^4, pos 1: pair 0 turns by 1 rad, pair 1 by
    10^4^(-2/4) = 0.01 rad (hand-computed)."""
    v = np.array([1.0, 0.0, 1.0, 0.0])
    got = rope(v, 1.0, 10000.0)
    want = np.array([math.cos(1.0), math.sin(1.0), math.cos(0.01), math.sin(0.01)])
    return float(np.max(np.abs(got - want)))


def test_rope_pins():
    assert check_rope_2d_closed_form() < 1e-14
    assert check_rope_frequency() < 1e-15
    v = rng.standard_normal((5, 64))
    # position 0 is the identity
    assert np.array_equal(O.rope(v, 0.0), v)
    # a rotation keeps the norm
    r = O.rope(v, np.arange(5) * 977.0)
    assert np.allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(v, axis=-1), rtol=1e-14)
    # the score depends on the relative position only
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    for m, n in ((5, 3), (4096, 17), (131071, 65536)):
        a = O.rope(q, m) @ O.rope(k, n)
        b = O.rope(q, m - n) @ k
        assert abs(a - b) < 1e-9 * max(1.0, abs(b))


def test_rope_planted_sign_error_is_caught():
    def bad_rope(v, pos, base=10000.0):  # rotates the wrong way
        return O.rope(v, -np.asarray(pos, float), base)
    assert check_rope_2d_closed_form(bad_rope) > 1e-3


def test_rope_planted_frequency_error_is_caught():
    def bad_rope(v, pos, base=10000.0):  # theta_i = base^(-i/d) instead of -2i/d
        v = np.asarray(v, float)
        d = v.shape[-1]
        ang = np.asarray(pos, float)[..., None] * np.power(base, -np.arange(d // 2) / d)
        out = np.empty_like(v)
        out[..., 0::2] = v[..., 0::2] * np.cos(ang) - v[..., 1::2] * np.sin(ang)
        out[..., 1::2] = v[..., 0::2] * np.sin(ang) + v[..., 1::2] * np.cos(ang)
        return out
    assert check_rope_frequency(bad_rope) > 1e-3


# ============================================================ append / query
def test_latent_cache_row_unit_vectors():
    """x = e_k picks column k of each matrix; at position 0 RoPE is the
    identity, at position p the key column is rotated (2-D closed form)."""
    d, d_c, d_r = 12, 6, 2
    w_dkv, w_kr = rng.standard_normal((d_c, d)), rng.standard_normal((d_r, d))
    for k in (0, 5, 11):
        x = np.zeros(d)
        x[k] = 1.0
        c, kr = O.latent_cache_row(x, w_dkv, w_kr, 0)
        assert np.array_equal(c, w_dkv[:, k]) and np.array_equal(kr, w_kr[:, k])
        c, kr = O.latent_cache_row(x, w_dkv, w_kr, 3.0)
        a, b = w_kr[:, k]
        want = [math.cos(3) * a - math.sin(3) * b, math.sin(3) * a + math.cos(3) * b]
        assert np.allclose(kr, want, atol=1e-15)


def test_project_query_unit_vectors():
    """x = e_k, no query compression, position 0: head h's parts are rows
    h*d_h.. of W^UQ and rows h*d_R.. of W^QR at column k. With W^DQ the
    composition runs through column k of W^DQ."""
    n_h, d_h, d_r, d = 3, 4, 2, 7
    w_uq, w_qr = rng.standard_normal((n_h * d_h, d)), rng.standard_normal((n_h * d_r, d))
    x = np.zeros(d)
    x[2] = 1.0
    qc, qr = O.project_query(x, w_uq, w_qr, 0, n_h)
    for h in range(n_h):
        assert np.array_equal(qc[h], w_uq[h * d_h:(h + 1) * d_h, 2])
        assert np.array_equal(qr[h], w_qr[h * d_r:(h + 1) * d_r, 2])
    d_cq = 5
    w_dq = np.zeros((d_cq, d))
    w_dq[1, 2] = 1.0                                      # c_Q = e_1
    w_uq2, w_qr2 = rng.standard_normal((n_h * d_h, d_cq)), rng.standard_normal((n_h * d_r, d_cq))
    qc, qr = O.project_query(x, w_uq2, w_qr2, 0, n_h, w_dq=w_dq)
    assert np.array_equal(qc.reshape(-1), w_uq2[:, 1])
    assert np.array_equal(qr.reshape(-1), w_qr2[:, 1])


def test_absorb_and_output_projection_unit_vectors():
    n_h, d_h, d_v, d_c, d = 3, 4, 5, 6, 7
    w_uk = rng.standard_normal((n_h * d_h, d_c))
    w_uv = rng.standard_normal((n_h * d_v, d_c))
    w_o = rng.standard_normal((d, n_h * d_v))
    for h, i in ((0, 0), (2, 3), (1, 1)):
        q = np.zeros((n_h, d_h))
        q[h, i] = 1.0
        got = O.absorb_query(q, w_uk)
        assert np.array_equal(got[h], w_uk[h * d_h + i]) and not got[np.arange(n_h) != h].any()
    for h, c in ((0, 5), (2, 0)):
        ol = np.zeros((n_h, d_c))
        ol[h, c] = 1.0
        got = O.absorb_output(ol, w_uv)
        assert np.array_equal(got[h], w_uv[h * d_v:(h + 1) * d_v, c])
    for h, v in ((0, 0), (2, 4), (1, 2)):
        o = np.zeros((n_h, d_v))
        o[h, v] = 1.0
        assert np.array_equal(O.output_projection(o, w_o), w_o[:, h * d_v + v])


# ================================================================ attention
def brute_force_attention(q_c, q_r, c, k_r, w_uk, w_uv, scale):
    """Pure-Python loops straight from the definition (tiny shapes only)."""
    n_h, d_h = len(q_c), len(q_c[0])
    d_c, N = len(c[0]), len(c)
    d_v = len(w_uv) // n_h
    out, lses = [], []
    for h in range(n_h):
        scores = []
        for j in range(N):
            s = 0.0
            for i in range(d_h):          # content part: q^C . (W^UK_h c_j)
                k_ij = sum(w_uk[h * d_h + i][t] * c[j][t] for t in range(d_c))
                s += q_c[h][i] * k_ij
            for r in range(len(k_r[j])):  # position part: q^R . k^R_j
                s += q_r[h][r] * k_r[j][r]
            scores.append(s * scale)
        mx = max(scores)
        e = [math.exp(s - mx) for s in scores]
        z = sum(e)
        o = []
        for v in range(d_v):
            acc = 0.0
            for j in range(N):
                vj = sum(w_uv[h * d_v + v][t] * c[j][t] for t in range(d_c))
                acc += e[j] / z * vj
            o.append(acc)
        out.append(o)
        lses.append(mx + math.log(z))
    return np.array(out), np.array(lses)


def tiny_case(n_h=2, d_h=3, d_r=2, d_c=4, d_v=3, N=5, seed=0):
    g = np.random.default_rng(seed)
    return dict(q_c=g.standard_normal((n_h, d_h)), q_r=g.standard_normal((n_h, d_r)),
                c=g.standard_normal((N, d_c)), k_r=g.standard_normal((N, d_r)),
                w_uk=g.standard_normal((n_h * d_h, d_c)),
                w_uv=g.standard_normal((n_h * d_v, d_c)),
                scale=1.0 / math.sqrt(d_h + d_r))


def check_brute_force(attn=O.attention_explicit):
    err = 0.0
    for seed, shape in enumerate([dict(), dict(n_h=3, d_h=2, d_r=4, d_c=5, d_v=2, N=7),
                                  dict(N=1), dict(n_h=1, d_c=1, N=3)]):
        case = tiny_case(seed=seed, **shape)
        o, lse = attn(**case)
        bo, blse = brute_force_attention(*[case[k].tolist() if hasattr(case[k], "tolist")
                                           else case[k] for k in
                                           ("q_c", "q_r", "c", "k_r", "w_uk", "w_uv", "scale")])
        err = max(err, rel(o, bo), float(np.max(np.abs(lse - blse))))
    return err


def check_mha_reduction_sdpa(attn=O.attention_explicit):
    """MHA special case: d_c = n_h*d_h, W^UK_h and W^UV_h select block h of
    the latent through (different) cyclic shifts, so K_h and V_h are column
    gathers of c. Torch's fp64 scaled_dot_product_attention (a library
    routine) on those gathers must agree with the oracle."""
    n_h, d_h, d_r, N = 4, 8, 4, 37
    d_c = d_v = None
    d_c = n_h * d_h
    g = np.random.default_rng(7)
    c, k_r = g.standard_normal((N, d_c)), g.standard_normal((N, d_r))
    q_c, q_r = g.standard_normal((n_h, d_h)), g.standard_normal((n_h, d_r))
    w_uk, w_uv = np.zeros((n_h * d_h, d_c)), np.zeros((n_h * d_h, d_c))
    idx_k = np.zeros((n_h, d_h), int)
    idx_v = np.zeros((n_h, d_h), int)
    for h in range(n_h):
        for i in range(d_h):
            idx_k[h, i] = h * d_h + (i + 1) % d_h
            idx_v[h, i] = h * d_h + (i + 3) % d_h
            w_uk[h * d_h + i, idx_k[h, i]] = 1.0
            w_uv[h * d_h + i, idx_v[h, i]] = 1.0
    scale = 1.0 / math.sqrt(d_h + d_r)
    o, lse = attn(q_c, q_r, c, k_r, w_uk, w_uv, scale)
    K = np.stack([np.concatenate([c[:, idx_k[h]], k_r], axis=1) for h in range(n_h)])
    V = np.stack([c[:, idx_v[h]] for h in range(n_h)])
    Q = np.concatenate([q_c, q_r], axis=1)[:, None, :]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q), torch.from_numpy(K), torch.from_numpy(V), scale=scale)
    return rel(o, ref.numpy()[:, 0, :])


def check_multi_token_sdpa(attn=O.attention_multi_token, lengths=O.multi_token_lengths):
    """MHA special case of decoding T new tokens together: the T queries sit
    at the last T cache positions, so torch's fp64 scaled_dot_product_attention
    with a boolean mask that lets query t see keys 0 .. N - T + t (a library
    routine with the causal mask aligned to the end) must agree."""
    n_h, d_h, d_r, N, T = 3, 4, 2, 23, 4
    d_c = n_h * d_h
    g = np.random.default_rng(17)
    c, k_r = g.standard_normal((N, d_c)), g.standard_normal((N, d_r))
    q_c, q_r = g.standard_normal((T, n_h, d_h)), g.standard_normal((T, n_h, d_r))
    w_uk, w_uv = np.zeros((n_h * d_h, d_c)), np.zeros((n_h * d_h, d_c))
    for h in range(n_h):
        for i in range(d_h):
            w_uk[h * d_h + i, h * d_h + (i + 1) % d_h] = 1.0
            w_uv[h * d_h + i, h * d_h + (i + 2) % d_h] = 1.0
    scale = 1.0 / math.sqrt(d_h + d_r)
    o, lse = attn(q_c, q_r, c, k_r, w_uk, w_uv, scale)
    K = np.stack([np.concatenate([c @ w_uk[h * d_h:(h + 1) * d_h].T, k_r], axis=1)
                  for h in range(n_h)])                               # [n_h, N, d_h + d_r]
    V = np.stack([c @ w_uv[h * d_h:(h + 1) * d_h].T for h in range(n_h)])
    Q = np.concatenate([q_c, q_r], axis=2).transpose(1, 0, 2)        # [n_h, T, d_h + d_r]
    mask = np.arange(N)[None, :] <= (N - T + np.arange(T))[:, None]   # [T, N]
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Q), torch.from_numpy(K), torch.from_numpy(V),
        attn_mask=torch.from_numpy(mask), scale=scale).numpy()        # [n_h, T, d_v]
    err = rel(o, ref.transpose(1, 0, 2))
    # lse: log sum_j exp(s_j) over the same visible keys
    s = np.einsum("htd,hnd->htn", Q, K) * scale
    s = np.where(mask[None], s, -np.inf)
    ref_lse = np.log(np.exp(s - s.max(-1, keepdims=True)).sum(-1)) + s.max(-1)
    return max(err, float(np.max(np.abs(lse - ref_lse.T))))


def test_multi_token_decode_matches_masked_sdpa():
    assert check_multi_token_sdpa() < 1e-12
    assert list(O.multi_token_lengths(10, 3)) == [8, 9, 10]
    assert list(O.multi_token_lengths(1, 1)) == [1]


def test_multi_token_planted_mistakes_are_caught():
    def top_left(n, t):  # token t sees rows 0..t (a mask aligned to the start)
        return 1 + np.arange(t)

    def without_own(n, t):  # token t does not see its own row
        return n - t + np.arange(t)

    for bad in (top_left, without_own):
        def attn(q_c, q_r, c, k_r, w_uk, w_uv, scale, bad=bad):
            outs, lses = [], []
            for t, n in enumerate(bad(len(c), len(q_c))):
                o, lse = O.attention_explicit(q_c[t], q_r[t], c[:n], k_r[:n], w_uk, w_uv, scale)
                outs.append(o)
                lses.append(lse)
            return np.stack(outs), np.stack(lses)
        assert check_multi_token_sdpa(attn) > 1e-3


def test_multi_token_one_token_and_forms_agree():
    case = tiny_case(n_h=2, N=9, seed=3)
    o1, l1 = O.attention_explicit(**case)
    om, lm = O.attention_multi_token(case["q_c"][None], case["q_r"][None], case["c"], case["k_r"],
                                     case["w_uk"], case["w_uv"], case["scale"])
    assert np.array_equal(om[0], o1) and np.array_equal(lm[0], l1)
    g = np.random.default_rng(4)
    q_c, q_r = g.standard_normal((3, 2, 3)), g.standard_normal((3, 2, 2))
    oe, le = O.attention_multi_token(q_c, q_r, case["c"], case["k_r"], case["w_uk"], case["w_uv"],
                                     case["scale"])
    oa, la = O.attention_multi_token(q_c, q_r, case["c"], case["k_r"], case["w_uk"], case["w_uv"],
                                     case["scale"], form="absorbed")
    assert rel(oe, oa) < 1e-10 and np.max(np.abs(le - la)) < 1e-10


def test_attention_brute_force():
    assert check_brute_force() < 1e-12


def test_attention_mha_reduction_matches_torch_sdpa():
    assert check_mha_reduction_sdpa() < 1e-12


def test_attention_special_cases():
    case = tiny_case(n_h=3, d_h=4, d_r=2, d_c=6, d_v=5, N=1, seed=3)
    o, lse = O.attention_explicit(**case)
    # one token: the output is that token's value whatever the query
    for h in range(3):
        assert np.allclose(o[h], case["w_uv"][h * 5:(h + 1) * 5] @ case["c"][0], rtol=1e-14)
    case = tiny_case(n_h=3, d_h=4, d_r=2, d_c=6, d_v=5, N=9, seed=4)
    zq = dict(case, q_c=np.zeros_like(case["q_c"]), q_r=np.zeros_like(case["q_r"]))
    o, lse = O.attention_explicit(**zq)
    # zero query: uniform weights, the mean value; lse = log N
    for h in range(3):
        assert np.allclose(o[h], case["w_uv"][h * 5:(h + 1) * 5] @ case["c"].mean(0), rtol=1e-13)
    assert np.allclose(lse, math.log(9), rtol=1e-15)
    # identical cached rows: the output does not depend on the query
    same = dict(case, c=np.repeat(case["c"][:1], 9, 0), k_r=np.repeat(case["k_r"][:1], 9, 0))
    o1, _ = O.attention_explicit(**same)
    o2, _ = O.attention_explicit(**dict(same, q_c=case["q_c"] * 5.0))
    assert np.allclose(o1, o2, rtol=1e-13)
    # the order of cached tokens does not matter
    perm = rng.permutation(9)
    o3, l3 = O.attention_explicit(**dict(case, c=case["c"][perm], k_r=case["k_r"][perm]))
    o4, l4 = O.attention_explicit(**case)
    assert np.allclose(o3, o4, rtol=1e-13) and np.allclose(l3, l4, rtol=1e-14)


def test_softmax_rows_sum_to_one_and_shift_invariance():
    s = rng.standard_normal((7, 300)) * 20
    p, lse = O.softmax(s)
    assert np.all(np.abs(p.sum(-1) - 1.0) < 1e-12)
    p2, lse2 = O.softmax(s + 1000.0)
    assert np.allclose(p, p2, rtol=1e-12) and np.allclose(lse2 - lse, 1000.0, rtol=1e-14)
    assert np.allclose(lse, np.log(np.exp(s).sum(-1)), rtol=1e-13)


def _drop_rope_term(q_c, q_r, c, k_r, w_uk, w_uv, scale, heads=None):
    return O.attention_explicit(q_c, np.zeros_like(q_r), c, k_r, w_uk, w_uv, scale, heads)


def _transposed_head_block(q_c, q_r, c, k_r, w_uk, w_uv, scale, heads=None):
    n_h, d_h = q_c.shape
    w = w_uk.reshape(n_h, d_h, -1)
    if w.shape[1] == w.shape[2]:
        w = w.transpose(0, 2, 1)
    else:  # read the head blocks in the wrong order instead
        w = w[::-1]
    return O.attention_explicit(q_c, q_r, c, k_r, w.reshape(w_uk.shape), w_uv, scale, heads)


def _wrong_scale(q_c, q_r, c, k_r, w_uk, w_uv, scale, heads=None):
    return O.attention_explicit(q_c, q_r, c, k_r, w_uk, w_uv, 1.0 / math.sqrt(q_c.shape[1]), heads)


@pytest.mark.parametrize("bug", [_drop_rope_term, _transposed_head_block, _wrong_scale])
def test_attention_planted_mistakes_are_caught(bug):
    assert max(check_brute_force(bug), check_mha_reduction_sdpa(bug)) > 1e-3


# =============================================================== absorption
def test_absorbed_equals_explicit():
    """[MLA-V2] 2.2: folding W^UK into the query and W^UV after the softmax
    changes nothing but rounding -- to 1e-10 in fp64."""
    for seed, shape in enumerate([dict(n_h=4, d_h=8, d_r=4, d_c=16, d_v=8, N=50),
                                  dict(n_h=16, d_h=128, d_r=64, d_c=512, d_v=128, N=300),
                                  dict(n_h=8, d_h=32, d_r=16, d_c=64, d_v=32, N=256)]):
        case = tiny_case(seed=seed, **shape)
        o_e, l_e = O.attention_explicit(**case)
        o_a, o_lat, l_a = O.attention_absorbed(**case)
        assert rel(o_a, o_e) < 1e-10
        assert np.max(np.abs(l_a - l_e)) < 1e-10


# ===================================================================== merge
def test_merge_partials_hand_example():
    # two parts: lse 0 and log 3 -> weights 1/4 and 3/4
    o, lse = O.merge_partials(np.array([[1.0], [5.0]]), np.array([0.0, math.log(3.0)]))
    assert abs(o[0] - 4.0) < 1e-15 and abs(lse - math.log(4.0)) < 1e-15


def test_merge_partials_equals_attention_over_union():
    case = tiny_case(n_h=6, d_h=8, d_r=4, d_c=16, d_v=8, N=97, seed=11)
    q_abs = O.absorb_query(case["q_c"], case["w_uk"])
    full_o, full_lse = O.attention_latent(q_abs, case["q_r"], case["c"], case["k_r"], case["scale"])
    cuts = [0, 13, 13, 64, 97]     # includes an empty part
    parts_o, parts_l = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        if a == b:
            parts_o.append(np.zeros_like(full_o))
            parts_l.append(np.full(full_lse.shape, -np.inf))
            continue
        o, l = O.attention_latent(q_abs, case["q_r"], case["c"][a:b], case["k_r"][a:b], case["scale"])
        parts_o.append(o)
        parts_l.append(l)
    o, lse = O.merge_partials(np.stack(parts_o), np.stack(parts_l))
    assert rel(o, full_o) < 1e-13 and np.max(np.abs(lse - full_lse)) < 1e-13


# ======================================================= cache-size closed forms
def test_cache_sizes_match_the_pages():
    g = json.load(open(os.path.join(GOLDEN, "cache_sizes.json")))
    v2 = dict(n_h=128, d_h=128, d_c=512, d_r=64)
    assert O.kv_elements_per_token("mla", **v2) == g["mla_v2_per_layer"]["value"]
    assert O.kv_elements_per_token("mla", layers=60, **v2) == g["mla_v2_all_layers"]["value"]
    mha60 = O.kv_elements_per_token("mha", layers=60, **v2)
    assert mha60 == g["mha_v2_all_layers"]["value"]
    ratio = O.kv_elements_per_token("mha", **v2) / O.kv_elements_per_token("mla", **v2)
    assert round(ratio, 1) == g["mha_over_mla_ratio"]["value"]
    assert round(mha60 / O.kv_elements_per_token("mla", layers=60, **v2), 1) == g["mha_over_mla_ratio"]["value"]
    assert O.gqa_equivalent_groups(512, 64, 128) == g["gqa_equivalent_groups"]["value"]
    assert round(100 * 64 / O.kv_elements_per_token("mla", **v2), 1) == g["rope_key_share_percent"]["value"]
    d = g["demo_counts"]
    BL = d["B"] * d["L"]
    assert BL * O.kv_elements_per_token("mha", n_h=d["H"], d_h=d["D"]) == d["mha"]
    assert BL * O.kv_elements_per_token("mqa", d_h=d["D"]) == d["mqa"]
    assert BL * O.kv_elements_per_token("gqa", n_g=d["G"], d_h=d["D"]) == d["gqa"]
    assert BL * O.kv_elements_per_token("mla", d_c=d["D_c"], separate_latents=True) == d["mla_separate_latents"]
    q = g["qwen72b_bytes_per_token"]
    by = O.kv_elements_per_token("mha", n_h=q["n_h"], d_h=q["d_h"], layers=q["layers"]) * q["bytes_per_elem"]
    assert by / 2 ** 20 == q["value_mib"]
    assert O.kv_elements_per_token("mha", n_h=128, d_h=128) == g["r1_mha_per_layer"]["value"]
    r1 = g["r1_mla_separate_latents_per_layer"]
    mla_sep = O.kv_elements_per_token("mla", d_c=r1["r"], separate_latents=True)
    assert mla_sep == r1["value"]
    assert g["r1_mha_per_layer"]["value"] // mla_sep == r1["compression"]
    assert 100 * (1 - mla_sep / g["r1_mha_per_layer"]["value"]) == r1["saving_percent"]
