"""fp64 CPU oracle for Multi-head Latent Attention decode.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or runs
this file: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm may. It shares no code with the CUDA library and
imports nothing from the ``mla_latent_kv_67_b300`` package.

It states what the decode path computes in the plainest form, in float64:

* the latent cache row of a token (joint KV down-projection plus the decoupled
  RoPE key);
* the query (optionally low-rank compressed, then per-head up-projection plus
  the decoupled RoPE query);
* attention in the **explicit** form: per head it rebuilds
  ``K_h = [W^UK_h c_j ; k_R,j]`` and ``V_h = W^UV_h c_j`` for every cached token
  and runs ordinary softmax attention -- the non-absorbed definition;
* attention in the **absorbed** form (query folded through W^UK, softmax over
  the latent rows, latent output mapped back through W^UV), used as a cheap
  cross-check that covers every head of the large workloads;
* decode of several new tokens at once (each sees the cache up to its own
  position);
* the log-sum-exp merge of attention over disjoint token subsets;
* the output projection W^O;
* the cache-size closed forms the pages print.

Sources (page title, section):
  [MLA-V2]  "DeepSeek-V2: Multi-Head Latent Attention (MLA) 原理与工程实现"
            (PaperTrace), sections 1.1-1.2, 2.1-2.3, 3.2-3.3, 4.1, 5.2.
  [R1-MLA]  "DeepSeek R1的MLA：KV缓存的低秩压缩革命", sections 一, 二 2.1-2.2, 三.
  [KV-opt]  "kv-cache 的优化学习" (cnblogs), the MHA/MQA/GQA/MLA demo and its
            printed output.
  [KV-72B]  "大模型训练过程中KVCache与MLA" (csdn), 显存大小计算.

Conventions: column vectors as in [MLA-V2]; every weight is stored row-major as
``W in R^{out x in}``; per-head blocks are consecutive rows (head h owns rows
``h*d .. h*d+d-1``).

Readings where the pages are silent:
  * one joint latent ``c_KV`` (not separate C_k / C_v);
  * ``k_R`` comes from the token's hidden state through its own matrix W^KR,
    then RoPE; it is not derived from ``c_KV``;
  * RoPE rotates interleaved pairs ``(2i, 2i+1)`` by ``pos * base^(-2i/d_R)``;
  * softmax scale ``1/sqrt(d_h + d_R)``;
  * the decode token attends to every cached position including its own;
  * no norms, no biases.

Parity pins: every function here is checked against something other than
itself in ``tests/test_oracle_*.py`` (brute force on tiny inputs, torch's
fp64 scaled-dot-product attention on an MHA special case, closed forms,
invariants, the pages' printed numbers). None is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=F64)


# --------------------------------------------------------------------- RoPE
def rope_angles(pos, d_r: int, base: float = 10000.0) -> np.ndarray:
    """Rotation angles ``pos * theta_i`` with ``theta_i = base^(-2i/d_r)``,
    ``i = 0 .. d_r/2 - 1`` (RoFormer, the RoPE that [MLA-V2] section 6 cites;
    the pages strip the formula). Shape ``pos.shape + (d_r/2,)``."""
    assert d_r % 2 == 0
    i = np.arange(d_r // 2, dtype=F64)
    theta = np.power(F64(base), -2.0 * i / d_r)
    return _f64(pos)[..., None] * theta


def rope(v: np.ndarray, pos, base: float = 10000.0) -> np.ndarray:
    """Rotate the last axis of ``v`` (length d_r) pair by pair: the pair
    ``(v[2i], v[2i+1])`` turns by angle ``pos * theta_i``.

    ``pos`` broadcasts against ``v.shape[:-1]``. [MLA-V2] section 3.2: the
    decoupled query ``q^R`` and the shared key ``k^R`` carry RoPE; ``c^KV``
    does not."""
    v = _f64(v)
    d_r = v.shape[-1]
    ang = np.broadcast_to(rope_angles(pos, d_r, base), v.shape[:-1] + (d_r // 2,))
    cos, sin = np.cos(ang), np.sin(ang)
    even, odd = v[..., 0::2], v[..., 1::2]
    out = np.empty_like(v)
    out[..., 0::2] = even * cos - odd * sin
    out[..., 1::2] = even * sin + odd * cos
    return out


# ---------------------------------------------------------- cache append
def latent_cache_row(x, w_dkv, w_kr, pos, base: float = 10000.0):
    """What one token stores in the latent cache.

    [MLA-V2] section 2.1: ``c^KV_t = W^DKV h_t`` with ``W^DKV in R^{d_c x d}``
    (the joint down-projection; only ``c^KV`` is cached). Section 3.2: the
    shared key ``k^R_t = RoPE(W^KR h_t)`` is cached beside it (section 3.3:
    the row holds ``d_c + d_R`` elements).

    ``x``: ``[..., d]``; ``pos``: broadcastable to ``x.shape[:-1]``.
    Returns ``(c_kv [..., d_c], k_r [..., d_R])``."""
    x = _f64(x)
    c = x @ _f64(w_dkv).T
    k = rope(x @ _f64(w_kr).T, pos, base)
    return c, k


# ----------------------------------------------------------------- query
def project_query(x, w_uq, w_qr, pos, n_h: int, w_dq=None, base: float = 10000.0):
    """Per-head query parts of one or more tokens.

    [MLA-V2] section 2.3: ``c^Q_t = W^DQ h_t`` (``d_c'`` wide), then
    ``q^C_t = W^UQ c^Q_t``; section 3.2: ``q^R_t = RoPE(W^QR c^Q_t)``, one
    ``d_R`` slice per head. With ``w_dq=None`` the query is not compressed
    (``c^Q = h``), i.e. a direct W^Q.

    ``x``: ``[..., d]``. Returns ``(q_c [..., n_h, d_h], q_r [..., n_h, d_R])``."""
    x = _f64(x)
    cq = x if w_dq is None else x @ _f64(w_dq).T
    qc = cq @ _f64(w_uq).T
    qr = cq @ _f64(w_qr).T
    qc = qc.reshape(qc.shape[:-1] + (n_h, -1))
    qr = qr.reshape(qr.shape[:-1] + (n_h, -1))
    return qc, rope(qr, np.asarray(pos)[..., None], base)


# --------------------------------------------------------------- softmax
def softmax(s):
    """Row softmax over the last axis and its log-sum-exp, max-shifted."""
    s = _f64(s)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    z = e.sum(axis=-1, keepdims=True)
    return e / z, (m + np.log(z))[..., 0]


# ------------------------------------------------------ explicit attention
def explicit_kv(c, k_r, w_uk, w_uv, h: int, n_h: int):
    """Head ``h``'s full keys and values rebuilt from the latent cache.

    [MLA-V2] section 2.1: ``k^C_t = W^UK c^KV_t`` and ``v^C_t = W^UV c^KV_t``
    with ``W^UK, W^UV in R^{d_h n_h x d_c}``; head h is the h-th block of rows.
    Section 3.2: the attention key is ``[k^C_{t,h} ; k^R_t]``, the RoPE key
    being shared by all heads.

    ``c [N, d_c]``, ``k_r [N, d_R]``.
    Returns ``K_h [N, d_h + d_R]`` and ``V_h [N, d_v]``."""
    c, w_uk, w_uv = _f64(c), _f64(w_uk), _f64(w_uv)
    d_h = w_uk.shape[0] // n_h
    d_v = w_uv.shape[0] // n_h
    k_c = c @ w_uk[h * d_h:(h + 1) * d_h].T
    v = c @ w_uv[h * d_v:(h + 1) * d_v].T
    return np.concatenate([k_c, _f64(k_r)], axis=1), v


def attention_explicit(q_c, q_r, c, k_r, w_uk, w_uv, scale: float, heads=None):
    """Decode attention of one query token over ``N`` cached tokens, the
    non-absorbed way.

    For each head: ``s_j = [q^C_h ; q^R_h] . K_h[j] * scale``,
    ``p = softmax(s)``, ``o_h = sum_j p_j V_h[j]`` ([MLA-V2] sections 2.1 and
    3.2; in decoding the new token attends over every cached token).

    ``q_c [n_h, d_h]``, ``q_r [n_h, d_R]``, ``c [N, d_c]``, ``k_r [N, d_R]``.
    Returns ``o [len(heads), d_v]`` and ``lse [len(heads)]``, the natural log of
    ``sum_j exp(s_j)``."""
    n_h = q_c.shape[0]
    heads = range(n_h) if heads is None else heads
    outs, lses = [], []
    for h in heads:
        K, V = explicit_kv(c, k_r, w_uk, w_uv, h, n_h)
        q = np.concatenate([_f64(q_c[h]), _f64(q_r[h])])
        p, lse = softmax((K @ q) * scale)
        outs.append(p @ V)
        lses.append(lse)
    return np.stack(outs), np.asarray(lses)


# ------------------------------------------------------ absorbed attention
def absorb_query(q_c, w_uk):
    """``q_abs,h = (W^UK_h)^T q^C_h``, a ``d_c``-vector per head.

    [MLA-V2] section 2.2: ``q^T k^C = q^T W^UK c = (W^UK^T q)^T c``, so the key
    up-projection folds into the query; [R1-MLA] 二 2.2 precomputes the same
    product ``Q^h W_uk^{hT}``. ``q_c [..., n_h, d_h]`` -> ``[..., n_h, d_c]``."""
    q_c, w_uk = _f64(q_c), _f64(w_uk)
    n_h, d_h = q_c.shape[-2], q_c.shape[-1]
    w = w_uk.reshape(n_h, d_h, -1)                  # [h][i][c]
    return np.einsum("...hi,hic->...hc", q_c, w)


def absorb_output(o_lat, w_uv):
    """``o_h = W^UV_h o~_h``: the latent attention output of each head mapped
    back to ``d_v`` ([MLA-V2] section 2.2, the W^UV half of
    ``W~^O = W^O W^UV`` applied unfused). ``o_lat [..., n_h, d_c]`` ->
    ``[..., n_h, d_v]``."""
    o_lat, w_uv = _f64(o_lat), _f64(w_uv)
    n_h = o_lat.shape[-2]
    w = w_uv.reshape(n_h, -1, o_lat.shape[-1])     # [h][v][c]
    return np.einsum("...hc,hvc->...hv", o_lat, w)


def attention_latent(q_abs, q_r, c, k_r, scale: float):
    """Attention in the latent space for every head at once.

    [MLA-V2] section 3.2: the score splits into a content part computed in the
    compressed space (``q_abs,h . c_j``) and a position part
    (``q^R_h . k^R_j``). Returns the latent output ``o~ [n_h, d_c]`` (the
    softmax-weighted sum of latent rows) and ``lse [n_h]``."""
    s = (_f64(q_abs) @ _f64(c).T + _f64(q_r) @ _f64(k_r).T) * scale   # [n_h, N]
    p, lse = softmax(s)
    return p @ _f64(c), lse


def attention_absorbed(q_c, q_r, c, k_r, w_uk, w_uv, scale: float):
    """The absorbed decode path end to end: returns ``(o [n_h, d_v],
    o_lat [n_h, d_c], lse [n_h])``. Equal to :func:`attention_explicit` up to
    rounding ([MLA-V2] section 2.2)."""
    q_abs = absorb_query(q_c, w_uk)
    o_lat, lse = attention_latent(q_abs, q_r, c, k_r, scale)
    return absorb_output(o_lat, w_uv), o_lat, lse


# ------------------------------------------------- multi-token decode
def multi_token_lengths(n_cached: int, n_new: int) -> np.ndarray:
    """Cached rows each of ``n_new`` new tokens attends over when they are
    decoded together (multi-token prediction / speculative drafts, [MLA-V2]
    4.3 and 6): the new tokens hold the last ``n_new`` of ``n_cached`` cache
    positions, and token t sees every position up to and including its own,
    ``n_cached - n_new + t + 1`` rows."""
    assert 1 <= n_new <= n_cached
    return n_cached - n_new + 1 + np.arange(n_new)


def attention_multi_token(q_c, q_r, c, k_r, w_uk, w_uv, scale: float, form: str = "explicit"):
    """Decode attention of ``T`` new tokens at once: token t attends over the
    first :func:`multi_token_lengths` ``(N, T)[t]`` cached rows, the explicit
    (or absorbed) single-token attention on that prefix.

    ``q_c [T, n_h, d_h]``, ``q_r [T, n_h, d_R]``, ``c [N, d_c]``,
    ``k_r [N, d_R]``. Returns ``o [T, n_h, d_v]`` and ``lse [T, n_h]``."""
    T = len(q_c)
    outs, lses = [], []
    for t, n in enumerate(multi_token_lengths(len(c), T)):
        if form == "explicit":
            o, lse = attention_explicit(q_c[t], q_r[t], c[:n], k_r[:n], w_uk, w_uv, scale)
        else:
            o, _, lse = attention_absorbed(q_c[t], q_r[t], c[:n], k_r[:n], w_uk, w_uv, scale)
        outs.append(o)
        lses.append(lse)
    return np.stack(outs), np.stack(lses)


# ----------------------------------------------------- split-KV merge
def merge_partials(o_parts, lse_parts):
    """Merge attention computed over disjoint token subsets.

    Each part ``s`` holds its normalised output ``o_s`` and log-sum-exp
    ``lse_s``; over the union ``lse = log sum_s exp(lse_s)`` and
    ``o = sum_s exp(lse_s - lse) o_s``. Parts with ``lse = -inf`` (no tokens)
    contribute nothing. ``o_parts [S, ..., d]``, ``lse_parts [S, ...]``."""
    o_parts, lse_parts = _f64(o_parts), _f64(lse_parts)
    m = lse_parts.max(axis=0)
    w = np.exp(lse_parts - m)
    z = w.sum(axis=0)
    o = (w[..., None] * o_parts).sum(axis=0) / z[..., None]
    return o, m + np.log(z)


# ------------------------------------------------------ output projection
def output_projection(o, w_o):
    """``u_t = W^O [o_{t,1}; ...; o_{t,n_h}]``: the heads' outputs concatenated
    and projected ([MLA-V2] section 2.2, ``W^O``). ``o [..., n_h, d_v]`` ->
    ``[..., d]``."""
    o = _f64(o)
    flat = o.reshape(o.shape[:-2] + (-1,))
    return flat @ _f64(w_o).T


# ----------------------------------------------------- cache-size forms
def kv_elements_per_token(kind: str, n_h: int = 0, d_h: int = 0, layers: int = 1,
                          n_g: int = 0, d_c: int = 0, d_r: int = 0,
                          separate_latents: bool = False) -> int:
    """Cached elements per token, summed over ``layers``.

    [MLA-V2] 1.1: MHA caches ``2 n_h d_h`` per layer; 1.2: MQA ``2 d_h``, GQA
    ``2 n_g d_h``; 3.3: MLA ``d_c + d_R``. [KV-opt] (its demo) and [R1-MLA]
    (its table) cache two separate latents of width ``d_c`` with no RoPE key:
    ``separate_latents=True`` gives that count, ``2 d_c``."""
    if kind == "mha":
        per = 2 * n_h * d_h
    elif kind == "mqa":
        per = 2 * d_h
    elif kind == "gqa":
        per = 2 * n_g * d_h
    elif kind == "mla":
        per = 2 * d_c if separate_latents else d_c + d_r
    else:
        raise ValueError(kind)
    return per * layers


def gqa_equivalent_groups(d_c: int, d_r: int, d_h: int) -> float:
    """The GQA group count whose cache equals MLA's: ``(d_c+d_R)/(2 d_h)``
    ([MLA-V2] 4.1)."""
    return (d_c + d_r) / (2 * d_h)
