"""The tcgen05 GEMMs behind mla_append_latent, mla_project_q, mla_expand_kv
and mla_out_proj, through the C ABI: the weight-streaming GEMM for few
tokens and the tile GEMM for 256 tokens or more.

Each product is checked against a float64 product of the same bf16 values
(fp32 accumulation on the GPU: max |gpu - ref| / max |ref| <= 1e-5 before
the output rounding), across shapes that exercise one and several token
tiles (in the order the kernel assigns them), a ragged last weight tile, and
each cluster split of K; the RoPE and paged-store epilogues against the
oracle.
"""
import numpy as np
import pytest
import torch

from mla_latent_kv_67_b300 import binding as M
from mla_latent_kv_67_b300 import synth
from mla_latent_kv_67_b300.step import DecodeStep
from oracle import mla_oracle as O
from reference import Expected, rel_to_max

pytestmark = pytest.mark.gpu


def bf16(shape, gen, scale=1.0):
    return (torch.randn(shape, generator=gen) * scale).bfloat16()


# (tokens M, heads, d_v, d_model): K = heads * d_v, N = d_model
OUT_PROJ_SHAPES = [
    (64, 128, 128, 5120),   # the DeepSeek-V2 W^O: K = 16384, N = 5120
    (1, 128, 128, 5120),
    (3, 2, 32, 200),        # K = 64 (one chunk), ragged N
    (130, 12, 128, 1000),   # two token tiles, K = 1536
    (257, 1, 64, 96),       # three token tiles, K = 64
    (600, 4, 128, 384),     # five token tiles, ragged last, K = 512
    (512, 8, 64, 256),      # four full token tiles x two weight tiles
    # tile GEMM (>= 256 tokens): 128-token x 256-feature tiles
    (1024, 16, 128, 768),   # 8 x 3 tiles, K = 2048
    (2048, 8, 64, 4096),    # 256 tiles: each SM takes two, both accumulators in turn
    (383, 3, 64, 520),      # ragged last token and feature tiles, K = 192
    (300, 2, 64, 97),       # fp32 rows of 97 features: not in 16-byte pieces
]


@pytest.mark.parametrize("shape", OUT_PROJ_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_out_proj_matches_fp64(shape):
    T, n_h, d_v, d_model = shape
    g = torch.Generator().manual_seed(sum(shape))
    K = n_h * d_v
    o = bf16((T, K), g)
    w = bf16((d_model, K), g, K ** -0.5)
    dims = M.Dims(n_h, 128, 64, 512, d_v, d_model, 0, 64)
    u = torch.full((T, d_model), float("nan"), device="cuda")
    M.mla_out_proj(o.cuda(), w.cuda(), u, dims)
    torch.cuda.synchronize()
    ref = (o.double() @ w.double().T).numpy()
    assert rel_to_max(u.cpu().numpy(), ref) <= 1e-5
    # the CUDA-core GEMM on the same inputs agrees
    M.mla_force_decode_path(0)
    try:
        u2 = torch.full_like(u, float("nan"))
        M.mla_out_proj(o.cuda(), w.cuda(), u2, dims)
        torch.cuda.synchronize()
    finally:
        M.mla_force_decode_path(-1)
    assert rel_to_max(u2.cpu().numpy(), ref) <= 1e-5


def test_project_q_epilogue_against_oracle():
    """x W^DQ^T -> c_Q (bf16), then [W^UQ | W^QR] c_Q with RoPE on the q_R
    slice of every head: c_Q against x W^DQ^T, q against the oracle's query
    projection of the GPU's own c_Q (so only the final bf16 rounding
    separates them)."""
    wl = synth.WORKLOADS["dsv2_layer_b64_ctx32k"].replace(batch=5, lens=(1, 2, 700, 4096, 32768))
    st = DecodeStep(wl)
    st.project()
    torch.cuda.synchronize()
    assert st.status() == 0
    ex = Expected(wl)
    cq = st.c_q.double().cpu().numpy()
    cq_ref = ex.x @ ex.w["w_dq"].T
    assert np.all(np.abs(cq - cq_ref) <= 2.0 ** -8 * np.abs(cq_ref) + 1e-5 * np.abs(cq_ref).max())
    q = st.q.double().cpu().numpy()
    for b in range(wl.batch):
        q_c, q_r = O.project_query(cq[b], ex.w["w_uq"], ex.w["w_qr"], int(ex.lens[b]) - 1,
                                   wl.n_h, w_dq=None, base=wl.rope_base)
        ref = np.concatenate([q_c, q_r], axis=-1)
        assert np.all(np.abs(q[b] - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5 * np.abs(ref).max()), b


def test_project_q_many_tokens_tile_gemm():
    """A 300-token prompt's query projection (tile GEMM, RoPE epilogue on the
    q_R slice of every head): c_Q against x W^DQ^T, q against the oracle's
    query projection of the GPU's own c_Q, every token."""
    wl = synth.EXTRA_WORKLOADS["dsv2_prefill_4k"].replace(name="proj_300", ctx=300, seed=62)
    st = DecodeStep(wl)
    st.project()
    torch.cuda.synchronize()
    assert st.status() == 0
    x = synth.tokens(wl).astype(np.float64)
    w_dq = synth.weight(wl, "w_dq").astype(np.float64)
    cq = st.c_q.double().cpu().numpy()
    cq_ref = x @ w_dq.T
    assert np.all(np.abs(cq - cq_ref) <= 2.0 ** -8 * np.abs(cq_ref) + 1e-5 * np.abs(cq_ref).max())
    q_c, q_r = O.project_query(cq, synth.weight(wl, "w_uq").astype(np.float64),
                               synth.weight(wl, "w_qr").astype(np.float64), np.arange(wl.ctx),
                               wl.n_h, w_dq=None, base=wl.rope_base)
    ref = np.concatenate([q_c, q_r], axis=-1)
    q = st.q.double().cpu().numpy()
    assert np.all(np.abs(q - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5 * np.abs(ref).max())


def test_append_many_tokens_across_token_tiles():
    """300 tokens of one sequence appended at positions 0..299 (three token
    tiles): every cache row against the oracle's bf16-rounded row."""
    wl = synth.WORKLOADS["tiny_f32_ctx256"].replace(
        name="prefill_bf16", dtype="bf16", n_h=128, d_h=128, d_r=64, d_c=512, d_v=128,
        d_model=512, d_cq=0, page_size=64, ctx=300)
    st = DecodeStep(wl)
    st.append()
    torch.cuda.synchronize()
    assert st.status() == 0
    ex = Expected(wl)
    pos, c, k = ex.appended_rows(0)
    ref = np.concatenate([c, k], axis=1)
    rows = st.cache.double().cpu().numpy()
    got = np.stack([rows[st.bt_np[0, p // 64], p % 64] for p in pos])
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5 * np.abs(ref).max())


def test_append_bad_positions_many_tokens():
    """300 tokens appended through the tile GEMM with two positions outside
    the block table (negative, and past it): both are reported as
    MLA_DEV_BAD_POS and skipped, every other row is written as the oracle
    says, and no other cache slot changes."""
    wl = synth.WORKLOADS["tiny_f32_ctx256"].replace(
        name="prefill_bf16_bad", dtype="bf16", n_h=128, d_h=128, d_r=64, d_c=512, d_v=128,
        d_model=512, d_cq=0, page_size=64, ctx=300)
    st = DecodeStep(wl)
    bad = {5: -1, 200: st.max_pages * wl.page_size + 7}
    for t, v in bad.items():
        st.append_pos[t] = v
    before = st.cache.clone()
    st.append()
    torch.cuda.synchronize()
    assert st.status() & M.MLA_DEV_BAD_POS
    ex = Expected(wl)
    pos, c, k = ex.appended_rows(0)
    ref = np.concatenate([c, k], axis=1)
    after = st.cache
    changed = (before.view(torch.int16) != after.view(torch.int16)).any(dim=-1).cpu().numpy()
    expect = np.zeros_like(changed)
    rows = after.double().cpu().numpy()
    for i, p in enumerate(pos):
        if i in bad:
            continue
        blk, r = st.bt_np[0, p // 64], p % 64
        expect[blk, r] = True
        got = rows[blk, r]
        assert np.all(np.abs(got - ref[i]) <= 2.0 ** -8 * np.abs(ref[i]) + 1e-5 * np.abs(ref).max()), i
    # rows that the oracle writes as exact zeros may leave a slot unchanged
    assert not np.any(changed & ~expect)


def test_layer_step_tensor_core_matches_cuda_core():
    """The full layer step on both GEMM paths: the same u within the bf16
    pipeline's rounding."""
    wl = synth.WORKLOADS["dsv2_layer_b64_ctx32k"].replace(batch=4, ctx=500)
    a = DecodeStep(wl)
    a.run()
    torch.cuda.synchronize()
    M.mla_force_decode_path(0)
    try:
        b = DecodeStep(wl)
        b.run()
        torch.cuda.synchronize()
    finally:
        M.mla_force_decode_path(-1)
    assert a.status() == 0 and b.status() == 0
    assert rel_to_max(a.u.cpu().numpy(), b.u.cpu().numpy()) <= 2e-2
