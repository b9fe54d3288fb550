"""Decode of several new tokens per sequence at once (mla_plan_decode_mtp /
mla_decode_attn_mtp) against the oracle's multi-token attention: query row
b * q_len + t sees the first len_b - q_len + 1 + t cached rows. Every query
row and head against the absorbed oracle, a few heads against the explicit
definition, on every decode kernel."""
import numpy as np
import pytest
import torch

from mla_latent_kv_67_b300 import binding as M
from mla_latent_kv_67_b300 import synth
from mla_latent_kv_67_b300.step import DecodeStep
from reference import TOL, Expected, gate_errors, gate_failures, lse_tol

pytestmark = pytest.mark.gpu

BASE = synth.WORKLOADS["dsv2_b32_ctx4k"].replace(name="mtp", batch=6,
                                                 lens=(4, 63, 65, 128, 700, 4096), seed=41)


def host(st, v):
    wl = st.wl
    return {"o_lat": st.o_lat[v].double().cpu().numpy(), "lse": st.lse[v].double().cpu().numpy(),
            "o": st.o[v].double().cpu().numpy().reshape(wl.n_h, wl.d_v)}


@pytest.mark.parametrize("q_len", [2, 4])
@pytest.mark.parametrize("path", [1, 2, 0])
def test_multi_token_decode_matches_oracle(q_len, path):
    wl = BASE.replace(q_len=q_len)
    M.mla_force_decode_path(path)
    try:
        if path >= 1 and M.mla_decode_path(M.MLA_BF16, M.Dims.of(wl)) != path:
            pytest.skip("tensor-core decode kernel not available")
        st = DecodeStep(wl)
        st.run()
        torch.cuda.synchronize()
    finally:
        M.mla_force_decode_path(-1)
    assert st.status() == 0, f"status {st.status():#x}"
    ex = Expected(wl)
    for v in range(wl.batch * q_len):
        eh = [0, 127] if v % 5 == 0 else None
        errs = gate_errors(host(st, v), ex.seq(v, explicit_heads=eh), eh)
        bad = gate_failures(errs, TOL["bf16"], lse_tol(wl))
        assert not bad, (v, bad, errs)


def test_multi_token_last_row_equals_single_token_decode():
    """The last new token of each sequence sees the whole cache, so its row
    equals the single-token decode of the same query (up to the bf16
    rounding of probabilities taken against different running maxima: the
    two plans split the pages differently)."""
    wl = BASE.replace(q_len=3)
    st = DecodeStep(wl)
    st.run()
    torch.cuda.synchronize()
    assert st.status() == 0
    one = BASE.replace(q_len=1)
    s1 = DecodeStep(one)
    last = st.q[wl.q_len - 1::wl.q_len].clone()
    s1.q.copy_(last)
    s1.run()
    torch.cuda.synchronize()
    assert s1.status() == 0
    a = st.o_lat[wl.q_len - 1::wl.q_len].cpu().numpy()
    b = s1.o_lat.cpu().numpy()
    assert float(np.max(np.abs(a - b)) / np.max(np.abs(b))) < 1e-2


def test_multi_token_rejects_bad_q_len():
    wl = BASE.replace(q_len=2)
    st = DecodeStep(wl)
    with pytest.raises(M.MlaError):
        M.mla_decode_attn_mtp(st.q_cat[:0], st.cache, st.block_table, st.seq_lens, 0, wl.scale,
                              st.workspace, st.o_lat[:0], st.lse[:0], st.dims, st.dev_status)
    with pytest.raises(M.MlaError):
        M.mla_plan_decode_mtp(st.seq_lens, 9, st.max_pages,
                              st.workspace, st.dtype, st.dims, st.dev_status)
