"""The fused absorption form (W~^Q = W^UQ^T W^UK and W~^O = W^O W^UV folded
into the weights once) through the C ABI: the fused weights against fp64
products of the same bf16 inputs, q_cat from the fused projection against
the per-head path, and the whole fused layer step against the oracle."""
import numpy as np
import pytest
import torch

from mla_latent_kv_67_b300 import synth
from mla_latent_kv_67_b300.step import DecodeStep
from reference import TOL, Expected, gate_errors, gate_failures, lse_tol, rel_to_max

pytestmark = pytest.mark.gpu

LAYER = synth.WORKLOADS["dsv2_layer_b64_ctx32k"].replace(name="fused_small", batch=3, ctx=300,
                                                         d_model=512, d_cq=256, seed=51)


def test_fused_weights_match_fp64_products():
    wl = LAYER.replace(fused=True)
    st = DecodeStep(wl)
    torch.cuda.synchronize()
    uq = st.w_uq_qr.double().cpu().numpy().reshape(wl.n_h, wl.d_h + wl.d_r, -1)
    uk = st.w_uk.double().cpu().numpy().reshape(wl.n_h, wl.d_h, wl.d_c)
    fq = st.w_fused_q.double().cpu().numpy().reshape(wl.n_h, wl.d_c + wl.d_r, -1)
    ref = np.einsum("hic,hij->hcj", uk, uq[:, :wl.d_h])
    assert np.all(np.abs(fq[:, :wl.d_c] - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6 * np.abs(ref).max())
    assert np.array_equal(fq[:, wl.d_c:], uq[:, wl.d_h:])
    wo = st.w_o.double().cpu().numpy().reshape(wl.d_model, wl.n_h, wl.d_v)
    uv = st.w_uv.double().cpu().numpy().reshape(wl.n_h, wl.d_v, wl.d_c)
    fo = st.w_fused_o.double().cpu().numpy().reshape(wl.d_model, wl.n_h, wl.d_c)
    ref = np.einsum("nhv,hvc->nhc", wo, uv)
    assert np.all(np.abs(fo - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6 * np.abs(ref).max())


def test_fused_query_projection_matches_per_head_path():
    a = DecodeStep(LAYER)
    a.project()
    a.absorb_q()
    b = DecodeStep(LAYER.replace(fused=True))
    b.project_absorbed()
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    assert rel_to_max(b.q_cat.float().cpu().numpy(), a.q_cat.float().cpu().numpy()) <= 2e-2


@pytest.mark.parametrize("wl", [LAYER.replace(fused=True),
                                synth.EXTRA_WORKLOADS["dsv2_layer_b64_ctx32k_fused"].replace(
                                    batch=4, ctx=2000)], ids=["small", "dsv2_shapes"])
def test_fused_layer_step_against_oracle(wl):
    st = DecodeStep(wl)
    st.run()
    torch.cuda.synchronize()
    assert st.status() == 0, f"status {st.status():#x}"
    ex = Expected(wl)
    for b in range(wl.batch):
        got = {"o_lat": st.o_lat[b].double().cpu().numpy(), "lse": st.lse[b].double().cpu().numpy(),
               "u": st.u[b].double().cpu().numpy()}
        errs = gate_errors(got, ex.seq(b))
        assert not gate_failures(errs, TOL["bf16"], lse_tol(wl)), (b, errs)
