"""The tcgen05 decode kernel: its tensor-core data path on one page, then the
whole kernel against the CUDA-core kernel and the oracle."""
import numpy as np
import pytest
import torch

from mla_latent_kv_67_b300 import binding as M
from mla_latent_kv_67_b300 import synth
from mla_latent_kv_67_b300.step import DecodeStep
from reference import LSE_ABS, Expected, rel_to_max

pytestmark = pytest.mark.gpu

DIMS = M.Dims(128, 128, 64, 512, 128, 0, 0, 64)


def tc_available():
    return M.mla_decode_path(M.MLA_BF16, DIMS) == 1


@pytest.mark.parametrize("half", [0, 1])
def test_tc_page_selftest(half):
    """S = Q.Page^T (Q partly from TMEM, partly from SMEM; page K-major) and
    O = P.Page[:, half] (page read MN-major) on one page, against torch fp64
    products of the same bf16 values."""
    if not tc_available():
        pytest.skip("no sm_103 tensor-core path")
    g = torch.Generator().manual_seed(5 + half)
    q = torch.randn(128, 576, generator=g).bfloat16()
    page = torch.randn(64, 576, generator=g).bfloat16()
    pm = torch.rand(128, 64, generator=g).bfloat16()
    s_out = torch.full((128, 64), float("nan"), device="cuda")
    o_out = torch.full((128, 256), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.mla_tc_selftest(q.cuda(), page.cuda(), pm.cuda(), s_out, o_out, half, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    s_ref = q.double() @ page.double().T
    o_ref = pm.double() @ page.double()[:, 256 * half:256 * half + 256]
    es = rel_to_max(s_out.cpu().numpy(), s_ref.numpy())
    eo = rel_to_max(o_out.cpu().numpy(), o_ref.numpy())
    assert es < 1e-5 and eo < 1e-5, (es, eo)


CROSS = synth.WORKLOADS["dsv2_b32_ctx4k"].replace(
    name="tc_cross", batch=7, lens=(1, 63, 64, 65, 1000, 4096, 2500), seed=21)


def _run(wl, path):
    M.mla_force_decode_path(path)
    try:
        st = DecodeStep(wl)
        st.run()
        torch.cuda.synchronize()
        return st
    finally:
        M.mla_force_decode_path(-1)


def test_tc_matches_simt_and_oracle():
    """Both decode kernels on the same inputs; both against the oracle."""
    if not tc_available():
        pytest.skip("no sm_103 tensor-core path")
    a = _run(CROSS, 1)
    b = _run(CROSS, 0)
    assert a.status() == 0 and b.status() == 0
    assert rel_to_max(a.o_lat.cpu().numpy(), b.o_lat.cpu().numpy()) < 2e-2
    ex = Expected(CROSS)
    for i in range(CROSS.batch):
        e = ex.seq(i)
        err = rel_to_max(a.o_lat[i].cpu().numpy(), e["o_lat"])
        lerr = np.max(np.abs(a.lse[i].cpu().numpy() - e["lse"]))
        assert err < 2e-2 and lerr < LSE_ABS["bf16"], (i, err, lerr)


def test_tc_timeout_free_on_idle_workers():
    """More workers than pages: idle CTAs exit cleanly, results correct."""
    if not tc_available():
        pytest.skip("no sm_103 tensor-core path")
    wl = CROSS.replace(name="tc_tiny", batch=2, lens=(5, 70))
    st = _run(wl, 1)
    assert st.status() == 0
    ex = Expected(wl)
    for i in range(2):
        assert rel_to_max(st.o_lat[i].cpu().numpy(), ex.seq(i)["o_lat"]) < 2e-2
