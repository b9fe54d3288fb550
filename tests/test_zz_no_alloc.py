"""The allocation-free decode entry point (mla_decode_attn_static).

Some callers cannot hand the library a workspace: a plugin host or embedded
runtime that passes a stream but no allocator, or a serving loop that bans
device allocations once it has started so that no step ever waits on the
allocator. They call mla_decode_attn_static, which keeps the plan and the
split partials in a fixed device array inside the library. It must give the
same results as mla_decode_attn + mla_combine with a caller workspace, call
after call, match the oracle, and refuse a batch too large for its fixed
scratch with a clear error.

This file is named so that pytest collects it after every other test.
"""
import ctypes

import pytest
import torch

from mla_latent_kv_67_b300 import binding as M
from mla_latent_kv_67_b300 import synth
from mla_latent_kv_67_b300.step import DecodeStep
from reference import Expected, gate_errors, gate_failures, lse_tol, rel_to_max

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}
CASES = [
    synth.Workload(name="static_f32", batch=4, n_h=8, d_h=32, d_r=16, d_c=64, d_v=32,
                   page_size=16, lens=(1, 33, 200, 517), dtype="f32", seed=901),
    synth.WORKLOADS["dsv2_b32_ctx4k"].replace(name="static_bf16", batch=5, n_h=16,
                                              lens=(1, 64, 300, 1500, 4096), seed=902),
    # the DeepSeek-V2 shape: 128 heads, d_c 512, bf16 -> the tcgen05 pair
    # kernel runs on the static scratch
    synth.WORKLOADS["dsv2_b32_ctx4k"].replace(
        name="static_dsv2_b32", lens=tuple([1, 64, 65, 4096] + [97 * i + 13 for i in range(1, 29)]),
        seed=903),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_static_scratch_matches_workspace_decode(wl):
    st = DecodeStep(wl)
    if wl.n_h == 128 and wl.dtype == "bf16":
        assert M.mla_decode_path(st.dtype, st.dims) == 1, "expected the tensor-core kernel"
    st.absorb_q()
    st.plan()
    st.attend()
    st.combine()
    torch.cuda.synchronize()
    assert st.status() == 0
    ref_o, ref_l = st.o_lat.clone(), st.lse.clone()
    for call in range(2):
        o = torch.full_like(ref_o, float("nan"))
        l = torch.full_like(ref_l, float("nan"))
        M.mla_decode_attn_static(st.q_cat, st.cache, st.block_table, st.seq_lens, wl.scale, o, l,
                                 st.dims, st.dev_status)
        torch.cuda.synchronize()
        assert st.status() == 0
        err_o = rel_to_max(o.cpu().numpy(), ref_o.cpu().numpy())
        err_l = rel_to_max(l.cpu().numpy(), ref_l.cpu().numpy())
        assert err_o <= TOL[wl.dtype] and err_l <= TOL[wl.dtype], (call, err_o, err_l)
        if wl.n_h == 128:
            # same plan, same kernels: the same bits as the workspace path
            assert torch.equal(o, ref_o) and torch.equal(l, ref_l), call
    if wl.n_h == 128:
        ex = Expected(wl)
        for b in range(wl.batch):
            got = {"o_lat": o[b].double().cpu().numpy(), "lse": l[b].double().cpu().numpy()}
            errs = gate_errors(got, ex.seq(b))
            assert not gate_failures(errs, TOL["bf16"], lse_tol(wl)), (b, errs)


def test_static_scratch_refuses_a_plan_that_does_not_fit():
    # fp32 with 128 heads x 512 latent runs the CUDA-core kernel on one
    # worker per SM; its split partials alone exceed the fixed scratch.
    d = M.Dims(128, 128, 64, 512, 128, 0, 0, 64)
    if M.mla_decode_workspace_size(8, M.MLA_F32, d) <= (48 << 20):
        pytest.skip("on this device the plan fits the static scratch")
    dummy = torch.zeros(16, dtype=torch.float32, device="cuda")
    p = dummy.data_ptr()
    st = M.lib().mla_decode_attn_static(p, p, p, 1, 1, p, 8, 1.0, p, p, M.MLA_F32,
                                        ctypes.byref(d), None, None)
    assert st == M.MLA_ERR_WORKSPACE
    msg = M.lib().mla_last_error().decode()
    assert "static scratch" in msg and "bytes" in msg
