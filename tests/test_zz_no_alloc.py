"""The allocation-free decode entry point (mla_decode_attn_static).

Callers that cannot allocate device memory while decoding (stream capture in
global mode, plugin hosts without an allocator, serving loops that ban
allocations after start-up) use this call instead of the workspace one. It
must give the same results as mla_decode_attn + mla_combine with a caller
workspace, call after call, and refuse a batch too large for its fixed
scratch with a clear error.

This file is named so that pytest collects it after every other test.
"""
import ctypes

import pytest
import torch

from mla_latent_kv_67_b300 import binding as M
from mla_latent_kv_67_b300 import synth
from mla_latent_kv_67_b300.step import DecodeStep
from reference import rel_to_max

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}
CASES = [
    synth.Workload(name="static_f32", batch=4, n_h=8, d_h=32, d_r=16, d_c=64, d_v=32,
                   page_size=16, lens=(1, 33, 200, 517), dtype="f32", seed=901),
    synth.WORKLOADS["dsv2_b32_ctx4k"].replace(name="static_bf16", batch=5, n_h=16,
                                              lens=(1, 64, 300, 1500, 4096), seed=902),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_static_scratch_matches_workspace_decode(wl):
    st = DecodeStep(wl)
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
