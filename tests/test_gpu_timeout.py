"""Bounded device waits: every mbarrier wait of the tensor-core decode kernel
gives up after a time limit, reports MLA_DEV_TIMEOUT in the status word and
lets the kernel return, so a lost arrival never hangs the GPU.

The test loads the library's test build (libmla_b300_testhooks.so: the same
sources with the wait limit cut to 20 ms and mla_test_withhold_pages), makes
the page producer of each tensor-core decode kernel withhold every page --
before any copy or product is issued -- and checks that the call returns,
the status word says MLA_DEV_TIMEOUT, and a normal decode afterwards in the
same process still matches the oracle. Nothing faults and nothing is left
waiting.
"""
import ctypes
import time

import pytest
import torch

from mla_latent_kv_67_b300 import binding as M
from mla_latent_kv_67_b300 import build as B
from mla_latent_kv_67_b300 import synth
from mla_latent_kv_67_b300.step import DecodeStep
from reference import TOL, Expected, gate_errors, gate_failures, lse_tol

pytestmark = pytest.mark.gpu


def hook_lib():
    lib = ctypes.CDLL(B.build(hooks=True))
    for name, (res, args) in M._SIGS.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    lib.mla_test_withhold_pages.restype = None
    lib.mla_test_withhold_pages.argtypes = [ctypes.c_int]
    return lib


@pytest.mark.parametrize("path", [1, 2], ids=["score_value_pair", "latent_split"])
def test_withheld_pages_time_out_and_the_next_call_is_correct(monkeypatch, path):
    lib = hook_lib()
    monkeypatch.setattr(M, "_lib", lib)  # every binding call goes to the test build
    wl = synth.WORKLOADS["dsv2_b32_ctx4k"].replace(name="timeout", batch=3, lens=(100, 700, 4096),
                                                   seed=31)
    lib.mla_force_decode_path(path)
    st = DecodeStep(wl)
    if M.mla_decode_path(st.dtype, st.dims) != path:
        lib.mla_force_decode_path(-1)
        pytest.skip("tensor-core decode kernel not available")
    st.absorb_q()
    st.plan()
    torch.cuda.synchronize()
    assert st.status() == 0
    lib.mla_test_withhold_pages(1)
    try:
        t0 = time.perf_counter()
        st.attend()
        torch.cuda.synchronize()
        waited = time.perf_counter() - t0
    finally:
        lib.mla_test_withhold_pages(0)
    assert st.status() & M.MLA_DEV_TIMEOUT, f"status {st.status():#x}"
    assert waited < 5.0, f"the kernel took {waited:.2f} s to give up"
    # the context is intact: a normal step in the same process is correct
    st.dev_status.zero_()
    st.run()
    torch.cuda.synchronize()
    assert st.status() == 0, f"status {st.status():#x}"
    lib.mla_force_decode_path(-1)
    ex = Expected(wl)
    for b in range(wl.batch):
        got = {"o_lat": st.o_lat[b].double().cpu().numpy(), "lse": st.lse[b].double().cpu().numpy(),
               "o": st.o[b].double().cpu().numpy().reshape(wl.n_h, wl.d_v)}
        errs = gate_errors(got, ex.seq(b))
        assert not gate_failures(errs, TOL["bf16"], lse_tol(wl)), (b, errs)
