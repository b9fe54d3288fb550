"""mla_combine_absorb_out is mla_combine followed by mla_absorb_out, bit for
bit: o_lat, lse and o agree exactly with the two separate calls on the same
decode output, for split counts of one, a few (one load round), more than
the four of a round, and more than 32 (the lse reduction's extra pass)."""
import pytest
import torch

from mla_latent_kv_67_b300 import binding as M
from mla_latent_kv_67_b300 import synth
from mla_latent_kv_67_b300.step import DecodeStep

pytestmark = pytest.mark.gpu

BASE = synth.WORKLOADS["dsv2_b32_ctx4k"]
CASES = {
    "b32_ctx4k": BASE,
    "b40_ragged": BASE.replace(name="b40_ragged", batch=40, ctx=0, ctx_range=(64, 3000)),
    "b16_ctx20k": BASE.replace(name="b16_ctx20k", batch=16, ctx=20000),
    "b16_one_long": BASE.replace(name="b16_one_long", batch=16, ctx=0,
                                 lens=[131072] + [700 + 37 * i for i in range(15)]),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fused_equals_separate(name):
    wl = CASES[name]
    st = DecodeStep(wl)
    assert M.mla_decode_path(st.dtype, st.dims) == 1
    st.absorb_q()
    st.plan()
    st.attend()
    torch.cuda.synchronize()
    o_lat0, lse0 = st.o_lat.clone(), st.lse.clone()
    st.combine()
    st.absorb_out()
    torch.cuda.synchronize()
    sep = (st.o_lat.clone(), st.lse.clone(), st.o.clone())
    st.o_lat.copy_(o_lat0)
    st.lse.copy_(lse0)
    st.o.zero_()
    st.combine_absorb_out()
    torch.cuda.synchronize()
    assert st.status() == 0, f"device status {st.status():#x}"
    for what, a, b in zip(("o_lat", "lse", "o"), sep, (st.o_lat, st.lse, st.o)):
        assert torch.equal(a, b), f"{name}: {what} differs (max |d| {(a - b).abs().max().item()})"
