"""Decode over the FP8 latent cache (MLA_FP8_E4M3: E4M3 codes with one float
scale per row for c_KV, the RoPE key in bf16) against the oracle, which sees
the values the stored rows decode to (code * scale), exactly as the bf16
workloads' oracle sees the bf16-rounded inputs. Every sequence and head
against the absorbed oracle, sampled heads against the explicit one."""
import pytest
import torch

from mla_latent_kv_67_b300 import binding as M
from mla_latent_kv_67_b300 import synth
from mla_latent_kv_67_b300.step import DecodeStep
from reference import TOL, Expected, gate_errors, gate_failures, lse_tol

pytestmark = pytest.mark.gpu

FP8 = synth.EXTRA_WORKLOADS["dsv2_b32_ctx4k_fp8"]


@pytest.mark.parametrize("wl", [FP8.replace(name="fp8_ragged", batch=6,
                                            lens=(1, 63, 65, 700, 1500, 4096), seed=71),
                                FP8.replace(name="fp8_mtp", batch=3, lens=(5, 300, 2000), q_len=2,
                                            seed=72)], ids=["ragged", "two_new_tokens"])
def test_fp8_cache_decode_matches_oracle(wl):
    st = DecodeStep(wl)
    assert st.cache.dtype == torch.uint8
    st.run()
    torch.cuda.synchronize()
    assert st.status() == 0, f"status {st.status():#x}"
    ex = Expected(wl)
    for v in range(wl.batch * wl.q_len):
        eh = [0, 90] if v % 2 == 0 else None
        got = {"o_lat": st.o_lat[v].double().cpu().numpy(), "lse": st.lse[v].double().cpu().numpy(),
               "o": st.o[v].double().cpu().numpy().reshape(wl.n_h, wl.d_v)}
        errs = gate_errors(got, ex.seq(v, explicit_heads=eh), eh)
        assert not gate_failures(errs, TOL["bf16"], lse_tol(wl)), (v, errs)


@pytest.mark.parametrize("lens", [(1, 63, 65, 700, 1500, 4096), (64, 128, 129)],
                         ids=["ragged", "page_edges"])
def test_fp8_staged_matches_oracle(lens):
    """mla_decode_attn_fp8_staged: pages widened to bf16 rows, then the bf16
    decode kernels. The widening rounds code * scale to bf16, which the bf16
    gate covers."""
    wl = FP8.replace(name="fp8_staged", batch=len(lens), lens=lens, seed=73)
    st = DecodeStep(wl, fp8_staged=True)
    st.run()
    torch.cuda.synchronize()
    assert st.status() == 0, f"status {st.status():#x}"
    ex = Expected(wl)
    for v in range(wl.batch):
        eh = [0, 90] if v % 2 == 0 else None
        got = {"o_lat": st.o_lat[v].double().cpu().numpy(), "lse": st.lse[v].double().cpu().numpy(),
               "o": st.o[v].double().cpu().numpy().reshape(wl.n_h, wl.d_v)}
        errs = gate_errors(got, ex.seq(v, explicit_heads=eh), eh)
        assert not gate_failures(errs, TOL["bf16"], lse_tol(wl)), (v, errs)


def test_fp8_staged_agrees_with_cuda_core_kernel():
    """Both FP8 decode entry points on the same batch: the staged result
    differs from the CUDA-core kernel's only by the bf16 rounding of the
    widened rows and the bf16 partials."""
    wl = FP8.replace(name="fp8_both", batch=4, lens=(3, 640, 1025, 2048), seed=74)
    a, b = DecodeStep(wl), DecodeStep(wl, fp8_staged=True)
    a.run()
    b.run()
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    d = (a.o_lat - b.o_lat).abs().amax(dim=-1) / a.o_lat.abs().amax(dim=-1)
    assert float(d.max()) < 2e-2
    assert float((a.lse - b.lse).abs().max()) < 2e-2


def test_fp8_staged_refuses_short_workspace_and_reports_bad_block():
    wl = FP8.replace(name="fp8_err", batch=2, lens=(70, 200), seed=75)
    st = DecodeStep(wl, fp8_staged=True)
    short = st.workspace[: st.workspace.numel() - 256]
    with pytest.raises(M.MlaError) as e:
        M.mla_decode_attn_fp8_staged(st.q_cat, st.cache, st.block_table, st.seq_lens, wl.scale,
                                     short, st.o_lat, st.lse, st.dims, st.dev_status)
    assert e.value.status == M.MLA_ERR_WORKSPACE
    bt = st.block_table.clone()
    bt[1, 2] = st.cache.shape[0]  # one past the pool
    M.mla_decode_attn_fp8_staged(st.q_cat, st.cache, bt, st.seq_lens, wl.scale, st.workspace,
                                 st.o_lat, st.lse, st.dims, st.dev_status)
    torch.cuda.synchronize()
    assert st.status() & M.MLA_DEV_BAD_BLOCK


@pytest.mark.slow
@pytest.mark.parametrize("staged", [False, True], ids=["cuda_core", "staged"])
def test_fp8_full_b32_ctx4k(staged):
    st = DecodeStep(FP8, fp8_staged=staged)
    st.run()
    torch.cuda.synchronize()
    assert st.status() == 0
    ex = Expected(FP8)
    for b in range(FP8.batch):
        got = {"o_lat": st.o_lat[b].double().cpu().numpy(), "lse": st.lse[b].double().cpu().numpy()}
        errs = gate_errors(got, ex.seq(b))
        assert not gate_failures(errs, TOL["bf16"], lse_tol(FP8)), (b, errs)


def test_fp8_rejected_outside_decode():
    """The FP8 dtype is refused by calls that do not read the cache."""
    d = M.Dims(128, 128, 64, 512, 128, 0, 0, 64)
    t = torch.zeros(16, device="cuda")
    import ctypes
    st = M.lib().mla_absorb_q(t.data_ptr(), t.data_ptr(), t.data_ptr(), 1, M.MLA_FP8_E4M3,
                              ctypes.byref(d), None)
    assert st == M.MLA_ERR_INVALID_ARG
