"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs.

Tolerances (from the stated precision of each path):
  * fp32 path: max |gpu - ref| / max |ref| <= 1e-5;
  * bf16 path (bf16 cache and weights, bf16 q_cat and probabilities, fp32
    accumulation): max |gpu - ref| / max |ref| <= 2e-2.
"""
import numpy as np
import pytest
import torch

from mla_latent_kv_67_b300 import binding as M
from mla_latent_kv_67_b300 import synth
from mla_latent_kv_67_b300.step import DecodeStep
from reference import Expected, rel_to_max

pytestmark = pytest.mark.gpu

TOL_F32, TOL_BF16 = 1e-5, 2e-2


def run(wl, **kw):
    st = DecodeStep(wl, **kw)
    st.run()
    torch.cuda.synchronize()
    assert st.status() == 0, f"device status {st.status():#x}"
    return st


def check_seq(st, ex, b, tol, explicit_heads=None, what=("o_lat", "o", "lse")):
    e = ex.seq(b, explicit_heads=explicit_heads)
    errs = {}
    if "o_lat" in what:
        errs["o_lat"] = rel_to_max(st.o_lat[b].cpu().numpy(), e["o_lat"])
    if "o" in what:
        o = st.o[b].float().cpu().numpy().reshape(st.wl.n_h, st.wl.d_v)
        errs["o"] = rel_to_max(o, e["o"])
        if explicit_heads is not None:
            errs["o_explicit"] = rel_to_max(o[list(explicit_heads)], e["o_explicit"])
    if "lse" in what:
        errs["lse"] = float(np.max(np.abs(st.lse[b].cpu().numpy() - e["lse"]))
                            / max(1.0, np.max(np.abs(e["lse"]))))
    if "u" in what:
        errs["u"] = rel_to_max(st.u[b].cpu().numpy(), e["u"])
    for k, v in errs.items():
        assert v <= tol, f"seq {b}: {k} error {v:.3g} > {tol:g} ({errs})"
    return errs


# ------------------------------------------------------------ fp32 (cfg 1)
def test_tiny_f32_layer_full():
    """The tiny fp32 workload end to end: 256 tokens appended from x, query
    projected from the last one, attention, W^UV -- every output element
    against the explicit oracle."""
    wl = synth.WORKLOADS["tiny_f32_ctx256"]
    st = run(wl)
    ex = Expected(wl)
    check_seq(st, ex, 0, TOL_F32, explicit_heads=range(wl.n_h))
    # the cache rows the append step wrote
    pos, c, k = ex.appended_rows(0)
    rows = st.cache[0].cpu().numpy()
    assert rel_to_max(rows[:, :wl.d_c], c) <= TOL_F32
    assert rel_to_max(rows[:, wl.d_c:], k) <= TOL_F32
    # the projected query
    q_c, q_r = ex.query(0)
    q = st.q[0].cpu().numpy()
    assert rel_to_max(q[:, :wl.d_h], q_c) <= TOL_F32
    assert rel_to_max(q[:, wl.d_h:], q_r) <= TOL_F32


# ------------------------------------------------------- bf16, small sizes
RAGGED = synth.WORKLOADS["dsv2_b32_ctx4k"].replace(
    name="ragged_small", batch=6, lens=(1, 17, 64, 65, 64 * 5 + 17, 1000), seed=11)


@pytest.mark.parametrize("path", [0, 1])
def test_bf16_ragged_small(path):
    """Several pages and ragged tails (1, 17, 64, 65, 337, 1000 tokens):
    every head against the absorbed oracle, three heads against the explicit
    definition."""
    M.mla_force_decode_path(path)
    try:
        if path == 1 and M.mla_decode_path(M.MLA_BF16, M.Dims.of(RAGGED)) != 1:
            pytest.skip("tensor-core decode kernel not available")
        st = run(RAGGED)
        ex = Expected(RAGGED)
        for b in range(RAGGED.batch):
            check_seq(st, ex, b, TOL_BF16, explicit_heads=[0, 77, 127])
    finally:
        M.mla_force_decode_path(-1)


def test_bf16_paging_invariance():
    """A shuffled block table gives bit-identical results to a contiguous
    one (same plan, same reduction order)."""
    a = run(RAGGED)
    b = run(RAGGED.replace(shuffle_pages=False))
    assert torch.equal(a.o_lat, b.o_lat) and torch.equal(a.o, b.o)


def test_bf16_layer_small():
    """The full layer step (append, query projection with d_c'=1536, absorb,
    attention, W^UV, W^O) on 3 short sequences."""
    wl = synth.WORKLOADS["dsv2_layer_b64_ctx32k"].replace(batch=3, ctx=300)
    st = run(wl)
    ex = Expected(wl)
    for b in range(3):
        check_seq(st, ex, b, TOL_BF16, explicit_heads=[5], what=("o_lat", "o", "lse", "u"))


def test_bf16_append_slot_and_canaries():
    """The append step writes exactly the target rows, each equal to the
    oracle's fp64 row within one bf16 rounding; every other row (other
    sequences' rows, padding, spare pages) is untouched."""
    wl = synth.WORKLOADS["dsv2_layer_b64_ctx32k"].replace(batch=4, lens=(1, 64, 65, 200),
                                                          spare_pages=3, d_model=256, d_cq=64)
    st = DecodeStep(wl)
    before = st.cache.clone()
    st.append()
    torch.cuda.synchronize()
    assert st.status() == 0
    after = st.cache
    ex = Expected(wl)
    changed = (before.view(torch.int16) != after.view(torch.int16)).any(dim=-1)  # [pool, P]
    expect_changed = torch.zeros_like(changed)
    for b in range(wl.batch):
        p = int(ex.lens[b]) - 1
        blk, r = int(st.bt_np[b, p // wl.page_size]), p % wl.page_size
        expect_changed[blk, r] = True
        _, c, k = ex.appended_rows(b)
        row = after[blk, r].float().cpu().numpy().astype(np.float64)
        ref = np.concatenate([c[0], k[0]])
        # one rounding to bf16 (relative half-ulp 2^-9) plus fp32 accumulation
        assert np.all(np.abs(row - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-4 * np.abs(ref).max())
    assert torch.equal(changed, expect_changed)


def test_device_status_reports_bad_block_and_length():
    """A block id outside the pool and a length past the block table are
    reported in the status word; the kernels skip the access instead of
    faulting, and the rest of the batch is still computed."""
    wl = RAGGED.replace(name="bad", batch=3, lens=(100, 200, 50))
    st = DecodeStep(wl)
    st.block_table[1, 2] = st.pool + 5          # outside the pool
    st.seq_lens[2] = st.max_pages * wl.page_size + 1   # past the table
    st.run()
    torch.cuda.synchronize()
    s = st.status()
    assert s & M.MLA_DEV_BAD_BLOCK and s & M.MLA_DEV_BAD_LEN
    ex = Expected(wl)
    check_seq(st, ex, 0, TOL_BF16)               # sequence 0 unaffected
    assert torch.all(st.o_lat[2] == 0) and torch.all(torch.isinf(st.lse[2]))


def test_bf16_sequence_split_over_32_ways():
    """One 131072-token sequence among fifteen short ones: the plan splits it
    over more than 32 workers, so the merge takes its second pass over the
    split lse values; that sequence and a short one against the oracle."""
    wl = RAGGED.replace(name="many_splits", batch=16, shuffle_pages=True,
                        lens=tuple([131072] + [700 + 37 * i for i in range(15)]))
    st = run(wl)
    if M.mla_decode_path(st.dtype, st.dims) == 1:
        seq0 = st.workspace[256:256 + 32].cpu().numpy().view(np.int32)  # SeqPlan of sequence 0
        assert seq0[3] > 32, f"only {seq0[3]} splits"
    ex = Expected(wl)
    for b in (0, 7):
        check_seq(st, ex, b, TOL_BF16, explicit_heads=[33])


# ---------------------------------------------------- full-size workloads
def _sampled(name, seqs, explicit_heads, what=("o_lat", "o", "lse")):
    wl = synth.WORKLOADS[name]
    st = run(wl)
    ex = Expected(wl)
    worst = {}
    for b in seqs:
        errs = check_seq(st, ex, b, TOL_BF16, explicit_heads=explicit_heads, what=what)
        for k, v in errs.items():
            worst[k] = max(worst.get(k, 0.0), v)
    o = st.result()
    assert torch.isfinite(o).all()
    return worst


@pytest.mark.slow
def test_full_dsv2_b32_ctx4k():
    print(_sampled("dsv2_b32_ctx4k", range(0, 32, 3), explicit_heads=[0, 101]))


@pytest.mark.slow
def test_full_dsv2_b4_ctx128k():
    print(_sampled("dsv2_b4_ctx128k", range(4), explicit_heads=[64]))


@pytest.mark.slow
def test_full_dsv2_b128_ragged():
    print(_sampled("dsv2_b128_ragged", [0, 1, 63, 127], explicit_heads=[3]))


@pytest.mark.slow
def test_full_dsv2_layer_b64_ctx32k():
    print(_sampled("dsv2_layer_b64_ctx32k", [0, 63], explicit_heads=[9],
                   what=("o_lat", "o", "lse", "u")))
