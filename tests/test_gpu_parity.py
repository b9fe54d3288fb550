"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs.

Tolerances (``tests/reference.py`` states them and their derivation):
  * fp32 path: max |gpu - ref| / max |ref| <= 1e-5;
  * bf16 path (bf16 cache and weights, bf16 q_cat and probabilities, fp32
    accumulation): max |gpu - ref| / max |ref| <= 2e-2;
  * lse: an absolute bound (1e-5 fp32; 1e-2 bf16; 2e-2 on the full-layer
    workload, whose query passes through three more bf16 roundings).
"""
import numpy as np
import pytest
import torch

from mla_latent_kv_67_b300 import binding as M
from mla_latent_kv_67_b300 import synth
from mla_latent_kv_67_b300.step import DecodeStep
from reference import (Expected, TOL, gate_errors, gate_failures, lse_tol, rel_to_max)

pytestmark = pytest.mark.gpu

TOL_F32, TOL_BF16 = TOL["f32"], TOL["bf16"]


def run(wl, **kw):
    st = DecodeStep(wl, **kw)
    st.run()
    torch.cuda.synchronize()
    assert st.status() == 0, f"device status {st.status():#x}"
    return st


def host_outputs(st, b, what=("o_lat", "o", "lse")):
    """Sequence b's GPU outputs as host float64 arrays."""
    wl = st.wl
    got = {}
    if "o_lat" in what:
        got["o_lat"] = st.o_lat[b].double().cpu().numpy()
    if "o" in what:
        got["o"] = st.o[b].double().cpu().numpy().reshape(wl.n_h, wl.d_v)
    if "lse" in what:
        got["lse"] = st.lse[b].double().cpu().numpy()
    if "u" in what:
        got["u"] = st.u[b].double().cpu().numpy()
    return got


def check_seq(st, ex, b, tol, explicit_heads=None, what=("o_lat", "o", "lse")):
    e = ex.seq(b, explicit_heads=explicit_heads)
    errs = gate_errors(host_outputs(st, b, what), e, explicit_heads)
    bad = gate_failures(errs, tol, lse_tol(st.wl))
    assert not bad, f"seq {b}: {bad} ({errs})"
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


@pytest.mark.parametrize("path", [0, 1, 2])
def test_bf16_ragged_small(path):
    """Several pages and ragged tails (1, 17, 64, 65, 337, 1000 tokens):
    every head against the absorbed oracle, three heads against the explicit
    definition."""
    M.mla_force_decode_path(path)
    try:
        if path >= 1 and M.mla_decode_path(M.MLA_BF16, M.Dims.of(RAGGED)) != path:
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
def _full(name, explicit_seqs, explicit_heads, what=("o_lat", "o", "lse")):
    """Every sequence and every head of a full-size workload against the
    absorbed fp64 oracle; the explicit (non-absorbed) oracle on the sampled
    sequences and heads. Returns the run, the oracle and the worst errors."""
    wl = synth.WORKLOADS[name]
    st = run(wl)
    ex = Expected(wl)
    worst = {}
    for b in range(wl.batch):
        eh = explicit_heads if b in explicit_seqs else None
        errs = check_seq(st, ex, b, TOL_BF16, explicit_heads=eh, what=what)
        for k, v in errs.items():
            worst[k] = max(worst.get(k, 0.0), v)
    print(name, {k: f"{v:.3g}" for k, v in worst.items()})
    return st, ex, worst


@pytest.mark.slow
def test_full_dsv2_b32_ctx4k():
    """All 32 sequences; and the gate itself must reject two planted wrong
    answers on the same GPU output: the oracle with one 64-token page of one
    sequence left out, and the oracle with two heads swapped."""
    st, ex, _ = _full("dsv2_b32_ctx4k", (0, 13, 31), [0, 101])
    tol_l = lse_tol(st.wl)
    for b, page in ((3, 10), (17, 63)):
        got = host_outputs(st, b)
        wrong = ex.seq(b, drop_rows=slice(64 * page, 64 * page + 64))
        errs = gate_errors(got, wrong)
        assert gate_failures(errs, TOL_BF16, tol_l), f"a dropped page passed the gate: {errs}"
        assert errs["lse_abs"] > tol_l and errs["o_lat"] > TOL_BF16, errs
        right = ex.seq(b)
        swapped = dict(right)
        for k in ("o", "o_lat", "lse"):
            v = right[k].copy()
            v[[5, 90]] = v[[90, 5]]
            swapped[k] = v
        errs = gate_errors(got, swapped)
        assert errs["o"] > TOL_BF16 and errs["o_lat"] > TOL_BF16 and errs["lse_abs"] > tol_l, errs


@pytest.mark.slow
def test_full_dsv2_b4_ctx128k():
    _full("dsv2_b4_ctx128k", range(4), [64])


@pytest.mark.slow
def test_full_dsv2_b128_ragged():
    _full("dsv2_b128_ragged", (0, 1, 63, 127), [3])


@pytest.mark.slow
def test_full_dsv2_layer_b64_ctx32k():
    _full("dsv2_layer_b64_ctx32k", (0, 63), [9], what=("o_lat", "o", "lse", "u"))
