"""Prefill in the MHA form (mla_gather_latent -> mla_expand_kv ->
mla_prefill_attn) against the oracle: the prompt's latent rows come from
the append step, every token's query from the query projection, and token
i's output is the attention over tokens 0..i (the oracle's multi-token
attention with every token new). The expanded keys and values against the
oracle's explicit up-projection of the same rows; the attention output
against the absorbed oracle on every head and the explicit definition on
sampled heads."""
import numpy as np
import pytest
import torch

from mla_latent_kv_67_b300 import binding as M
from mla_latent_kv_67_b300 import synth
from mla_latent_kv_67_b300.step import DecodeStep
from oracle import mla_oracle as O
from reference import TOL, LSE_ABS, rel_to_max

pytestmark = pytest.mark.gpu

BASE = synth.EXTRA_WORKLOADS["dsv2_prefill_4k"]


class PrefillOracle:
    def __init__(self, wl):
        self.wl = wl
        self.w = {k: synth.weight(wl, k).astype(np.float64)
                  for k in ("w_dkv", "w_kr", "w_uq", "w_qr", "w_dq", "w_uk", "w_uv")}
        self.x = synth.tokens(wl).astype(np.float64)
        pos = np.arange(wl.ctx)
        self.c, self.k = O.latent_cache_row(self.x, self.w["w_dkv"], self.w["w_kr"], pos,
                                            wl.rope_base)
        self.q_c, self.q_r = O.project_query(self.x, self.w["w_uq"], self.w["w_qr"], pos, wl.n_h,
                                             w_dq=self.w["w_dq"], base=wl.rope_base)

    def row(self, i, explicit_heads=None):
        """Outputs of prompt token i: it attends to tokens 0..i."""
        wl = self.wl
        n = int(O.multi_token_lengths(wl.ctx, wl.ctx)[i])
        o, _, lse = O.attention_absorbed(self.q_c[i], self.q_r[i], self.c[:n], self.k[:n],
                                         self.w["w_uk"], self.w["w_uv"], wl.scale)
        out = {"o": o, "lse": lse}
        if explicit_heads is not None:
            out["o_explicit"], out["lse_explicit"] = O.attention_explicit(
                self.q_c[i], self.q_r[i], self.c[:n], self.k[:n], self.w["w_uk"], self.w["w_uv"],
                wl.scale, heads=explicit_heads)
        return out


def run(wl):
    st = DecodeStep(wl)
    if M.mla_decode_path(st.dtype, st.dims) != 1:
        pytest.skip("tensor-core kernels not available")
    st.run()
    torch.cuda.synchronize()
    assert st.status() == 0, f"status {st.status():#x}"
    return st


def check_rows(st, ora, rows, explicit_every=7):
    wl = st.wl
    o = st.o_pf.double().cpu().numpy()
    lse = st.lse_pf.double().cpu().numpy()
    worst = {}
    for n, i in enumerate(rows):
        eh = [0, 64, 127] if n % explicit_every == 0 else None
        ref = ora.row(i, explicit_heads=eh)
        errs = {"o": rel_to_max(o[i], ref["o"]),
                "lse_abs": float(np.max(np.abs(lse[i] - ref["lse"])))}
        if eh is not None:
            errs["o_explicit"] = rel_to_max(o[i][eh], ref["o_explicit"])
        for k, v in errs.items():
            worst[k] = max(worst.get(k, 0.0), v)
        assert errs["o"] <= TOL["bf16"] and errs.get("o_explicit", 0) <= TOL["bf16"], (i, errs)
        assert errs["lse_abs"] <= LSE_ABS["bf16_layer"], (i, errs)
    return worst


def test_prefill_small_every_row():
    """300 prompt tokens (three query tiles, a ragged last one): every row,
    every head."""
    wl = BASE.replace(name="prefill_300", ctx=300, seed=61)
    st = run(wl)
    ora = PrefillOracle(wl)
    # the expanded keys and values of sampled tokens against the explicit
    # up-projection of the GPU's own (bf16) latent rows
    rows = st.rows.double().cpu().numpy()
    kn = st.k_nope.double().cpu().numpy()
    vv = st.v.double().cpu().numpy()
    for t in (0, 1, 150, 299):
        for h in (0, 77, 127):
            K, V = O.explicit_kv(rows[t:t + 1, :wl.d_c], rows[t:t + 1, wl.d_c:], ora.w["w_uk"],
                                 ora.w["w_uv"], h, wl.n_h)
            assert rel_to_max(kn[t, h], K[0, :wl.d_h]) <= 2.0 ** -7
            assert rel_to_max(vv[t, h], V[0]) <= 2.0 ** -7
    print(check_rows(st, ora, range(wl.ctx)))


def test_prefill_4k_sampled_rows():
    """The 4096-token prompt: the first, last and diagonal-tile edge rows,
    and a seeded sample, every head."""
    st = run(BASE)
    ora = PrefillOracle(BASE)
    g = np.random.default_rng(7)
    rows = sorted(set([0, 1, 63, 127, 128, 129, 255, 1000, 2047, 2048, 4094, 4095] +
                      g.integers(0, BASE.ctx, 20).tolist()))
    print(check_rows(st, ora, rows))
