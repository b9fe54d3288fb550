"""Expected values for a workload's sequences, computed by the fp64 oracle
from the seeded inputs, and the parity gate that compares the GPU's outputs
with them. Imports only ``oracle`` and ``synth`` (never the CUDA path)."""
from __future__ import annotations

import numpy as np

from oracle import mla_oracle as O
from mla_latent_kv_67_b300 import synth

# Tolerances of the parity gate.
#  * Tensors (o_lat, o, u): max |gpu - ref| / max |ref| -- 1e-5 on the fp32
#    path, 2e-2 on the bf16 path (bf16 cache and weights, bf16 q_cat and
#    probabilities, fp32 accumulation).
#  * lse (natural log of the softmax normaliser) is gated on its ABSOLUTE
#    error, since an error in it is an error of the normaliser itself. The
#    bf16 rounding of q_abs moves every score s_j by scale * (dq . c_j); lse
#    moves by the p-weighted mean of those shifts, which is largest when one
#    token dominates (a one-token context: lse = s_0). A simulation of the
#    bf16 roundings in fp64 gives a worst |d lse| of 4.9e-3 on attention-only
#    workloads (q_abs rounded) and 9.0e-3 on the full layer (c_Q, q, q_cat
#    and the appended row rounded as well), both at one-token contexts, and
#    2.7e-4 / 1.2e-3 at 4096 tokens. The gates sit at twice the worst case;
#    one dropped 64-token page of a 4096-token context moves lse by 0.023 to
#    0.028 (max over heads), which the attention-only gate rejects.
TOL = {"f32": 1e-5, "bf16": 2e-2}
LSE_ABS = {"f32": 1e-5, "bf16": 1e-2, "bf16_layer": 2e-2}


def rel_to_max(got, ref) -> float:
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def lse_tol(wl: synth.Workload) -> float:
    if wl.dtype == "f32":
        return LSE_ABS["f32"]
    return LSE_ABS["bf16_layer"] if wl.mode == "layer" else LSE_ABS["bf16"]


def gate_errors(got: dict, ref: dict, explicit_heads=None) -> dict:
    """Errors of one sequence's GPU outputs ``got`` (host arrays: any of
    o_lat [n_h, d_c], o [n_h, d_v], lse [n_h], u [d_model]) against the
    oracle's ``ref`` (from :meth:`Expected.seq`)."""
    errs = {}
    for k in ("o_lat", "o", "u"):
        if k in got:
            errs[k] = rel_to_max(got[k], ref[k])
    if "o" in got and explicit_heads is not None and "o_explicit" in ref:
        errs["o_explicit"] = rel_to_max(np.asarray(got["o"])[list(explicit_heads)],
                                        ref["o_explicit"])
    if "lse" in got:
        errs["lse_abs"] = float(np.max(np.abs(np.asarray(got["lse"], np.float64) - ref["lse"])))
        if explicit_heads is not None and "lse_explicit" in ref:
            errs["lse_explicit_abs"] = float(np.max(np.abs(
                np.asarray(got["lse"], np.float64)[list(explicit_heads)] - ref["lse_explicit"])))
    return errs


def gate_failures(errs: dict, tol: float, lse_abs: float) -> list[str]:
    """The gate's verdict: the names of the errors above their bound."""
    bad = []
    for k, v in errs.items():
        bound = lse_abs if k.startswith("lse") else tol
        if not v <= bound:
            bad.append(f"{k}={v:.3g}>{bound:g}")
    return bad


class Expected:
    """Oracle inputs and outputs for one workload (weights drawn once)."""

    def __init__(self, wl: synth.Workload):
        self.wl = wl
        self.lens = synth.seq_lens(wl)
        self.w = {k: synth.weight(wl, k).astype(np.float64) for k in ("w_uk", "w_uv")}
        if wl.mode in ("layer", "prefill"):
            for k in ("w_dkv", "w_kr", "w_uq", "w_qr"):
                self.w[k] = synth.weight(wl, k).astype(np.float64)
            if wl.d_cq:
                self.w["w_dq"] = synth.weight(wl, "w_dq").astype(np.float64)
            if wl.mode == "layer":
                self.w["w_o"] = synth.weight(wl, "w_o").astype(np.float64)
            self.x = synth.tokens(wl).astype(np.float64)
        else:
            self.q = synth.query(wl).astype(np.float64)

    def appended_rows(self, b: int):
        """Rows the append step writes for sequence b: (positions, c, k_r)."""
        wl = self.wl
        if wl.mode == "layer":
            pos = np.array([self.lens[b] - 1])
            x = self.x[b:b + 1]
        else:
            pos = np.arange(wl.ctx)
            x = self.x
        c, k = O.latent_cache_row(x, self.w["w_dkv"], self.w["w_kr"], pos, wl.rope_base)
        return pos, c, k

    def query(self, b: int):
        """(q_c [n_h, d_h], q_r [n_h, d_r]) of query row b (sequence b, or
        with several new tokens per sequence row b = sequence * q_len + t)."""
        wl = self.wl
        if wl.mode == "attn":
            return self.q[b, :, :wl.d_h], self.q[b, :, wl.d_h:]
        x = self.x[b] if wl.mode == "layer" else self.x[-1]
        pos = self.lens[b] - 1 if wl.mode == "layer" else wl.ctx - 1
        return O.project_query(x, self.w["w_uq"], self.w["w_qr"], pos, wl.n_h,
                               w_dq=self.w.get("w_dq"), base=wl.rope_base)

    def cache_rows(self, b: int):
        """(c [N, d_c], k_r [N, d_r]) of sequence b as the oracle sees them."""
        wl = self.wl
        n = int(self.lens[b])
        nd = int(synth.drawn_rows(wl, self.lens)[b])
        rows = synth.cache_rows(wl, b, nd).astype(np.float64)
        c, k = rows[:, :wl.d_c], rows[:, wl.d_c:]
        if nd < n:
            _, c2, k2 = self.appended_rows(b)
            c, k = np.concatenate([c, c2]), np.concatenate([k, k2])
        return c, k

    def seq(self, b: int, explicit_heads=None, drop_rows=None):
        """Oracle outputs of query row b (sequence b; with q_len new tokens
        per sequence, row b = sequence * q_len + t, which sees the first
        ``multi_token_lengths(len, q_len)[t]`` cached rows): absorbed (all
        heads) and, for ``explicit_heads``, the explicit non-absorbed
        definition. ``drop_rows`` (a slice of token indices) removes those
        cached tokens from the oracle's input: a planted mistake for checking
        that the parity gate rejects a wrong answer."""
        wl = self.wl
        q_c, q_r = self.query(b)
        seq, t = divmod(b, wl.q_len)
        c, k = self.cache_rows(seq)
        if wl.q_len > 1:
            n = int(O.multi_token_lengths(len(c), wl.q_len)[t])
            c, k = c[:n], k[:n]
        if drop_rows is not None:
            keep = np.ones(len(c), bool)
            keep[drop_rows] = False
            c, k = c[keep], k[keep]
        o, o_lat, lse = O.attention_absorbed(q_c, q_r, c, k, self.w["w_uk"], self.w["w_uv"], wl.scale)
        out = dict(o=o, o_lat=o_lat, lse=lse, q_c=q_c, q_r=q_r)
        if explicit_heads is not None:
            oe, le = O.attention_explicit(q_c, q_r, c, k, self.w["w_uk"], self.w["w_uv"],
                                          wl.scale, heads=explicit_heads)
            out["o_explicit"], out["lse_explicit"] = oe, le
        if wl.mode == "layer":
            out["u"] = O.output_projection(o, self.w["w_o"])
        return out
