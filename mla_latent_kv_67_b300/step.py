"""One decode step of a workload, as the sequence of C-ABI calls.

:class:`DecodeStep` uploads a workload's seeded inputs into device memory
(torch only allocates), then :meth:`DecodeStep.run` enqueues the calls of one
step on the current stream:

  attn    : absorb_q -> plan -> decode_attn -> combine -> absorb_out
            (with q_len > 1: q_len new tokens per sequence, B * q_len query
            rows, the _mtp plan and decode calls)
  layer   : append_latent -> project_q -> absorb_q -> plan -> decode_attn
            -> combine -> absorb_out -> out_proj
  prefill : append_latent (all ctx tokens) -> project_q (last token) ->
            absorb_q -> plan -> decode_attn -> combine -> absorb_out
  layer, fused weights: append_latent -> project_q_absorbed (writes q_cat)
            -> plan -> decode_attn -> combine -> out_proj_absorbed
  prefill_mha : append_latent (all ctx tokens) -> project_q (all tokens) ->
            gather_latent -> expand_kv -> prefill_attn
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as M
from . import synth


def to_device(arr: np.ndarray, wl: synth.Workload, device) -> torch.Tensor:
    """Storage-form numpy array -> device tensor (bf16 bits or float32)."""
    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


class DecodeStep:
    def __init__(self, wl: synth.Workload, device="cuda", out_dtype=None, fp8_staged=False):
        """fp8_staged: on the FP8 cache (one new token per sequence), decode
        with mla_decode_attn_fp8_staged (pages widened to bf16, then the bf16
        decode kernels) instead of the CUDA-core FP8 kernel."""
        self.wl, self.device = wl, torch.device(device)
        assert not fp8_staged or (wl.dtype == "fp8" and wl.q_len == 1)
        self.fp8_staged = fp8_staged
        self.dims = M.Dims.of(wl)
        self.dtype = {"bf16": M.MLA_BF16, "f32": M.MLA_F32, "fp8": M.MLA_FP8_E4M3}[wl.dtype]
        tdt = M.torch_dtype(self.dtype)
        dev = self.device
        lens = synth.seq_lens(wl)
        bt, pool = synth.block_table(wl, lens)
        self.lens_np, self.bt_np, self.pool = lens, bt, pool
        self.seq_lens = torch.from_numpy(lens).to(dev)
        self.block_table = torch.from_numpy(bt).to(dev)
        self.cache = to_device(synth.paged_cache(wl, lens, bt, pool), wl, dev)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
        B, n_h = wl.batch, wl.n_h
        W = lambda name: to_device(synth.storage(wl, synth.weight(wl, name)), wl, dev)
        self.w_uk, self.w_uv = W("w_uk"), W("w_uv")
        if wl.mode in ("layer", "prefill", "prefill_mha"):
            self.w_dkv_kr = to_device(synth.storage(wl, synth.joint_w_dkv_kr(
                synth.weight(wl, "w_dkv"), synth.weight(wl, "w_kr"))), wl, dev)
            self.w_uq_qr = to_device(synth.storage(wl, synth.joint_w_uq_qr(
                synth.weight(wl, "w_uq"), synth.weight(wl, "w_qr"), n_h)), wl, dev)
            self.w_dq = W("w_dq") if wl.d_cq else None
            self.x = to_device(synth.storage(wl, synth.tokens(wl)), wl, dev)
            max_pos = int(lens.max())
            self.rope = torch.empty((max_pos, wl.d_r // 2, 2), dtype=torch.float32, device=dev)
            M.mla_rope_table(self.rope, wl.rope_base)
            if wl.mode == "layer":
                self.append_pos = (self.seq_lens - 1).contiguous()
                self.append_seq = None
                self.q_pos = self.append_pos
                self.x_q = self.x
            elif wl.mode == "prefill":
                self.append_pos = torch.arange(wl.ctx, dtype=torch.int32, device=dev)
                self.append_seq = torch.zeros(wl.ctx, dtype=torch.int32, device=dev)
                self.q_pos = self.append_pos[-1:].contiguous()
                self.x_q = self.x[-1:].contiguous()
            else:  # prefill_mha: every prompt token is a query
                self.append_pos = torch.arange(wl.ctx, dtype=torch.int32, device=dev)
                self.append_seq = torch.zeros(wl.ctx, dtype=torch.int32, device=dev)
                self.q_pos = self.append_pos
                self.x_q = self.x
            T = wl.ctx if wl.mode == "prefill_mha" else B
            self.c_q = (torch.empty((T, wl.d_cq), dtype=tdt, device=dev) if wl.d_cq else None)
            self.q = torch.empty((T, n_h, wl.d_h + wl.d_r), dtype=tdt, device=dev)
            self.w_o = W("w_o") if wl.mode == "layer" else None
            if wl.fused:
                # W^UK and W^UV folded into the neighbouring weights once
                assert wl.mode == "layer"
                K = wl.d_cq or wl.d_model
                self.w_fused_q = torch.empty((n_h * (wl.d_c + wl.d_r), K), dtype=tdt, device=dev)
                M.mla_fuse_query_weights(self.w_uq_qr, self.w_uk, self.w_fused_q, self.dims)
                self.w_fused_o = torch.empty((wl.d_model, n_h * wl.d_c), dtype=tdt, device=dev)
                M.mla_fuse_output_weights(self.w_o, self.w_uv, self.w_fused_o, self.dims)
                self.o_lat_lowp = torch.empty((B, n_h * wl.d_c), dtype=tdt, device=dev)
        else:
            self.q = to_device(synth.storage(wl, synth.query(wl)), wl, dev)
        assert wl.q_len == 1 or wl.mode == "attn", "several new tokens: attention-only workloads"
        assert wl.dtype != "fp8" or wl.mode == "attn", "the FP8 cache: attention-only workloads"
        if wl.mode == "prefill_mha":
            N = wl.ctx
            self.rows = torch.empty((N, wl.d_c + wl.d_r), dtype=tdt, device=dev)
            self.k_nope = torch.empty((N, n_h, wl.d_h), dtype=tdt, device=dev)
            self.v = torch.empty((N, n_h, wl.d_v), dtype=tdt, device=dev)
            self.o_pf = torch.empty((N, n_h, wl.d_v), dtype=torch.bfloat16, device=dev)
            self.lse_pf = torch.empty((N, n_h), dtype=torch.float32, device=dev)
        R = B * wl.q_len  # query rows
        self.q_cat = torch.empty((R, n_h, wl.d_c + wl.d_r), dtype=tdt, device=dev)
        ws = (M.mla_decode_fp8_staged_workspace_size(R, bt.shape[1], self.dims) if fp8_staged
              else M.mla_decode_workspace_size(R, self.dtype, self.dims))
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=dev)
        self.o_lat = torch.empty((R, n_h, wl.d_c), dtype=torch.float32, device=dev)
        self.lse = torch.empty((R, n_h), dtype=torch.float32, device=dev)
        if out_dtype is None:
            out_dtype = tdt if wl.mode == "layer" else torch.float32
        self.o = torch.empty((R, n_h * wl.d_v), dtype=out_dtype, device=dev)
        self.u = (torch.empty((B, wl.d_model), dtype=torch.float32, device=dev)
                  if wl.mode == "layer" else None)
        self.max_pages = bt.shape[1]
        self._side = None  # side stream of run(), made on first use
        # mla_combine_absorb_out instead of the two calls: bit-identical, but
        # measured slower on B300 (dsv2_b32_ctx4k step 80 vs 79 us) -- the
        # merge inside the W^UV kernel serialises partial loads that the
        # separate merge kernel spreads over all SMs. Off by default.
        self.fuse_out = False

    # ------------------------------------------------------------- stages
    def append(self):
        M.mla_append_latent(self.x, self.w_dkv_kr, self.append_seq, self.append_pos,
                            self.block_table, self.rope, self.cache, self.dims, self.dev_status)

    def project(self):
        M.mla_project_q(self.x_q, self.w_dq, self.w_uq_qr, self.q_pos, self.rope, self.c_q,
                        self.q, self.dims, self.dev_status)

    def absorb_q(self):
        M.mla_absorb_q(self.q, self.w_uk, self.q_cat, self.dims)

    def plan(self):
        if self.wl.q_len > 1:
            M.mla_plan_decode_mtp(self.seq_lens, self.wl.q_len, self.max_pages, self.workspace,
                                  self.dtype, self.dims, self.dev_status)
        else:
            M.mla_plan_decode(self.seq_lens, self.max_pages, self.workspace, self.dtype,
                              self.dims, self.dev_status)

    def attend(self):
        if self.wl.q_len > 1:
            M.mla_decode_attn_mtp(self.q_cat, self.cache, self.block_table, self.seq_lens,
                                  self.wl.q_len, self.wl.scale, self.workspace, self.o_lat,
                                  self.lse, self.dims, self.dev_status)
        else:
            M.mla_decode_attn(self.q_cat, self.cache, self.block_table, self.seq_lens,
                              self.wl.scale, self.workspace, self.o_lat, self.lse, self.dims,
                              self.dev_status)

    def attend_fp8_staged(self):
        M.mla_decode_attn_fp8_staged(self.q_cat, self.cache, self.block_table, self.seq_lens,
                                     self.wl.scale, self.workspace, self.o_lat, self.lse,
                                     self.dims, self.dev_status)

    def combine(self):
        M.mla_combine(self.workspace, self.o_lat, self.lse, self.dtype, self.dims)

    def absorb_out(self):
        M.mla_absorb_out(self.o_lat, self.w_uv, self.o, self.dims)

    def combine_absorb_out(self):
        M.mla_combine_absorb_out(self.workspace, self.o_lat, self.lse, self.w_uv, self.o, self.dims,
                                 self.dev_status)

    def out_proj(self):
        M.mla_out_proj(self.o, self.w_o, self.u, self.dims)

    def gather(self):
        M.mla_gather_latent(self.cache, self.block_table, 0, self.rows, self.dims, self.dev_status)

    def expand(self):
        M.mla_expand_kv(self.rows, self.w_uk, self.w_uv, self.k_nope, self.v, self.dims)

    def prefill(self):
        M.mla_prefill_attn(self.q, self.k_nope, self.rows, self.v, self.o_pf, self.lse_pf,
                           self.wl.scale, self.dims, self.dev_status)

    def project_absorbed(self):
        M.mla_project_q_absorbed(self.x_q, self.w_dq, self.w_fused_q, self.q_pos, self.rope,
                                 self.c_q, self.q_cat, self.dims, self.dev_status)

    def out_absorbed(self):
        M.mla_out_proj_absorbed(self.o_lat, self.o_lat_lowp, self.w_fused_o, self.u, self.dims)

    def stages(self):
        if self.wl.mode == "prefill_mha":
            return [self.append, self.project, self.gather, self.expand, self.prefill]
        if self.fp8_staged:  # plan and merge inside the call
            return [self.absorb_q, self.attend_fp8_staged, self.absorb_out]
        if self.wl.fused:
            return [self.append, self.project_absorbed, self.plan, self.attend, self.combine,
                    self.out_absorbed]
        s = []
        if self.wl.mode in ("layer", "prefill"):
            s += [self.append, self.project]
        s += [self.absorb_q, self.plan, self.attend]
        if self.fuse_out:
            s.append(self.combine_absorb_out)
        else:
            s += [self.combine, self.absorb_out]
        if self.wl.mode == "layer":
            s.append(self.out_proj)
        return s

    def run(self):
        """One step. The split plan depends only on the lengths, so it runs on
        a side stream next to the stages before attention (both streams
        join before the decode kernel; this also captures into a graph)."""
        if self.wl.mode == "prefill_mha" or self.fp8_staged:
            for f in self.stages():
                f()
            return
        main = torch.cuda.current_stream(self.q_cat.device)
        if self._side is None:
            self._side = torch.cuda.Stream(device=self.q_cat.device)
        self._side.wait_stream(main)
        with torch.cuda.stream(self._side):
            self.plan()
        for f in self.stages():
            if f.__name__ == "plan":
                main.wait_stream(self._side)
            else:
                f()

    def result(self) -> torch.Tensor:
        if self.wl.mode == "prefill_mha":
            return self.o_pf
        return self.u if self.wl.mode == "layer" else self.o

    def status(self) -> int:
        return int(self.dev_status.item())
