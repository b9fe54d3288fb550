"""Thin Python binding of ``libmla_b300.so`` (the C ABI in include/mla_b300.h).

Argument marshalling only: every function takes torch tensors that already
live on the GPU, checks their dtype/shape/contiguity against the C ABI,
passes raw device pointers and the current CUDA stream, and raises
:class:`MlaError` on a non-OK status. All arithmetic runs in the library's
kernels. If the library is missing this module raises -- there is no
fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE, MLA_ERR_CUDA = range(5)
MLA_F32, MLA_BF16, MLA_FP8_E4M3 = 0, 1, 2
MLA_DEV_BAD_BLOCK, MLA_DEV_BAD_POS, MLA_DEV_BAD_LEN, MLA_DEV_TIMEOUT = 1, 2, 4, 8

LIB_PATH = _build.LIB


class MlaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("n_h", "d_h", "d_r", "d_c", "d_v", "d_model", "d_cq", "page_size")]

    @classmethod
    def of(cls, wl) -> "Dims":
        """Dims of a :class:`synth.Workload` (or anything with those fields)."""
        return cls(wl.n_h, wl.d_h, wl.d_r, wl.d_c, wl.d_v, wl.d_model, wl.d_cq, wl.page_size)


_lib = None
_P, _I, _S, _F, _D = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float, ctypes.c_double
_DIMS = ctypes.POINTER(Dims)
_SIGS = {
    "mla_status_string": (ctypes.c_char_p, [_I]),
    "mla_last_error": (ctypes.c_char_p, []),
    "mla_abi_version": (_I, []),
    "mla_force_decode_path": (None, [_I]),
    "mla_decode_path": (_I, [_I, _DIMS]),
    "mla_rope_table": (_I, [_P, _I, _I, _D, _P]),
    "mla_append_latent": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _I, _P, _I, _DIMS, _P, _P]),
    "mla_project_q": (_I, [_P, _P, _P, _P, _I, _P, _I, _P, _P, _I, _DIMS, _P, _P]),
    "mla_absorb_q": (_I, [_P, _P, _P, _I, _I, _DIMS, _P]),
    "mla_decode_workspace_size": (_S, [_I, _I, _DIMS]),
    "mla_plan_decode": (_I, [_P, _I, _I, _P, _S, _I, _DIMS, _P, _P]),
    "mla_decode_attn": (_I, [_P, _P, _P, _I, _I, _P, _I, _F, _P, _S, _P, _P, _I, _DIMS, _P, _P]),
    "mla_plan_decode_mtp": (_I, [_P, _I, _I, _I, _P, _S, _I, _DIMS, _P, _P]),
    "mla_decode_attn_mtp": (_I, [_P, _P, _P, _I, _I, _P, _I, _I, _F, _P, _S, _P, _P, _I, _DIMS, _P,
                                 _P]),
    "mla_combine": (_I, [_P, _S, _I, _P, _P, _I, _DIMS, _P]),
    "mla_decode_attn_static": (_I, [_P, _P, _P, _I, _I, _P, _I, _F, _P, _P, _I, _DIMS, _P, _P]),
    "mla_decode_fp8_staged_workspace_size": (_S, [_I, _I, _DIMS]),
    "mla_decode_attn_fp8_staged": (_I, [_P, _P, _P, _I, _I, _P, _I, _F, _P, _S, _P, _P, _DIMS, _P,
                                        _P]),
    "mla_absorb_out": (_I, [_P, _P, _P, _I, _I, _I, _DIMS, _P]),
    "mla_combine_absorb_out": (_I, [_P, _S, _I, _P, _P, _P, _P, _I, _I, _DIMS, _P, _P]),
    "mla_tc_selftest": (_I, [_P, _P, _P, _P, _P, _I, _P, _P]),
    "mla_out_proj": (_I, [_P, _P, _P, _I, _I, _DIMS, _P]),
    "mla_fuse_query_weights": (_I, [_P, _P, _P, _I, _DIMS, _P]),
    "mla_gather_latent": (_I, [_P, _P, _I, _I, _I, _I, _P, _I, _DIMS, _P, _P]),
    "mla_expand_kv": (_I, [_P, _P, _P, _P, _P, _I, _I, _DIMS, _P]),
    "mla_prefill_attn": (_I, [_P, _P, _P, _P, _P, _P, _I, _F, _I, _DIMS, _P, _P]),
    "mla_project_q_absorbed": (_I, [_P, _P, _P, _P, _I, _P, _I, _P, _P, _I, _DIMS, _P, _P]),
    "mla_fuse_output_weights": (_I, [_P, _P, _P, _I, _DIMS, _P]),
    "mla_out_proj_absorbed": (_I, [_P, _P, _P, _P, _I, _I, _DIMS, _P]),
}


def lib() -> ctypes.CDLL:
    """Load the library once (torch first, so one CUDA runtime is shared)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MlaError(MLA_ERR_UNSUPPORTED,
                           f"{LIB_PATH} is missing: run `python -m mla_latent_kv_67_b300.build`")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(l, name)
            f.restype, f.argtypes = res, args
        _lib = l
    return _lib


def _check(st: int) -> None:
    if st != MLA_OK:
        raise MlaError(st, lib().mla_last_error().decode())


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MLA_F32
    if t.dtype == torch.bfloat16:
        return MLA_BF16
    if t.dtype == torch.uint8:  # the FP8 latent cache (row format of the header)
        return MLA_FP8_E4M3
    raise MlaError(MLA_ERR_INVALID_ARG, f"unsupported dtype {t.dtype}")


def _ptr(t: torch.Tensor | None, dtype=None, shape=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise MlaError(MLA_ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise MlaError(MLA_ERR_INVALID_ARG, f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise MlaError(MLA_ERR_INVALID_ARG, f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise MlaError(MLA_ERR_INVALID_ARG, f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def torch_dtype(dtype: int):
    """Element type of the queries, weights and activations for `dtype` (the
    FP8 cache comes with bf16 everything else)."""
    return torch.float32 if dtype == MLA_F32 else torch.bfloat16


def fp8_row_bytes(d_c: int, d_r: int) -> int:
    """MLA_FP8_ROW_BYTES of the header."""
    return (d_c + 2 * d_r + 4 + 15) // 16 * 16


def _cache_shape(cache, dims: Dims):
    w = fp8_row_bytes(dims.d_c, dims.d_r) if cache.dtype == torch.uint8 else dims.d_c + dims.d_r
    return (cache.shape[0], dims.page_size, w)


def _q_dtype(cache):
    return torch.bfloat16 if cache.dtype == torch.uint8 else cache.dtype


# ------------------------------------------------------------- entry points
def mla_abi_version() -> int:
    return lib().mla_abi_version()


def mla_force_decode_path(path: int) -> None:
    lib().mla_force_decode_path(path)


def mla_decode_path(dtype: int, dims: Dims) -> int:
    return lib().mla_decode_path(dtype, ctypes.byref(dims))


def mla_tc_selftest(q_cat, page, pmat, s_out, o_out, half: int, dev_status=None,
                    stream=None) -> None:
    """One page through the tensor-core decode data path (diagnostic)."""
    bf = torch.bfloat16
    _check(lib().mla_tc_selftest(
        _ptr(q_cat, bf, (128, 576), "q_cat"), _ptr(page, bf, (64, 576), "page"),
        _ptr(pmat, bf, (128, 64), "pmat"), _ptr(s_out, torch.float32, (128, 64), "s_out"),
        _ptr(o_out, torch.float32, (128, 256), "o_out"), half,
        _ptr(dev_status, torch.int32, name="dev_status"), _stream(stream)))


def mla_rope_table(cos_sin: torch.Tensor, base: float = 10000.0, stream=None) -> None:
    max_pos, half, two = cos_sin.shape
    assert two == 2
    _check(lib().mla_rope_table(_ptr(cos_sin, torch.float32, name="cos_sin"), max_pos, 2 * half,
                                base, _stream(stream)))


def mla_append_latent(x, w_dkv_kr, seq_idx, pos, block_table, rope, cache, dims: Dims,
                      dev_status=None, stream=None) -> None:
    dt = _dt(cache)
    T = x.shape[0]
    B, max_pages = block_table.shape
    _check(lib().mla_append_latent(
        _ptr(x, cache.dtype, (T, dims.d_model), "x"),
        _ptr(w_dkv_kr, cache.dtype, (dims.d_c + dims.d_r, dims.d_model), "w_dkv_kr"),
        _ptr(seq_idx, torch.int32, (T,), "seq_idx"), _ptr(pos, torch.int32, (T,), "pos"),
        _ptr(block_table, torch.int32, name="block_table"), B, max_pages, cache.shape[0], T,
        _ptr(rope, torch.float32, name="rope"), rope.shape[0] if rope is not None else 0,
        _ptr(cache, shape=(cache.shape[0], dims.page_size, dims.d_c + dims.d_r), name="cache"),
        dt, ctypes.byref(dims), _ptr(dev_status, torch.int32, name="dev_status"), _stream(stream)))


def mla_project_q(x, w_dq, w_uq_qr, pos, rope, c_q, q, dims: Dims, dev_status=None,
                  stream=None) -> None:
    dt = _dt(q)
    T = x.shape[0]
    K = dims.d_cq or dims.d_model
    _check(lib().mla_project_q(
        _ptr(x, q.dtype, (T, dims.d_model), "x"),
        _ptr(w_dq, q.dtype, (dims.d_cq, dims.d_model), "w_dq") if dims.d_cq else None,
        _ptr(w_uq_qr, q.dtype, (dims.n_h * (dims.d_h + dims.d_r), K), "w_uq_qr"),
        _ptr(pos, torch.int32, (T,), "pos"), T,
        _ptr(rope, torch.float32, name="rope"), rope.shape[0] if rope is not None else 0,
        _ptr(c_q, q.dtype, (T, dims.d_cq), "c_q") if dims.d_cq else None,
        _ptr(q, shape=(T, dims.n_h, dims.d_h + dims.d_r), name="q"), dt, ctypes.byref(dims),
        _ptr(dev_status, torch.int32, name="dev_status"), _stream(stream)))


def mla_absorb_q(q, w_uk, q_cat, dims: Dims, stream=None) -> None:
    B = q.shape[0]
    dt = _dt(q_cat)
    _check(lib().mla_absorb_q(
        _ptr(q, q_cat.dtype, (B, dims.n_h, dims.d_h + dims.d_r), "q"),
        _ptr(w_uk, q_cat.dtype, (dims.n_h * dims.d_h, dims.d_c), "w_uk"),
        _ptr(q_cat, shape=(B, dims.n_h, dims.d_c + dims.d_r), name="q_cat"), B, dt,
        ctypes.byref(dims), _stream(stream)))


def mla_decode_workspace_size(B: int, dtype: int, dims: Dims) -> int:
    return int(lib().mla_decode_workspace_size(B, dtype, ctypes.byref(dims)))


def mla_plan_decode(seq_lens, max_pages: int, workspace, dtype: int, dims: Dims,
                    dev_status=None, stream=None) -> None:
    B = seq_lens.shape[0]
    _check(lib().mla_plan_decode(
        _ptr(seq_lens, torch.int32, (B,), "seq_lens"), B, max_pages,
        _ptr(workspace, torch.uint8, name="workspace"), workspace.numel(), dtype,
        ctypes.byref(dims), _ptr(dev_status, torch.int32, name="dev_status"), _stream(stream)))


def mla_decode_attn(q_cat, cache, block_table, seq_lens, scale: float, workspace, o_lat, lse,
                    dims: Dims, dev_status=None, stream=None) -> None:
    B, max_pages = block_table.shape
    dt = _dt(cache)
    _check(lib().mla_decode_attn(
        _ptr(q_cat, _q_dtype(cache), (B, dims.n_h, dims.d_c + dims.d_r), "q_cat"),
        _ptr(cache, shape=_cache_shape(cache, dims), name="cache"),
        _ptr(block_table, torch.int32, name="block_table"), max_pages, cache.shape[0],
        _ptr(seq_lens, torch.int32, (B,), "seq_lens"), B, scale,
        _ptr(workspace, torch.uint8, name="workspace"), workspace.numel(),
        _ptr(o_lat, torch.float32, (B, dims.n_h, dims.d_c), "o_lat"),
        _ptr(lse, torch.float32, (B, dims.n_h), "lse"), dt, ctypes.byref(dims),
        _ptr(dev_status, torch.int32, name="dev_status"), _stream(stream)))


def mla_plan_decode_mtp(seq_lens, q_len: int, max_pages: int, workspace, dtype: int, dims: Dims,
                        dev_status=None, stream=None) -> None:
    """Plan for q_len new tokens per sequence (query rows B * q_len)."""
    B = seq_lens.shape[0]
    _check(lib().mla_plan_decode_mtp(
        _ptr(seq_lens, torch.int32, (B,), "seq_lens"), B, q_len, max_pages,
        _ptr(workspace, torch.uint8, name="workspace"), workspace.numel(), dtype,
        ctypes.byref(dims), _ptr(dev_status, torch.int32, name="dev_status"), _stream(stream)))


def mla_decode_attn_mtp(q_cat, cache, block_table, seq_lens, q_len: int, scale: float, workspace,
                        o_lat, lse, dims: Dims, dev_status=None, stream=None) -> None:
    """Decode q_len new tokens per sequence; q_cat [B * q_len, n_h, d_c + d_r]."""
    B, max_pages = block_table.shape
    dt = _dt(cache)
    R = B * q_len
    _check(lib().mla_decode_attn_mtp(
        _ptr(q_cat, _q_dtype(cache), (R, dims.n_h, dims.d_c + dims.d_r), "q_cat"),
        _ptr(cache, shape=_cache_shape(cache, dims), name="cache"),
        _ptr(block_table, torch.int32, name="block_table"), max_pages, cache.shape[0],
        _ptr(seq_lens, torch.int32, (B,), "seq_lens"), B, q_len, scale,
        _ptr(workspace, torch.uint8, name="workspace"), workspace.numel(),
        _ptr(o_lat, torch.float32, (R, dims.n_h, dims.d_c), "o_lat"),
        _ptr(lse, torch.float32, (R, dims.n_h), "lse"), dt, ctypes.byref(dims),
        _ptr(dev_status, torch.int32, name="dev_status"), _stream(stream)))


def mla_combine(workspace, o_lat, lse, dtype: int, dims: Dims, stream=None) -> None:
    B = o_lat.shape[0]
    _check(lib().mla_combine(
        _ptr(workspace, torch.uint8, name="workspace"), workspace.numel(), B,
        _ptr(o_lat, torch.float32, (B, dims.n_h, dims.d_c), "o_lat"),
        _ptr(lse, torch.float32, (B, dims.n_h), "lse"), dtype, ctypes.byref(dims), _stream(stream)))


def mla_absorb_out(o_lat, w_uv, o, dims: Dims, stream=None) -> None:
    B = o_lat.shape[0]
    _check(lib().mla_absorb_out(
        _ptr(o_lat, torch.float32, (B, dims.n_h, dims.d_c), "o_lat"),
        _ptr(w_uv, shape=(dims.n_h * dims.d_v, dims.d_c), name="w_uv"),
        _ptr(o, shape=(B, dims.n_h * dims.d_v), name="o"), B, _dt(w_uv), _dt(o),
        ctypes.byref(dims), _stream(stream)))


def mla_combine_absorb_out(workspace, o_lat, lse, w_uv, o, dims: Dims, dev_status=None,
                           stream=None) -> None:
    B = o_lat.shape[0]
    _check(lib().mla_combine_absorb_out(
        _ptr(workspace, torch.uint8, name="workspace"), workspace.numel(), B,
        _ptr(o_lat, torch.float32, (B, dims.n_h, dims.d_c), "o_lat"),
        _ptr(lse, torch.float32, (B, dims.n_h), "lse"),
        _ptr(w_uv, shape=(dims.n_h * dims.d_v, dims.d_c), name="w_uv"),
        _ptr(o, shape=(B, dims.n_h * dims.d_v), name="o"), _dt(w_uv), _dt(o),
        ctypes.byref(dims), _ptr(dev_status, torch.int32, name="dev_status"), _stream(stream)))


def mla_out_proj(o, w_o, u, dims: Dims, stream=None) -> None:
    B = o.shape[0]
    _check(lib().mla_out_proj(
        _ptr(o, w_o.dtype, (B, dims.n_h * dims.d_v), "o"),
        _ptr(w_o, shape=(dims.d_model, dims.n_h * dims.d_v), name="w_o"),
        _ptr(u, torch.float32, (B, dims.d_model), "u"), B, _dt(w_o), ctypes.byref(dims),
        _stream(stream)))


def mla_decode_attn_static(q_cat, cache, block_table, seq_lens, scale: float, o_lat, lse,
                           dims: Dims, dev_status=None, stream=None) -> None:
    """Plan, decode and combine with the library's static device scratch, for
    callers that cannot allocate a workspace (see the header)."""
    B, max_pages = block_table.shape
    dt = _dt(cache)
    _check(lib().mla_decode_attn_static(
        _ptr(q_cat, _q_dtype(cache), (B, dims.n_h, dims.d_c + dims.d_r), "q_cat"),
        _ptr(cache, shape=_cache_shape(cache, dims), name="cache"),
        _ptr(block_table, torch.int32, name="block_table"), max_pages, cache.shape[0],
        _ptr(seq_lens, torch.int32, (B,), "seq_lens"), B, scale,
        _ptr(o_lat, torch.float32, (B, dims.n_h, dims.d_c), "o_lat"),
        _ptr(lse, torch.float32, (B, dims.n_h), "lse"), dt, ctypes.byref(dims),
        _ptr(dev_status, torch.int32, name="dev_status"), _stream(stream)))


def mla_decode_fp8_staged_workspace_size(B: int, max_pages: int, dims: Dims) -> int:
    return int(lib().mla_decode_fp8_staged_workspace_size(B, max_pages, ctypes.byref(dims)))


def mla_decode_attn_fp8_staged(q_cat, cache, block_table, seq_lens, scale: float, workspace,
                               o_lat, lse, dims: Dims, dev_status=None, stream=None) -> None:
    """Decode on the FP8 latent cache by widening the batch's pages to bf16
    rows in `workspace` and running the bf16 decode on them (see the header)."""
    B, max_pages = block_table.shape
    if cache.dtype != torch.uint8:
        raise MlaError(MLA_ERR_INVALID_ARG, "cache must be the FP8 row format (uint8)")
    _check(lib().mla_decode_attn_fp8_staged(
        _ptr(q_cat, torch.bfloat16, (B, dims.n_h, dims.d_c + dims.d_r), "q_cat"),
        _ptr(cache, shape=_cache_shape(cache, dims), name="cache"),
        _ptr(block_table, torch.int32, name="block_table"), max_pages, cache.shape[0],
        _ptr(seq_lens, torch.int32, (B,), "seq_lens"), B, scale,
        _ptr(workspace, torch.uint8, name="workspace"), workspace.numel(),
        _ptr(o_lat, torch.float32, (B, dims.n_h, dims.d_c), "o_lat"),
        _ptr(lse, torch.float32, (B, dims.n_h), "lse"), ctypes.byref(dims),
        _ptr(dev_status, torch.int32, name="dev_status"), _stream(stream)))


# ------------------------------------------------------- fused absorption
def mla_fuse_query_weights(w_uq_qr, w_uk, w_fused_q, dims: Dims, stream=None) -> None:
    K = dims.d_cq or dims.d_model
    dt = _dt(w_fused_q)
    _check(lib().mla_fuse_query_weights(
        _ptr(w_uq_qr, w_fused_q.dtype, (dims.n_h * (dims.d_h + dims.d_r), K), "w_uq_qr"),
        _ptr(w_uk, w_fused_q.dtype, (dims.n_h * dims.d_h, dims.d_c), "w_uk"),
        _ptr(w_fused_q, shape=(dims.n_h * (dims.d_c + dims.d_r), K), name="w_fused_q"), dt,
        ctypes.byref(dims), _stream(stream)))


def mla_project_q_absorbed(x, w_dq, w_fused_q, pos, rope, c_q, q_cat, dims: Dims,
                           dev_status=None, stream=None) -> None:
    dt = _dt(q_cat)
    T = x.shape[0]
    K = dims.d_cq or dims.d_model
    _check(lib().mla_project_q_absorbed(
        _ptr(x, q_cat.dtype, (T, dims.d_model), "x"),
        _ptr(w_dq, q_cat.dtype, (dims.d_cq, dims.d_model), "w_dq") if dims.d_cq else None,
        _ptr(w_fused_q, q_cat.dtype, (dims.n_h * (dims.d_c + dims.d_r), K), "w_fused_q"),
        _ptr(pos, torch.int32, (T,), "pos"), T,
        _ptr(rope, torch.float32, name="rope"), rope.shape[0] if rope is not None else 0,
        _ptr(c_q, q_cat.dtype, (T, dims.d_cq), "c_q") if dims.d_cq else None,
        _ptr(q_cat, shape=(T, dims.n_h, dims.d_c + dims.d_r), name="q_cat"), dt,
        ctypes.byref(dims), _ptr(dev_status, torch.int32, name="dev_status"), _stream(stream)))


def mla_fuse_output_weights(w_o, w_uv, w_fused_o, dims: Dims, stream=None) -> None:
    dt = _dt(w_fused_o)
    _check(lib().mla_fuse_output_weights(
        _ptr(w_o, w_fused_o.dtype, (dims.d_model, dims.n_h * dims.d_v), "w_o"),
        _ptr(w_uv, w_fused_o.dtype, (dims.n_h * dims.d_v, dims.d_c), "w_uv"),
        _ptr(w_fused_o, shape=(dims.d_model, dims.n_h * dims.d_c), name="w_fused_o"), dt,
        ctypes.byref(dims), _stream(stream)))


def mla_out_proj_absorbed(o_lat, o_lat_lowp, w_fused_o, u, dims: Dims, stream=None) -> None:
    B = o_lat.shape[0]
    dt = _dt(w_fused_o)
    _check(lib().mla_out_proj_absorbed(
        _ptr(o_lat, torch.float32, (B, dims.n_h, dims.d_c), "o_lat"),
        _ptr(o_lat_lowp, w_fused_o.dtype, (B, dims.n_h * dims.d_c), "o_lat_lowp")
        if dt == MLA_BF16 else None,
        _ptr(w_fused_o, shape=(dims.d_model, dims.n_h * dims.d_c), name="w_fused_o"),
        _ptr(u, torch.float32, (B, dims.d_model), "u"), B, dt, ctypes.byref(dims),
        _stream(stream)))


# ----------------------------------------------------------------- prefill
def mla_gather_latent(cache, block_table, seq: int, rows, dims: Dims, dev_status=None,
                      stream=None) -> None:
    N = rows.shape[0]
    B, max_pages = block_table.shape
    _check(lib().mla_gather_latent(
        _ptr(cache, shape=(cache.shape[0], dims.page_size, dims.d_c + dims.d_r), name="cache"),
        _ptr(block_table, torch.int32, name="block_table"), max_pages, cache.shape[0], seq, N,
        _ptr(rows, cache.dtype, (N, dims.d_c + dims.d_r), "rows"), _dt(cache), ctypes.byref(dims),
        _ptr(dev_status, torch.int32, name="dev_status"), _stream(stream)))


def mla_expand_kv(rows, w_uk, w_uv, k_nope, v, dims: Dims, stream=None) -> None:
    N = rows.shape[0]
    dt = _dt(rows)
    _check(lib().mla_expand_kv(
        _ptr(rows, shape=(N, dims.d_c + dims.d_r), name="rows"),
        _ptr(w_uk, rows.dtype, (dims.n_h * dims.d_h, dims.d_c), "w_uk"),
        _ptr(w_uv, rows.dtype, (dims.n_h * dims.d_v, dims.d_c), "w_uv"),
        _ptr(k_nope, rows.dtype, (N, dims.n_h, dims.d_h), "k_nope"),
        _ptr(v, rows.dtype, (N, dims.n_h, dims.d_v), "v"), N, dt, ctypes.byref(dims),
        _stream(stream)))


def mla_prefill_attn(q, k_nope, rows, v, o, lse, scale: float, dims: Dims, dev_status=None,
                     stream=None) -> None:
    N = q.shape[0]
    dt = _dt(q)
    _check(lib().mla_prefill_attn(
        _ptr(q, shape=(N, dims.n_h, dims.d_h + dims.d_r), name="q"),
        _ptr(k_nope, q.dtype, (N, dims.n_h, dims.d_h), "k_nope"),
        _ptr(rows, q.dtype, (N, dims.d_c + dims.d_r), "rows"),
        _ptr(v, q.dtype, (N, dims.n_h, dims.d_v), "v"),
        _ptr(o, torch.bfloat16, (N, dims.n_h, dims.d_v), "o"),
        _ptr(lse, torch.float32, (N, dims.n_h), "lse"), N, scale, dt, ctypes.byref(dims),
        _ptr(dev_status, torch.int32, name="dev_status"), _stream(stream)))
