"""Python binding of the C ABI (include/mla_dcp.h) for torch CUDA tensors.

Argument marshalling only: every call checks shapes, allocates outputs the
caller did not pass (torch owns device memory), and hands raw pointers to the
CUDA library on the current (or given) stream.  No arithmetic of the method
happens here and there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional

import torch

from . import _ffi

D_LATENT, D_ROPE, D_QK, D_V = 512, 64, 576, 128
DEFAULT_SCALE = 1.0 / math.sqrt(128 + D_ROPE)

_TORCH_DT = {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float32: "fp32"}
_DT_TORCH = {v: k for k, v in _TORCH_DT.items()}


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _code(dtype: torch.dtype) -> int:
    try:
        return _ffi.DTYPE[_TORCH_DT[dtype]]
    except KeyError:
        raise TypeError(f"unsupported dtype {dtype}") from None


def _need(t: torch.Tensor, name: str):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


_WORKSPACES = {}


def partial_workspace(device, B: int, q_len: int, num_shards: int, has_current: bool,
                      stream=None):
    """The default workspace of mla_dcp_decode_partial on `device` for calls on
    `stream` (one per (device, stream), grown as needed), or None for sizes
    the library rejects.  Calls on one stream run one after another, so they
    can share it; calls on different streams get different workspaces.  Two
    calls that may overlap in time on the same stream handle (graphs replayed
    concurrently, say) must pass workspaces of their own."""
    device = torch.device(device)
    with torch.cuda.device(device):
        need = int(_ffi.lib().mla_dcp_decode_partial_workspace_size(
            B, q_len, num_shards, 1 if has_current else 0))
        s = stream if stream is not None else torch.cuda.current_stream()
    if need == 0:
        return None      # invalid sizes: the call itself reports them
    key = (device.index, s.cuda_stream)
    ws = _WORKSPACES.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.empty(need, dtype=torch.uint8, device=device)
        _WORKSPACES[key] = ws
    return ws


def is_fp8_cache(kv_cache) -> bool:
    """An E4M3 cache: uint8 bytes or torch.float8_e4m3fn."""
    return kv_cache.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8))


def mla_dcp_decode_partial(q_abs, q_pe, kv_cache, block_table, seq_lens, num_shards: int, *,
                           kv_cur=None, scale: float = DEFAULT_SCALE, part_dtype=None,
                           o_part=None, lse_part=None, err_flag=None, stream=None,
                           workspace="default", head_slices: int = 1, kv_scale=None):
    """Partial attention of every (sequence, query token, shard [, CURRENT]).

    q_abs [B, q, H, 512], q_pe [B, q, H, 64], kv_cache [num_blocks, bs, 576],
    block_table [B, max_blocks] int32, seq_lens [B] int32 (history lengths),
    kv_cur [B, q, 576] or None.  A kv_cache of E4M3 bytes (torch.uint8 or
    torch.float8_e4m3fn; kv_cur likewise) goes to mla_dcp_decode_partial_fp8
    with kv_scale (default 1.0).  Returns o_part [B, q, P, H, 512] and
    lse_part [B, q, P, H] (float32), P = num_shards + (kv_cur is not None);
    with head_slices = N > 1 they are [N, B*q, P, H/N, 512] and
    [N, B*q, P, H/N] (mla_dcp_decode_partial_sliced: block n is what rank n
    receives in a head-scattered all-to-all).
    workspace: "default" (one kept per device and stream, see
    partial_workspace), a uint8 CUDA tensor of at least
    mla_dcp_decode_partial_workspace_size bytes, or None (pairs of CTAs then
    take whole shards)."""
    B, q_len, H, _ = q_abs.shape
    num_blocks, bs, _ = kv_cache.shape
    P = num_shards + (1 if kv_cur is not None else 0)
    part_dtype = part_dtype or q_abs.dtype
    for t, n in ((q_abs, "q_abs"), (q_pe, "q_pe"), (kv_cache, "kv_cache"),
                 (block_table, "block_table"), (seq_lens, "seq_lens")):
        _need(t, n)
    if head_slices == 1:
        o_shape, l_shape = (B, q_len, P, H, D_LATENT), (B, q_len, P, H)
    else:
        hs = H // head_slices
        o_shape = (head_slices, B * q_len, P, hs, D_LATENT)
        l_shape = (head_slices, B * q_len, P, hs)
    if o_part is None:
        o_part = torch.empty(o_shape, dtype=part_dtype, device=q_abs.device)
    if lse_part is None:
        lse_part = torch.empty(l_shape, dtype=torch.float32, device=q_abs.device)
    if isinstance(workspace, str):
        if workspace != "default":
            raise ValueError("workspace must be 'default', a tensor or None")
        workspace = partial_workspace(q_abs.device, B, q_len, num_shards, kv_cur is not None,
                                      stream)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if is_fp8_cache(kv_cache):
        if kv_cur is not None and not is_fp8_cache(kv_cur):
            raise TypeError("kv_cur must be E4M3 bytes like kv_cache")
        st = _ffi.lib().mla_dcp_decode_partial_fp8(
            _p(q_abs), _p(q_pe), _p(kv_cache), _p(block_table), _p(seq_lens), _p(kv_cur),
            B, q_len, H, num_blocks, bs, block_table.shape[1], num_shards, float(scale),
            float(1.0 if kv_scale is None else kv_scale), _code(q_abs.dtype),
            _code(o_part.dtype), _p(o_part), _p(lse_part), _p(err_flag), _p(workspace), ws_bytes,
            int(head_slices), _s(stream))
        _ffi.check("mla_dcp_decode_partial_fp8", st)
        return o_part, lse_part
    if kv_scale is not None:
        raise TypeError("kv_scale applies to an E4M3 cache only")
    st = _ffi.lib().mla_dcp_decode_partial_sliced(
        _p(q_abs), _p(q_pe), _p(kv_cache), _p(block_table), _p(seq_lens), _p(kv_cur),
        B, q_len, H, num_blocks, bs, block_table.shape[1], num_shards, float(scale),
        _code(q_abs.dtype), _code(o_part.dtype), _p(o_part), _p(lse_part), _p(err_flag),
        _p(workspace), ws_bytes, int(head_slices), _s(stream))
    _ffi.check("mla_dcp_decode_partial_sliced", st)
    return o_part, lse_part


def mla_dcp_combine_exchanged(o_recv, lse_recv, *, hist_parts: int, local_src: int = -1,
                              out_dtype=None, o_latent=None, lse_out=None, stream=None):
    """Combine on one GPU after the head-scattered exchange: o_recv
    [N, T, P, Hs, 512] and lse_recv [N, T, P, Hs] as delivered by the
    all-to-all; parts p < hist_parts of every source plus (if local_src >= 0)
    part hist_parts of source local_src.  Returns o_latent [T, Hs, 512] and
    lse [T, Hs]."""
    N, T, P, Hs, _ = o_recv.shape
    _need(o_recv, "o_recv")
    _need(lse_recv, "lse_recv")
    out_dtype = out_dtype or o_recv.dtype
    if o_latent is None:
        o_latent = torch.empty((T, Hs, D_LATENT), dtype=out_dtype, device=o_recv.device)
    if lse_out is None:
        lse_out = torch.empty((T, Hs), dtype=torch.float32, device=o_recv.device)
    st = _ffi.lib().mla_dcp_combine_exchanged(
        _p(o_recv), _p(lse_recv), N, P, int(hist_parts), int(local_src), T, Hs,
        _code(o_recv.dtype), _code(o_latent.dtype), _p(o_latent), _p(lse_out), _s(stream))
    _ffi.check("mla_dcp_combine_exchanged", st)
    return o_latent, lse_out


def mla_dcp_decode_partial_noalloc(q_abs, q_pe, kv_cache, block_table, seq_lens,
                                   num_shards: int, *, o_part, lse_part, kv_cur=None,
                                   scale: float = DEFAULT_SCALE, err_flag=None, stream=None):
    """mla_dcp_decode_partial with the library's fixed scratch array instead of
    a workspace: allocates nothing (o_part / lse_part are required), for
    callers that cannot lend the library device memory.  Calls that may
    overlap in time share that array and must be serialised."""
    B, q_len, H, _ = q_abs.shape
    num_blocks, bs, _ = kv_cache.shape
    for t, n in ((q_abs, "q_abs"), (q_pe, "q_pe"), (kv_cache, "kv_cache"),
                 (block_table, "block_table"), (seq_lens, "seq_lens"), (o_part, "o_part"),
                 (lse_part, "lse_part")):
        _need(t, n)
    st = _ffi.lib().mla_dcp_decode_partial_noalloc(
        _p(q_abs), _p(q_pe), _p(kv_cache), _p(block_table), _p(seq_lens), _p(kv_cur),
        B, q_len, H, num_blocks, bs, block_table.shape[1], num_shards, float(scale),
        _code(q_abs.dtype), _code(o_part.dtype), _p(o_part), _p(lse_part), _p(err_flag),
        _s(stream))
    _ffi.check("mla_dcp_decode_partial_noalloc", st)
    return o_part, lse_part


def _rows(o_part, lse_part):
    """View [..., P, H, 512] partials as T rows."""
    P, H = o_part.shape[-3], o_part.shape[-2]
    T = o_part.numel() // (P * H * D_LATENT)
    return T, P, H


def mla_lse_combine(o_part, lse_part, *, o_local=None, lse_local=None, out_dtype=None,
                    o_latent=None, lse_out=None, stream=None):
    """LSE-weighted merge of partials [..., P, H, 512] (+ optional local
    [..., H, 512]) -> o_latent [T, H, 512], lse [T, H]."""
    T, P, H = _rows(o_part, lse_part)
    _need(o_part, "o_part")
    _need(lse_part, "lse_part")
    out_dtype = out_dtype or o_part.dtype
    if o_latent is None:
        o_latent = torch.empty((T, H, D_LATENT), dtype=out_dtype, device=o_part.device)
    if lse_out is None:
        lse_out = torch.empty((T, H), dtype=torch.float32, device=o_part.device)
    st = _ffi.lib().mla_lse_combine(
        _p(o_part), _p(lse_part), P, _p(o_local), _p(lse_local), T, H, _code(o_part.dtype),
        _code(o_latent.dtype), _p(o_latent), _p(lse_out), _s(stream))
    _ffi.check("mla_lse_combine", st)
    return o_latent, lse_out


def mla_vup(o_latent, W_UV, *, out=None, err_flag=None, stream=None):
    """out [T, H*128] = per-head o_latent[:, h, :] @ W_UV[h]."""
    H = W_UV.shape[0]
    T = o_latent.numel() // (H * D_LATENT)
    _need(o_latent, "o_latent")
    _need(W_UV, "W_UV")
    if out is None:
        out = torch.empty((T, H * D_V), dtype=W_UV.dtype, device=W_UV.device)
    st = _ffi.lib().mla_vup(_p(o_latent), _p(W_UV), T, H, _code(W_UV.dtype), _p(out),
                            _p(err_flag), _s(stream))
    _ffi.check("mla_vup", st)
    return out


def mla_lse_combine_vup(o_part, lse_part, W_UV, *, o_local=None, lse_local=None, out=None,
                        o_latent=None, lse_out=None, err_flag=None, stream=None):
    """Combine + V-up in one launch -> out [T, H*128] (and optionally the
    combined latent / LSE if o_latent / lse_out are given)."""
    T, P, H = _rows(o_part, lse_part)
    _need(o_part, "o_part")
    _need(W_UV, "W_UV")
    if out is None:
        out = torch.empty((T, H * D_V), dtype=W_UV.dtype, device=W_UV.device)
    st = _ffi.lib().mla_lse_combine_vup(
        _p(o_part), _p(lse_part), P, _p(o_local), _p(lse_local), _p(W_UV), T, H,
        _code(o_part.dtype), _code(W_UV.dtype), _p(out), _p(o_latent), _p(lse_out),
        _p(err_flag), _s(stream))
    _ffi.check("mla_lse_combine_vup", st)
    return out


def mla_gather_kv(kv_cache, block_table, seq_lens, max_len: int, *, dst=None, err_flag=None,
                  stream=None):
    """dst [B, max_len, 576]: each sequence's paged history, bit-exact."""
    B = block_table.shape[0]
    num_blocks, bs, _ = kv_cache.shape
    if dst is None:
        dst = torch.empty((B, max_len, D_QK), dtype=kv_cache.dtype, device=kv_cache.device)
    st = _ffi.lib().mla_gather_kv(_p(kv_cache), _p(block_table), _p(seq_lens), B, num_blocks, bs,
                                  block_table.shape[1], max_len, _p(dst), _p(err_flag),
                                  _s(stream))
    _ffi.check("mla_gather_kv", st)
    return dst


def decode_step(q_abs, q_pe, kv_cache, block_table, seq_lens, W_UV, num_shards: int, *,
                kv_cur=None, scale: float = DEFAULT_SCALE, part_dtype=None, o_part=None,
                lse_part=None, out=None, err_flag=None, stream=None, workspace="default",
                kv_scale=None):
    """One decode step of the attention layer: partials, then the fused
    combine + V-up.  Returns out [B*q, H*128]."""
    o_part, lse_part = mla_dcp_decode_partial(
        q_abs, q_pe, kv_cache, block_table, seq_lens, num_shards, kv_cur=kv_cur, scale=scale,
        part_dtype=part_dtype, o_part=o_part, lse_part=lse_part, err_flag=err_flag,
        stream=stream, workspace=workspace, kv_scale=kv_scale)
    return mla_lse_combine_vup(o_part, lse_part, W_UV, out=out, err_flag=err_flag, stream=stream)


def torch_dtype(name: str) -> torch.dtype:
    return _DT_TORCH[name]
