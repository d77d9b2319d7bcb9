"""Decode context parallelism across GPUs (one rank per GPU).

The history of every sequence is split along the sequence over the N ranks
of a process group; each rank keeps its piece of the paged latent cache.
This follows the vllm-ascend PR #16977 study page: glossary "DCP", and its
third change, in which the HISTORY partials of all ranks go through one
all-to-all that scatters heads (scatter_dim = 1) and every rank then merges
all shards plus the local CURRENT partial exactly once for its H / N heads.

One decode step on rank r:

1. ``mla_dcp_decode_partial_sliced`` over the rank's own history (and the
   CURRENT chunk, which every rank holds alike): partials laid out as
   [N, T, P, H/N, 512], block n being what rank n needs;
2. one all-to-all of equal splits of those partials and their LSEs (NCCL on
   GPUs; any torch.distributed backend with ``all_to_all_single``);
3. ``mla_dcp_combine_exchanged``: the history shards of every rank plus the
   CURRENT partial once (from this rank's own block);
4. ``mla_vup`` with this rank's heads of W_UV.

Only step 2 is torch.distributed (plain copies between GPUs: no multicast,
no remote memory access by any kernel); every step on the data runs in this
library's kernels.  The block-table split below is host-side integer logic.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

from . import api


def history_split(seq_lens: np.ndarray, block_size: int, world: int, rank: int):
    """Token range [start, end) of ``rank``'s piece of each history: block-aligned
    contiguous pieces, piece r = [r*n, min(L, (r+1)*n)), n = bs*ceil(L/(world*bs)).
    Trailing pieces may be empty (the same rule as the shards of one GPU)."""
    L = np.asarray(seq_lens, dtype=np.int64)
    chunk = world * block_size
    n = block_size * ((L + chunk - 1) // chunk)
    start = np.minimum(L, rank * n)
    end = np.minimum(L, (rank + 1) * n)
    return start, end


def local_block_table(block_table: np.ndarray, seq_lens: np.ndarray, block_size: int,
                      world: int, rank: int):
    """Block table and history lengths of ``rank``'s piece: the same physical
    blocks, each row shifted so the piece starts at logical block 0; entries
    past the piece are -1.  (In a deployment each rank's cache holds only its
    own blocks; the ids are then that cache's.)"""
    table = np.asarray(block_table, dtype=np.int32)
    start, end = history_split(seq_lens, block_size, world, rank)
    lens = (end - start).astype(np.int32)
    nb = (lens.astype(np.int64) + block_size - 1) // block_size
    width = max(1, int(nb.max()) if nb.size else 1)
    out = np.full((table.shape[0], width), -1, dtype=np.int32)
    for b in range(table.shape[0]):
        first = int(start[b]) // block_size
        out[b, :nb[b]] = table[b, first:first + nb[b]]
    return out, lens


def exchange_partials(o_send: torch.Tensor, lse_send: torch.Tensor, group=None):
    """The all-to-all of DCP: block n (dimension 0) of the sliced partials goes
    to rank n; returns, in the same shapes, the blocks every rank sent here
    (block src = rank src's partials for this rank's heads)."""
    world = dist.get_world_size(group)
    if o_send.shape[0] != world or lse_send.shape[0] != world:
        raise ValueError("dimension 0 of the partials must equal the group size")
    o_recv = torch.empty_like(o_send)
    lse_recv = torch.empty_like(lse_send)
    dist.all_to_all_single(o_recv, o_send.contiguous(), group=group)
    dist.all_to_all_single(lse_recv, lse_send.contiguous(), group=group)
    return o_recv, lse_recv


def dcp_decode_step(q_abs, q_pe, kv_cache, block_table, seq_lens, W_UV, num_shards: int, *,
                    kv_cur=None, group=None, scale: float = api.DEFAULT_SCALE, part_dtype=None,
                    err_flag=None, stream=None, workspace="default", kv_scale=None):
    """One decode step of MLA with the history split over the ranks of ``group``.

    Every rank passes the same q_abs [B, q, H, 512], q_pe, kv_cur and W_UV,
    and its own piece of the history: kv_cache, block_table and seq_lens of
    that piece (``local_block_table`` builds them from a whole table), split
    into ``num_shards`` shards on this GPU.  H must be a multiple of the group
    size N.  An E4M3 cache (uint8 / float8_e4m3fn bytes, with ``kv_scale``)
    takes the FP8 partial kernel, as in ``api.mla_dcp_decode_partial``.  Returns this rank's heads [r*H/N, (r+1)*H/N): the output
    [B*q, (H/N)*128], the combined latent [B*q, H/N, 512] and its LSE
    [B*q, H/N]."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    H = q_abs.shape[2]
    if H % world != 0:
        raise ValueError(f"{H} heads cannot be split over {world} ranks")
    hs = H // world
    o_send, lse_send = api.mla_dcp_decode_partial(
        q_abs, q_pe, kv_cache, block_table, seq_lens, num_shards, kv_cur=kv_cur, scale=scale,
        part_dtype=part_dtype, err_flag=err_flag, stream=stream, workspace=workspace,
        head_slices=world, kv_scale=kv_scale)
    if world == 1:
        o_send = o_send.view(1, -1, *o_send.shape[2:])
        lse_send = lse_send.view(1, -1, *lse_send.shape[2:])
    o_recv, lse_recv = exchange_partials(o_send, lse_send, group)
    o_lat, lse = api.mla_dcp_combine_exchanged(
        o_recv, lse_recv, hist_parts=num_shards, local_src=rank if kv_cur is not None else -1,
        out_dtype=W_UV.dtype, stream=stream)
    out = api.mla_vup(o_lat, W_UV[rank * hs:(rank + 1) * hs].contiguous(), err_flag=err_flag,
                      stream=stream)
    return out, o_lat, lse


def partials_per_rank(num_shards: int, has_current: bool) -> int:
    """Parts per rank in the exchange: the rank's history shards (+ CURRENT)."""
    return num_shards + (1 if has_current else 0)


def exchange_bytes(T: int, H: int, world: int, num_shards: int, has_current: bool,
                   part_bytes: int = 2) -> int:
    """Bytes one rank sends per step (the pages count 512*2 + 4 per head row)."""
    P = partials_per_rank(num_shards, has_current)
    return T * P * H * (512 * part_bytes + 4) * (world - 1) // world if world > 1 else 0


__all__ = ["history_split", "local_block_table", "exchange_partials", "dcp_decode_step",
           "partials_per_rank", "exchange_bytes"]
