"""Decode context parallelism across ranks, on CPU (no GPU): the history of
every sequence split over two gloo ranks, each rank's partials laid out
head-sliced as mla_dcp_decode_partial_sliced writes them, the head-scattered
all-to-all of dcp.exchange_partials, then the combine in the order
mla_dcp_combine_exchanged documents (every rank's history shards, then the
CURRENT partial once).  The fp64 oracle stands in for the GPU kernels; the
result for each rank's heads must equal one softmax over the whole sequence.
"""
import dataclasses
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

from mla_decode_attention_kv_gb300 import dcp, inputs
from oracle import mla_oracle as om

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CFG = inputs.DecodeConfig(name="dcp", batch=3, heads=8, q_len=2, num_shards=2, block_size=16,
                          ragged=(1, 150), current=True, seed=301)


def sliced(o_part, lse_part, N):
    """[B, q, P, H, 512] -> [N, B*q, P, H/N, 512], the layout of the sliced
    partial entry point (block n = heads [n*H/N, (n+1)*H/N))."""
    B, q, P, H, D = o_part.shape
    hs = H // N
    o = o_part.reshape(B * q, P, N, hs, D).transpose(2, 0, 1, 3, 4)
    lse = lse_part.reshape(B * q, P, N, hs).transpose(2, 0, 1, 3)
    return np.ascontiguousarray(o), np.ascontiguousarray(lse)


def local_problem(prob, world, rank):
    table, lens = dcp.local_block_table(prob.block_table, prob.seq_lens, prob.cfg.block_size,
                                        world, rank)
    return dataclasses.replace(prob, block_table=table, seq_lens=lens)


def combine_exchanged(o_recv, lse_recv, hist, local_src):
    """The documented part order: (src 0, p < hist), (src 1, ...), ..., then
    part `hist` of `local_src`; merged by the oracle's LSE combine."""
    N = o_recv.shape[0]
    po = [o_recv[s, :, p] for s in range(N) for p in range(hist)]
    pl = [lse_recv[s, :, p] for s in range(N) for p in range(hist)]
    if local_src >= 0:
        po.append(o_recv[local_src, :, hist])
        pl.append(lse_recv[local_src, :, hist])
    return om.lse_combine(np.stack(po, axis=1), np.stack(pl, axis=1))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        prob = inputs.make_problem(CFG)
        o, lse = om.decode_partials(local_problem(prob, world, rank))
        o_s, l_s = sliced(o, lse, world)
        o_r, l_r = dcp.exchange_partials(torch.from_numpy(o_s), torch.from_numpy(l_s))
        o_c, lse_c = combine_exchanged(o_r.numpy(), l_r.numpy(), CFG.num_shards, rank)
        hs = CFG.heads // world
        ref_o, ref_l, _ = om.decode_reference(prob, heads=range(rank * hs, (rank + 1) * hs),
                                              with_vup=False)
        T = CFG.batch * CFG.q_len
        ref_o = ref_o.reshape(T, hs, 512)
        ref_l = ref_l.reshape(T, hs)
        # what this rank received from each source is that source's block for these heads
        ok_blocks = all(np.array_equal(o_r.numpy()[src], sliced(*om.decode_partials(
            local_problem(prob, world, src)), world)[0][rank]) for src in range(world))
        q.put((rank, float(np.abs(o_c - ref_o).max()), float(np.abs(lse_c - ref_l).max()),
               ok_blocks))
    finally:
        dist.destroy_process_group()


def test_dcp_two_gloo_ranks_equal_one_softmax():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {r: (eo, el, ob) for r, eo, el, ob in (q.get(timeout=240) for _ in procs)}
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        err_o, err_l, ok_blocks = res[r]
        assert ok_blocks, f"rank {r} received the wrong blocks"
        assert err_o < 1e-10 and err_l < 1e-10, (r, err_o, err_l)


@pytest.mark.parametrize("world", [1, 2, 3, 4])
def test_history_split_covers_every_token_once(world):
    """The pieces of the ranks tile [0, L) in order, block-aligned, and each
    rank's local block table reads exactly its piece's tokens."""
    prob = inputs.make_problem(CFG.with_(batch=6, ragged=(1, 300), seed=302))
    bs = CFG.block_size
    for b in range(CFG.batch):
        L = int(prob.seq_lens[b])
        full = om.gather_history(prob.kv_cache, prob.block_table[b], bs, L)
        got = []
        prev_end = 0
        for r in range(world):
            start, end = dcp.history_split(prob.seq_lens, bs, world, r)
            assert start[b] == prev_end and start[b] % bs == 0 or start[b] == L
            prev_end = int(end[b])
            table, lens = dcp.local_block_table(prob.block_table, prob.seq_lens, bs, world, r)
            assert lens[b] == end[b] - start[b]
            got.append(om.gather_history(prob.kv_cache, table[b], bs, int(lens[b])))
        assert prev_end == L
        assert np.array_equal(np.concatenate(got, axis=0), full)


def test_exchange_bytes_of_the_pages_row_format():
    """Per head row the exchange carries 512 values and one fp32 LSE."""
    assert dcp.exchange_bytes(T=4, H=128, world=8, num_shards=2, has_current=True) == \
        4 * 3 * 128 * (1024 + 4) * 7 // 8
    assert dcp.exchange_bytes(T=4, H=128, world=1, num_shards=2, has_current=False) == 0
