"""The E4M3-cache partial kernel (mla_dcp_decode_partial_fp8) versus the fp64
oracle, through the C ABI.

Two comparisons per case:
* against the oracle fed the kernel's two-term query q' (split_query), under
  the 16-bit tolerances: everything but the query rounding must agree as
  closely as the 16-bit path does;
* against the oracle on the exact query, under the documented bound: the
  LSE within LSE_ATOL + D and the outputs within OUT_RTOL * max|ref| +
  (e^(2D) - 1) * max|c|, D = fp8_score_bound (the largest score change the
  query error |q - q'| <= 2^-8 |q| + 2^-17 max|q row| allows).
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

from mla_decode_attention_kv_gb300 import api, inputs
from oracle import mla_oracle as om

from gpu_util import (LSE_ATOL, OUT_RTOL, DeviceProblem, assert_lse_close, assert_out_close, f64,
                      fp8_score_bound, max_latent, split_partials)

pytestmark = pytest.mark.gpu

F8 = dict(kv_dtype="e4m3")
CASES = {
    # several tiles per shard with ragged tails, shuffled pages, CURRENT
    "ragged_bf16_cur": inputs.DecodeConfig(
        name="f1", batch=3, heads=128, q_len=1, num_shards=3, block_size=32, ragged=(1, 400),
        current=True, kv_scale=2.0 ** -8, seed=121, **F8),
    # two query tokens, fp16, a kv_scale that is not a power of two
    "mtp_fp16": inputs.DecodeConfig(
        name="f2", batch=2, heads=128, q_len=2, num_shards=2, block_size=64, history=300,
        current=True, dtype="fp16", part_dtype="fp16", kv_scale=0.0123, seed=122, **F8),
    # few heads (rows past H), fp32 partials, 16-token pages
    "heads16_fp32part": inputs.DecodeConfig(
        name="f3", batch=2, heads=16, q_len=1, num_shards=4, block_size=16, ragged=(20, 200),
        part_dtype="fp32", kv_scale=2.0 ** -6, seed=123, **F8),
    # 256-token pages (two tiles per page), peaked logits
    "bs256_peaked": inputs.DecodeConfig(
        name="f4", batch=2, heads=64, q_len=1, num_shards=2, block_size=256, history=700,
        q_gain=6.0, kv_scale=2.0 ** -8, seed=124, **F8),
    # a long CURRENT chunk (16 query tokens) over a short history
    "current16": inputs.DecodeConfig(
        name="f5", batch=2, heads=128, q_len=16, num_shards=2, block_size=32, history=90,
        current=True, kv_scale=2.0 ** -7, seed=125, **F8),
}


def _check_split(dp, o_part, lse_part):
    ref_o, ref_l = split_partials(dp.prob)
    got_o, got_l = f64(o_part), f64(lse_part)
    assert_lse_close(got_l, ref_l, "lse_part vs q'")
    for s in range(ref_o.shape[2]):
        assert_out_close(got_o[:, :, s], ref_o[:, :, s], f"o_part shard {s} vs q'")


def _check_bound(dp, o_part, lse_part):
    D = fp8_score_bound(dp.prob)
    ref_o, ref_l = om.decode_partials(dp.prob)
    got_o, got_l = f64(o_part), f64(lse_part)
    assert_lse_close(got_l, ref_l, "lse_part", atol=LSE_ATOL + D)
    extra = math.expm1(2 * D) * max_latent(dp.prob)
    for s in range(ref_o.shape[2]):
        ref = ref_o[:, :, s]
        tol = OUT_RTOL + extra / max(np.abs(ref).max(), 1e-30)
        assert_out_close(got_o[:, :, s], ref, f"o_part shard {s}", rtol=tol)
    return D


@pytest.mark.parametrize("name", list(CASES))
def test_fp8_partials_match_oracle(name):
    dp = DeviceProblem(inputs.make_problem(CASES[name]))
    o_part, lse_part = dp.partial()
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    _check_split(dp, o_part, lse_part)
    _check_bound(dp, o_part, lse_part)


@pytest.mark.parametrize("name", ["ragged_bf16_cur", "mtp_fp16"])
def test_fp8_decode_step_matches_oracle(name):
    """Partials, then the fused combine + V-up, against one softmax over the
    decoded cache (documented bound)."""
    dp = DeviceProblem(inputs.make_problem(CASES[name]))
    out = dp.step()
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    _, _, ref = om.decode_reference(dp.prob)
    D = fp8_score_bound(dp.prob)
    W = om.to_f64(dp.prob.W_UV, dp.prob.cfg.dtype)
    # |delta out| <= sum_j |delta o_j| |W_jk| <= (e^(2D) - 1) max|c| * max_h,k sum_j |W_hjk|
    extra = math.expm1(2 * D) * max_latent(dp.prob) * float(np.abs(W).sum(axis=1).max())
    got = f64(out)
    assert_out_close(got, ref, "out", rtol=OUT_RTOL + extra / np.abs(ref).max())


@pytest.mark.parametrize("lens", [[0, 0], [1, 0], [127, 128], [129, 255], [0, 1000]])
def test_fp8_edge_lengths(lens):
    cfg = inputs.DecodeConfig(name="fe", batch=2, heads=128, q_len=1, num_shards=4,
                              block_size=32, history=1, current=True, kv_scale=2.0 ** -8,
                              seed=131, **F8)
    dp = DeviceProblem(inputs.make_problem(cfg, seq_lens=np.array(lens, np.int32)))
    o_part, lse_part = dp.partial()
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    _check_split(dp, o_part, lse_part)


def test_fp8_stale_bytes_past_the_history_are_ignored():
    """Slots of a last page past L_b may hold any finite codes (stale tokens,
    values up to +-448): they get weight 0."""
    cfg = inputs.DecodeConfig(name="fn", batch=3, heads=128, q_len=1, num_shards=2,
                              block_size=64, history=1, kv_scale=2.0 ** -8, seed=132, **F8)
    lens = np.array([70, 129, 5], np.int32)
    prob = inputs.make_problem(cfg, seq_lens=lens)
    for b in range(cfg.batch):
        L = int(lens[b])
        last = prob.block_table[b, (L - 1) // cfg.block_size]
        tail = prob.kv_cache[last, L % cfg.block_size or cfg.block_size:, :]
        tail[:] = np.where(np.arange(tail.size).reshape(tail.shape) % 2, 0x7E, 0xFE)
    dp = DeviceProblem(prob)
    o_part, lse_part = dp.partial()
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    assert torch.isfinite(o_part.float()).all()
    _check_split(dp, o_part, lse_part)


@pytest.mark.parametrize("workspace", ["default", None])
def test_fp8_split_and_whole_shards_agree(workspace):
    """One long shard per sequence: with a workspace the pairs cut it into
    exact tile shares (merge kernel), without one each pair takes whole
    shards; both match the oracle."""
    cfg = inputs.DecodeConfig(name="fs", batch=2, heads=128, q_len=1, num_shards=1,
                              block_size=64, history=9000, current=True, kv_scale=2.0 ** -8,
                              seed=133, **F8)
    dp = DeviceProblem(inputs.make_problem(cfg))
    o_part, lse_part = dp.partial(workspace=workspace)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    _check_split(dp, o_part, lse_part)


def test_fp8_head_slices_are_the_same_rows():
    """head_slices = 2 writes the rows of the plain layout, regrouped."""
    dp = DeviceProblem(inputs.make_problem(CASES["ragged_bf16_cur"]))
    o1, l1 = dp.partial()
    o2, l2 = dp.partial(head_slices=2)
    torch.cuda.synchronize()
    B, q, P, H, D = o1.shape
    o1s = o1.reshape(B * q, P, 2, H // 2, D).permute(2, 0, 1, 3, 4)
    l1s = l1.reshape(B * q, P, 2, H // 2).permute(2, 0, 1, 3)
    assert torch.equal(o1s, o2) and torch.equal(l1s, l2)


def test_fp8_bad_block_id_sets_device_error():
    cfg = inputs.DecodeConfig(name="fb", batch=2, heads=16, q_len=1, num_shards=2,
                              block_size=32, history=100, kv_scale=2.0 ** -8, seed=134, **F8)
    prob = inputs.make_problem(cfg)
    prob.block_table[1, 1] = prob.num_blocks + 5
    dp = DeviceProblem(prob)
    dp.partial()
    torch.cuda.synchronize()
    assert dp.err.item() == 1


def test_fp8_full_size_sampled():
    """The very long context over an E4M3 cache at full size, in the launch
    configuration the bench times (default workspace), sampled sequences and
    heads against the oracle."""
    cfg = inputs.CONFIGS["verylong_fp8"]
    prob = inputs.make_problem(cfg)
    dp = DeviceProblem(prob)
    o_part, lse_part = dp.partial()
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    batch = [0, cfg.batch - 1]
    heads = [0, 77, cfg.heads - 1]
    ref_o, ref_l = om.decode_partials(prob, batch=batch, heads=heads)
    got_o = f64(o_part[batch][:, :, :, heads])
    got_l = f64(lse_part[batch][:, :, :, heads])
    # the sampled rows as a problem of their own, for the bound
    sub = dataclasses.replace(prob, cfg=cfg.with_(batch=len(batch), heads=len(heads)),
                              seq_lens=prob.seq_lens[batch],
                              q_abs=prob.q_abs[batch][:, :, heads],
                              q_pe=prob.q_pe[batch][:, :, heads],
                              block_table=prob.block_table[batch])
    D = fp8_score_bound(sub)
    assert_lse_close(got_l, ref_l, "lse_part", atol=LSE_ATOL + D)
    extra = math.expm1(2 * D) * max_latent(sub)
    for s in range(ref_o.shape[2]):
        ref = ref_o[:, :, s]
        assert_out_close(got_o[:, :, s], ref, f"o_part shard {s}",
                         rtol=OUT_RTOL + extra / np.abs(ref).max())


def test_fp8_many_short_units_per_pair():
    """The E4M3-cache kernel over 512 short histories in 16 shards: more units
    per CTA pair than the pair's table of units holds."""
    cfg = inputs.DecodeConfig(name="fmu", batch=512, heads=16, q_len=1, num_shards=16,
                              block_size=16, ragged=(1, 200), kv_scale=2.0 ** -8, seed=142, **F8)
    dp = DeviceProblem(inputs.make_problem(cfg))
    o_part, lse_part = dp.partial()
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    _check_split(dp, o_part, lse_part)
