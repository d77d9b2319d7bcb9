"""CUDA path versus the fp64 oracle, through the C ABI.

Small cases are compared element by element (every shard partial, every
LSE, the combined latent and the V-up output); the full-size workloads are
run in the launch configuration the bench times and compared on sampled
sequences and heads.
"""
import numpy as np
import pytest
import torch

from mla_decode_attention_kv_gb300 import api, inputs
from oracle import mla_oracle as om

from gpu_util import DeviceProblem, assert_lse_close, assert_out_close, f64

pytestmark = pytest.mark.gpu

SMALL = {
    # several 32-token tiles per shard with ragged tails, shuffled pages
    "ragged_bf16_cur": inputs.DecodeConfig(
        name="s1", batch=3, heads=128, q_len=1, num_shards=3, block_size=32,
        ragged=(1, 400), current=True, seed=21),
    # MTP-like: two query tokens, causal CURRENT chunk, fp16, 64-token pages
    "mtp_fp16": inputs.DecodeConfig(
        name="s2", batch=2, heads=128, q_len=2, num_shards=2, block_size=64,
        history=300, current=True, dtype="fp16", part_dtype="fp16", seed=22),
    # few heads (padded MMA rows), fp32 partials, 16-token pages
    "heads16_fp32part": inputs.DecodeConfig(
        name="s3", batch=2, heads=16, q_len=1, num_shards=4, block_size=16,
        ragged=(20, 200), dtype="bf16", part_dtype="fp32", seed=23),
    "tiny": inputs.CONFIGS["tiny"],
}


def _check_partials(dp, o_part, lse_part):
    ref_o, ref_l = om.decode_partials(dp.prob)
    got_o, got_l = f64(o_part), f64(lse_part)
    assert_lse_close(got_l, ref_l, "lse_part")
    for s in range(ref_o.shape[2]):
        assert_out_close(got_o[:, :, s], ref_o[:, :, s], f"o_part shard {s}")


@pytest.mark.parametrize("name", list(SMALL))
def test_partials_match_oracle(name):
    dp = DeviceProblem(inputs.make_problem(SMALL[name]))
    o_part, lse_part = dp.partial()
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    _check_partials(dp, o_part, lse_part)


@pytest.mark.parametrize("name", list(SMALL))
def test_decode_step_matches_oracle(name):
    dp = DeviceProblem(inputs.make_problem(SMALL[name]))
    H = dp.prob.cfg.heads
    o_latent = torch.empty((dp.prob.cfg.batch * dp.prob.cfg.q_len, H, 512), dtype=dp.dt,
                           device=dp.dev)
    lse = torch.empty((dp.prob.cfg.batch * dp.prob.cfg.q_len, H), dtype=torch.float32,
                      device=dp.dev)
    o_part, lse_part = dp.partial()
    out = api.mla_lse_combine_vup(o_part, lse_part, dp.W, o_latent=o_latent, lse_out=lse,
                                  err_flag=dp.err)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    ref_o, ref_l, ref_out = om.decode_reference(dp.prob)
    B, q = dp.prob.cfg.batch, dp.prob.cfg.q_len
    assert_out_close(f64(o_latent).reshape(B, q, H, 512), ref_o, "o_latent")
    assert_lse_close(f64(lse).reshape(B, q, H), ref_l, "lse")
    assert_out_close(f64(out), ref_out, "out")


@pytest.mark.parametrize("part", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("local", [False, True])
def test_combine_dtypes_and_local(part, local):
    """Combine alone on oracle partials rounded to each partial dtype (the
    BF16 / FP16 / FP32 history-output parametrisation), with and without
    the CURRENT partial passed separately."""
    cfg = inputs.DecodeConfig(name="c", batch=2, heads=128, q_len=2, num_shards=5,
                              block_size=32, ragged=(1, 300), current=True, seed=31)
    prob = inputs.make_problem(cfg, seq_lens=[0, 270])      # sequence 0: all shards empty
    ref_o, ref_l = om.decode_partials(prob)
    dev = torch.device("cuda:0")
    pdt = api.torch_dtype(part)
    o_part = torch.tensor(ref_o, dtype=torch.float32).to(pdt).to(dev)
    lse_part = torch.tensor(ref_l, dtype=torch.float32).to(dev)
    T = cfg.batch * cfg.q_len
    if local:
        S = cfg.num_shards
        o_hist = o_part[:, :, :S].contiguous()
        l_hist = lse_part[:, :, :S].contiguous()
        o_loc = o_part[:, :, S].contiguous()
        l_loc = lse_part[:, :, S].contiguous()
        got_o, got_l = api.mla_lse_combine(o_hist, l_hist, o_local=o_loc, lse_local=l_loc,
                                           out_dtype=torch.float32)
    else:
        got_o, got_l = api.mla_lse_combine(o_part, lse_part, out_dtype=torch.float32)
    torch.cuda.synchronize()
    exp_o, exp_l = om.lse_combine(f64(o_part.float()), ref_l)
    assert_out_close(f64(got_o).reshape(exp_o.shape), exp_o, "o")
    assert_lse_close(f64(got_l).reshape(exp_l.shape), exp_l, "lse")
    assert got_o.shape == (T, cfg.heads, 512)


@pytest.mark.parametrize("P,local,T,H", [(7, True, 37, 8), (20, False, 5, 3), (40, True, 70, 2),
                                         (64, False, 16, 4), (64, True, 9, 2)])
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_combine_vup_of_parts(P, local, T, H, dt):
    """The fused combine + V-up with partials in W_UV's dtype (the up-projection
    of every part, then the LSE-weighted sum): 1 to 9 blocks of rows, 8 to 65
    parts (65 is past what that form takes and goes the register-combine way),
    against combine-then-V-up in fp64.  An empty part (lse = -inf) holds NaN
    rows that must not reach the output; row 0 of head 0 has no part at all."""
    rng = np.random.default_rng(P * 1000 + T)
    tdt = api.torch_dtype(dt)
    o = rng.standard_normal((T, P, H, 512)).astype(np.float32)
    lse = rng.uniform(-3.0, 3.0, (T, P, H)).astype(np.float32)
    lse[:, 1, :] = -np.inf
    o[:, 1] = np.nan
    lse[0, :, 0] = -np.inf
    W = (rng.standard_normal((H, 512, 128)) * 0.05).astype(np.float32)
    o_t = torch.tensor(o).to(tdt).cuda()
    lse_t = torch.tensor(lse).cuda()
    W_t = torch.tensor(W).to(tdt).cuda()
    kw = {}
    o_loc = l_loc = None
    if local:
        o_loc = rng.standard_normal((T, H, 512)).astype(np.float32)
        l_loc = rng.uniform(-3.0, 3.0, (T, H)).astype(np.float32)
        l_loc[0, 0] = -np.inf
        kw = dict(o_local=torch.tensor(o_loc).to(tdt).cuda(), lse_local=torch.tensor(l_loc).cuda())
        o_loc = f64(kw["o_local"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lse_out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    out = api.mla_lse_combine_vup(o_t, lse_t, W_t, lse_out=lse_out, err_flag=err, **kw)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref_o, ref_l = om.lse_combine(np.nan_to_num(f64(o_t), nan=0.0), lse, o_loc, l_loc)
    ref = om.v_up(ref_o, f64(W_t))
    got = f64(out)
    assert np.isfinite(got).all()
    assert not got.reshape(T, H, 128)[0, 0].any()
    assert_out_close(got, ref, "out")
    assert_lse_close(f64(lse_out), ref_l, "lse_out")


def test_vup_matches_oracle():
    rng = np.random.default_rng(5)
    for T, H in ((1, 1), (37, 8), (130, 128)):
        o = rng.standard_normal((T, H, 512)).astype(np.float32)
        W = (rng.standard_normal((H, 512, 128)) * 0.05).astype(np.float32)
        o_t = torch.tensor(o).to(torch.bfloat16).cuda()
        W_t = torch.tensor(W).to(torch.bfloat16).cuda()
        out = api.mla_vup(o_t, W_t)
        torch.cuda.synchronize()
        ref = om.v_up(f64(o_t), f64(W_t))
        assert_out_close(f64(out), ref, f"vup T={T} H={H}")


def test_gather_bit_exact():
    cfg = inputs.DecodeConfig(name="g", batch=5, heads=16, q_len=1, num_shards=2,
                              block_size=16, ragged=(1, 150), seed=41)
    prob = inputs.make_problem(cfg, seq_lens=[0, 1, 16, 17, 149])
    dp = DeviceProblem(prob)
    max_len = 160
    dst = api.mla_gather_kv(dp.cache, dp.table, dp.lens, max_len, err_flag=dp.err)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    got = dst.view(torch.int16).cpu().numpy().view(np.uint16)
    for b in range(cfg.batch):
        L = int(prob.seq_lens[b])
        want = om.gather_history(prob.kv_cache, prob.block_table[b], cfg.block_size, L)
        assert np.array_equal(got[b, :L], want)
        assert not got[b, L:].any()


# ------------------------------------------------------------------ edge cases
@pytest.mark.parametrize("lens", [[0, 0], [1, 31], [32, 64], [33, 97]])
def test_edge_lengths(lens):
    """Empty history (only the CURRENT part is visible), one token, exact
    tile multiples and one-past-a-tile lengths."""
    cfg = inputs.DecodeConfig(name="e", batch=2, heads=128, q_len=2, num_shards=3,
                              block_size=32, ragged=(1, 100), current=True, seed=51)
    dp = DeviceProblem(inputs.make_problem(cfg, seq_lens=lens))
    o_part, lse_part = dp.partial()
    out = api.mla_lse_combine_vup(o_part, lse_part, dp.W, err_flag=dp.err)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    _check_partials(dp, o_part, lse_part)
    _, _, ref_out = om.decode_reference(dp.prob)
    assert_out_close(f64(out), ref_out, "out")


@pytest.mark.parametrize("gain", [30.0, 300.0])
def test_peaked_logits_rescale(gain):
    """q scaled up so the running max moves by many units across tiles: the
    lazy O rescale must keep the result exact."""
    cfg = inputs.DecodeConfig(name="pk", batch=2, heads=128, q_len=1, num_shards=2,
                              block_size=32, history=700, q_gain=gain, seed=61)
    dp = DeviceProblem(inputs.make_problem(cfg))
    o_part, lse_part = dp.partial(part_dtype=torch.float32)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    _check_partials(dp, o_part, lse_part)


def test_extreme_tile_late_in_shard():
    """One tile late in a shard holds logits far above the rest (the slice
    whose max dwarfs the others)."""
    cfg = inputs.DecodeConfig(name="x", batch=1, heads=128, q_len=1, num_shards=2,
                              block_size=32, history=512, shuffle_table=False, seed=71)
    prob = inputs.make_problem(cfg)
    # plant: q_abs[..., 0] = 4 for every head, and tokens 200..231 (tiles 6-7
    # of shard 0, identity page table) carry c[0] large enough to lift their
    # logits by about +30 over the rest
    q = om.to_f64(prob.q_abs, "bf16")
    q[0, 0, :, 0] = 4.0
    prob.q_abs = inputs.round_to_bits(q.astype(np.float32), "bf16")
    kv = om.to_f64(prob.kv_cache, "bf16")
    flat = kv.reshape(-1, 576)
    flat[200:232, 0] = 30.0 / (4.0 * cfg.scale)
    prob.kv_cache = inputs.round_to_bits(kv.astype(np.float32), "bf16")
    dp = DeviceProblem(prob)
    o_part, lse_part = dp.partial(part_dtype=torch.float32)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    _check_partials(dp, o_part, lse_part)


def test_equal_logit_rows():
    """A sequence whose query is all zero: every logit is 0, so each part's
    LSE is ln(tokens) and the combined LSE is ln(L).  Checked on every shard
    partial, the combined LSE and the output."""
    cfg = inputs.DecodeConfig(name="eq", batch=3, heads=128, q_len=1, num_shards=4,
                              block_size=32, ragged=(40, 500), dtype="fp16",
                              part_dtype="fp16", equal_logit_rows=(1,), seed=81)
    dp = DeviceProblem(inputs.make_problem(cfg))
    o_part, lse_part = dp.partial()
    lse = torch.empty((cfg.batch, cfg.heads), dtype=torch.float32, device=dp.dev)
    out = api.mla_lse_combine_vup(o_part, lse_part, dp.W, lse_out=lse, err_flag=dp.err)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    _check_partials(dp, o_part, lse_part)
    _, ref_l, ref_out = om.decode_reference(dp.prob)
    assert_lse_close(f64(lse).reshape(ref_l.shape), ref_l, "lse")
    # the closed form of the all-equal row, independent of the oracle
    L = int(dp.prob.seq_lens[1])
    assert np.abs(f64(lse)[1] - np.log(L)).max() <= 2e-3
    assert_out_close(f64(out), ref_out, "out")


# ------------------------------------------------------------------ page sizes and query counts
@pytest.mark.parametrize("bs", [128, 256])
def test_large_pages(bs):
    """128- and 256-token pages: one TMA box per chunk on the QK CTA, and
    partial tiles at the ends of shards that start inside a page."""
    cfg = inputs.DecodeConfig(name=f"pg{bs}", batch=3, heads=128, q_len=1, num_shards=3,
                              block_size=bs, ragged=(400, 3000), current=True, seed=111)
    dp = DeviceProblem(inputs.make_problem(cfg))
    o_part, lse_part = dp.partial()
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    _check_partials(dp, o_part, lse_part)


def test_many_query_tokens_few_heads():
    """q_len 4 with the causal CURRENT chunk and 64 heads (half-filled MMA rows)."""
    cfg = inputs.DecodeConfig(name="q4", batch=2, heads=64, q_len=4, num_shards=2,
                              block_size=64, ragged=(50, 700), current=True, seed=121)
    dp = DeviceProblem(inputs.make_problem(cfg))
    out = dp.step()
    o_part, lse_part = dp.partial()
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    _check_partials(dp, o_part, lse_part)
    _, _, ref_out = om.decode_reference(dp.prob)
    assert_out_close(f64(out), ref_out, "out")


@pytest.mark.parametrize("q_len,bs", [(16, 32), (64, 16), (64, 64)])
def test_long_current_chunk(q_len, bs):
    """CURRENT chunks of 16 and 64 query tokens (a chunked-prefill step)
    with 128 heads: query i sees history plus current tokens 0..i; every
    shard partial, the CURRENT partial and the combined output."""
    cfg = inputs.DecodeConfig(name=f"q{q_len}", batch=2, heads=128, q_len=q_len, num_shards=2,
                              block_size=bs, ragged=(60, 500), current=True, seed=141 + q_len)
    dp = DeviceProblem(inputs.make_problem(cfg))
    o_part, lse_part = dp.partial()
    out = api.mla_lse_combine_vup(o_part, lse_part, dp.W, err_flag=dp.err)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    _check_partials(dp, o_part, lse_part)
    _, _, ref_out = om.decode_reference(dp.prob)
    assert_out_close(f64(out), ref_out, "out")


@pytest.mark.parametrize("batch,shards", [(3, 4), (32, 8), (5, 64)])
def test_all_parts_empty(batch, shards):
    """No history and no CURRENT chunk: every partial is o = 0, lse = -inf,
    and the combined output is 0 (with and without a workspace).  The
    outputs start as NaN, so a part that no CTA pair wrote would show."""
    cfg = inputs.DecodeConfig(name="em", batch=batch, heads=128, q_len=1, num_shards=shards,
                              block_size=32, ragged=(1, 100), current=False, seed=131)
    dp = DeviceProblem(inputs.make_problem(cfg, seq_lens=[0] * batch))
    for ws in ("default", None):
        o_part = torch.full((batch, 1, shards, 128, 512), float("nan"), dtype=dp.part_dt,
                            device=dp.dev)
        lse_part = torch.full((batch, 1, shards, 128), float("nan"), device=dp.dev)
        dp.partial(workspace=ws, o_part=o_part, lse_part=lse_part)
        out = api.mla_lse_combine_vup(o_part, lse_part, dp.W, err_flag=dp.err)
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        assert torch.isneginf(lse_part).all()
        assert not o_part.float().abs().sum().item()
        assert not out.float().abs().sum().item()


@pytest.mark.parametrize("name", ["ragged_bf16_cur", "heads16_fp32part"])
def test_partials_at_16_byte_offsets(name):
    """q_abs, q_pe and o_part 16-byte aligned but not 32-byte aligned: the
    TMA maps take any 16-byte base and the epilogue falls back from its
    32-byte stores; same results."""
    dp = DeviceProblem(inputs.make_problem(SMALL[name]))

    def shifted(t, dtype=None):
        dtype = dtype or t.dtype
        pad = 16 // torch.empty((), dtype=dtype).element_size()
        buf = torch.empty(t.numel() + pad, dtype=dtype, device=t.device)
        out = buf[pad:].view(t.shape)
        assert out.data_ptr() % 32 == 16
        return out

    dp.q_abs = shifted(dp.q_abs).copy_(dp.q_abs)
    dp.q_pe = shifted(dp.q_pe).copy_(dp.q_pe)
    cfg = dp.prob.cfg
    P = cfg.num_shards + (1 if cfg.current else 0)
    o_part = shifted(torch.empty((cfg.batch, cfg.q_len, P, cfg.heads, 512), dtype=dp.part_dt,
                                 device=dp.dev))
    for ws in ("default", None):
        o_part.fill_(float("nan"))
        o, lse_part = dp.partial(o_part=o_part, workspace=ws)
        torch.cuda.synchronize()
        assert o.data_ptr() == o_part.data_ptr()
        assert dp.err.item() == 0
        _check_partials(dp, o, lse_part)


# ------------------------------------------------------------------ work split across CTA pairs
@pytest.mark.parametrize("name", ["ragged_bf16_cur", "mtp_fp16", "heads16_fp32part"])
def test_whole_shards_without_workspace(name):
    """Without a workspace every CTA pair takes whole shards; same results."""
    dp = DeviceProblem(inputs.make_problem(SMALL[name]))
    o_part, lse_part = dp.partial(workspace=None)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    _check_partials(dp, o_part, lse_part)


@pytest.mark.parametrize("history,q_len,cur", [(40000, 1, False), (9000, 2, True),
                                                  (3000, 1, False)])
def test_shard_split_over_many_pairs(history, q_len, cur):
    """Few long shards cut into pieces of a few tiles for every CTA pair (with
    3000 tokens there are fewer tiles than pairs, so pairs with empty shares
    sit between the pieces): the merged pieces must equal the oracle, and a
    second call on the same (uninitialised) workspace gives identical results."""
    cfg = inputs.DecodeConfig(name="sp", batch=1, heads=128, q_len=q_len, num_shards=1,
                              block_size=64, history=history, current=cur, seed=101)
    dp = DeviceProblem(inputs.make_problem(cfg))
    nbytes = api._ffi.lib().mla_dcp_decode_partial_workspace_size(1, q_len, 1, int(cur))
    ws = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device=dp.dev)
    o1, l1 = dp.partial(workspace=ws, part_dtype=torch.float32)
    o2, l2 = dp.partial(workspace=ws, part_dtype=torch.float32)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    _check_partials(dp, o1, l1)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("workspace", ["default", None])
def test_many_short_units_per_pair(workspace):
    """512 short histories in 16 shards of 16 tokens: about 108 units per CTA
    pair, most of them empty or one tile, more than the pair's shared-memory
    table of units holds (the rest are looked up as they come), and share
    boundaries that fall between, inside and at the ends of tiny units.
    Every partial matches the oracle, with and without a workspace."""
    cfg = inputs.DecodeConfig(name="mu", batch=512, heads=16, q_len=1, num_shards=16,
                              block_size=16, ragged=(1, 200), seed=141)
    dp = DeviceProblem(inputs.make_problem(cfg))
    o_part, lse_part = dp.partial(workspace=workspace)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    _check_partials(dp, o_part, lse_part)


def test_workspace_too_small_is_rejected():
    dp = DeviceProblem(inputs.make_problem(SMALL["tiny"]))
    ws = torch.zeros(1024, dtype=torch.uint8, device=dp.dev)
    with pytest.raises(api._ffi.MlaError) as e:
        dp.partial(workspace=ws)
    assert e.value.status == 2


# ------------------------------------------------------------------ decode context parallelism
@pytest.mark.parametrize("world", [2, 4])
def test_dcp_kernels_with_the_exchange_done_by_hand(world):
    """The GPU steps of a DCP decode step across `world` ranks, with the
    all-to-all done by hand on one GPU: each rank's sliced partials over its
    piece of the history (the sliced layout must be the plain one with heads
    regrouped, bit for bit), block r of every rank stacked (what rank r
    receives), then mla_dcp_combine_exchanged and mla_vup with rank r's
    heads: equal to one softmax over the whole sequence for those heads."""
    import dataclasses
    from mla_decode_attention_kv_gb300 import dcp
    cfg = inputs.DecodeConfig(name="dcpg", batch=3, heads=128, q_len=2, num_shards=2,
                              block_size=32, ragged=(1, 700), current=True, seed=311)
    prob = inputs.make_problem(cfg)
    T, P, hs = cfg.batch * cfg.q_len, cfg.num_shards + 1, cfg.heads // world
    sends = []
    for r in range(world):
        table, lens = dcp.local_block_table(prob.block_table, prob.seq_lens, cfg.block_size,
                                            world, r)
        dp = DeviceProblem(dataclasses.replace(prob, block_table=table, seq_lens=lens))
        o_s, l_s = dp.partial(head_slices=world)
        o_p, l_p = dp.partial()
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        assert torch.equal(o_s, o_p.reshape(T, P, world, hs, 512).permute(2, 0, 1, 3, 4))
        assert torch.equal(l_s, l_p.reshape(T, P, world, hs).permute(2, 0, 1, 3))
        sends.append((o_s, l_s))
    W = DeviceProblem(prob).W
    for r in range(world):
        o_recv = torch.stack([s[0][r] for s in sends]).contiguous()
        l_recv = torch.stack([s[1][r] for s in sends]).contiguous()
        o_lat, lse = api.mla_dcp_combine_exchanged(o_recv, l_recv, hist_parts=cfg.num_shards,
                                                   local_src=r, out_dtype=W.dtype)
        out = api.mla_vup(o_lat, W[r * hs:(r + 1) * hs].contiguous())
        torch.cuda.synchronize()
        ref_o, ref_l, ref_out = om.decode_reference(prob, heads=range(r * hs, (r + 1) * hs))
        assert_out_close(f64(o_lat).reshape(ref_o.shape), ref_o, f"o_latent rank {r}")
        assert_lse_close(f64(lse).reshape(ref_l.shape), ref_l, f"lse rank {r}")
        assert_out_close(f64(out), ref_out, f"out rank {r}")


# ------------------------------------------------------------------ streams and errors
def test_user_stream_no_implicit_sync():
    dp = DeviceProblem(inputs.make_problem(SMALL["ragged_bf16_cur"]))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = dp.step(stream=s)
    s.synchronize()
    _, _, ref_out = om.decode_reference(dp.prob)
    assert_out_close(f64(out), ref_out, "out")


def test_bad_block_id_sets_device_error():
    cfg = inputs.DecodeConfig(name="bb", batch=2, heads=128, q_len=1, num_shards=2,
                              block_size=32, history=100, seed=91)
    prob = inputs.make_problem(cfg)
    prob.block_table[1, 2] = prob.num_blocks + 5        # corrupt one entry
    dp = DeviceProblem(prob)
    dp.partial()
    torch.cuda.synchronize()
    assert dp.err.item() == 1
    # the context is still usable
    dp.err.zero_()
    dp2 = DeviceProblem(inputs.make_problem(cfg))
    dp2.partial()
    torch.cuda.synchronize()
    assert dp2.err.item() == 0


@pytest.mark.parametrize("bad", [-1, "over"])
def test_bad_seq_len_sets_device_error(bad):
    """A history length outside [0, max_blocks * block_size] (a corrupt
    length, set on the host) is reported through the device error word by
    the partial kernel and by the gather; the context stays usable."""
    cfg = inputs.DecodeConfig(name="bl", batch=3, heads=128, q_len=1, num_shards=2,
                              block_size=32, history=100, seed=92)
    prob = inputs.make_problem(cfg)
    cap = prob.max_blocks * cfg.block_size
    prob.seq_lens[1] = cap + 1 if bad == "over" else bad
    dp = DeviceProblem(prob)
    dp.partial()
    torch.cuda.synchronize()
    assert dp.err.item() == 3
    dp.err.zero_()
    api.mla_gather_kv(dp.cache, dp.table, dp.lens, 128, err_flag=dp.err)
    torch.cuda.synchronize()
    assert dp.err.item() == 3
    dp2 = DeviceProblem(inputs.make_problem(cfg))
    o_part, lse_part = dp2.partial()
    torch.cuda.synchronize()
    assert dp2.err.item() == 0
    _check_partials(dp2, o_part, lse_part)


def test_wait_timeout_sets_device_error_and_context_survives():
    """The failure path of a pipeline wait, made to run out on purpose: with
    the waits' poll budget cut to a few polls (a test hook, nothing faults),
    the partial kernel records MLA_DEV_WAIT_TIMEOUT, drains what it issued and
    returns; a normal call on the same context then matches the oracle.  Both
    work splits (with and without a workspace) and two calls in a row."""
    lib = api._ffi.lib()
    dp = DeviceProblem(inputs.make_problem(SMALL["ragged_bf16_cur"]))
    try:
        lib.mla_debug_set_spin_limit(8)
        for ws in ("default", None, "default"):
            dp.err.zero_()
            dp.partial(workspace=ws)
            torch.cuda.synchronize()
            assert dp.err.item() == 2
    finally:
        lib.mla_debug_set_spin_limit(0)
    dp.err.zero_()
    o_part, lse_part = dp.partial()
    out = api.mla_lse_combine_vup(o_part, lse_part, dp.W, err_flag=dp.err)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    _check_partials(dp, o_part, lse_part)
    _, _, ref_out = om.decode_reference(dp.prob)
    assert_out_close(f64(out), ref_out, "out")


def test_host_errors_launch_nothing():
    dp = DeviceProblem(inputs.make_problem(inputs.CONFIGS["tiny"]))
    with pytest.raises(api._ffi.MlaError) as e:
        api.mla_dcp_decode_partial(dp.q_abs, dp.q_pe, dp.cache, dp.table, dp.lens, 65)
    assert e.value.status == 5
    with pytest.raises(api._ffi.MlaError) as e:
        api.mla_dcp_decode_partial(dp.q_abs, dp.q_pe, dp.cache, dp.table, dp.lens, 2,
                                   scale=-1.0)
    assert e.value.status == 2


# ------------------------------------------------------------------ full-size workloads
@pytest.mark.parametrize("name", ["dsv3", "mtp", "ragged", "verylong"])
def test_full_size_sampled(name):
    """Full workload in the bench's launch configuration; checked on sampled
    sequences and heads (every shard partial of those, and the final output)."""
    cfg = inputs.CONFIGS[name]
    prob = inputs.make_problem(cfg)
    dp = DeviceProblem(prob)
    o_part, lse_part = dp.partial()
    out = api.mla_lse_combine_vup(o_part, lse_part, dp.W, err_flag=dp.err)
    torch.cuda.synchronize()
    assert dp.err.item() == 0
    rng = np.random.default_rng(7)
    batch = sorted(set([0, cfg.batch - 1] + rng.integers(0, cfg.batch, 2).tolist()))
    if cfg.equal_logit_rows:
        batch = sorted(set(batch + [cfg.equal_logit_rows[0]]))
    heads = sorted(set([0, cfg.heads - 1] + rng.integers(0, cfg.heads, 4).tolist()))
    ref_po, ref_pl = om.decode_partials(prob, batch=batch, heads=heads)
    got_po = f64(o_part[batch][:, :, :, heads])
    got_pl = f64(lse_part[batch][:, :, :, heads])
    assert_lse_close(got_pl, ref_pl, "lse_part")
    assert_out_close(got_po, ref_po, "o_part")
    ref_o, ref_l, ref_out = om.decode_reference(prob, batch=batch, heads=heads)
    got = f64(out).reshape(cfg.batch, cfg.q_len, cfg.heads, 128)[batch][:, :, heads]
    assert_out_close(got.reshape(ref_out.shape), ref_out, "out")
