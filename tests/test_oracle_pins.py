"""Pins for the fp64 oracle, each against something other than the oracle.

* sizes the pages print (tests/golden/page_sizes.json)
* a two-token closed form (tests/golden/two_token_closed_form.json)
* brute force with literal loops and no max subtraction on tiny inputs
* the explicitly materialised per-head form (K = [W_UK c ; k_R], V = W_UV^T c)
  and torch's scaled_dot_product_attention on that form, in float64
* sharded + LSE combine equal to one unsharded softmax
* closed-form special cases (one token, constant latent, equal logits)
* planted mistakes: a wrong oracle must fail at least one of these pins
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import mla_oracle as om
from mla_decode_attention_kv_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def _rand(*shape, s=1.0):
    return RNG.standard_normal(shape) * s


# ----------------------------------------------------------------- sizes
def test_page_size_pins():
    g = json.load(open(os.path.join(GOLDEN, "page_sizes.json")))
    assert oracle.D_LATENT == g["d_c"] and oracle.D_ROPE == g["d_R"]
    assert oracle.D_QK == g["values_per_token"]
    per_token = oracle.D_QK * 2
    assert abs(per_token / 1000 - g["bytes_per_token_approx_kb"]) < 0.01
    for bs, kb in g["block_bytes_kb"].items():
        assert int(bs) * per_token == kb * 1024


def test_two_token_closed_form():
    g = json.load(open(os.path.join(GOLDEN, "two_token_closed_form.json")))
    q_abs = np.zeros((1, 512))
    q_abs[0, g["q_abs_nonzero"]["index"]] = g["q_abs_nonzero"]["value"]
    toks = np.zeros((2, 576))
    toks[0, 0], toks[0, 1] = g["token0"]["c0"], g["token0"]["c1"]
    toks[1, 0], toks[1, 1] = math.log(3.0), g["token1"]["c1"]
    o, lse = om.segment_attention(q_abs, np.zeros((1, 64)), toks, g["scale"])
    w = g["expected"]["weights"]
    assert o[0, 1] == pytest.approx(g["expected"]["o_c1"], abs=1e-14)
    assert o[0, 0] == pytest.approx(w[1] * math.log(3.0), abs=1e-14)
    assert lse[0] == pytest.approx(math.log(4.0), abs=1e-14)


# ----------------------------------------------------------------- decode
def test_bits_decode_exact():
    x = np.array([0.0, 1.0, -2.5, 0.1, 65504.0, 1e-3], dtype=np.float32)
    for dt in ("bf16", "fp16"):
        bits = inputs.round_to_bits(x, dt)
        back = om.to_f64(bits, dt)
        if dt == "fp16":
            ref = x.astype(np.float16).astype(np.float64)
        else:
            ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            # bf16 keeps 8 significant bits: relative error <= 2^-9
            assert np.all(np.abs(back - x) <= np.abs(x) * 2.0 ** -8 + 1e-30)
        assert np.array_equal(back, ref)
    assert om.to_f64(np.array([0x3F80], np.uint16), "bf16")[0] == 1.0
    assert om.to_f64(np.array([0x3C00], np.uint16), "fp16")[0] == 1.0


# ----------------------------------------------------------------- E4M3 cache
def test_e4m3_decode_special_codes():
    """Codes whose values follow directly from the E4M3 definition (bias 7,
    3 mantissa bits, subnormals at exponent field 0, 0x7F / 0xFF NaN)."""
    cases = {0x00: 0.0, 0x38: 1.0, 0xB8: -1.0, 0x40: 2.0, 0x3C: 1.5, 0x7E: 448.0,
             0xFE: -448.0, 0x08: 2.0 ** -6, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9,
             0x77: 240.0, 0x30: 0.5, 0x28: 0.25}
    got = om.e4m3_to_f64(np.array(list(cases), dtype=np.uint8))
    assert np.array_equal(got, np.array(list(cases.values())))
    neg0 = om.e4m3_to_f64(np.array([0x80], np.uint8))[0]
    assert neg0 == 0.0 and np.signbit(neg0)
    assert np.all(np.isnan(om.e4m3_to_f64(np.array([0x7F, 0xFF], np.uint8))))


def test_e4m3_decode_equals_torch_float8():
    """All 256 codes against torch's float8_e4m3fn conversion (a separate
    implementation of the same format)."""
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = om.e4m3_to_f64(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_e4m3_codes_monotone_and_spaced():
    """Positive codes 0x00..0x7E increase; the step up from code c is the ulp
    2^(e-10) of c's binade e (exponent field; the subnormal step 2^-9 equals
    the first normal binade's)."""
    v = om.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    d = np.diff(v)
    assert np.all(d > 0)
    e = np.maximum(np.arange(0, 0x7E) >> 3, 1)
    assert np.array_equal(d, np.ldexp(1.0, e - 10))


def test_e4m3_generator_rounds_to_nearest_even():
    """The input generator's E4M3 rounding, by brute force over all codes:
    the nearest finite value, ties to the even code, saturation at 448."""
    vals = om.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    x = np.concatenate([RNG.standard_normal(4000) * 30, RNG.standard_normal(2000) * 0.01,
                        (vals[1:] + vals[:-1]) / 2, vals, [500.0, -1e6, 464.0]])
    codes = inputs.round_to_bits(x.astype(np.float32), "e4m3")
    got = om.e4m3_to_f64(codes)
    xf = x.astype(np.float32).astype(np.float64)
    a = np.minimum(np.abs(xf), 448.0)
    dist = np.abs(a[:, None] - vals[None, :])
    best = dist.min(axis=1)
    assert np.all(np.abs(np.abs(got) - a) == best)
    ties = (dist == best[:, None]).sum(axis=1) == 2
    assert np.all((codes[ties] & 1) == 0)
    nz = got != 0
    assert np.all(np.sign(got[nz]) == np.sign(xf[nz]))


def test_e4m3_cache_attention_equals_decoded_16bit_cache():
    """An E4M3 problem attends over byte * kv_scale: the same problem with the
    cache stored as those exact values in bf16 (every E4M3 value times a power
    of two is a bf16 value), decoded by torch, gives identical results."""
    torch = pytest.importorskip("torch")
    cfg = inputs.DecodeConfig(name="f8", batch=2, heads=4, q_len=2, num_shards=2, block_size=16,
                              ragged=(3, 90), current=True, kv_dtype="e4m3", kv_scale=2.0 ** -7,
                              seed=41)
    p8 = inputs.make_problem(cfg)

    def as_bf16(bits):
        v = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        v = v * cfg.kv_scale
        out = inputs.round_to_bits(v.astype(np.float32), "bf16")
        assert np.array_equal(om.to_f64(out, "bf16"), v)
        return out

    import dataclasses
    p16 = dataclasses.replace(p8, cfg=cfg.with_(kv_dtype=""), kv_cache=as_bf16(p8.kv_cache),
                              kv_cur=as_bf16(p8.kv_cur))
    o8, l8, y8 = om.decode_reference(p8)
    o16, l16, y16 = om.decode_reference(p16)
    assert np.array_equal(o8, o16) and np.array_equal(l8, l16) and np.array_equal(y8, y16)
    a8, b8 = om.decode_partials(p8)
    a16, b16 = om.decode_partials(p16)
    assert np.array_equal(a8, a16) and np.array_equal(b8, b16)


# ----------------------------------------------------------------- gather
def test_gather_tags_through_shuffled_table():
    cfg = inputs.DecodeConfig(name="g", batch=3, heads=2, q_len=1,
                              num_shards=2, block_size=4, ragged=(3, 20), seed=5)
    p = inputs.make_problem(cfg)
    # tag every physical slot with a unique id, then read the ids back
    tags = np.arange(p.num_blocks * 4, dtype=np.uint16).reshape(p.num_blocks, 4, 1)
    cache = np.broadcast_to(tags, (p.num_blocks, 4, 576)).copy()
    for b in range(cfg.batch):
        L = int(p.seq_lens[b])
        got = om.gather_history(cache, p.block_table[b], 4, L)[:, 0]
        want = [p.block_table[b][t // 4] * 4 + t % 4 for t in range(L)]
        assert list(got) == want
        fast = om.gather_history_fast(cache, p.block_table[b], 4, L)
        assert np.array_equal(fast, om.gather_history(cache, p.block_table[b], 4, L))
    for gather in (om.gather_history, om.gather_history_fast):
        assert gather(cache, p.block_table[0], 4, 0).shape == (0, 576)
    # every physical block is used by exactly one sequence
    used = p.block_table[p.block_table >= 0]
    assert sorted(used.tolist()) == list(range(p.num_blocks))


def test_shard_bounds_worked_cases():
    assert om.shard_bounds(4096, 8, 64) == [(512 * s, 512 * (s + 1)) for s in range(8)]
    assert om.shard_bounds(256, 2, 64) == [(0, 128), (128, 256)]
    assert om.shard_bounds(100, 4, 32) == [(0, 32), (32, 64), (64, 96), (96, 100)]
    assert om.shard_bounds(10, 4, 32) == [(0, 10), (10, 10), (10, 10), (10, 10)]
    assert om.shard_bounds(0, 3, 32) == [(0, 0)] * 3
    for L in (1, 31, 32, 33, 1000, 65536, 54321):
        for S in (1, 2, 8, 16):
            for bs in (32, 64):
                b = om.shard_bounds(L, S, bs)
                assert b[0][0] == 0 and b[-1][1] == L
                for (lo, hi), (lo2, _) in zip(b, b[1:]):
                    assert hi == lo2 and lo <= hi
                    assert lo % bs == 0 or lo == L
                per = bs * -(-L // (S * bs))
                sizes = [hi - lo for lo, hi in b]
                assert all(sz == per for sz in sizes[:L // per])
                assert sum(sizes) == L


# ----------------------------------------------------------------- brute force (C3)
def _brute(q_abs, q_pe, toks, scale, visible=None):
    R, N = len(q_abs), len(toks)
    o = [[0.0] * 512 for _ in range(R)]
    lse = [-math.inf] * R
    for r in range(R):
        num = [0.0] * 512
        den = 0.0
        for t in range(N):
            if visible is not None and not visible[r][t]:
                continue
            dot = 0.0
            for d in range(512):
                dot += q_abs[r][d] * toks[t][d]
            for d in range(64):
                dot += q_pe[r][d] * toks[t][512 + d]
            w = math.exp(scale * dot)
            den += w
            for d in range(512):
                num[d] += w * toks[t][d]
        if den > 0:
            o[r] = [x / den for x in num]
            lse[r] = math.log(den)
    return np.array(o), np.array(lse)


@pytest.mark.parametrize("N", [1, 2, 5, 8])
def test_segment_attention_brute_force(N):
    qa, qp, toks = _rand(2, 512, s=0.3), _rand(2, 64, s=0.3), _rand(N, 576, s=0.3)
    vis = RNG.random((2, N)) < 0.7
    vis[:, 0] = True
    for mask in (None, vis):
        o, lse = om.segment_attention(qa, qp, toks, 0.07, mask)
        ob, lb = _brute(qa.tolist(), qp.tolist(), toks.tolist(), 0.07,
                        None if mask is None else mask.tolist())
        assert np.max(np.abs(o - ob)) < 1e-12
        assert np.max(np.abs(lse - lb)) < 1e-12


def test_decode_reference_brute_force_tiny():
    cfg = inputs.DecodeConfig(name="t", batch=2, heads=2, q_len=2, num_shards=2,
                              block_size=2, ragged=(2, 7), current=True, seed=3,
                              std=0.5)
    p = inputs.make_problem(cfg)
    o, lse, _ = om.decode_reference(p, with_vup=False)
    for b in range(2):
        hist = [om.to_f64(p.kv_cache[p.block_table[b][t // 2], t % 2], "bf16").tolist()
                for t in range(int(p.seq_lens[b]))]
        cur = om.to_f64(p.kv_cur[b], "bf16").tolist()
        for i in range(2):
            toks = hist + cur[:i + 1]
            qa = om.to_f64(p.q_abs[b, i], "bf16").tolist()
            qp = om.to_f64(p.q_pe[b, i], "bf16").tolist()
            ob, lb = _brute(qa, qp, toks, cfg.scale)
            assert np.max(np.abs(o[b, i] - ob)) < 1e-12
            assert np.max(np.abs(lse[b, i] - lb)) < 1e-12


# ----------------------------------------------------------------- explicit form (C1)
def _explicit_problem(H=4, L=37, T=3, seed=7):
    rng = np.random.default_rng(seed)
    q_nope = rng.standard_normal((T, H, 128)) * 0.2
    q_pe = rng.standard_normal((T, H, 64)) * 0.2
    W_UK = rng.standard_normal((H, 128, 512)) * 0.05     # c (512) -> k_nope (128)
    W_UV = rng.standard_normal((H, 512, 128)) * 0.05     # c (512) -> v (128)
    c = rng.standard_normal((L, 512)) * 0.3
    k_r = rng.standard_normal((L, 64)) * 0.3
    return q_nope, q_pe, W_UK, W_UV, c, k_r


def _explicit_attention(q_nope, q_pe, W_UK, W_UV, c, k_r):
    """Textbook per-head attention on materialised 192-dim keys, 128-dim values."""
    T, H, _ = q_nope.shape
    out = np.zeros((T, H, 128))
    for h in range(H):
        K = np.concatenate([c @ W_UK[h].T, k_r], axis=1)       # [L, 192]
        V = c @ W_UV[h]                                         # [L, 128]
        q = np.concatenate([q_nope[:, h], q_pe[:, h]], axis=1)  # [T, 192]
        s = q @ K.T / math.sqrt(192.0)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        out[:, h] = p @ V
    return out.reshape(T, H * 128)


def _absorbed(q_nope, q_pe, W_UK, W_UV, c, k_r):
    T, H, _ = q_nope.shape
    toks = np.concatenate([c, k_r], axis=1)
    o = np.zeros((T, H, 512))
    for t in range(T):
        q_abs = np.einsum("hn,hnc->hc", q_nope[t], W_UK)       # W_UK^T q_nope
        o[t], _ = om.segment_attention(q_abs, q_pe[t], toks, 1.0 / math.sqrt(192.0))
    return om.v_up(o, W_UV)


def test_absorbed_equals_explicit():
    args = _explicit_problem()
    ref = _explicit_attention(*args)
    got = _absorbed(*args)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_absorbed_equals_library_sdpa():
    torch = pytest.importorskip("torch")
    q_nope, q_pe, W_UK, W_UV, c, k_r = _explicit_problem(H=3, L=29, T=2, seed=9)
    T, H = q_nope.shape[:2]
    q = torch.from_numpy(np.concatenate([q_nope, q_pe], axis=2)).permute(1, 0, 2)
    K = torch.from_numpy(np.stack([np.concatenate([c @ W_UK[h].T, k_r], 1) for h in range(H)]))
    V = torch.from_numpy(np.stack([c @ W_UV[h] for h in range(H)]))
    ref = torch.nn.functional.scaled_dot_product_attention(
        q[None], K[None], V[None], scale=1.0 / math.sqrt(192.0))[0]
    ref = ref.permute(1, 0, 2).reshape(T, H * 128).numpy()
    got = _absorbed(q_nope, q_pe, W_UK, W_UV, c, k_r)
    assert np.max(np.abs(got - ref)) <= 1e-12 * np.max(np.abs(ref))


# ----------------------------------------------------------------- sharded == unsharded (C2)
@pytest.mark.parametrize("S", [1, 2, 8, 16])
def test_sharded_combine_equals_single_softmax(S):
    cfg = inputs.DecodeConfig(name="c2", batch=3, heads=3, q_len=2, num_shards=S,
                              block_size=4, ragged=(1, 60), current=True,
                              seed=11 + S, std=0.4)
    p = inputs.make_problem(cfg)
    o_ref, lse_ref, out_ref = om.decode_reference(p)
    o_part, lse_part = om.decode_partials(p)
    o, lse = om.lse_combine(o_part, lse_part)
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert np.max(np.abs(lse - lse_ref)) < 1e-12
    # the CURRENT partial passed separately as the local input
    o2, lse2 = om.lse_combine(o_part[:, :, :S], lse_part[:, :, :S],
                              o_part[:, :, S], lse_part[:, :, S])
    assert np.max(np.abs(o2 - o_ref)) < 1e-12
    out = om.v_up(o.reshape(-1, 3, 512), om.to_f64(p.W_UV, "bf16"))
    assert np.max(np.abs(out - out_ref)) < 1e-12


def test_combine_random_boundaries_and_empty_shards():
    qa, qp, toks = _rand(3, 512, s=0.2), _rand(3, 64, s=0.2), _rand(50, 576, s=0.4)
    o_ref, lse_ref = om.segment_attention(qa, qp, toks, 0.3)
    cuts = sorted(RNG.integers(0, 51, size=9).tolist())
    bounds = list(zip([0] + cuts, cuts + [50]))          # some empty
    parts = [om.segment_attention(qa, qp, toks[lo:hi], 0.3) for lo, hi in bounds]
    o_part = np.stack([p[0] for p in parts])
    lse_part = np.stack([p[1] for p in parts])
    o, lse = om.lse_combine(o_part, lse_part)
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert np.max(np.abs(lse - lse_ref)) < 1e-12


# ----------------------------------------------------------------- closed forms
def test_single_token_gives_its_latent():
    qa, qp, tok = _rand(4, 512), _rand(4, 64), _rand(1, 576)
    o, lse = om.segment_attention(qa, qp, tok, 0.05)
    assert np.allclose(o, tok[0, :512][None], atol=1e-15)
    s0 = 0.05 * (qa @ tok[0, :512] + qp @ tok[0, 512:])
    assert np.allclose(lse, s0, atol=1e-13)


def test_constant_latent_any_logits():
    qa, qp = _rand(3, 512), _rand(3, 64)
    toks = _rand(20, 576)
    toks[:, :512] = 0.37
    o, _ = om.segment_attention(qa, qp, toks, 0.9)
    assert np.max(np.abs(o - 0.37)) < 1e-14


def test_equal_logits_mean_and_log_count():
    toks = _rand(33, 576)
    o, lse = om.segment_attention(np.zeros((2, 512)), np.zeros((2, 64)), toks, 0.1)
    assert np.max(np.abs(o - toks[:, :512].mean(0))) < 1e-14
    assert np.allclose(lse, math.log(33.0), atol=1e-14)


def test_extreme_shard_dominates():
    """One shard's logits sit +30 above the rest: its partial must dominate
    and the combine must still equal the single softmax."""
    qa = np.zeros((1, 512)); qa[0, 0] = 1.0
    toks = _rand(64, 576, s=0.1)
    toks[40:48, 0] += 30.0
    o_ref, lse_ref = om.segment_attention(qa, np.zeros((1, 64)), toks, 1.0)
    parts = [om.segment_attention(qa, np.zeros((1, 64)), toks[s:s + 16], 1.0)
             for s in range(0, 64, 16)]
    o, lse = om.lse_combine(np.stack([p[0] for p in parts]),
                            np.stack([p[1] for p in parts]))
    assert np.max(np.abs(o - o_ref)) < 1e-11
    assert abs(lse[0] - lse_ref[0]) < 1e-12
    assert np.max(np.abs(o[0] - parts[2][0][0])) < 1e-10


def test_all_empty_parts_give_zero_and_minus_inf():
    o, lse = om.lse_combine(np.ones((3, 2, 512)), np.full((3, 2), -np.inf))
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    o, lse = om.segment_attention(_rand(2, 512), _rand(2, 64), np.zeros((0, 576)), 1.0)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


def test_combine_two_equal_parts_closed_form():
    a, b = _rand(1, 2, 512), _rand(1, 2, 512)
    o, lse = om.lse_combine(np.concatenate([a, b]), np.full((2, 2), 1.5))
    assert np.allclose(o, (a[0] + b[0]) / 2, atol=1e-15)
    assert np.allclose(lse, 1.5 + math.log(2.0), atol=1e-15)


def test_vup_identity_blocks_and_head_order():
    """W_UV[h] = (h+1) * [I_128 ; 0]: output head h must be (h+1) times the
    first 128 latent values of head h, laid out head-major in each row."""
    T, H = 3, 5
    o = _rand(T, H, 512)
    W = np.zeros((H, 512, 128))
    for h in range(H):
        W[h, :128, :] = (h + 1) * np.eye(128)
    out = om.v_up(o, W)
    assert out.shape == (T, H * 128)
    for t in range(T):
        for h in range(H):
            assert np.array_equal(out[t, h * 128:(h + 1) * 128], (h + 1) * o[t, h, :128])


def test_vup_of_parts_equals_combine_then_vup():
    """The up-projection is linear, so projecting each part and taking the
    LSE-weighted sum in the 128-wide V space equals combine-then-V-up (the
    fused call's form for partials in the model dtype).  The per-part side
    is written here with plain numpy: weights exp(lse_p - LSE), empty parts
    (lse = -inf) weight 0, a row with no part gives 0."""
    rng = np.random.default_rng(17)
    T, P, H = 5, 6, 3
    o = rng.standard_normal((T, P, H, 512))
    lse = rng.uniform(-4.0, 4.0, (T, P, H))
    lse[:, 2, :] = -np.inf
    lse[1, :, 0] = -np.inf
    W = rng.standard_normal((H, 512, 128)) * 0.05
    o_c, l_c = om.lse_combine(o, lse)
    want = om.v_up(o_c, W).reshape(T, H, 128)
    got = np.zeros((T, H, 128))
    for t in range(T):
        for h in range(H):
            fin = np.isfinite(lse[t, :, h])
            if not fin.any():
                continue
            m = lse[t, fin, h].max()
            w = np.where(fin, np.exp(np.where(fin, lse[t, :, h], m) - m), 0.0)
            w /= w.sum()
            for p in range(P):
                if w[p]:
                    got[t, h] += w[p] * (o[t, p, h] @ W[h])
    assert not got[1, 0].any() and not want[1, 0].any()
    assert np.max(np.abs(got - want)) < 1e-12 * max(1.0, np.abs(want).max())


def test_shuffled_table_same_result_as_identity():
    base = inputs.DecodeConfig(name="p", batch=2, heads=2, q_len=1, num_shards=3,
                               block_size=8, history=50, seed=4)
    a = inputs.make_problem(base.with_(shuffle_table=False))
    b = inputs.make_problem(base)
    # same random values, different page placement: move pages to match
    b_cache = np.empty_like(a.kv_cache)
    for s in range(2):
        for j in range((50 + 7) // 8):
            b_cache[b.block_table[s, j]] = a.kv_cache[a.block_table[s, j]]
    b.kv_cache = b_cache
    oa, la, _ = om.decode_reference(a)
    ob, lb, _ = om.decode_reference(b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


# ----------------------------------------------------------------- planted mistakes
def _pins_pass():
    try:
        test_segment_attention_brute_force(5)
        test_absorbed_equals_explicit()
        test_sharded_combine_equals_single_softmax(2)
        test_vup_identity_blocks_and_head_order()
        test_combine_random_boundaries_and_empty_shards()
        test_e4m3_decode_equals_torch_float8()
        test_e4m3_cache_attention_equals_decoded_16bit_cache()
    except AssertionError:
        return False
    return True


def test_pins_pass_unmodified():
    assert _pins_pass()


@pytest.mark.parametrize("mutant", ["drop_rope", "rope_sign", "scale_sqrt128",
                                    "transposed_wuv", "combine_no_weights",
                                    "lse_log2", "e4m3_bias8", "e4m3_no_subnormals",
                                    "kv_scale_dropped"])
def test_planted_mistake_is_caught(monkeypatch, mutant):
    real_seg, real_comb, real_vup = om.segment_attention, om.lse_combine, om.v_up
    real_e4m3, real_cache = om.e4m3_to_f64, om.cache_values

    def e4m3(bits):
        v = real_e4m3(bits)
        b = np.asarray(bits, dtype=np.uint8)
        if mutant == "e4m3_bias8":
            v = v / 2.0
        if mutant == "e4m3_no_subnormals":
            v = np.where((b & 0x78) == 0, 0.0, v)
        return v

    def cache(bits, cfg):
        if mutant == "kv_scale_dropped" and cfg.cache_dtype == "e4m3":
            return om.e4m3_to_f64(bits)
        return real_cache(bits, cfg)

    def seg(q_abs, q_pe, tokens, scale, visible=None):
        if mutant == "drop_rope":
            q_pe = np.zeros_like(q_pe)
        if mutant == "rope_sign":
            q_pe = -q_pe
        if mutant == "scale_sqrt128":
            scale = scale * math.sqrt(192.0 / 128.0)
        o, lse = real_seg(q_abs, q_pe, tokens, scale, visible)
        if mutant == "lse_log2":
            lse = lse / math.log(2.0)
        return o, lse

    def comb(o_part, lse_part, o_local=None, lse_local=None):
        if mutant == "combine_no_weights":
            lse_part = np.where(np.isfinite(lse_part), 0.0, lse_part)
        return real_comb(o_part, lse_part, o_local, lse_local)

    def vup(o_latent, W_UV):
        if mutant == "transposed_wuv":
            W_UV = np.ascontiguousarray(np.swapaxes(W_UV.reshape(W_UV.shape[0], 4, 128, 128), 2, 3)
                                        ).reshape(W_UV.shape)
        return real_vup(o_latent, W_UV)

    monkeypatch.setattr(om, "segment_attention", seg)
    monkeypatch.setattr(om, "lse_combine", comb)
    monkeypatch.setattr(om, "v_up", vup)
    monkeypatch.setattr(om, "e4m3_to_f64", e4m3)
    monkeypatch.setattr(om, "cache_values", cache)
    assert not _pins_pass()
