"""Helpers for the GPU tests: move a seeded problem to the device and compare
with the oracle under the stated tolerances."""
import numpy as np
import torch

from mla_decode_attention_kv_gb300 import api, inputs
from oracle import mla_oracle as om

# Tolerances of the decode path (bf16/fp16 inputs, fp32 accumulation):
#   max|out - ref| <= 1e-2 * max|ref|;  |lse - ref| <= 2e-3
OUT_RTOL = 1e-2
LSE_ATOL = 2e-3


class DeviceProblem:
    def __init__(self, prob: inputs.DecodeProblem, device="cuda:0"):
        self.prob = prob
        cfg = prob.cfg
        self.dev = torch.device(device)
        self.dt = api.torch_dtype(cfg.dtype)
        self.part_dt = api.torch_dtype(cfg.part_dtype)
        self.q_abs = self.t16(prob.q_abs)
        self.q_pe = self.t16(prob.q_pe)
        self.fp8 = cfg.cache_dtype == "e4m3"
        tk = self.t8 if self.fp8 else self.t16
        self.cache = tk(prob.kv_cache)
        self.kv_cur = tk(prob.kv_cur) if prob.kv_cur is not None else None
        self.kv_scale = cfg.kv_scale if self.fp8 else None
        self.W = self.t16(prob.W_UV)
        self.table = torch.from_numpy(prob.block_table).to(self.dev)
        self.lens = torch.from_numpy(prob.seq_lens).to(self.dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=self.dev)

    def t16(self, a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(self.dev).view(self.dt)

    def t8(self, a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(self.dev)

    def partial(self, **kw):
        kw.setdefault("part_dtype", self.part_dt)
        if self.fp8:
            kw.setdefault("kv_scale", self.kv_scale)
        return api.mla_dcp_decode_partial(
            self.q_abs, self.q_pe, self.cache, self.table, self.lens, self.prob.cfg.num_shards,
            kv_cur=self.kv_cur, scale=self.prob.cfg.scale, err_flag=self.err, **kw)

    def step(self, **kw):
        kw.setdefault("part_dtype", self.part_dt)
        if self.fp8:
            kw.setdefault("kv_scale", self.kv_scale)
        return api.decode_step(
            self.q_abs, self.q_pe, self.cache, self.table, self.lens, self.W,
            self.prob.cfg.num_shards, kv_cur=self.kv_cur, scale=self.prob.cfg.scale,
            err_flag=self.err, **kw)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_out_close(got, ref, what="out", rtol=OUT_RTOL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    scale = np.abs(ref).max()
    diff = np.abs(got - ref).max()
    assert diff <= rtol * scale + 1e-30, f"{what}: max|got-ref| = {diff:.3e} > {rtol} * {scale:.3e}"


def assert_lse_close(got, ref, what="lse", atol=LSE_ATOL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    inf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf_ref), f"{what}: -inf pattern differs"
    fin = ~inf_ref
    if fin.any():
        diff = np.abs(got[fin] - ref[fin]).max()
        assert diff <= atol, f"{what}: max|lse-ref| = {diff:.3e} > {atol}"


# ---------------------------------------------------------------- E4M3 cache
# The E4M3-cache kernel multiplies the cache bytes by the query in two E4M3
# terms: per row a power-of-two scale sq = 2^(E-8) (max|q| = f 2^E, f in
# [0.5, 1)), hi = rn(q / sq), lo = rn(q / sq - hi), both rounded to nearest
# even with saturation, and uses q' = sq (hi + lo).  split_query computes q'
# the same way (the rounding decisions in the same precision: q / sq and the
# remainder are exact in fp32), so the kernel can be held to the 16-bit
# tolerances against the oracle fed q'.  The documented bound of the query
# error, |q - q'| <= 2^-8 |q| + 2^-17 max|q row|, gives the tolerance against
# the oracle on the exact q (fp8_score_bound).


def _e4m3_round(x):
    return om.e4m3_to_f64(inputs.round_to_bits(np.asarray(x, np.float32), "e4m3"))


def split_query(prob):
    """q' rows of every (b, i, h): q_abs' [B, q, H, 512], q_pe' [B, q, H, 64]."""
    dt = prob.cfg.dtype
    q = np.concatenate([om.to_f64(prob.q_abs, dt), om.to_f64(prob.q_pe, dt)], axis=-1)
    amax = np.abs(q).max(axis=-1, keepdims=True)
    _, E = np.frexp(amax)
    sq = np.where(amax > 0, np.ldexp(1.0, E - 8), 1.0)
    x = q / sq
    hi = _e4m3_round(x)
    lo = _e4m3_round(x - hi)
    qs = sq * (hi + lo)
    return qs[..., :512], qs[..., 512:]


def split_partials(prob):
    """Oracle partials with the kernel's two-term query."""
    qa, qp = split_query(prob)
    return om.decode_partials(prob, queries=lambda b, i, h: (qa[b, i][h], qp[b, i][h]))


def fp8_score_bound(prob):
    """Largest change of a score s_t that the documented query error allows:
    scale * sum_i |k_i| (2^-8 |q_i| + 2^-17 max|q row|), over every row and
    every token the row may see."""
    dt = prob.cfg.dtype
    q = np.abs(np.concatenate([om.to_f64(prob.q_abs, dt), om.to_f64(prob.q_pe, dt)], axis=-1))
    dq = 2.0 ** -8 * q + 2.0 ** -17 * q.max(axis=-1, keepdims=True)    # [B, q, H, 576]
    worst = 0.0
    for b in range(prob.cfg.batch):
        toks = np.abs(np.concatenate([om._history(prob, b), om._current(prob, b)], axis=0))
        if toks.shape[0]:
            worst = max(worst, float((dq[b].reshape(-1, 576) @ toks.T).max()))
    return prob.cfg.scale * worst


def max_latent(prob):
    """max |c_t| over the latent values of every token some row sees."""
    m = 0.0
    for b in range(prob.cfg.batch):
        toks = np.concatenate([om._history(prob, b), om._current(prob, b)], axis=0)
        if toks.shape[0]:
            m = max(m, float(np.abs(toks[:, :512]).max()))
    return m
