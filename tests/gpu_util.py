"""Helpers for the GPU tests: move a seeded problem to the device and compare
with the oracle under the stated tolerances."""
import numpy as np
import torch

from mla_decode_attention_kv_gb300 import api, inputs

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
        self.cache = self.t16(prob.kv_cache)
        self.kv_cur = self.t16(prob.kv_cur) if prob.kv_cur is not None else None
        self.W = self.t16(prob.W_UV)
        self.table = torch.from_numpy(prob.block_table).to(self.dev)
        self.lens = torch.from_numpy(prob.seq_lens).to(self.dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=self.dev)

    def t16(self, a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(self.dev).view(self.dt)

    def partial(self, **kw):
        kw.setdefault("part_dtype", self.part_dt)
        return api.mla_dcp_decode_partial(
            self.q_abs, self.q_pe, self.cache, self.table, self.lens, self.prob.cfg.num_shards,
            kv_cur=self.kv_cur, scale=self.prob.cfg.scale, err_flag=self.err, **kw)

    def step(self, **kw):
        kw.setdefault("part_dtype", self.part_dt)
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
