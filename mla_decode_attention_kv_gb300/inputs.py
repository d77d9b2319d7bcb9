"""Seeded synthetic inputs for decode-step MLA over a paged latent KV cache.

This module is the one thing the oracle and the CUDA path share.  It draws
random numbers, rounds them to the storage dtype and lays them out in the
paged-cache format; it holds none of the attention arithmetic.  It imports
numpy only.

Every tensor is returned as raw 16-bit storage bits (``np.uint16``) plus a
dtype tag, so the very same bytes feed the fp64 oracle (which decodes them
itself) and the GPU (which reinterprets them as bf16/fp16).

Layouts (all C-contiguous):

=============  ==========================  =====================================
name           shape                       meaning
=============  ==========================  =====================================
q_abs          [B, q_len, H, 512]          query already absorbed into latent
                                           space (q_nope times W_UK)
q_pe           [B, q_len, H, 64]           RoPE part of the query (pre-rotated)
kv_cache       [num_blocks, bs, 576]       c_KV in [0:512), k_R in [512:576)
block_table    [B, max_blocks] int32       physical block of logical block j;
                                           entries past a sequence's last
                                           block are -1
seq_lens       [B] int32                   HISTORY length of each sequence
kv_cur         [B, q_len, 576] or None     CURRENT-chunk latent + RoPE key
W_UV           [H, 512, 128]               per-head V up-projection
=============  ==========================  =====================================

Recipe: ``numpy.random.default_rng(seed)``; values are N(0, 1) * 0.1 drawn in
float32 and rounded to nearest-even in the storage dtype.  An FP8 latent
cache (``kv_dtype="e4m3"``) stores the cache and CURRENT values divided by
``kv_scale`` (a power of two) as E4M3 bytes, rounded to nearest-even and
saturated at +-448; q and W_UV keep the model dtype.  Draw order:
(ragged history lengths), q_abs, q_pe, kv_cache, kv_cur, W_UV, block-table
permutation.  The block table is a random permutation of all physical blocks
cut per sequence (or the identity), so a sequence's pages are scattered over
the pool as in a paged serving cache.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

D_LATENT = 512          # kv_lora_rank: width of c_KV
D_ROPE = 64             # width of the decoupled RoPE key k_R
D_QK = D_LATENT + D_ROPE
D_V = 128               # per-head V width after the up-projection

_CHUNK = 1 << 24        # values drawn per call when filling big tensors


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    """One synthetic decode workload (all sizes explicit)."""
    name: str
    batch: int
    heads: int
    q_len: int
    num_shards: int
    block_size: int
    history: int = 0                 # fixed history length (ignored if ragged)
    ragged: tuple = ()               # (lo, hi): log-uniform history lengths
    current: bool = False            # CURRENT segment present (kv_cur)
    dtype: str = "bf16"              # storage dtype of q, cache, W_UV
    part_dtype: str = "bf16"         # dtype of the per-shard partial outputs
    kv_dtype: str = ""               # cache / kv_cur storage dtype ("" = dtype, or "e4m3")
    kv_scale: float = 1.0            # e4m3 cache: value = decoded byte * kv_scale
    shuffle_table: bool = True
    equal_logit_rows: tuple = ()     # sequences whose q is all zero
    q_gain: float = 1.0              # test-only: scales q to sharpen softmax
    std: float = 0.1
    seed: int = 0

    @property
    def cache_dtype(self) -> str:
        return self.kv_dtype or self.dtype

    @property
    def scale(self) -> float:
        # softmax scale of the explicit per-head form: 128 nope + 64 rope dims
        return 1.0 / math.sqrt(128 + D_ROPE)

    def with_(self, **kw) -> "DecodeConfig":
        return dataclasses.replace(self, **kw)


# The workloads that define this library's test and bench surface.
CONFIGS = {
    "tiny": DecodeConfig(
        name="tiny", batch=1, heads=16, q_len=1, num_shards=2, block_size=64,
        history=256, current=True, shuffle_table=False),
    "dsv3": DecodeConfig(
        name="dsv3", batch=32, heads=128, q_len=1, num_shards=8, block_size=64,
        history=4096),
    "mtp": DecodeConfig(
        name="mtp", batch=8, heads=128, q_len=2, num_shards=8, block_size=32,
        history=32768, current=True),
    "ragged": DecodeConfig(
        name="ragged", batch=64, heads=128, q_len=1, num_shards=16,
        block_size=32, ragged=(512, 65536), dtype="fp16", part_dtype="fp16",
        equal_logit_rows=(5, 21, 37, 53)),
    "verylong": DecodeConfig(
        name="verylong", batch=16, heads=128, q_len=1, num_shards=16,
        block_size=64, history=131072),
    # the very long context over an FP8 (E4M3) latent cache, kv_scale 2^-8
    # (stored values ~ N(0, 25.6): no saturation at 448)
    "verylong_fp8": DecodeConfig(
        name="verylong_fp8", batch=16, heads=128, q_len=1, num_shards=16,
        block_size=64, history=131072, kv_dtype="e4m3", kv_scale=2.0 ** -8),
}


@dataclasses.dataclass
class DecodeProblem:
    cfg: DecodeConfig
    seq_lens: np.ndarray          # [B] int32
    q_abs: np.ndarray             # uint16 bits
    q_pe: np.ndarray
    kv_cache: np.ndarray
    kv_cur: Optional[np.ndarray]
    W_UV: np.ndarray
    block_table: np.ndarray       # [B, max_blocks] int32

    @property
    def num_blocks(self) -> int:
        return self.kv_cache.shape[0]

    @property
    def max_blocks(self) -> int:
        return self.block_table.shape[1]

    @property
    def num_parts(self) -> int:
        return self.cfg.num_shards + (1 if self.kv_cur is not None else 0)


def _round_e4m3(x: np.ndarray) -> np.ndarray:
    """float32 -> E4M3 bytes (sign bit, 4 exponent bits with bias 7, 3 mantissa
    bits, exponent field 0 subnormal): nearest value, ties to the even code,
    magnitudes past 448 saturate to 448 (0x7E); -0 and values that round to
    zero give 0x00.  Below 2^-6 the codes are the subnormal steps m * 2^-9,
    m = rint(|x| * 2^9) (8 is the first normal code); above, the float32
    mantissa is rounded to 3 bits on the integer bits (a carry moves into the
    exponent) and the exponent rebased from 127 to 7."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32) & np.uint32(0x7FFFFFFF)
    a = u.view(np.float32)
    small = a < np.float32(2.0 ** -6)
    sub = np.rint(np.where(small, a, 0) * np.float32(512.0)).astype(np.int32)
    r = u + (np.uint32(0x7FFFF) + ((u >> np.uint32(20)) & np.uint32(1)))
    norm = (r >> np.uint32(20)).view(np.int32) - np.int32(120 << 3)
    code = np.where(small, sub, np.minimum(norm, 0x7E)).astype(np.uint8)
    neg = (x.view(np.uint32) >> np.uint32(31)).astype(np.uint8) & (code != 0)
    return code | (neg << np.uint8(7))


def round_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 -> storage bits, round to nearest even."""
    if dtype == "e4m3":
        return _round_e4m3(x)
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "fp16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = x.view(np.uint32)
        u = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
        return (u >> np.uint32(16)).astype(np.uint16)
    raise ValueError(f"unknown storage dtype {dtype!r}")


def _normal_bits(rng, shape, std, dtype, gain=1.0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint8 if dtype == "e4m3" else np.uint16)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        v = rng.standard_normal(hi - lo, dtype=np.float32)
        v *= np.float32(std * gain)
        out[lo:hi] = round_to_bits(v, dtype)
    return out.reshape(shape)


def history_lengths(cfg: DecodeConfig, rng) -> np.ndarray:
    if cfg.ragged:
        lo, hi = cfg.ragged
        u = rng.uniform(math.log(lo), math.log(hi), size=cfg.batch)
        return np.floor(np.exp(u)).astype(np.int32)
    return np.full(cfg.batch, cfg.history, dtype=np.int32)


def make_problem(cfg: DecodeConfig, seq_lens: Optional[np.ndarray] = None
                 ) -> DecodeProblem:
    """Draw one problem.  ``seq_lens`` overrides the configured lengths
    (used by edge-case tests: zero-length or one-token histories)."""
    rng = np.random.default_rng(cfg.seed)
    lens = history_lengths(cfg, rng)
    if seq_lens is not None:
        lens = np.asarray(seq_lens, dtype=np.int32).reshape(cfg.batch)
    B, q, H, bs = cfg.batch, cfg.q_len, cfg.heads, cfg.block_size

    q_abs = _normal_bits(rng, (B, q, H, D_LATENT), cfg.std, cfg.dtype, cfg.q_gain)
    q_pe = _normal_bits(rng, (B, q, H, D_ROPE), cfg.std, cfg.dtype, cfg.q_gain)
    for b in cfg.equal_logit_rows:
        if b < B:
            q_abs[b] = 0
            q_pe[b] = 0

    blocks_per_seq = [(int(L) + bs - 1) // bs for L in lens]
    num_blocks = max(1, sum(blocks_per_seq))
    # an e4m3 cache stores value / kv_scale
    kv_gain = 1.0 / cfg.kv_scale if cfg.cache_dtype == "e4m3" else 1.0
    kv_cache = _normal_bits(rng, (num_blocks, bs, D_QK), cfg.std, cfg.cache_dtype, kv_gain)
    kv_cur = (_normal_bits(rng, (B, q, D_QK), cfg.std, cfg.cache_dtype, kv_gain)
              if cfg.current else None)
    W_UV = _normal_bits(rng, (H, D_LATENT, D_V), cfg.std, cfg.dtype)

    perm = (rng.permutation(num_blocks) if cfg.shuffle_table
            else np.arange(num_blocks))
    max_blocks = max(1, max(blocks_per_seq))
    table = np.full((B, max_blocks), -1, dtype=np.int32)
    pos = 0
    for b, nb in enumerate(blocks_per_seq):
        table[b, :nb] = perm[pos:pos + nb]
        pos += nb
    return DecodeProblem(cfg=cfg, seq_lens=lens, q_abs=q_abs, q_pe=q_pe,
                         kv_cache=kv_cache, kv_cur=kv_cur, W_UV=W_UV,
                         block_table=table)


def kv_bytes(problem: DecodeProblem) -> int:
    """Bytes of latent KV one decode step must read (history + current)."""
    cur = problem.cfg.q_len if problem.kv_cur is not None else 0
    tokens = int(problem.seq_lens.astype(np.int64).sum()) + problem.cfg.batch * cur
    return tokens * D_QK * (1 if problem.cfg.cache_dtype == "e4m3" else 2)
