"""fp64 CPU oracle for decode-step MLA over a sequence-sharded latent KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this
module; only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.  It shares no code with the CUDA library: it reads
the raw storage bits produced by the seeded input generator and decodes them
itself.

What it computes, and where the pages define it
------------------------------------------------
Sources are the four web pages on this subject; each is cited by its title
and the section it falls in:

* [K3] "RTPLLM推理优化：K3芯片上MLA注意力的DCP与通算融合实践" (zwxr.cn news 254603)
* [PR] the vllm-ascend PR #16977 study page, "DCP decode: streams and V-up"
  (huashanblogllm.xyz, study-dcp-decode-streams-vup)
* [TP] the MLA multi-GPU TP configuration article (hncyxsy.com news 238223)

1. Cache entry.  Each token stores a 512-wide latent c_KV plus a 64-wide
   decoupled RoPE key k_R, 576 values shared by every query head
   ([TP] "物理矛盾" equation for c_t^KV and k_t^R; [TP] route A: 576 values,
   about 1.15 KB per token).
2. Paged history.  The HISTORY segment is read through ``block_table`` and
   ``block_size`` with ``cp_history_seq_len`` valid tokens ([PR] code block B,
   the HISTORY attention call).  Token t sits at
   kv_cache[block_table[t // bs], t % bs].
3. Absorbed scores.  The QK product is not taken on materialised per-head
   keys: the latent key and the RoPE key are handled separately
   ([K3] section 2.1), s_t = scale * (q_abs . c_t + q_pe . k_R_t), and the
   value is the latent itself, so attention yields a 512-wide latent output
   that the V-up turns into per-head values ([PR] glossary: MLA; code block A).
4. Sharding.  The KV sequence is split along the sequence into dcp_size
   shards; each shard yields a partial output and its log-sum-exp
   ([PR] glossary: DCP, LSE).  The pages give no boundary rule; the plain
   reading used here is contiguous, block-aligned shards of
   bs * ceil(L / (S * bs)) tokens, trailing shards possibly empty.
5. CURRENT segment.  The current chunk's keys are attended with a causal
   window mask (query i sees current tokens 0..i) and produce one more
   partial ([PR] code block C, ``sparse_mode=3``).  History is fully visible.
6. LSE combine.  Merging the partials by their LSEs equals one softmax over
   the whole sequence ([PR] section describing the two-segment decode step).
   Partials with no visible token (lse = -inf) carry weight zero.
7. V-up.  The combined output stays batch-major [T, H, 512]; each head is
   multiplied by W_UV[h] (512 x 128) and the result reshaped to [T, H*128]
   ([PR] code block A, ``_v_up_proj_batch_major``).

Readings where the pages are silent: natural-log LSE; scale 1/sqrt(192)
(the 128 + 64 head width of the explicit form); fp32-width LSE outputs;
all-empty rows give o = 0 and lse = -inf.

FP8 latent cache (a variant the pages only point towards: the compressed KV
direction of the Kthena x Mooncake page, sections 3.2 and 5.2).  The plain
reading taken: every cached value (history and CURRENT, latent and RoPE) is
one E4M3 byte e times one per-tensor scale kv_scale; the attention itself is
unchanged and runs on the decoded values e * kv_scale.  E4M3 is the OCP FP8
format: sign bit, 4 exponent bits with bias 7, 3 mantissa bits, exponent
field 0 subnormal, no infinities, 0x7F / 0xFF NaN.

Every function below is pinned by tests that do not reuse its arithmetic:
brute force on tiny inputs, the explicitly materialised per-head form, a
library attention routine, sharded-versus-unsharded equality and closed-form
special cases.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

D_LATENT = 512      # d_c, width of c_KV            ([TP] "物理矛盾")
D_ROPE = 64         # d_R, width of k_R             ([TP] "物理矛盾")
D_QK = D_LATENT + D_ROPE
D_V = 128           # per-head V width after V-up   ([PR] code block A)


# ---------------------------------------------------------------- decoding
def e4m3_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact float64 value of E4M3 bytes, from the format's definition:
    (-1)^s * 2^(e-7) * (1 + m/8) for e > 0, (-1)^s * 2^-6 * (m/8) for e = 0,
    NaN for e = 15, m = 7."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    s = np.where(b >> 7, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 7).astype(np.float64)
    mag = np.where(e == 0, 2.0 ** -6 * (m / 8.0), np.ldexp(1.0 + m / 8.0, e - 7))
    return np.where((e == 15) & (m == 7), np.nan, s * mag)


def to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of raw bf16 / fp16 / E4M3 storage bits."""
    if dtype == "e4m3":
        return e4m3_to_f64(bits)
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


# ---------------------------------------------------------------- step 2
def gather_history(kv_cache_bits, block_table_row, block_size: int, L: int):
    """Raw bits of history tokens 0..L-1 of one sequence, in sequence order.

    Token t is slot t % bs of physical block block_table[t // bs]."""
    out = np.empty((L, kv_cache_bits.shape[-1]), dtype=kv_cache_bits.dtype)
    for t in range(L):
        out[t] = kv_cache_bits[block_table_row[t // block_size], t % block_size]
    return out


def gather_history_fast(kv_cache_bits, block_table_row, block_size, L):
    """Same as ``gather_history`` one block at a time (used at large L)."""
    nb = (L + block_size - 1) // block_size
    if nb == 0:
        return np.empty((0, kv_cache_bits.shape[-1]), dtype=kv_cache_bits.dtype)
    pages = kv_cache_bits[np.asarray(block_table_row[:nb], dtype=np.int64)]
    return pages.reshape(nb * block_size, -1)[:L]


# ---------------------------------------------------------------- step 4
def shard_bounds(L: int, num_shards: int, block_size: int):
    """[start, end) of each history shard: contiguous, block aligned."""
    per = block_size * (-(-L // (num_shards * block_size))) if L > 0 else 0
    out = []
    for s in range(num_shards):
        lo = min(L, s * per)
        hi = min(L, (s + 1) * per)
        out.append((lo, hi))
    return out


# ---------------------------------------------------------------- step 3/5
def segment_attention(q_abs, q_pe, tokens, scale, visible=None):
    """Softmax attention of R query rows over N cached tokens (absorbed form).

    q_abs [R, 512], q_pe [R, 64], tokens [N, 576] (float64);
    visible: optional bool [R, N] mask.
    Returns o [R, 512] (softmax-weighted mean of c_KV) and lse [R]."""
    R = q_abs.shape[0]
    N = tokens.shape[0]
    o = np.zeros((R, D_LATENT))
    lse = np.full(R, -np.inf)
    if N == 0:
        return o, lse
    c = tokens[:, :D_LATENT]
    k_r = tokens[:, D_LATENT:]
    s = scale * (q_abs @ c.T + q_pe @ k_r.T)            # [R, N]
    if visible is None:
        visible = np.ones((R, N), dtype=bool)
    for r in range(R):
        v = visible[r]
        if not v.any():
            continue
        m = s[r, v].max()
        e = np.where(v, np.exp(s[r] - m), 0.0)
        l = e.sum()
        o[r] = (e @ c) / l
        lse[r] = m + math.log(l)
    return o, lse


def _queries(problem, b, i, heads):
    q_abs = to_f64(problem.q_abs[b, i, heads], problem.cfg.dtype)
    q_pe = to_f64(problem.q_pe[b, i, heads], problem.cfg.dtype)
    return q_abs, q_pe


def cache_values(bits, cfg):
    """Values of cached tokens: the storage bits decoded, times kv_scale for
    an E4M3 cache."""
    if cfg.cache_dtype == "e4m3":
        return e4m3_to_f64(bits) * cfg.kv_scale
    return to_f64(bits, cfg.cache_dtype)


def _history(problem, b):
    L = int(problem.seq_lens[b])
    bits = gather_history_fast(problem.kv_cache, problem.block_table[b],
                               problem.cfg.block_size, L)
    return cache_values(bits, problem.cfg)


def _current(problem, b):
    if problem.kv_cur is None:
        return np.zeros((0, D_QK))
    return cache_values(problem.kv_cur[b], problem.cfg)


def _all_heads(problem):
    return np.arange(problem.cfg.heads)


# ---------------------------------------------------------------- partials
def decode_partials(problem, batch: Optional[Sequence[int]] = None,
                    heads: Optional[Sequence[int]] = None, queries=None):
    """Per-shard (and CURRENT) partial outputs and LSEs.

    Returns o_part [nb, q, P, nh, 512] and lse_part [nb, q, P, nh] for the
    requested sequences and heads, P = num_shards (+1 for CURRENT, last).
    queries: optional (b, i, heads) -> (q_abs, q_pe) float64 rows used in
    place of the problem's stored queries."""
    cfg = problem.cfg
    batch = list(range(cfg.batch)) if batch is None else list(batch)
    heads = _all_heads(problem) if heads is None else np.asarray(heads)
    P = problem.num_parts
    o_part = np.zeros((len(batch), cfg.q_len, P, len(heads), D_LATENT))
    lse_part = np.full((len(batch), cfg.q_len, P, len(heads)), -np.inf)
    for bi, b in enumerate(batch):
        hist = _history(problem, b)
        cur = _current(problem, b)
        bounds = shard_bounds(hist.shape[0], cfg.num_shards, cfg.block_size)
        for i in range(cfg.q_len):
            qa, qp = (queries or (lambda b_, i_, h_: _queries(problem, b_, i_, h_)))(b, i, heads)
            for s, (lo, hi) in enumerate(bounds):
                o_part[bi, i, s], lse_part[bi, i, s] = segment_attention(
                    qa, qp, hist[lo:hi], cfg.scale)
            if problem.kv_cur is not None:
                vis = np.zeros((len(heads), cur.shape[0]), dtype=bool)
                vis[:, :i + 1] = True
                o_part[bi, i, P - 1], lse_part[bi, i, P - 1] = segment_attention(
                    qa, qp, cur, cfg.scale, vis)
    return o_part, lse_part


# ---------------------------------------------------------------- step 6
def lse_combine(o_part, lse_part, o_local=None, lse_local=None):
    """Merge partials along axis -3 of o_part / -2 of lse_part.

    o_part [..., P, H, 512], lse_part [..., P, H]; optional o_local
    [..., H, 512] / lse_local [..., H] is one more partial taken after the
    P stored ones.  Returns o [..., H, 512] and lse [..., H]."""
    o_part = np.asarray(o_part, dtype=np.float64)
    lse_part = np.asarray(lse_part, dtype=np.float64)
    if o_local is not None:
        o_part = np.concatenate([o_part, np.asarray(o_local, np.float64)[..., None, :, :]], axis=-3)
        lse_part = np.concatenate([lse_part, np.asarray(lse_local, np.float64)[..., None, :]], axis=-2)
    finite = np.isfinite(lse_part)
    m = np.where(finite, lse_part, -np.inf).max(axis=-2, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.where(finite, np.exp(lse_part - m_safe), 0.0)       # [..., P, H]
    tot = w.sum(axis=-2, keepdims=True)
    any_part = tot > 0
    lse = np.where(any_part, m_safe + np.log(np.where(any_part, tot, 1.0)), -np.inf)
    w = w / np.where(any_part, tot, 1.0)
    o = (w[..., None] * o_part).sum(axis=-3)
    return o, lse[..., 0, :]


# ---------------------------------------------------------------- step 7
def v_up(o_latent, W_UV):
    """Batch-major V-up: o_latent [T, H, 512] x W_UV [H, 512, 128] -> [T, H*128]."""
    o_latent = np.asarray(o_latent, dtype=np.float64)
    T, H, _ = o_latent.shape
    out = np.empty((T, H, D_V))
    for h in range(H):
        out[:, h, :] = o_latent[:, h, :] @ W_UV[h]
    return out.reshape(T, H * D_V)


# ---------------------------------------------------------------- reference
def decode_reference(problem, batch: Optional[Sequence[int]] = None,
                     heads: Optional[Sequence[int]] = None, with_vup: bool = True):
    """One softmax over every visible token, no sharding.

    Returns o_latent [nb, q, nh, 512], lse [nb, q, nh] and, if with_vup,
    out [nb*q, nh*128] using W_UV of the requested heads."""
    cfg = problem.cfg
    batch = list(range(cfg.batch)) if batch is None else list(batch)
    heads = _all_heads(problem) if heads is None else np.asarray(heads)
    o = np.zeros((len(batch), cfg.q_len, len(heads), D_LATENT))
    lse = np.full((len(batch), cfg.q_len, len(heads)), -np.inf)
    for bi, b in enumerate(batch):
        hist = _history(problem, b)
        cur = _current(problem, b)
        toks = np.concatenate([hist, cur], axis=0)
        for i in range(cfg.q_len):
            qa, qp = _queries(problem, b, i, heads)
            vis = np.ones((len(heads), toks.shape[0]), dtype=bool)
            vis[:, hist.shape[0] + i + 1:] = False
            o[bi, i], lse[bi, i] = segment_attention(qa, qp, toks, cfg.scale, vis)
    if not with_vup:
        return o, lse, None
    W = to_f64(problem.W_UV[heads], cfg.dtype)
    out = v_up(o.reshape(-1, len(heads), D_LATENT), W)
    return o, lse, out
