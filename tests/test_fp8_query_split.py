"""The two-term E4M3 form of the query that the E4M3-cache kernel multiplies
the cache by (emulated in gpu_util.split_query): its error stays within the
bound the header documents, |q - q'| <= 2^-8 |q| + 2^-17 max|q row|, on
queries of every magnitude, and it is exact where q itself has few bits."""
import numpy as np
import pytest

from mla_decode_attention_kv_gb300 import inputs
from oracle import mla_oracle as om

from gpu_util import split_query


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("gain", [1e-3, 1.0, 40.0])
def test_split_error_within_documented_bound(dtype, gain):
    cfg = inputs.DecodeConfig(name="qs", batch=3, heads=32, q_len=2, num_shards=1,
                              block_size=16, history=16, dtype=dtype, q_gain=gain, seed=77)
    prob = inputs.make_problem(cfg)
    qa, qp = split_query(prob)
    q = np.concatenate([om.to_f64(prob.q_abs, dtype), om.to_f64(prob.q_pe, dtype)], axis=-1)
    qs = np.concatenate([qa, qp], axis=-1)
    bound = 2.0 ** -8 * np.abs(q) + 2.0 ** -17 * np.abs(q).max(axis=-1, keepdims=True)
    assert np.all(np.abs(q - qs) <= bound)
    # the error is far below the bound on average (about 2^-11 relative)
    rel = np.abs(q - qs).sum() / np.abs(q).sum()
    assert rel < 2.0 ** -9


def test_split_exact_for_short_mantissas():
    """Values with at most 4 significant bits in the E4M3 range of the row
    scale are carried by hi alone: q' = q exactly."""
    cfg = inputs.DecodeConfig(name="qx", batch=1, heads=4, q_len=1, num_shards=1,
                              block_size=16, history=16, seed=78)
    prob = inputs.make_problem(cfg)
    vals = np.array([0.5, -0.75, 0.0625, 1.875, -0.25, 0.0], np.float32)
    row = np.resize(vals, 576).astype(np.float32)
    prob.q_abs[:] = inputs.round_to_bits(row[:512], "bf16")
    prob.q_pe[:] = inputs.round_to_bits(row[512:], "bf16")
    qa, qp = split_query(prob)
    assert np.array_equal(np.concatenate([qa, qp], axis=-1)[0, 0, 0], row.astype(np.float64))
