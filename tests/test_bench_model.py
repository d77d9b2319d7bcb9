"""bench.py's algorithmic work model (the numerators of every roofline
fraction and of the KV-read TB/s) against the per-workload figures of the
scope table: KV bytes (1152 B per cached token at bf16/fp16), flops
(2 * H * (576 + 512) per visible query/key pair) and the step's total
algorithmic bytes (KV + queries + the partials written and read back + W_UV +
the output), as tabulated there to 0.1 MB / 0.1 GFLOP.  CPU only."""
import numpy as np
import pytest

import bench
from mla_decode_attention_kv_gb300 import inputs


def _light_problem(cfg):
    """The workload's history lengths and table shape (the generator's first
    draw), without the cache and query arrays the work model does not read."""
    lens = inputs.history_lengths(cfg, np.random.default_rng(cfg.seed))
    bs = cfg.block_size
    max_blocks = max(1, max((int(L) + bs - 1) // bs for L in lens))
    z = np.zeros(1, np.uint16)
    cur = np.zeros((cfg.batch, cfg.q_len, inputs.D_QK), np.uint16) if cfg.current else None
    return inputs.DecodeProblem(cfg=cfg, seq_lens=lens, q_abs=z, q_pe=z, kv_cache=z, kv_cur=cur,
                                W_UV=z, block_table=np.zeros((cfg.batch, max_blocks), np.int32))


# workload: (KV MB, GFLOP, total algorithmic MB, relative tolerance)
TABLE = {
    "tiny": (0.30, 0.01, 2.5, 0.05),
    "dsv3": (151.0, 36.5, 240.9, 0.002),
    "mtp": (302.0, 146.0, 359.6, 0.002),
    "verylong": (2416.0, 584.0, 2500.0, 0.002),
    # the ragged lengths are drawn, so its row is approximate (mean L ~ 13.4K)
    "ragged": (988.0, 239.0, 1290.0, 0.03),
}


def test_light_problem_is_the_generated_one():
    cfg = inputs.CONFIGS["tiny"]
    full, light = inputs.make_problem(cfg), _light_problem(cfg)
    assert np.array_equal(full.seq_lens, light.seq_lens)
    assert full.block_table.shape == light.block_table.shape
    assert bench.work_model(full) == bench.work_model(light)


@pytest.mark.parametrize("name", list(TABLE))
def test_work_model_matches_scope_table(name):
    kv_mb, gflop, total_mb, rel = TABLE[name]
    wm = bench.work_model(_light_problem(inputs.CONFIGS[name]))
    assert wm["kv_bytes"] / 1e6 == pytest.approx(kv_mb, rel=rel, abs=0.01)
    assert wm["partial_flops"] / 1e9 == pytest.approx(gflop, rel=rel, abs=0.01)
    assert wm["step_bytes"] / 1e6 == pytest.approx(total_mb, rel=rel, abs=0.05)


def test_work_model_parts_add_up():
    """The step's bytes are the partial kernel's plus the combine/V-up's, with
    the partials counted once written and once read."""
    wm = bench.work_model(_light_problem(inputs.CONFIGS["dsv3"]))
    assert wm["step_bytes"] == wm["partial_bytes"] + wm["combine_vup_bytes"]
    assert wm["step_flops"] > wm["partial_flops"]
