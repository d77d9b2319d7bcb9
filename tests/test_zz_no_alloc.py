"""mla_dcp_decode_partial_noalloc (the entry point whose split-shard scratch is
a fixed device array inside the library) against mla_dcp_decode_partial with
a workspace, on two calls in a row.  Kept in a file of its own, collected
last, so it runs both alone and after every other test in one process."""
import pytest
import torch

from mla_decode_attention_kv_gb300 import api, inputs

from gpu_util import DeviceProblem

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 24 << 20

CASES = {
    # one long shard cut into pieces for every CTA pair (split path)
    "split": inputs.DecodeConfig(name="na1", batch=1, heads=128, q_len=1, num_shards=1,
                                 block_size=64, history=20000, seed=201),
    # several sequences, shards of unequal length, CURRENT chunk, fp16
    "ragged": inputs.DecodeConfig(name="na2", batch=5, heads=128, q_len=2, num_shards=3,
                                  block_size=32, ragged=(100, 9000), current=True,
                                  dtype="fp16", part_dtype="fp16", seed=202),
}


def _outputs(dp, part_dtype):
    cfg = dp.prob.cfg
    P = cfg.num_shards + (1 if cfg.current else 0)
    o = torch.empty((cfg.batch, cfg.q_len, P, cfg.heads, 512), dtype=part_dtype, device=dp.dev)
    l = torch.empty((cfg.batch, cfg.q_len, P, cfg.heads), dtype=torch.float32, device=dp.dev)
    return o, l


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_workspace_entry_point_twice(name):
    dp = DeviceProblem(inputs.make_problem(CASES[name]))
    pdt = dp.part_dt
    ref_o, ref_l = dp.partial()                       # workspace entry point
    for _ in range(2):                                # two calls in a row on the shared array
        o, l = _outputs(dp, pdt)
        api.mla_dcp_decode_partial_noalloc(
            dp.q_abs, dp.q_pe, dp.cache, dp.table, dp.lens, dp.prob.cfg.num_shards,
            o_part=o, lse_part=l, kv_cur=dp.kv_cur, scale=dp.prob.cfg.scale, err_flag=dp.err)
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        assert torch.equal(o, ref_o) and torch.equal(l, ref_l)


def test_noalloc_rejects_what_the_array_cannot_hold():
    """FP32 partials need twice the scratch of 16-bit ones; the call is
    refused (MLA_ERR_BAD_SHAPE) exactly when that exceeds the 24 MiB array."""
    dp = DeviceProblem(inputs.make_problem(CASES["split"]))
    need_fp32 = api._ffi.lib().mla_dcp_decode_partial_workspace_size(1, 1, 1, 0)
    o, l = _outputs(dp, torch.float32)
    call = lambda: api.mla_dcp_decode_partial_noalloc(
        dp.q_abs, dp.q_pe, dp.cache, dp.table, dp.lens, 1, o_part=o, lse_part=l,
        scale=dp.prob.cfg.scale, err_flag=dp.err)
    if need_fp32 > SCRATCH_BYTES:
        with pytest.raises(api._ffi.MlaError) as e:
            call()
        assert e.value.status == 2
    else:
        call()
        torch.cuda.synchronize()
        ref_o, ref_l = dp.partial(part_dtype=torch.float32)
        assert torch.equal(o, ref_o) and torch.equal(l, ref_l)
