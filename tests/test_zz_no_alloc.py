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


def test_noalloc_fp32_partials():
    """FP32 partials need twice the scratch of 16-bit ones.  When that exceeds
    the 24 MiB array (a GPU with more than 47 resident CTA pairs) the call
    takes whole shards with no scratch, so it matches the workspace-free
    entry point; otherwise the workspace one.  Two calls in a row."""
    dp = DeviceProblem(inputs.make_problem(CASES["split"]))
    need_fp32 = api._ffi.lib().mla_dcp_decode_partial_workspace_size(1, 1, 1, 0)
    ws = None if need_fp32 > SCRATCH_BYTES else "default"
    ref_o, ref_l = dp.partial(part_dtype=torch.float32, workspace=ws)
    for _ in range(2):
        o, l = _outputs(dp, torch.float32)
        api.mla_dcp_decode_partial_noalloc(
            dp.q_abs, dp.q_pe, dp.cache, dp.table, dp.lens, 1, o_part=o, lse_part=l,
            scale=dp.prob.cfg.scale, err_flag=dp.err)
        torch.cuda.synchronize()
        assert dp.err.item() == 0
        assert torch.equal(o, ref_o) and torch.equal(l, ref_l)


def test_noalloc_checks_arguments_like_the_workspace_entry_point():
    """Bad arguments get the same status from both entry points."""
    dp = DeviceProblem(inputs.make_problem(CASES["ragged"]))
    o, l = _outputs(dp, dp.part_dt)
    for kw in (dict(num_shards=65), dict(scale=-1.0)):
        args = dict(num_shards=dp.prob.cfg.num_shards, scale=dp.prob.cfg.scale)
        args.update(kw)
        with pytest.raises(api._ffi.MlaError) as e1:
            api.mla_dcp_decode_partial(dp.q_abs, dp.q_pe, dp.cache, dp.table, dp.lens,
                                       args["num_shards"], kv_cur=dp.kv_cur, scale=args["scale"],
                                       o_part=o, lse_part=l)
        with pytest.raises(api._ffi.MlaError) as e2:
            api.mla_dcp_decode_partial_noalloc(dp.q_abs, dp.q_pe, dp.cache, dp.table, dp.lens,
                                               args["num_shards"], o_part=o, lse_part=l,
                                               kv_cur=dp.kv_cur, scale=args["scale"])
        assert e1.value.status == e2.value.status
