"""Benchmark of one decode step of MLA attention over a sharded latent KV cache.

A step is the whole hot path on one batch: the per-shard partial attention
kernel (with its split-shard merge), then the fused LSE combine + V-up
kernel.  The default workload is the very long context decode (batch 16,
128 heads, 131072 history tokens per sequence in 16 shards, 64-token pages
with a shuffled block table, bf16, 2.4 GB of latent KV per layer): the
largest single-GPU workload, and one of those at L >= 32K.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config NAME] [--extra NAMES|none]

Prints one JSON line (rank 0).  `value` is the KV-read rate in TB/s: the
latent-KV bytes every step must read, divided by the device time per step.
Inputs are larger than L2: each step uses the next of several layer caches
(and W_UV copies), so no step finds the previous step's KV in L2.  The
other workloads (--extra) are timed the same way, device-only, and reported
under "extra_workloads".

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload on this machine's host cores (the CPU baseline arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

# BLAS threads of the CPU oracle: every host core, stated in the output.
_CPU_THREADS = os.cpu_count() or 1
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CPU_THREADS))

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mla_decode_attention_kv_gb300 import inputs  # noqa: E402

METRIC = "MLA decode attn: KV-read TB/s, tokens/s, % of roofline at 1 GB300"
L2_BYTES = 129 * 2 ** 20
PROFILES = os.path.join(ROOT, "profiles")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

WORKLOAD_TEXT = {
    "dsv3": "DeepSeek-V3-shaped decode: batch 32, 128 heads, latent 512 + rope 64, 4096 KV "
            "tokens each, 8 shards, paged cache block 64 with a shuffled block table, bf16 "
            "N(0,1)*0.1, W_UV [128,512,128]",
    "mtp": "long context MTP: batch 8, 128 heads, 32768 history tokens in 8 shards + current "
           "chunk q_len 2 with a causal mask, bf16, block 32",
    "ragged": "ragged mixed batch: batch 64, 128 heads, seq_lens log-uniform in [512,65536], "
              "16 shards, block 32, random block table, fp16 cache",
    "verylong": "very long context: batch 16, 128 heads, 131072 KV tokens, 16 shards, bf16, "
                "fused combine + V-up",
    "verylong_fp8": "very long context over an FP8 (E4M3) latent cache, kv_scale 2^-8: batch 16, "
                    "128 heads, 131072 KV tokens, 16 shards, bf16 queries, fused combine + V-up",
    "tiny": "tiny: batch 1, 16 heads, 256 history tokens in 2 shards + 1 current token",
}


# ------------------------------------------------------------------ work model
def work_model(prob: inputs.DecodeProblem) -> dict:
    """Algorithmic bytes / flops of one step (each byte the method must move
    once; KV read once for all heads)."""
    cfg = prob.cfg
    B, q, H, P = cfg.batch, cfg.q_len, cfg.heads, prob.num_parts
    T = B * q
    esz = 2
    psz = 4 if cfg.part_dtype == "fp32" else 2
    kv = inputs.kv_bytes(prob)
    q_bytes = T * H * inputs.D_QK * esz
    opart = T * P * H * inputs.D_LATENT * psz
    lsep = T * P * H * 4
    w = H * inputs.D_LATENT * inputs.D_V * esz
    out = T * H * inputs.D_V * esz
    hist = prob.seq_lens.astype(np.int64)
    cur = q if prob.kv_cur is not None else 0
    # visible (query, key) pairs; each costs 2*H*(576 + 512) flops
    pairs = int(hist.sum()) * q + B * (q * (q + 1) // 2 if cur else 0)
    attn_flops = 2 * H * (inputs.D_QK + inputs.D_LATENT) * pairs
    vup_flops = 2 * T * H * inputs.D_LATENT * inputs.D_V
    return {
        "kv_bytes": kv,
        "partial_bytes": kv + q_bytes + opart + lsep,
        "partial_flops": attn_flops,
        "combine_vup_bytes": opart + lsep + w + out,
        "step_bytes": kv + q_bytes + 2 * (opart + lsep) + w + out,
        "step_flops": attn_flops + vup_flops,
        "query_tokens": T,
        "h2d_bytes": q_bytes + prob.block_table.nbytes + prob.seq_lens.nbytes
        + (prob.kv_cur.nbytes if prob.kv_cur is not None else 0),
        "d2h_bytes": out,
    }


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, \
            "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha(fp8: bool = False) -> str:
    """Hash of the partial kernel's sources (the 16-bit or the E4M3-cache
    kernel) with comments and blank lines removed, so that editing a comment
    does not disown the ncu counters."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_decode_attention_kv_gb300", "csrc")
    main = "partial_fp8.cu" if fp8 else "partial.cu"
    for name in (main, "partial_sched.cuh", "ptx.cuh", "common.cuh", "kernels.cuh"):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(code.encode())
    return h.hexdigest()[:16]


def profile_counters(config_name: str):
    """The committed ncu counters of the partial kernel on this workload
    (profiles/partial_kernel_<config>.json), if they were taken on the
    current kernel source; else None."""
    try:
        with open(os.path.join(PROFILES, f"partial_kernel_{config_name}.json")) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_sha") != kernel_source_sha(inputs.CONFIGS[config_name].kv_dtype == "e4m3"):
        return None
    return d


def traffic_from_profile(config_name: str):
    """DRAM bytes (read + write) per launch of the partial kernel, scaled to
    a full launch when the capture was taken on a smaller case; else None."""
    d = profile_counters(config_name)
    if not d:
        return None
    try:
        return float(d["dram_bytes_per_launch"])
    except (KeyError, TypeError, ValueError):
        return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append({"t": ts + frac, "sm": float(parts[2]), "max": float(parts[3]),
                             "power": float(parts[4]) if parts[4] not in ("[N/A]", "") else None,
                             "hw": parts[6], "hw_thermal": parts[7], "sw_thermal": parts[8],
                             "sw_power": parts[9]})
            except (ValueError, IndexError):
                continue
        os.unlink(self.path)
        return rows

    @staticmethod
    def summarize(rows, t0, t1):
        if not rows:
            return None
        inside = [r for r in rows if t0 - 0.06 <= r["t"] <= t1 + 0.06]
        used = inside or sorted(rows, key=lambda r: abs(r["t"] - (t0 + t1) / 2))[:3]
        reasons = set()
        for r in used:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in used),
                "sm_max_mhz": max(r["max"] for r in used),
                "reasons": sorted(reasons), "samples": len(used),
                "samples_in_timed_region": len(inside)}


# ------------------------------------------------------------------ our arm
def max_over_ranks(values, world: int, device="cpu"):
    """Each timing's maximum over the ranks: N replicas take as long as the
    slowest one.  Collective over the default process group when world > 1."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def replica_throughput(world: int, units_per_replica: float, ms_per_step: float) -> float:
    """Whole-job rate of N replicas: every rank's units over the slowest rank's
    time per step (weak scaling)."""
    return world * units_per_replica / (ms_per_step * 1e-3)


class DeviceWorkload:
    """One workload resident on the device: the seeded problem, `layers`
    rotated copies of the cache and W_UV (more bytes than L2 holds), and the
    output buffers of a step."""

    def __init__(self, name: str, dev, layers: int = 0):
        import torch
        from mla_decode_attention_kv_gb300 import api
        self.api = api
        self.name = name
        self.cfg = cfg = inputs.CONFIGS[name]
        self.prob = prob = inputs.make_problem(cfg)
        self.wm = work_model(prob)
        self.dev = dev
        self.dt = api.torch_dtype(cfg.dtype)
        pdt = api.torch_dtype(cfg.part_dtype)

        def t16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(self.dt)

        def t8(a):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(dev)

        self.fp8 = cfg.cache_dtype == "e4m3"
        self.kv_scale = cfg.kv_scale if self.fp8 else None
        tk = t8 if self.fp8 else t16
        self.q_abs, self.q_pe, W0 = t16(prob.q_abs), t16(prob.q_pe), t16(prob.W_UV)
        cache0 = tk(prob.kv_cache)
        self.kv_cur = tk(prob.kv_cur) if prob.kv_cur is not None else None
        self.table = torch.from_numpy(prob.block_table).to(dev)
        self.lens = torch.from_numpy(prob.seq_lens).to(dev)
        self.per_layer = cache0.numel() * cache0.element_size() + W0.numel() * 2
        self.layers = layers or max(2, math.ceil(4 * L2_BYTES / self.per_layer))
        self.caches = [cache0] + [cache0.clone() for _ in range(self.layers - 1)]
        self.Ws = [W0] + [W0.clone() for _ in range(self.layers - 1)]
        B, q, H, P = cfg.batch, cfg.q_len, cfg.heads, prob.num_parts
        self.o_part = torch.empty((B, q, P, H, 512), dtype=pdt, device=dev)
        self.lse_part = torch.empty((B, q, P, H), dtype=torch.float32, device=dev)
        self.out = torch.empty((B * q, H * 128), dtype=self.dt, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(self, i, stream, ev=None):
        li = i % self.layers
        if ev is not None:
            ev[0].record(stream)
        self.api.mla_dcp_decode_partial(
            self.q_abs, self.q_pe, self.caches[li], self.table, self.lens, self.cfg.num_shards,
            kv_cur=self.kv_cur, scale=self.cfg.scale, o_part=self.o_part,
            lse_part=self.lse_part, err_flag=self.err, stream=stream, kv_scale=self.kv_scale)
        if ev is not None:
            ev[1].record(stream)
        self.api.mla_lse_combine_vup(self.o_part, self.lse_part, self.Ws[li], out=self.out,
                                     err_flag=self.err, stream=stream)

    def time_device(self, steps, warmup, stream, barrier):
        """(ms of all `steps` steps, mean partial-kernel ms per step), device
        time by CUDA events on the launching stream.  The steps are timed
        twice: once as they run (the step time), then again with an event pair
        around every partial launch (its time, for the roofline).  An event
        recorded between the merge kernel and the fused V-up breaks the
        V-up's programmatic dependent launch, so the second loop's steps are
        a few microseconds slower and do not give the step time."""
        import torch
        for i in range(warmup):
            self.step(i, stream)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        e0.record(stream)
        for i in range(steps):
            self.step(warmup + i, stream)
        e1.record(stream)
        barrier()
        total_ms = e0.elapsed_time(e1)
        kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        barrier()
        for i in range(steps):
            self.step(warmup + i, stream, kev[i])
        barrier()
        partial_ms = sum(a.elapsed_time(b) for a, b in kev) / steps
        if self.err.item() != 0:
            raise RuntimeError(f"{self.name}: device error {self.err.item()} in the timed region")
        return total_ms, partial_ms

    def time_e2e(self, steps, warmup, stream, barrier):
        """ms of `steps` steps end to end through the public API: every step
        copies its inputs from pinned host memory and its output back.  Two
        sets of device input / output buffers alternate, and the copies run
        on a second stream, so step i's copies overlap the kernels of its
        neighbours (as a serving loop would run them).  Each direction has
        its own copy stream, so step i + 1's inputs are not queued behind
        step i's output copy (which waits for step i's kernels).  One
        cudaMemcpyAsync per direction and step; returns (ms, h2d bytes,
        d2h bytes)."""
        import torch
        prob, cfg, dev = self.prob, self.cfg, self.dev
        parts = [("q_abs", prob.q_abs.view(np.int16)), ("q_pe", prob.q_pe.view(np.int16)),
                 ("table", prob.block_table), ("lens", prob.seq_lens)]
        if prob.kv_cur is not None:
            parts.append(("kv_cur", prob.kv_cur))
        offs, off = {}, 0
        for name, a in parts:
            offs[name] = off
            off += (a.nbytes + 255) // 256 * 256
        h_in = torch.empty(off, dtype=torch.uint8).pin_memory()
        for name, a in parts:
            h_in[offs[name]:offs[name] + a.nbytes].copy_(
                torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1)))
        d_in = [torch.empty(off, dtype=torch.uint8, device=dev) for _ in range(2)]
        d_out = [torch.empty_like(self.out) for _ in range(2)]
        h_out = [torch.empty(self.out.shape, dtype=torch.int16).pin_memory() for _ in range(2)]
        likes = {"q_abs": self.q_abs, "q_pe": self.q_pe, "table": self.table, "lens": self.lens,
                 "kv_cur": self.kv_cur}

        def dview(k, name):
            like = likes[name]
            n = like.numel() * like.element_size()
            return d_in[k][offs[name]:offs[name] + n].view(like.dtype).view(like.shape)

        views = [{name: dview(k, name) for name, _ in parts} for k in range(2)]
        h2d = torch.cuda.Stream(device=dev)
        d2h = torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]      # inputs of buffer k landed
        ev_used = [torch.cuda.Event() for _ in range(2)]    # kernels done with buffer k
        ev_out = [torch.cuda.Event() for _ in range(2)]     # output k copied to the host
        for k in range(2):
            ev_used[k].record(stream)
            ev_out[k].record(stream)

        def e2e_step(i):
            k, li = i % 2, i % self.layers
            v = views[k]
            with torch.cuda.stream(h2d):
                h2d.wait_event(ev_used[k])
                d_in[k].copy_(h_in, non_blocking=True)
                ev_in[k].record(h2d)
            stream.wait_event(ev_in[k])
            stream.wait_event(ev_out[k])
            self.api.decode_step(v["q_abs"], v["q_pe"], self.caches[li], v["table"], v["lens"],
                                 self.Ws[li], cfg.num_shards, kv_cur=v.get("kv_cur"),
                                 scale=cfg.scale, o_part=self.o_part, lse_part=self.lse_part,
                                 out=d_out[k], err_flag=self.err, stream=stream,
                                 kv_scale=self.kv_scale)
            ev_used[k].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(ev_used[k])
                h_out[k].copy_(d_out[k].view(torch.int16), non_blocking=True)
                ev_out[k].record(d2h)

        for i in range(warmup):
            e2e_step(i)
        barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        h2d.wait_event(f0)
        d2h.wait_event(f0)
        for i in range(steps):
            e2e_step(warmup + i)
        stream.wait_event(ev_out[0])
        stream.wait_event(ev_out[1])
        f1.record(stream)
        barrier()
        if self.err.item() != 0:
            raise RuntimeError(f"{self.name}: device error {self.err.item()} in the e2e region")
        return f0.elapsed_time(f1), off, self.wm["d2h_bytes"]

    def roofline(self, partial_ms):
        """Roofline of the partial kernel (+ its merge) from its own
        CUDA-event time, against the measured peaks."""
        wm = self.wm
        peaks, peak_src = load_peaks()
        part_s = partial_ms * 1e-3
        hbm_ach = wm["partial_bytes"] / part_s / 1e9
        tc_ach = wm["partial_flops"] / part_s / 1e12
        hbm_frac = hbm_ach / peaks["hbm_gbs"]
        tc_frac = tc_ach / peaks["bf16_tflops"]
        if hbm_frac >= tc_frac:
            roof = {"bound": "hbm", "achieved": round(hbm_ach, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(hbm_frac, 4)}
        else:
            roof = {"bound": "tensor", "achieved": round(tc_ach, 1), "peak": peaks["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": round(tc_frac, 4)}
        roof["traffic"] = traffic_from_profile(self.name)
        roof["kernel"] = ("mla_partial_fp8_kernel" if self.fp8 else "mla_partial_kernel") + \
            " (+ mla_partial_merge_kernel)"
        roof["kernel_ms"] = round(partial_ms, 5)
        roof["alg_bytes_per_launch"] = wm["partial_bytes"]
        roof["alg_flops_per_launch"] = wm["partial_flops"]
        roof["tensor_frac"] = round(tc_frac, 4)
        roof["hbm_frac"] = round(hbm_frac, 4)
        roof["peak_source"] = ("measured (MEASURED_PEAKS.json, burst figures)"
                               if peak_src == "measured" else "fallback")
        return roof

    def step_roofline(self, ms_per_step):
        peaks, _ = load_peaks()
        wm = self.wm
        return max(wm["step_bytes"] / (peaks["hbm_gbs"] * 1e9),
                   wm["step_flops"] / (peaks["bf16_tflops"] * 1e12)) / (ms_per_step * 1e-3)

    def free(self):
        for k in ("caches", "Ws", "o_part", "lse_part", "out", "q_abs", "q_pe", "kv_cur"):
            setattr(self, k, None)


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from mla_decode_attention_kv_gb300 import build as mbuild
    from mla_decode_attention_kv_gb300 import _ffi

    mbuild.build()
    _ffi.lib()
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    wl = DeviceWorkload(args.config, dev, args.layers)
    sampler = ClockSampler(local_rank) if rank == 0 else None
    w0 = time.time()
    total_ms, partial_ms = wl.time_device(args.steps, args.warmup, stream, barrier)
    w1 = time.time()
    e2e_ms, h2d_bytes, d2h_bytes = wl.time_e2e(args.steps, args.warmup, stream, barrier)
    clocks = ClockSampler.summarize(sampler.stop(), w0, w1) if sampler else None
    total_ms, e2e_ms, partial_ms = max_over_ranks([total_ms, e2e_ms, partial_ms], world, dev)

    extras = {}
    names = [] if args.extra == "none" else [n for n in args.extra.split(",") if n]
    prob_for_cpu = wl.prob
    wm = wl.wm
    line_roof = wl.roofline(partial_ms)
    step_roof = wl.step_roofline(total_ms / args.steps)
    layers, per_layer = wl.layers, wl.per_layer
    wl.free()
    del wl
    torch.cuda.empty_cache()
    for name in names:
        if name == args.config:
            continue
        x = DeviceWorkload(name, dev)
        steps = max(20, min(args.steps, 200))
        t_ms, p_ms = x.time_device(steps, max(3, args.warmup), stream, barrier)
        t_ms, p_ms = max_over_ranks([t_ms, p_ms], world, dev)
        ms = t_ms / steps
        extras[name] = {
            "workload": WORKLOAD_TEXT[name],
            "value": round(replica_throughput(world, x.wm["kv_bytes"], ms) / 1e12, 4),
            "unit": "TB/s",
            "tokens_per_s": round(replica_throughput(world, x.wm["query_tokens"], ms), 1),
            "ms_per_step": round(ms, 5), "steps": steps,
            "step_roofline_frac": round(x.step_roofline(ms), 4),
            "roofline": x.roofline(p_ms),
        }
        x.free()
        del x
        torch.cuda.empty_cache()
    if rank != 0:
        return None

    ms_per_step = total_ms / args.steps
    kv_tbs = replica_throughput(world, wm["kv_bytes"], ms_per_step) / 1e12
    tok_s = replica_throughput(world, wm["query_tokens"], ms_per_step)
    e2e_tbs = replica_throughput(world, wm["kv_bytes"], e2e_ms / args.steps) / 1e12
    line = {
        "metric": METRIC,
        "value": round(kv_tbs, 4),
        "unit": "TB/s",
        "tokens_per_s": round(tok_s, 1),
        "step_roofline_frac": round(step_roof, 4),
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": inputs.CONFIGS[args.config].dtype,
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.config], "name": args.config,
                   "query_tokens_per_step": wm["query_tokens"],
                   "kv_bytes_per_step": wm["kv_bytes"],
                   "l2": f"inputs larger than L2: {layers} rotated layer caches + W_UV "
                         f"({layers * per_layer / 1e6:.0f} MB)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": line_roof,
        "e2e": {"value": round(e2e_tbs, 4), "unit": "TB/s",
                "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
                "copies": "double-buffered inputs/outputs, copies on one stream per direction"},
        # per step: partial kernel, its split-shard merge kernel, fused combine + V-up;
        # the same three per step in the e2e leg (which also runs the copies)
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
    }
    if extras:
        line["extra_workloads"] = extras
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(prob_for_cpu, args.cpu_seconds)
    return line


# ------------------------------------------------------------------ CPU oracle
def _oracle_sample(prob, batch):
    from oracle import mla_oracle as om
    om.decode_reference(prob, batch=batch)


def cpu_baseline(prob, budget_s: float):
    """The oracle as it stands on the host cores, on a bounded sample of the
    workload (whole sequences, all heads), scaled to KV-read TB/s."""
    cfg = prob.cfg
    t0 = time.perf_counter()
    _oracle_sample(prob, [0])
    one = time.perf_counter() - t0
    n = int(max(1, min(cfg.batch, budget_s / max(one, 1e-3))))
    batch = list(range(n))
    t0 = time.perf_counter()
    _oracle_sample(prob, batch)
    dt = time.perf_counter() - t0
    kv = int(prob.seq_lens[:n].astype(np.int64).sum()) * inputs.D_QK * 2
    return {"value": round(kv / dt / 1e12, 9), "unit": "TB/s", "cores": _CPU_THREADS,
            "kind": "oracle",
            "sample": f"{n} of {cfg.batch} sequences (all {cfg.heads} heads, full history) "
                      f"in {dt:.1f} s, fp64 numpy oracle, {_CPU_THREADS} BLAS threads",
            "value_1thread": _cpu_one_thread(cfg.name, budget_s / 3)}


def _cpu_one_thread(config: str, budget_s: float):
    """The same oracle sample with BLAS limited to one thread (a child process,
    since the thread count is fixed when numpy loads); None if it fails."""
    env = dict(os.environ)
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = "1"
    try:
        res = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-probe", config,
                              str(budget_s)], env=env, capture_output=True, text=True,
                             timeout=max(60.0, 6 * budget_s))
        return json.loads(res.stdout.strip().splitlines()[-1])["value"]
    except Exception:
        return None


def _cpu_probe(config: str, budget_s: float):
    """Child of _cpu_one_thread: time the oracle on whole sequences of `config`."""
    prob = inputs.make_problem(inputs.CONFIGS[config])
    t0 = time.perf_counter()
    _oracle_sample(prob, [0])
    one = time.perf_counter() - t0
    n = int(max(1, min(prob.cfg.batch, budget_s / max(one, 1e-3))))
    t0 = time.perf_counter()
    _oracle_sample(prob, list(range(n)))
    dt = time.perf_counter() - t0
    kv = int(prob.seq_lens[:n].astype(np.int64).sum()) * inputs.D_QK * 2
    print(json.dumps({"value": round(kv / dt / 1e12, 9)}))


def run_reference(args, rank, world):
    """CPU baseline arm: the oracle timed as it stands on the host cores."""
    if rank != 0:
        return None
    cfg = inputs.CONFIGS[args.config]
    prob = inputs.make_problem(cfg)
    per_seq = int(prob.seq_lens[0]) * inputs.D_QK * 2
    for i in range(args.warmup):
        _oracle_sample(prob, [i % cfg.batch])
    times = []
    kv = 0
    for i in range(args.steps):
        b = (args.warmup + i) % cfg.batch
        t0 = time.perf_counter()
        _oracle_sample(prob, [b])
        times.append(time.perf_counter() - t0)
        kv += int(prob.seq_lens[b]) * inputs.D_QK * 2
    total = sum(times)
    value = kv / total / 1e12
    sample = (f"each step: 1 of {cfg.batch} sequences (all {cfg.heads} heads, "
              f"{int(prob.seq_lens[0])} history tokens, {per_seq / 1e6:.1f} MB KV)")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 9), "unit": "TB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.config], "name": args.config,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 9), "unit": "TB/s", "cores": _CPU_THREADS,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 9), "unit": "TB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=sorted(inputs.CONFIGS), default="verylong")
    ap.add_argument("--extra", default="dsv3,mtp,ragged,verylong_fp8",
                    help="other workloads timed device-only (comma list, or none)")
    ap.add_argument("--layers", type=int, default=0, help="layer caches rotated (0 = auto)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="budget of the CPU-oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-probe", nargs=2, metavar=("CONFIG", "SECONDS"), help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_probe:
        _cpu_probe(args.cpu_probe[0], float(args.cpu_probe[1]))
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
        line = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
