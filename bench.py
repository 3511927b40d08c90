"""Benchmark of MLA chunked prefill over a paged packed-latent KV cache.

One step = one whole mla_prefill_ctx call (plan, fused gather + up-projection +
attention kernel, merge of the KV splits) for one layer of one workload, with
every input already resident in HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config reloc_256k]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

The default workload is the largest one that fits a GPU: 16 relocated
documents of 16K tokens (256K cached) and 4K new tokens, 128 heads.  The same
line carries `target_128k`: the 128K-token FP8 cache with 4K new tokens, timed
the same way, with its own fused-kernel roofline.

Multi-GPU: the path is run as independent replicas (one process per GPU, the
same workload each; no collective on the data path), so scaling is weak and
`value` is the work of all ranks divided by the slowest rank's time.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "MLA chunked-prefill TFLOP/s & prefill tok/s at 1 GB300; % of dense BF16 peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20          # > 2x the 129 MB L2


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def gpu_delay(ms: float = 1.0) -> None:
    """A spin of about `ms` on the GPU, queued after the L2 flush and before a
    start event: the host then queues the event and the timed launches while
    the GPU still spins, so no host time falls between the events."""
    import torch
    torch.cuda._sleep(int(ms * 2.0e6))   # clock cycles, ~2 GHz


def max_over_ranks(value: float, world: int, device="cpu") -> float:
    """The largest value over the ranks (replicas: the job ends when its
    slowest rank does); the process group must exist when world > 1."""
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(units_per_rank_step: float, steps: int, world: int, max_total_ms: float) -> float:
    """Whole-job throughput of `world` replicas: every rank's units over the
    slowest rank's time, per second."""
    return units_per_rank_step * steps * world / (max_total_ms / 1e3)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), with the architecture."""
    import platform
    name = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        fields = dict(line.split(":", 1) for line in out.splitlines() if ":" in line)
        fields = {k.strip(): v.strip() for k, v in fields.items()}
        name = fields.get("Model name", "")
        if fields.get("Vendor ID") and fields["Vendor ID"] not in name:
            name = f"{fields['Vendor ID']} {name}".strip()
    except (OSError, subprocess.SubprocessError, ValueError):
        name = ""
    if not name:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith(("model name", "cpu part")):
                        name = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return f"{name or 'unknown'} ({platform.machine()})"


def executed_flops(wl) -> float:
    """Tensor-core FLOPs the fused kernel issues for one call, as its planner
    cuts the work: per (piece, head) every producer pass up-projects 256
    tokens (M = 256 per CTA pair, the last pass's second half included), and
    every consumer pair runs M = 256 (its two query tiles) x N = 128 score and
    PV MMAs over as many 128-key tiles as the longer of its two tiles needs
    (masked columns of the causal diagonal and of the piece edges included).
    The algorithmic count (wl.algorithmic_flops) takes each unmasked pair once."""
    H = wl.num_heads
    max_keys = max(wl.chunk, 16384)
    f = 0.0
    for r in range(wl.num_reqs):
        C, E = int(wl.ctx_lens[r]), int(wl.ext_lens[r])
        if E == 0:
            continue
        if wl.segments is None:
            ranges = [(c0, min(c0 + wl.chunk, C), 0) for c0 in range(0, C, wl.chunk)]
        else:
            ranges = []
            for req, start, length, off in wl.segments.tolist():
                if req == r:
                    ranges += [(c0, min(c0 + wl.chunk, start + length), off)
                               for c0 in range(start, start + length, wl.chunk)]
        ranges.append((C, C + E, 0))
        ranges.sort(key=lambda x: x[0])
        pieces = []
        for k0, k1, off in ranges:
            if k1 <= k0:
                continue
            if pieces and pieces[-1][2] == off and pieces[-1][1] == k0 and pieces[-1][1] - pieces[-1][0] < max_keys:
                pieces[-1][1] = k1
            else:
                pieces.append([k0, k1, off])
        n_cons = (E + 127) // 128
        for k0, k1, _ in pieces:
            t0 = k0 & ~63
            n_tiles = (k1 - t0 + 127) // 128
            f += H * ((n_tiles + 1) // 2) * 256 * 2.0 * 512 * 256

            def tiles(ci):
                q0 = 128 * ci
                nq = min(128, E - q0)
                if nq <= 0:
                    return 0
                ke = min(k1, C + q0 + nq)
                return 0 if ke <= k0 else (ke - t0 + 127) // 128

            for k in range((n_cons + 1) // 2):
                n = max(tiles(2 * k), tiles(2 * k + 1) if 2 * k + 1 < n_cons else 0)
                f += H * n * 256 * 128 * 2.0 * (192 + 128)
    return f


def workload_config(wl, extra=None):
    c = {"workload": wl.name, "heads": wl.num_heads, "requests": wl.num_reqs,
         "context_tokens": int(wl.ctx_lens.sum()), "extend_tokens": int(wl.ext_lens.sum()),
         "chunk": wl.chunk, "kv_dtype": wl.kv_dtype,
         "segments": 0 if wl.segments is None else int(len(wl.segments)),
         "d_c": 512, "d_rope": 64, "d_nope": 128, "d_v": 128, "block": 64,
         "algorithmic_flops_per_step": wl.algorithmic_flops()}
    if extra:
        c.update(extra)
    return c


# ---------------------------------------------------------------- CPU oracle timing

def oracle_sample(wl, n_heads):
    """Runs the oracle for the first n_heads heads, all query rows; returns
    (seconds, algorithmic flops of that sample)."""
    from oracle import mla_oracle
    heads = list(range(n_heads))
    t0 = time.perf_counter()
    mla_oracle.mla_prefill(**mla_oracle.workload_args(wl), heads=heads)
    dt = time.perf_counter() - t0
    return dt, wl.algorithmic_flops() * n_heads / wl.num_heads


def cpu_baseline(wl, budget_s=15.0):
    """The oracle as it stands on the host cores, on a bounded sample of the
    workload: whole heads (all rows, all keys) until ~budget_s of work."""
    dt1, f1 = oracle_sample(wl, 1)
    n = max(1, min(wl.num_heads, int(budget_s / max(dt1, 1e-3))))
    if n > 1:
        dt, f = oracle_sample(wl, n)
    else:
        dt, f = dt1, f1
    return {"value": f / dt / 1e12, "unit": UNIT, "cores": host_cores(), "cpu": cpu_model(), "kind": "oracle",
            "sample": f"{n} of {wl.num_heads} heads x all {wl.total_q} query rows x all keys of "
                      f"{wl.name} (numpy fp32, {dt:.1f} s)"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from mla_prefix_cache_gb300 import workload
    wl = workload.by_name(args.config)
    dt1, _ = oracle_sample(wl, 1)
    per_step = min(args.ref_step_s, 150.0 / (args.steps + args.warmup))   # whole run within a few minutes
    n = max(1, min(wl.num_heads, int(per_step / max(dt1, 1e-3))))
    for _ in range(args.warmup):
        oracle_sample(wl, n)
    times, flops = [], 0.0
    for _ in range(args.steps):
        dt, f = oracle_sample(wl, n)
        times.append(dt)
        flops = f
    total = sum(times)
    value = flops * len(times) / total / 1e12
    sample = f"{n} of {wl.num_heads} heads x all {wl.total_q} query rows x all keys of {wl.name} per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded)", "config": workload_config(wl),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(), "cpu": cpu_model(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 20 ms; `stop(t0, t1)` keeps
    the samples whose own timestamps fall inside the timed region [t0, t1]
    (wall clock), widened by one sampling period."""
    FIELDS = ("timestamp,index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_S = 0.02

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.proc = None
        self.path = os.path.join("/tmp", f"mla_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", str(int(self.PERIOD_S * 1000))], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        time.sleep(0.3)   # let the sampler come up before the timed region starts

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        time.sleep(2 * self.PERIOD_S)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        import datetime
        lo = datetime.datetime.fromtimestamp(t0 - self.PERIOD_S)
        hi = datetime.datetime.fromtimestamp(t1 + self.PERIOD_S)
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 11:
                    continue
                if self.uuid and parts[2] != self.uuid:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                except ValueError:
                    continue
                if lo <= ts <= hi:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        mx = [float(r[4]) for r in rows if r[4].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[7 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "period_ms": int(self.PERIOD_S * 1000)}


# ---------------------------------------------------------------- our arm

def fused_kernel_name():
    """The fused kernel mla_prefill_ctx launches."""
    return "fused2_prefill_kernel"


KERNEL_SOURCES = {
    "fused": ("fused2.cu", "fused_common.cuh", "ptx.cuh", "internal.h"),
    "absorbed": ("absorb.cu", "absorb.h", "ptx.cuh", "internal.h"),
}


def kernel_sha(path="fused"):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[path]:
        with open(os.path.join(ROOT, "mla_prefix_cache_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload_name, path="fused"):
    """DRAM bytes per launch of the timed kernel from a committed ncu summary,
    valid only while the kernel source is the one that was profiled."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if path not in KERNEL_SOURCES or not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload_name if path == "fused" else f"{workload_name}/{path}")
    kernel = fused_kernel_name() if path == "fused" else "absorb_attn_kernel"
    if not e or e.get("kernel_sha") != kernel_sha(path) or e.get("kernel") != kernel:
        return None
    return e.get("dram_bytes_per_launch")


def hbm_kernels(dev, flush, peak_gbs, reps=10):
    """HBM rooflines of the bandwidth-bound entry points, each timed alone with
    CUDA events (L2 flushed before every launch, median of `reps`), on inputs
    shaped like the long-context workloads: a 128K-token paged gather (BF16
    and FP8 rows), merge_attn_states of 4096 tokens x 128 heads of fp32
    states, RoPE relocation of a [4096, 128, 192] bf16 query in place, and
    the block store's content hash of all 2304 bf16 blocks of the pool and
    byte comparison of 1152 block pairs.
    Bytes are algorithmic (each byte the operation must read or write once)."""
    import torch
    from mla_prefix_cache_gb300 import api

    g = torch.Generator(device=dev)
    g.manual_seed(7)
    n_tok, n_blocks = 131072, 2304
    perm = torch.randperm(n_blocks, generator=g, device=dev)[: n_tok // 64].to(torch.int32)
    bf16_cache = torch.randn((n_blocks, 64, 576), generator=g, device=dev).to(torch.bfloat16)
    fp8_cache = torch.randint(0, 256, (n_blocks, 64, 640), generator=g, device=dev, dtype=torch.uint8)
    fp8_cache[..., 512:] = bf16_cache[..., 512:].contiguous().view(torch.uint8)
    dst = torch.empty((n_tok, 576), dtype=torch.bfloat16, device=dev)
    rows = 4096 * 128
    oa = torch.randn((rows, 128), generator=g, device=dev)
    ob = torch.randn((rows, 128), generator=g, device=dev)
    la = torch.randn((rows,), generator=g, device=dev)
    lb = torch.randn((rows,), generator=g, device=dev)
    om, lm = torch.empty_like(oa), torch.empty_like(la)
    q = torch.randn((4096, 128, 192), generator=g, device=dev).to(torch.bfloat16)
    pos = torch.arange(4096, dtype=torch.int32, device=dev) + 262144
    all_ids = torch.randperm(n_blocks, generator=g, device=dev).to(torch.int32)
    pair_a, pair_b = all_ids[: n_blocks // 2].contiguous(), all_ids[n_blocks // 2:].contiguous()

    cases = {
        "gather_bf16": (lambda: api.gather_latent(bf16_cache, perm, 0, n_tok, dst=dst),
                        n_tok * (1152 + 1152) + 4 * (n_tok // 64)),
        "gather_fp8": (lambda: api.gather_latent(fp8_cache, perm, 0, n_tok, kv_scale=0.05, dst=dst),
                       n_tok * (640 + 1152) + 4 * (n_tok // 64)),
        "merge_states": (lambda: api.merge_states(oa, la, ob, lb, out=om, lse=lm),
                         rows * (2 * (128 * 4 + 4) + (128 * 4 + 4))),
        "rope_relocate": (lambda: api.rope_relocate(q, pos, 65536, 10000.0, y=q),
                          4096 * 128 * 64 * 2 * 2 + 4096 * 4),
        "block_hash": (lambda: api.block_hash(bf16_cache, all_ids), n_blocks * (64 * 1152 + 4 + 8)),
        "block_compare": (lambda: api.block_compare(bf16_cache, pair_a, pair_b),
                          (n_blocks // 2) * (2 * 64 * 1152 + 8 + 4)),
    }
    stream = torch.cuda.current_stream(dev)
    res = {}
    for name, (fn, nbytes) in cases.items():
        for _ in range(3):
            fn()
        ms = []
        for _ in range(reps):
            flush.zero_()
            gpu_delay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms.append(e0.elapsed_time(e1))
        t = statistics.median(ms)
        gbs = nbytes / (t / 1e3) / 1e9
        res[name] = {"achieved": gbs, "peak": peak_gbs, "unit": "GB/s", "frac": gbs / peak_gbs,
                     "bytes": int(nbytes), "us": t * 1e3}
    return res


def absorbed_compare(dev, flush, peak, source, reps=10, config="short_ext_32k", fp8_scores=False):
    """A short-extend workload (default: 128 heads, 32K cached + 64 new
    tokens) through the up-projected and the absorbed entry points (with
    fp8_scores, the FP8-score one: FP8 caches) on the same inputs: median
    CUDA-event time of a whole call (L2 flushed before each), and the latent
    attention kernel's tensor-core roofline."""
    import torch
    from mla_prefix_cache_gb300 import api, workload

    wl = workload.by_name(config)
    mode = "fp8" if fp8_scores else True
    dw = api.DeviceWorkload(wl, dev)
    T_q, H = wl.total_q, wl.num_heads
    out = torch.empty((T_q, H, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((T_q, H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    res = {}
    for absorbed in (False, mode):
        if absorbed:
            nbytes = api.absorbed_workspace_size(wl.seq_lens, wl.cu_q, H, wl.segments, wl.chunk,
                                                 fp8_scores=fp8_scores)
        else:
            nbytes = api.prefill_workspace_size(wl.seq_lens, wl.cu_q, H, wl.segments, wl.chunk)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        for _ in range(3):
            flush.zero_()
            dw.run(out=out, lse=lse, workspace=ws, absorbed=absorbed)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for k in range(reps):
            flush.zero_()
            gpu_delay()
            api.set_kernel_events(*kev[k])
            ev[k][0].record(stream)
            dw.run(out=out, lse=lse, workspace=ws, absorbed=absorbed)
            ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        api.set_kernel_events(None, None)
        if api.device_error(ws) != 0:
            raise RuntimeError("device error word set in the absorbed comparison")
        res[absorbed] = (float(statistics.median([a.elapsed_time(b) for a, b in ev])),
                         float(statistics.median([a.elapsed_time(b) for a, b in kev])))
        del ws
    (ms_f, _), (ms_a, kms_a) = res[False], res[mode]
    att = wl.absorbed_attention_flops()
    achieved = att / (kms_a / 1e3) / 1e12
    return {"workload": workload_config(wl), "ms_fused": ms_f, "ms_absorbed": ms_a, "speedup": ms_f / ms_a,
            "prefill_tok_s_absorbed": T_q / (ms_a / 1e3), "prefill_tok_s_fused": T_q / (ms_f / 1e3),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak,
                         "traffic": None if fp8_scores else measured_traffic(wl.name, "absorbed"),
                         "kernel": "absorb_attn_kernel",
                         "kernel_ms": kms_a, "peak_source": f"bf16_tflops (burst) of {source} peaks",
                         "note": "tensor-core FLOPs of the latent attention, 2 (576 + 512) per visible "
                                 "query-key-head, / its event time" + ("; the 512-wide score part on E4M3 "
                                 "tensor cores, counted at the bf16 peak" if fp8_scores else "")},
            "path": "absorbed_fp8" if fp8_scores else "absorbed"}


def fp8w_compare(dev, flush, peak, source, reps=5, config="fp8_128k"):
    """The FP8 cache workload through mla_prefill_ctx (bf16 up-projection of
    the dequantised rows) and mla_prefill_ctx_fp8w (E4M3 rows as stored times
    an E4M3 copy of kv_b_proj on the FP8 tensor cores): median CUDA-event time
    of a whole call (L2 flushed before each) and of the fused kernel; the
    E4M3 copy of kv_b_proj is made once, outside the timing (a model constant)."""
    import torch
    from mla_prefix_cache_gb300 import api, workload

    wl = workload.by_name(config)
    dw = api.DeviceWorkload(wl, dev)
    T_q, H = wl.total_q, wl.num_heads
    out = torch.empty((T_q, H, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((T_q, H), dtype=torch.float32, device=dev)
    w_scale = api.kv_b_proj_absmax(dw.kv_b_proj) / 448.0
    w8 = api.kv_b_proj_to_e4m3(dw.kv_b_proj, w_scale)
    ws = torch.empty(api.prefill_workspace_size(wl.seq_lens, wl.cu_q, H, wl.segments, wl.chunk),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    res = {}
    for fp8w in (False, True):
        kw = dict(kv_b_proj_e4m3=w8, w_scale=w_scale) if fp8w else {}
        for _ in range(3):
            flush.zero_()
            dw.run(out=out, lse=lse, workspace=ws, **kw)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for k in range(reps):
            flush.zero_()
            torch.cuda.synchronize(dev)
            api.set_kernel_events(*kev[k])
            ev[k][0].record(stream)
            dw.run(out=out, lse=lse, workspace=ws, **kw)
            ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        api.set_kernel_events(None, None)
        if api.device_error(ws) != 0:
            raise RuntimeError("device error word set in the FP8 up-projection comparison")
        res[fp8w] = (float(statistics.median([a.elapsed_time(b) for a, b in ev])),
                     float(statistics.median([a.elapsed_time(b) for a, b in kev])))
    (ms_b, kms_b), (ms_8, kms_8) = res[False], res[True]
    flops = wl.algorithmic_flops()
    del ws, w8
    torch.cuda.empty_cache()
    return {"workload": config, "ms_bf16_proj": ms_b, "ms_fp8_proj": ms_8, "speedup": ms_b / ms_8,
            "kernel_ms_bf16_proj": kms_b, "kernel_ms_fp8_proj": kms_8,
            "tflops_fp8_proj": flops / (ms_8 / 1e3) / 1e12,
            "kernel_frac_fp8_proj": flops / (kms_8 / 1e3) / 1e12 / peak,
            "note": "algorithmic FLOPs over the kernel time against the bf16 peak; the up-projection "
                    "(9% of the FLOPs here) runs on E4M3 tensor cores"}


def auto_compare(dev, flush, reps=5, config="mixed_32k"):
    """Per-request dispatch against the up-projected path alone, on a mixed
    batch of long and short requests: median CUDA-event time of a whole call,
    L2 flushed before each."""
    import torch
    from mla_prefix_cache_gb300 import api, workload

    wl = workload.by_name(config)
    dw = api.DeviceWorkload(wl, dev)
    T_q, H = wl.total_q, wl.num_heads
    out = torch.empty((T_q, H, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((T_q, H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    res = {}
    for mode in (False, "auto"):
        nbytes = (api.absorbed_workspace_size(wl.seq_lens, wl.cu_q, H, wl.segments, wl.chunk, fp8_scores="auto")
                  if mode else api.prefill_workspace_size(wl.seq_lens, wl.cu_q, H, wl.segments, wl.chunk))
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        for _ in range(3):
            flush.zero_()
            dw.run(out=out, lse=lse, workspace=ws, absorbed=mode)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            flush.zero_()
            gpu_delay()
            a.record(stream)
            dw.run(out=out, lse=lse, workspace=ws, absorbed=mode)
            b.record(stream)
        torch.cuda.synchronize(dev)
        if api.device_error(ws) != 0:
            raise RuntimeError("device error word set in the dispatch comparison")
        res[mode] = float(statistics.median([a.elapsed_time(b) for a, b in ev]))
        del ws
    short = int(sum(1 for e in wl.ext_lens.tolist() if 0 < e <= 128))
    return {"workload": workload_config(wl), "requests_absorbed": short, "ms_fused": res[False],
            "ms_auto": res["auto"], "speedup": res[False] / res["auto"],
            "prefill_tok_s_auto": T_q / (res["auto"] / 1e3)}


def reuse_compare(dev, flush, reps=5, config="v3_8k", n_global=16, protected_frac=0.10):
    """Head-split reuse against full recomputation on the same inputs: the
    Global heads (every 8th head: 16 of 128, the RedKnot page's 8 of 64) and
    a seeded share of the query rows (`protected_frac`) recomputed, the rest
    taken from an artifact.  Median CUDA-event time of a whole call, L2
    flushed before each."""
    import torch
    from mla_prefix_cache_gb300 import api, workload

    wl = workload.by_name(config)
    dw = api.DeviceWorkload(wl, dev)
    T_q, H = wl.total_q, wl.num_heads
    glob = list(range(0, H, max(1, H // n_global)))[:n_global]
    rng = np.random.default_rng(9)
    prot = np.sort(rng.choice(T_q, size=max(1, int(round(protected_frac * T_q))), replace=False))
    g = torch.Generator(device=dev)
    g.manual_seed(9)
    art_out = torch.randn((T_q, H, 128), generator=g, device=dev)
    art_lse = torch.randn((T_q, H), generator=g, device=dev)
    out = torch.empty((T_q, H, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((T_q, H), dtype=torch.float32, device=dev)
    ws_f = torch.empty(api.prefill_workspace_size(wl.seq_lens, wl.cu_q, H, wl.segments, wl.chunk), dtype=torch.uint8,
                       device=dev)
    ws_r = torch.empty(api.reuse_workspace_size(wl.seq_lens, wl.cu_q, H, glob, prot, wl.segments, wl.chunk),
                       dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def full():
        dw.run(out=out, lse=lse, workspace=ws_f)

    def reuse():
        api.prefill_reuse(dw.q, dw.q_pos, dw.kv_cache, dw.block_table, wl.seq_lens, wl.cu_q, dw.kv_b_proj,
                          art_out, art_lse, global_heads=glob, protected_rows=prot, chunk=wl.chunk,
                          softmax_scale=wl.softmax_scale, rope_theta=wl.rope_theta, kv_scale=wl.kv_scale,
                          segments=wl.segments, out=out, lse=lse, workspace=ws_r)

    res = {}
    for name, fn in (("full", full), ("reuse", reuse)):
        for _ in range(3):
            flush.zero_()
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            flush.zero_()
            gpu_delay()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        res[name] = float(statistics.median([a.elapsed_time(b) for a, b in ev]))
    if api.device_error(ws_r) != 0:
        raise RuntimeError("device error word set in the reuse comparison")
    recomputed = (len(glob) * T_q + (H - len(glob)) * len(prot)) / (H * T_q)
    return {"workload": config, "global_heads": len(glob), "protected_rows": int(len(prot)),
            "recomputed_fraction": recomputed, "ms_full": res["full"], "ms_reuse": res["reuse"],
            "speedup": res["full"] / res["reuse"]}


def time_prefill(wl, dev, flush, steps, warmup, world, absorbed=False, with_e2e=True):
    """Times `steps` whole calls of the prefill entry point on `wl` (inputs
    resident, L2 flushed before each step, outside its events), with the
    fused (or latent attention) kernel's own events, the host time of each
    call (planning and launches, from entry to return), the clocks sampled
    during the timed region and, with_e2e, the end-to-end loop through the
    public API with host buffers."""
    import torch
    import torch.distributed as dist
    from mla_prefix_cache_gb300 import api

    dw = api.DeviceWorkload(wl, dev)
    T_q, H = wl.total_q, wl.num_heads
    out = torch.empty((T_q, H, 128), dtype=torch.float32, device=dev)
    lse = torch.empty((T_q, H), dtype=torch.float32, device=dev)
    if absorbed:
        nbytes = api.absorbed_workspace_size(wl.seq_lens, wl.cu_q, H, wl.segments, wl.chunk,
                                             fp8_scores=absorbed == "fp8")
    else:
        nbytes = api.prefill_workspace_size(wl.seq_lens, wl.cu_q, H, wl.segments, wl.chunk)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        dw.run(out=out, lse=lse, workspace=ws, absorbed=absorbed)

    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if api.device_error(ws) != 0:
        raise RuntimeError("device error word set during warm-up")

    K = steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler(getattr(torch.cuda.get_device_properties(dev), "uuid", None))
    uuid = clocks.uuid
    clocks.uuid = ("GPU-" + str(uuid)) if uuid is not None and not str(uuid).startswith("GPU-") else uuid
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    n0 = api.launch_count()
    host_us = []
    for k in range(K):
        flush.zero_()                       # L2 flush, outside the step events
        torch.cuda.synchronize(dev)         # the step's events then also hold the call's host time
        api.set_kernel_events(*kev[k])
        ev[k][0].record(stream)
        h0 = time.perf_counter()
        step()
        host_us.append((time.perf_counter() - h0) * 1e6)
        ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    launches = api.launch_count() - n0
    api.set_kernel_events(None, None)
    if world > 1:
        dist.barrier()
    clk = clocks.stop(t_wall0, t_wall1)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    kern_ms = [a.elapsed_time(b) for a, b in kev]
    if api.device_error(ws) != 0:
        raise RuntimeError("device error word set during the timed steps")
    res = {"step_ms": step_ms, "kern_ms": kern_ms, "launches": launches, "clocks": clk,
           "host_us": statistics.median(host_us), "ws_bytes": int(nbytes), "e2e_ms": None}

    # ---- end to end through the public API: pinned host inputs in, result out.
    # A serving loop: step k's inputs go up (one copy stream) while step k-1
    # computes and step k-2's result comes down (another copy stream); two
    # device buffer sets alternate, and events order each buffer's reuse.
    if with_e2e:
        import copy
        names = ("q", "q_pos", "kv_cache", "block_table", "kv_b_proj")
        host = {n: torch.empty(getattr(dw, n).shape, dtype=getattr(dw, n).dtype, pin_memory=True).copy_(getattr(dw, n))
                for n in names}
        sets = [dw, copy.copy(dw)]
        for n in names:
            setattr(sets[1], n, torch.empty_like(getattr(dw, n)))
        outs = [out, torch.empty_like(out)]
        lses = [lse, torch.empty_like(lse)]
        out_h = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
        lse_h = [torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True) for _ in range(2)]
        res["h2d_bytes"] = sum(v.numel() * v.element_size() for v in host.values())
        res["d2h_bytes"] = out_h[0].numel() * out_h[0].element_size() + lse_h[0].numel() * lse_h[0].element_size()
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        mk = lambda: torch.cuda.Event()
        done_compute = [mk(), mk()]
        done_down = [mk(), mk()]
        for e_ in done_compute + done_down:
            e_.record(stream)

        def e2e_step(k):
            b = k & 1
            up.wait_event(done_compute[b])            # step k-2 no longer reads these inputs
            with torch.cuda.stream(up):
                for n in names:
                    getattr(sets[b], n).copy_(host[n], non_blocking=True)
            uploaded = mk()
            uploaded.record(up)
            stream.wait_event(uploaded)
            stream.wait_event(done_down[b])           # step k-2's result has left this buffer
            sets[b].run(out=outs[b], lse=lses[b], workspace=ws, absorbed=absorbed)
            done_compute[b].record(stream)
            down.wait_event(done_compute[b])
            with torch.cuda.stream(down):
                out_h[b].copy_(outs[b], non_blocking=True)
                lse_h[b].copy_(lses[b], non_blocking=True)
            done_down[b].record(down)

        for k in range(max(1, warmup)):
            e2e_step(k)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        e0.record(up)
        stream.wait_event(e0)
        down.wait_event(e0)
        for k in range(K):
            e2e_step(k)
        stream.wait_event(done_down[(K - 1) & 1])
        stream.wait_event(done_down[K & 1])
        e1.record(stream)
        torch.cuda.synchronize(dev)
        res["e2e_ms"] = e0.elapsed_time(e1)
        del sets, outs, lses, out_h, lse_h, host
    del dw, out, lse, ws
    torch.cuda.empty_cache()
    return res


def kernel_roofline(wl, res, peak, source, path="fused"):
    """The timed kernel's roofline: algorithmic FLOPs (latent attention for the
    absorbed paths) over its mean event time per call, against the measured
    bf16 burst peak, with the executed FLOPs of the fused kernel beside it."""
    k_ms = sum(res["kern_ms"]) / len(res["kern_ms"])
    if path == "fused":
        kflops, xflops = wl.algorithmic_flops(), executed_flops(wl)
    else:
        kflops, xflops = wl.absorbed_attention_flops(), None
    achieved = kflops / (k_ms / 1e3) / 1e12
    r = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
         "traffic": measured_traffic(wl.name, path), "kernel": "absorb_attn_kernel" if path != "fused" else fused_kernel_name(),
         "peak_source": f"bf16_tflops (burst) of {source} peaks", "kernel_ms": k_ms,
         "algorithmic_flops": kflops}
    if xflops is not None:
        r["executed_flops"] = xflops
        r["executed_tflops"] = xflops / (k_ms / 1e3) / 1e12
    return r


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    from mla_prefix_cache_gb300 import workload

    wl = workload.by_name(args.config)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.cpu_budget_s)

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    absorbed = {"fused": False, "absorbed": True, "absorbed_fp8": "fp8"}[args.path]
    res = time_prefill(wl, dev, flush, args.steps, args.warmup, world, absorbed, with_e2e=not args.no_e2e)
    K = args.steps
    total_ms = max_over_ranks(sum(res["step_ms"]), world, dev)
    flops = wl.algorithmic_flops()
    value = weak_scaling_value(flops, K, world, total_ms) / 1e12
    tok_s = weak_scaling_value(wl.total_q, K, world, total_ms)
    scan_tok_s = weak_scaling_value(int(wl.ctx_lens.sum()), K, world, total_ms)   # cached tokens attended per s
    e2e = None
    if res["e2e_ms"] is not None:
        ems = max_over_ranks(res["e2e_ms"], world, dev)
        e2e = {"value": weak_scaling_value(flops, K, world, ems) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": int(res["h2d_bytes"]), "d2h_bytes_per_step": int(res["d2h_bytes"]),
               "ms_per_step": ems / K,
               "note": "pinned host inputs copied up and results copied down every step, on two copy streams "
                       "overlapping the neighbouring steps' compute (two device buffer sets)"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peaks, source = load_peaks()
    peak = float(peaks["bf16_tflops"])
    path = "fused" if not absorbed else args.path
    roof = kernel_roofline(wl, res, peak, source, path)
    # the 128K FP8 configuration, timed the same way (its own fused-kernel roofline)
    target = None
    if not args.no_target and world == 1 and not absorbed and args.config != "fp8_128k":
        wt = workload.by_name("fp8_128k")
        rt = time_prefill(wt, dev, flush, max(3, min(K, 10)), args.warmup, 1, False, with_e2e=False)
        tms = sum(rt["step_ms"]) / len(rt["step_ms"])
        target = {"workload": "fp8_128k", "value": wt.algorithmic_flops() / (tms / 1e3) / 1e12, "unit": UNIT,
                  "ms_per_step": tms, "prefill_tok_s": wt.total_q / (tms / 1e3), "steps": len(rt["step_ms"]),
                  "roofline": kernel_roofline(wt, rt, peak, source), "host_us_per_call": rt["host_us"],
                  "clocks": rt["clocks"]}
        del wt
    hbm = None if args.no_hbm_kernels else hbm_kernels(dev, flush, float(peaks["hbm_gbs"]))
    cmp_abs = cmp_abs8 = None
    if not args.no_absorbed and world == 1 and not absorbed:
        cmp_abs = absorbed_compare(dev, flush, peak, source)
        cmp_abs8 = absorbed_compare(dev, flush, peak, source, reps=5, config="short_ext_fp8_128k", fp8_scores=True)
    cmp_fp8w = None
    if not args.no_fp8w and world == 1 and not absorbed:
        cmp_fp8w = fp8w_compare(dev, flush, peak, source)
    cmp_reuse = cmp_auto = None
    if not args.no_reuse and world == 1:
        cmp_reuse = reuse_compare(dev, flush)
        # few protected rows (61 of 2048): the call takes them through the absorbed path
        cmp_reuse["small_protected_set"] = reuse_compare(dev, flush, protected_frac=0.03)
    if not args.no_auto and world == 1 and not absorbed:
        cmp_auto = auto_compare(dev, flush)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded; shapes of the workload, random values)",
        "config": workload_config(wl, {"parallelism": f"replicas x{world}",
                                       "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB memset and a "
                                             "synchronize outside the step events; the events hold the "
                                             "call's host planning and launches too)"}),
        "prefill_tok_s": tok_s,
        "context_scan_tok_s": scan_tok_s,
        "frac_of_bf16_peak": value / world / peak,
        "roofline": roof,
        "host_us_per_call": res["host_us"],
        "workspace_bytes": res["ws_bytes"],
        "path": args.path,
        "gpu_launches": int(res["launches"]),
        "hbm_kernels": hbm,
        "hbm_peak_source": f"hbm_gbs of {source} peaks",
        "absorbed": cmp_abs,
        "absorbed_fp8": cmp_abs8,
        "reuse": cmp_reuse,
        "auto": cmp_auto,
        "fp8w": cmp_fp8w,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": res["clocks"],
        "target_128k": target,
    }
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="reloc_256k")
    ap.add_argument("--path", choices=["fused", "absorbed", "absorbed_fp8"], default="fused",
                    help="entry point timed: mla_prefill_ctx (up-projected, fused), mla_prefill_ctx_absorbed, or "
                         "mla_prefill_ctx_absorbed_fp8 (FP8 caches)")
    ap.add_argument("--no-absorbed", action="store_true",
                    help="skip the absorbed-vs-fused comparison on the short-extend workload")
    ap.add_argument("--no-auto", action="store_true",
                    help="skip the per-request dispatch comparison on the mixed batch")
    ap.add_argument("--no-fp8w", action="store_true",
                    help="skip the FP8 up-projection comparison on fp8_128k (mla_prefill_ctx_fp8w)")
    ap.add_argument("--no-reuse", action="store_true",
                    help="skip the head-split reuse comparison (16 Global heads, 10% protected rows on v3_8k)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-target", action="store_true",
                    help="skip the second timed line on the 128K FP8 configuration (target_128k)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-hbm-kernels", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--ref-step-s", type=float, default=8.0)
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)      # at least 3 untimed warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
