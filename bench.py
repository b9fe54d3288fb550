#!/usr/bin/env python3
"""Absorbed paged MLA decode benchmark (one JSON line on stdout).

A step is one pass of the decode path over one batch of synthetic input
(default workload: DeepSeek-V2 shapes, batch 32, 4096-token contexts, bf16
paged cache): absorb_q -> plan -> decode_attn -> combine -> absorb_out, all
through the C ABI. ``--workload`` picks another workload (the FP8 cache
workload with the suffix ``_staged`` goes through mla_decode_attn_fp8_staged);
the line also carries ``other_workloads``: the long-context, ragged,
full-layer, multi-token, prefill and FP8 workloads measured the same way,
each with its own roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Timing: W untimed warm-up steps, then K steps, each preceded by an L2 flush
(a read of a buffer twice the L2 size, outside the timed events) and timed
with CUDA events on the launching stream; barrier + synchronize on both sides
of the timed loop; max over ranks. Inputs are resident in HBM. The step's
calls are recorded once into a CUDA graph and ``value`` times its replays
(the eager, call-by-call time is reported beside it). Each stage is also
recorded into a graph of its own and timed alone after a flush: the decode
kernel's duration (``roofline.kernel_us``) comes from that, so host launch
overhead never enters it. The ``e2e`` figure times the same step with the
per-step inputs copied host->device from pinned memory before it and the
result copied back after it, all inside the timed region, and splits the
time into those three parts.

``--impl reference`` times the fp64 explicit oracle on the host cores, each
step one whole oracle step of the workload (every sequence and head).

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path does not shard); there is no collective on the data path.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode μs/step and achieved fraction of roofline (HBM GB/s, TFLOP/s)"
UNIT = "us/step"
DEFAULT_WORKLOAD = "dsv2_b32_ctx4k"

# DRAM bytes (read + write) of one tcgen05 decode launch, from an ncu
# capture of that kernel on the workload. Valid only for the kernel source
# the capture measured: drop the entry whenever the decode kernel changes,
# until it is captured again.
DECODE_TRAFFIC = {"dsv2_b32_ctx4k": 157_358_336 + 4_366_592}
DECODE_KERNELS = {0: "simt", 1: "tcgen05 score/value pair", 2: "tcgen05 latent-split pair"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other", action="store_true",
                    help="measure only --workload (skip the other_workloads entries)")
    ap.add_argument("--ctx", type=int, default=0,
                    help="override the workload's context length (small cases for profiling)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6400.0, 1800.0, "fallback"


def algorithmic_prefill(wl):
    """Algorithmic bytes and FLOPs of one prefill attention launch over a
    prompt of N tokens: q, k_nope, v and the latent rows read once, o
    written once; FLOPs of the causal products (token i: i + 1 keys, scores
    over d_h + d_r, output over d_v)."""
    N = wl.ctx
    b = N * wl.n_h * ((wl.d_h + wl.d_r) + wl.d_h + wl.d_v + wl.d_v) * 2 + N * (wl.d_c + wl.d_r) * 2
    pairs = N * (N + 1) // 2
    return b, pairs * wl.n_h * 2 * (wl.d_h + wl.d_r + wl.d_v)


def algorithmic(wl, lens):
    """Algorithmic bytes and FLOPs of one decode_attn launch: each cached row
    (c_kv | k_R) read once, q_cat read once, o_lat written once; FLOPs of the
    two contractions (scores over d_c + d_r, latent output over d_c). With
    q_len new tokens per sequence the rows are still read once, and new
    token t of a sequence of length L attends over L - q_len + 1 + t rows."""
    esz = 4 if wl.dtype == "f32" else 2
    lens = np.asarray(lens, np.int64)
    tokens = int(np.sum(lens))
    R = len(lens) * wl.q_len
    seen = int(np.sum(lens)) * wl.q_len - len(lens) * (wl.q_len * (wl.q_len - 1) // 2)
    if wl.dtype == "fp8":  # the FP8 row: codes, bf16 RoPE key, scale, padding
        cache = tokens * ((wl.d_c + 2 * wl.d_r + 4 + 15) // 16 * 16)
    else:
        cache = tokens * (wl.d_c + wl.d_r) * esz
    q = R * wl.n_h * (wl.d_c + wl.d_r) * esz
    o = R * wl.n_h * wl.d_c * 4
    flops = seen * (2 * wl.n_h * (wl.d_c + wl.d_r) + 2 * wl.n_h * wl.d_c)
    return cache + q + o, flops


def max_over_ranks(vals, device):
    """Element-wise max of a list of floats over the ranks of the default
    process group (the list itself when there is none or only one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in vals]
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


# --------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock and throttle reasons while the timed loop runs:
    through NVML when the Python binding is importable, else by polling
    ``nvidia-smi`` (read-only queries in both cases)."""
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int, period=0.02):
        self.index, self.samples, self.reasons, self.period = index, [], set(), period
        self.max_mhz, self.err, self.nv, self.proc = None, None, None, None
        self._stop = threading.Event()
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
        except Exception as e:  # noqa: BLE001
            self.nv, self.err = None, f"nvml: {e}"

    def _run_nvml(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM))
                r = self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                for bit, name in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(name)
            except Exception:  # noqa: BLE001
                pass
            time.sleep(self.period)

    def __enter__(self):
        self._stop.clear()
        if self.nv:
            self.t = threading.Thread(target=self._run_nvml, daemon=True)
            self.t.start()
        else:
            import subprocess
            q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap")
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception as e:  # noqa: BLE001
                self.err = f"{self.err}; nvidia-smi: {e}"
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self.nv:
            self.t.join()
        elif self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in out.splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 6:
                    continue
                try:
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                except ValueError:
                    continue
                for name, v in zip(names, f[2:6]):
                    if v.lower() == "active":
                        self.reasons.add(name)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                    "error": self.err or "no samples"}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples),
                "source": "nvml" if self.nv else "nvidia-smi"}


# ---------------------------------------------------------- CPU oracle
def oracle_step(wl):
    """One whole step of the fp64 explicit oracle on this host's cores: for
    every sequence, its cached rows (drawn, plus the rows the append step
    writes on the full-layer and prefill workloads), its query (drawn, or
    projected from the token), then every head rebuilt as
    K_h = [c W^UK_h^T | k_R], V_h = c W^UV_h^T and attended with plain
    softmax, and W^O on the full-layer workload. Returns the seconds spent
    inside the oracle (drawing the seeded inputs is outside the clock)."""
    from oracle import mla_oracle as O
    from mla_latent_kv_67_b300 import synth
    lens = synth.seq_lens(wl)
    w = {k: synth.weight(wl, k).astype(np.float64) for k in ("w_uk", "w_uv")}
    if wl.mode == "attn":
        q = synth.query(wl).astype(np.float64)
    else:
        for k in ("w_dkv", "w_kr", "w_uq", "w_qr") + (("w_dq",) if wl.d_cq else ()) + \
                (("w_o",) if wl.mode == "layer" else ()):
            w[k] = synth.weight(wl, k).astype(np.float64)
        x = synth.tokens(wl).astype(np.float64)
    drawn = synth.drawn_rows(wl, lens)
    spent = 0.0
    for b in range(wl.batch):
        rows = synth.cache_rows(wl, b, int(drawn[b])).astype(np.float64)
        t = time.perf_counter()
        c, k = rows[:, :wl.d_c], rows[:, wl.d_c:]
        if wl.mode == "attn":
            q_c, q_r = q[b, :, :wl.d_h], q[b, :, wl.d_h:]
        else:
            xs = x[b:b + 1] if wl.mode == "layer" else x
            pos = np.arange(int(drawn[b]), int(lens[b]))
            c2, k2 = O.latent_cache_row(xs, w["w_dkv"], w["w_kr"], pos, wl.rope_base)
            c, k = np.concatenate([c, c2]), np.concatenate([k, k2])
            q_c, q_r = O.project_query(xs[-1], w["w_uq"], w["w_qr"], int(lens[b]) - 1, wl.n_h,
                                       w_dq=w.get("w_dq"), base=wl.rope_base)
        o, _ = O.attention_explicit(q_c, q_r, c, k, w["w_uk"], w["w_uv"], wl.scale)
        if wl.mode == "layer":
            O.output_projection(o, w["w_o"])
        spent += time.perf_counter() - t
    return spent


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        return max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
    except Exception:  # noqa: BLE001
        return os.cpu_count() or 1


def oracle_sample_text(wl):
    return (f"one whole step: the fp64 explicit (non-absorbed) oracle over all "
            f"{wl.batch} x {wl.n_h} (sequence, head) pairs of {wl.name}")


def cpu_baseline_entry(wl):
    """The oracle timed on this host's cores over one whole step."""
    spent = oracle_step(wl)
    return {"value": spent * 1e6, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": oracle_sample_text(wl)}


# -------------------------------------------------------------- reference
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from mla_latent_kv_67_b300 import synth
    wl = synth.WORKLOADS[args.workload]
    lens = synth.seq_lens(wl)
    t_run = time.perf_counter()
    times = []
    for i in range(args.warmup + args.steps):
        spent = oracle_step(wl)
        if i >= args.warmup:
            times.append(spent)
    us = sum(times) / len(times) * 1e6
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name, "batch": wl.batch,
                                            "ctx": int(lens.max()), "n_h": wl.n_h, "d_c": wl.d_c,
                                            "d_r": wl.d_r, "page_size": wl.page_size},
            "cpu_baseline": {"value": us, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                             "sample": oracle_sample_text(wl)},
            "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": time.perf_counter() - t_run}
    print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------------- ours
def weight_bytes(wl):
    """Bytes of the weights one step of the workload reads (bf16 or fp32)."""
    esz = 4 if wl.dtype == "f32" else 2
    if wl.fused:
        k = wl.d_cq or wl.d_model
        n = (wl.d_c + wl.d_r) * wl.d_model + wl.d_cq * wl.d_model   # W^DKV | W^KR, W^DQ
        n += wl.n_h * (wl.d_c + wl.d_r) * k                         # W^UK^T W^UQ | W^QR
        n += wl.d_model * wl.n_h * wl.d_c                           # W^O W^UV
        return n * esz, n
    n = wl.n_h * wl.d_h * wl.d_c + wl.n_h * wl.d_v * wl.d_c     # W^UK, W^UV
    if wl.mode == "layer":
        k = wl.d_cq or wl.d_model
        n += (wl.d_c + wl.d_r) * wl.d_model                      # W^DKV | W^KR
        n += wl.d_cq * wl.d_model                                # W^DQ
        n += wl.n_h * (wl.d_h + wl.d_r) * k                      # W^UQ | W^QR
        n += wl.d_model * wl.n_h * wl.d_v                        # W^O
    return n * esz, n


def step_roofline(wl, lens, hbm, tflops, step_us):
    """Roofline of the whole step: the decode launch's algorithmic bytes and
    FLOPs plus every weight read once and its product with the batch."""
    b, f = algorithmic(wl, lens)
    wb, wn = weight_bytes(wl)
    b += wb
    f += 2 * wl.batch * wn
    t = max(b / (hbm * 1e9), f / (tflops * 1e12))
    return {"alg_bytes": b, "alg_flops": f, "roofline_us": t * 1e6,
            "frac": t * 1e6 / step_us if step_us else None}


def time_graph(g, K, flush, stream):
    """Mean CUDA-event time (ms) of K replays of graph g, L2 flushed before each."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    for a, b in evs:
        flush()
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / K


def capture(fn):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        fn()
    return g


def measure_workload(wl, dev, K, W, flush, stream, hbm, tflops, barrier=None, sampler=None,
                     fp8_staged=False):
    """Step and per-stage times of one workload: the step as one CUDA graph
    (value), each stage as a graph of its own timed alone, the decode
    kernel's roofline. fp8_staged: the FP8 cache through the widening entry
    point (its attention stage then holds widen, plan, decode and merge)."""
    import torch
    from mla_latent_kv_67_b300 import binding as M
    from mla_latent_kv_67_b300.step import DecodeStep
    st = DecodeStep(wl, device=dev, fp8_staged=fp8_staged)
    for _ in range(W):
        flush()
        st.run()
    torch.cuda.synchronize()
    assert st.status() == 0, f"{wl.name}: device status {st.status():#x}"
    g = capture(st.run)
    for _ in range(W):
        flush()
        g.replay()
    torch.cuda.synchronize()
    assert st.status() == 0, f"{wl.name}: device status {st.status():#x}"
    if barrier:
        barrier()
    if sampler is not None:
        with sampler:
            step_ms = time_graph(g, K, flush, stream)
    else:
        step_ms = time_graph(g, K, flush, stream)
    stages = {}
    for f in st.stages():
        gs = capture(f)
        for _ in range(2):
            flush()
            gs.replay()
        stages[f.__name__] = time_graph(gs, K, flush, stream) * 1e3
    torch.cuda.synchronize()
    assert st.status() == 0, f"{wl.name}: device status {st.status():#x}"
    prefill = wl.mode == "prefill_mha"
    kernel_us = stages["prefill" if prefill else
                       ("attend_fp8_staged" if fp8_staged else "attend")]
    alg_bytes, alg_flops = algorithmic_prefill(wl) if prefill else algorithmic(wl, st.lens_np)
    t_hbm = alg_bytes / (hbm * 1e9)
    t_flop = alg_flops / (tflops * 1e12)
    achieved = alg_bytes / (kernel_us * 1e-6) / 1e9
    tensor = alg_flops / (kernel_us * 1e-6) / 1e12
    path = M.mla_decode_path(st.dtype, st.dims)
    tensor_bound = t_flop > t_hbm
    roof = {"bound": "tensor" if tensor_bound else "hbm",
            "achieved": tensor if tensor_bound else achieved,
            "peak": tflops if tensor_bound else hbm,
            "unit": "TFLOP/s" if tensor_bound else "GB/s",
            "frac": tensor / tflops if tensor_bound else achieved / hbm,
            "traffic": DECODE_TRAFFIC.get(wl.name) if path == 1 else None,
            "kernel": "mla_prefill_attn" if prefill else
                      ("mla_decode_attn_fp8_staged" if fp8_staged else "mla_decode_attn"),
            "kernel_us": kernel_us,
            "alg_bytes": alg_bytes, "alg_flops": alg_flops,
            "tensor_tflops": tensor, "tensor_peak": tflops, "tensor_frac": tensor / tflops,
            "roofline_us": max(t_hbm, t_flop) * 1e6,
            "frac_of_roofline": max(t_hbm, t_flop) * 1e6 / kernel_us}
    return st, g, {"step_us": step_ms * 1e3, "stages_us": stages, "roofline": roof,
                   "decode_kernel": (DECODE_KERNELS.get(M.mla_decode_path(M.MLA_BF16, st.dims))
                                     + " on bf16-widened pages") if fp8_staged else
                                    DECODE_KERNELS.get(path, "simt"),
                   "step_roofline": None if prefill else
                   step_roofline(wl, st.lens_np, hbm, tflops, step_ms * 1e3)}


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from mla_latent_kv_67_b300 import build as mbuild
    mbuild.build()
    from mla_latent_kv_67_b300 import synth

    staged = args.workload.endswith(STAGED)  # an FP8 workload through the widening entry
    base = args.workload[:-len(STAGED)] if staged else args.workload
    wl = synth.WORKLOADS.get(base) or synth.EXTRA_WORKLOADS[base]
    if staged:
        wl = wl.replace(name=args.workload)
    if args.ctx:
        wl = wl.replace(name=f"{wl.name}_ctx{args.ctx}", ctx=args.ctx, ctx_range=None, lens=None)
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.ones(2 * l2 // 4, dtype=torch.float32, device=dev)

    def flush():
        flush_buf.sum()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    hbm, tflops, peak_kind = peaks()
    K = args.steps
    sampler = ClockSampler(local)
    st, graph, res = measure_workload(wl, dev, K, args.warmup, flush, stream, hbm, tflops,
                                      barrier=barrier, sampler=sampler, fp8_staged=staged)
    stages = st.stages()

    # the same step, call by call (eager), for comparison
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    barrier()
    for i in range(K):
        flush()
        ev[i][0].record(stream)
        st.run()
        ev[i][1].record(stream)
    barrier()
    eager_ms = sum(a.elapsed_time(b) for a, b in ev) / K
    step_ms = res["step_us"] / 1e3
    kernel_ms = res["roofline"]["kernel_us"] / 1e3
    step_ms, kernel_ms, eager_ms = max_over_ranks([step_ms, kernel_ms, eager_ms], dev)

    # ---- end to end with host buffers: pinned H2D of the step's inputs, the
    # step, D2H of its result, all inside the timed region. The three are
    # recorded into one CUDA graph (copies as memcpy nodes) when the runtime
    # allows it, else issued one after the other; each part is also timed
    # alone.
    # The step's host inputs (queries or hidden states, lengths, block
    # table) sit back to back in one pinned buffer and go over in one copy
    # into one device buffer whose views the step then reads.
    q_name = "q" if wl.mode == "attn" else "x"
    parts = [getattr(st, q_name), st.seq_lens, st.block_table]
    offs, total = [], 0
    for t in parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    stage_dev = torch.empty(total, dtype=torch.uint8, device=dev)
    stage_host = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    views = []
    for t, o in zip(parts, offs):
        n = t.numel() * t.element_size()
        v = stage_dev[o:o + n].view(t.dtype).view(t.shape)
        v.copy_(t)
        stage_host[o:o + n].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
        views.append(v)
    setattr(st, q_name, views[0])
    st.seq_lens, st.block_table = views[1], views[2]
    out = st.result()
    out_host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)

    def h2d():
        stage_dev.copy_(stage_host, non_blocking=True)

    def d2h():
        out_host.copy_(out, non_blocking=True)

    def e2e_body():
        h2d()
        st.run()
        d2h()

    Ke = min(K, 100)
    e2e_launch = "one CUDA graph: one pinned H2D copy of the packed inputs + the step + D2H copy"
    try:
        ge = capture(e2e_body)
        g_h2d, g_d2h = capture(h2d), capture(d2h)
        for _ in range(3):
            flush()
            ge.replay()
        torch.cuda.synchronize()
        e2e_ms = time_graph(ge, Ke, flush, stream)
        h2d_ms = time_graph(g_h2d, Ke, flush, stream)
        d2h_ms = time_graph(g_d2h, Ke, flush, stream)
    except Exception as exc:  # noqa: BLE001
        e2e_launch = f"eager copies + step graph ({type(exc).__name__})"
        parts = []
        for i in range(Ke + 2):
            flush()
            torch.cuda.synchronize()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            e[0].record(stream)
            h2d()
            e[1].record(stream)
            st.run()
            e[2].record(stream)
            d2h()
            e[3].record(stream)
            e[3].synchronize()
            if i >= 2:
                parts.append([e[0].elapsed_time(e[1]), e[2].elapsed_time(e[3]), e[0].elapsed_time(e[3])])
        h2d_ms, d2h_ms, e2e_ms = (sum(p[j] for p in parts) / len(parts) for j in range(3))
    torch.cuda.synchronize()
    assert st.status() == 0, f"device status {st.status():#x}"
    e2e_ms, = max_over_ranks([e2e_ms], dev)
    h2d = total
    d2h = out_host.numel() * out_host.element_size()

    roof = dict(res["roofline"])
    roof["kernel_us"] = kernel_ms * 1e3
    roof["tensor_tflops"] = roof["alg_flops"] / (kernel_ms * 1e-3) / 1e12
    roof["tensor_frac"] = roof["tensor_tflops"] / tflops
    if roof["bound"] == "tensor":  # the kernel's own bound decides the unit
        roof["achieved"], roof["frac"] = roof["tensor_tflops"], roof["tensor_frac"]
    else:
        roof["achieved"] = roof["alg_bytes"] / (kernel_ms * 1e-3) / 1e9
        roof["frac"] = roof["achieved"] / hbm
    roof["frac_of_roofline"] = roof["roofline_us"] / (kernel_ms * 1e3)
    roof["peak_source"] = peak_kind
    roof["timing"] = "decode launch alone in its own CUDA graph, L2 flushed before each"
    launches = sum({"absorb_q": 1 if res["decode_kernel"] != "simt" else 2,
                    "project": 2 if wl.d_cq else 1, "project_absorbed": 2 if wl.d_cq else 1,
                    "out_absorbed": 2, "expand": 2}.get(f.__name__, 1) for f in stages)
    line = {
        "metric": METRIC, "value": step_ms * 1e3, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.batch, "ctx": int(st.lens_np.max()),
                   "ctx_total": int(st.lens_np.sum()), "n_h": wl.n_h, "d_c": wl.d_c,
                   "d_r": wl.d_r, "page_size": wl.page_size,
                   "l2": f"flushed before every timed step (read of a {2 * l2 >> 20} MiB buffer, untimed)",
                   "decode_kernel": res["decode_kernel"], "step_launch": "cuda_graph",
                   "e2e_launch": e2e_launch,
                   "eager_us_per_step": eager_ms * 1e3,
                   "stages_us": res["stages_us"],
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roof,
        "step_roofline": res["step_roofline"],
        "e2e": {"value": e2e_ms * 1e3, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "h2d_alone_us": h2d_ms * 1e3,
                "step_alone_us": step_ms * 1e3, "d2h_alone_us": d2h_ms * 1e3},
        "gpu_launches": launches * K,
        "clocks": sampler.summary(),
    }
    del st, graph, out
    torch.cuda.empty_cache()
    if not args.no_other and world == 1:
        others = {}
        for name in OTHER_WORKLOADS:
            if name == wl.name:
                continue
            staged = name.endswith(STAGED)
            base = name[:-len(STAGED)] if staged else name
            ow = synth.WORKLOADS.get(base) or synth.EXTRA_WORKLOADS[base]
            ost, og, ores = measure_workload(ow, dev, max(3, min(K, 20)), max(3, min(args.warmup, 5)),
                                             flush, stream, hbm, tflops, fp8_staged=staged)
            ores["roofline"]["peak_source"] = peak_kind
            ores["config"] = {"batch": ow.batch, "ctx_total": int(ost.lens_np.sum()),
                              "ctx_max": int(ost.lens_np.max()), "mode": ow.mode,
                              "new_tokens_per_seq": ow.q_len}
            others[name] = ores
            del ost, og
            torch.cuda.empty_cache()
        line["other_workloads"] = others
    if rank == 0 and world == 1 and not args.no_cpu_baseline and wl.mode == "attn" and not args.ctx:
        line["cpu_baseline"] = cpu_baseline_entry(wl)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# measured beside the headline workload in the same run (the tiny fp32
# workload is a parity case only)
OTHER_WORKLOADS = ("dsv2_b4_ctx128k", "dsv2_b128_ragged", "dsv2_layer_b64_ctx32k",
                   "dsv2_layer_b64_ctx32k_fused", "dsv2_b32_ctx4k_mtp2", "dsv2_prefill_4k",
                   "dsv2_b32_ctx4k_fp8", "dsv2_b32_ctx4k_fp8_staged")
# an entry named <workload> + STAGED: that FP8 workload through
# mla_decode_attn_fp8_staged instead of the CUDA-core FP8 kernel
STAGED = "_staged"


if __name__ == "__main__":
    sys.exit(main())
