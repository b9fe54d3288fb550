#!/usr/bin/env python3
"""Absorbed paged MLA decode benchmark (one JSON line on stdout).

A step is one pass of the decode path over one batch of synthetic input
(default workload: DeepSeek-V2 shapes, batch 32, 4096-token contexts, bf16
paged cache): absorb_q -> plan -> decode_attn -> combine -> absorb_out, all
through the C ABI. ``--workload`` picks another of the five workloads.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Timing: W untimed warm-up steps, then K steps, each preceded by an L2 flush
(a read of a buffer twice the L2 size, outside the timed events) and timed
with CUDA events on the launching stream; barrier + synchronize on both sides
of the timed loop; max over ranks. Inputs are resident in HBM. The step's
calls are recorded once into a CUDA graph and ``value`` times its replays
(the eager, call-by-call time is reported beside it); the decode kernel's
own time comes from events around its call in the eager loop. The ``e2e``
figure times the same step (the same graph, else the eager calls) with the
per-step inputs copied host->device from pinned memory before it and the
result copied back after it, all inside the timed region.

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

# DRAM bytes (read + write) of one tcgen05 decode launch, from the ncu
# capture summarised in profiles/decode_pair_dsv2_b32_ctx4k.md. Valid only
# for the kernel source that capture measured: set to None whenever the
# decode kernel changes, until it is captured again.
DECODE_TRAFFIC = {"dsv2_b32_ctx4k": 157_475_840 + 5_623_296}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle sample")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6400.0, 1800.0, "fallback"


def algorithmic(wl, lens):
    """Algorithmic bytes and FLOPs of one decode_attn launch: each cached row
    (c_kv | k_R) read once, q_cat read once, o_lat written once; FLOPs of the
    two contractions (scores over d_c + d_r, latent output over d_c)."""
    esz = 2 if wl.dtype == "bf16" else 4
    tokens = int(np.sum(lens))
    B = len(lens)
    cache = tokens * (wl.d_c + wl.d_r) * esz
    q = B * wl.n_h * (wl.d_c + wl.d_r) * esz
    o = B * wl.n_h * wl.d_c * 4
    flops = tokens * (2 * wl.n_h * (wl.d_c + wl.d_r) + 2 * wl.n_h * wl.d_c)
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
def cpu_oracle_sample(wl, target_s: float, seqs_heads=None):
    """Time the fp64 explicit oracle on a bounded sample of the workload:
    (sequence, head) pairs in a fixed order until ``target_s`` seconds have
    been spent. Returns (seconds, pairs done, token-heads done)."""
    from oracle import mla_oracle as O
    from mla_latent_kv_67_b300 import synth
    lens = synth.seq_lens(wl)
    w_uk = synth.weight(wl, "w_uk").astype(np.float64)
    w_uv = synth.weight(wl, "w_uv").astype(np.float64)
    q = synth.query(wl).astype(np.float64)
    # heads in a spread order (0, 16, 32, ..., 1, 17, ...), sequences inner
    order = [h0 + k for h0 in range(16) for k in range(0, wl.n_h, 16) if h0 + k < wl.n_h]
    pairs = seqs_heads or [(b, h) for h in order for b in range(wl.batch)]
    spent, done, tok, rows_cache = 0.0, 0, 0, {}
    for b, h in pairs:
        if b not in rows_cache:
            rows_cache = {b: synth.cache_rows(wl, b, int(lens[b])).astype(np.float64)}
        rows = rows_cache[b]
        t = time.perf_counter()
        O.attention_explicit(q[b, :, :wl.d_h], q[b, :, wl.d_h:], rows[:, :wl.d_c], rows[:, wl.d_c:],
                             w_uk, w_uv, wl.scale, heads=[h])
        spent += time.perf_counter() - t
        done += 1
        tok += int(lens[b])
        if spent >= target_s:
            break
    return spent, done, tok


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        return max((i.get("num_threads", 1) for i in threadpool_info()), default=1)
    except Exception:  # noqa: BLE001
        return os.cpu_count() or 1


def cpu_baseline_entry(wl, target_s):
    """The oracle timed on this host's cores on a bounded sample, extrapolated
    by token-heads to one full step."""
    from mla_latent_kv_67_b300 import synth
    lens = synth.seq_lens(wl)
    spent, pairs, tok = cpu_oracle_sample(wl, target_s)
    full = float(np.sum(lens)) * wl.n_h
    us = spent * full / tok * 1e6
    return {"value": us, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": f"fp64 explicit (non-absorbed) oracle on {pairs} of {wl.batch * wl.n_h} "
                      f"(sequence, head) pairs ({spent:.1f} s), extrapolated by token-heads "
                      f"to the full step"}


# -------------------------------------------------------------- reference
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from mla_latent_kv_67_b300 import synth
    wl = synth.WORKLOADS[args.workload]
    lens = synth.seq_lens(wl)
    # each step: one (sequence, head) pair of the explicit oracle, rotating
    pairs = [(b, h) for h in range(wl.n_h) for b in range(wl.batch)]
    spent_t, tok_t = 0.0, 0
    for i in range(args.warmup + args.steps):
        b, h = pairs[i % len(pairs)]
        spent, _, tok = cpu_oracle_sample(wl, 0.0, seqs_heads=[(b, h)])
        if i >= args.warmup:
            spent_t, tok_t = spent_t + spent, tok_t + tok
    us = spent_t / tok_t * float(np.sum(lens)) * wl.n_h * 1e6
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name, "batch": wl.batch,
                                            "ctx": int(lens.max()), "n_h": wl.n_h, "d_c": wl.d_c,
                                            "d_r": wl.d_r, "page_size": wl.page_size},
            "cpu_baseline": {"value": us, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                             "sample": f"each step: the fp64 explicit oracle on one (sequence, head) "
                                       f"pair, extrapolated by token-heads to the full step"},
            "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------------- ours
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
    from mla_latent_kv_67_b300 import binding as M
    from mla_latent_kv_67_b300 import synth
    from mla_latent_kv_67_b300.step import DecodeStep

    wl = synth.WORKLOADS[args.workload]
    st = DecodeStep(wl, device=dev)
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.ones(2 * l2 // 4, dtype=torch.float32, device=dev)

    def do_flush():
        flush.sum()

    tc = M.mla_decode_path(st.dtype, st.dims) == 1
    launches_per_step = 0
    for f in st.stages():
        launches_per_step += {"absorb_q": 1 if tc else 2,
                              "project": 2 if wl.d_cq else 1}.get(f.__name__, 1)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        do_flush()
        st.run()
    barrier()
    assert st.status() == 0, f"device status {st.status():#x}"

    # The step's calls recorded once into a CUDA graph (the library allocates
    # nothing and only enqueues work, so the calls capture as they are).
    graph, graph_err = None, None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            st.run()
        for _ in range(args.warmup):
            do_flush()
            g.replay()
        barrier()
        assert st.status() == 0, f"device status {st.status():#x}"
        graph = g
    except Exception as e:  # noqa: BLE001
        graph_err = f"{type(e).__name__}: {e}"[:200]

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    ka = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(local)
    stages = st.stages()
    with sampler:
        barrier()
        t_wall = time.perf_counter()
        for i in range(K):
            do_flush()
            ev[i][0].record(stream)
            for f in stages:
                if f.__name__ == "attend":
                    ka[i][0].record(stream)
                    f()
                    ka[i][1].record(stream)
                else:
                    f()
            ev[i][1].record(stream)
        barrier()
        t_wall = time.perf_counter() - t_wall
    step_ms = sum(a.elapsed_time(b) for a, b in ev) / K
    attn_ms = sum(a.elapsed_time(b) for a, b in ka) / K
    eager_ms = step_ms
    if graph is not None:
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        with sampler:
            barrier()
            for i in range(K):
                do_flush()
                gev[i][0].record(stream)
                graph.replay()
                gev[i][1].record(stream)
            barrier()
        step_ms = sum(a.elapsed_time(b) for a, b in gev) / K
    step_ms, attn_ms = max_over_ranks([step_ms, attn_ms], dev)

    # ---- end to end through the C ABI with host buffers
    q_host = st.q.cpu().pin_memory() if wl.mode == "attn" else st.x.cpu().pin_memory()
    q_dev = st.q if wl.mode == "attn" else st.x
    lens_host = st.seq_lens.cpu().pin_memory()
    bt_host = st.block_table.cpu().pin_memory()
    res = st.result()
    out_host = torch.empty(res.shape, dtype=res.dtype, pin_memory=True)
    Ke = min(K, 100)
    e2e = []
    for i in range(Ke + 2):
        do_flush()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        q_dev.copy_(q_host, non_blocking=True)
        st.seq_lens.copy_(lens_host, non_blocking=True)
        st.block_table.copy_(bt_host, non_blocking=True)
        if graph is not None:
            graph.replay()
        else:
            st.run()
        out_host.copy_(res, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= 2:
            e2e.append(a.elapsed_time(b))
    e2e_ms = sum(e2e) / len(e2e)
    e2e_ms, = max_over_ranks([e2e_ms], dev)
    h2d = q_host.numel() * q_host.element_size() + lens_host.numel() * 4 + bt_host.numel() * 4
    d2h = out_host.numel() * out_host.element_size()

    hbm, tflops, peak_kind = peaks()
    alg_bytes, alg_flops = algorithmic(wl, st.lens_np)
    achieved = alg_bytes / (attn_ms * 1e-3) / 1e9
    tensor_achieved = alg_flops / (attn_ms * 1e-3) / 1e12
    t_hbm = alg_bytes / (hbm * 1e9)
    t_flop = alg_flops / (tflops * 1e12)
    path = M.mla_decode_path(st.dtype, st.dims)
    line = {
        "metric": METRIC, "value": step_ms * 1e3, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.batch, "ctx": int(st.lens_np.max()),
                   "ctx_total": int(st.lens_np.sum()), "n_h": wl.n_h, "d_c": wl.d_c,
                   "d_r": wl.d_r, "page_size": wl.page_size,
                   "l2": f"flushed before every timed step (read of a {2 * l2 >> 20} MiB buffer, untimed)",
                   "decode_kernel": "tcgen05" if path == 1 else "simt",
                   "step_launch": "cuda_graph" if graph is not None else f"eager ({graph_err})",
                   "e2e_launch": "pinned copies + cuda_graph + copy back" if graph is not None
                   else "pinned copies + eager calls + copy back",
                   "eager_us_per_step": eager_ms * 1e3,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm" if t_hbm >= t_flop else "tensor", "achieved": achieved,
                     "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": DECODE_TRAFFIC.get(wl.name) if path == 1 else None,
                     "kernel": "mla_decode_attn", "kernel_us": attn_ms * 1e3,
                     "alg_bytes": alg_bytes, "alg_flops": alg_flops,
                     "tensor_tflops": tensor_achieved, "tensor_peak": tflops,
                     "tensor_frac": tensor_achieved / tflops,
                     "roofline_us": max(t_hbm, t_flop) * 1e6,
                     "frac_of_roofline": max(t_hbm, t_flop) / (attn_ms * 1e-3),
                     "peak_source": peak_kind},
        "e2e": {"value": e2e_ms * 1e3, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * K * (2 if graph is not None else 1),
        "clocks": sampler.summary(),
        "wall_s_timed": t_wall,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and wl.mode == "attn":
        line["cpu_baseline"] = cpu_baseline_entry(wl, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
