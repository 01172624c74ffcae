"""Benchmark of the SSD forward scan on B300: tokens/s, TFLOP/s, fraction of
roofline, next to the fp64 CPU oracle.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 2] [--algo auto|simt|tc|tc2]

A step is one ssd_scan() over the whole workload (default: the 2.7B-shaped
SSD layer, batch 4 x 8192 tokens, 80 heads, P=64, N=128, chunk 256, bf16),
inputs resident in HBM.  Under torchrun each rank runs its own full copy of
the workload (independent problems: weak scaling, no collective on the data
path); rank 0 prints one JSON line.
``--impl reference`` times the CPU oracle on the host cores instead (a bounded
sample of the same workload per step).

``--op step`` measures the decode step instead (ssd_step: one token for each
of 64 sequences of the 2.7B-shaped layer, the fp32 state updated in place),
with its own JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import ssd_synth  # noqa: E402

L2_BYTES = 126 * 1024 * 1024


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0,
                    source="fallback")


def workload_cost(inp):
    """Algorithmic bytes and FLOPs of one scan over ``inp``.

    bytes: x, y, B, C, dt (+ initial/final states, A, D) each moved once.
    FLOPs (causal count): per token and head (Q+1)P for the masked intra-chunk
    product and 4NP for the chunk state and the output from the carried state;
    per token and group (Q+1)N for C B^T.  The dense count is what square
    tensor-core tiles execute: 2QP + 4NP per token-head and 2QN per token-group.
    """
    b, L, H, P, N, G, Q = (inp[k] for k in ("batch", "seqlen", "nheads", "headdim", "dstate",
                                            "ngroups", "chunk"))
    esz = 2 if inp["dtype"] == "bf16" else 4
    T = b * L
    nbytes = 2 * T * H * P * esz + 2 * T * G * N * esz + T * H * 4 + 2 * H * 4
    nstates = inp["nseq"] * H * P * N * 4
    if inp["initial_states"] is not None:
        nbytes += nstates
    nbytes += nstates  # final_states written
    causal = T * (H * ((Q + 1) * P + 4 * N * P) + G * (Q + 1) * N)
    dense = T * (H * (2 * Q * P + 4 * N * P) + G * 2 * Q * N)
    return nbytes, causal, dense


class ClockSampler:
    """Samples SM clock and clock-event (throttle) reasons while the timed
    region runs: NVML when the Python bindings are present, else a
    background `nvidia-smi --query-gpu ... -lms` process."""

    REASONS = {
        0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
        0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
        0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
        0x100: "display_clock_setting",
    }

    def __init__(self, index: int):
        self.index = index
        self.samples = []          # (host time, sm MHz, reasons bitmask)
        self.max_mhz = None
        self._stop = threading.Event()
        self._proc = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.source = "nvml"
        except Exception:
            self.source = "nvidia-smi"

    def _run_nvml(self):
        nv = self.nv
        while not self._stop.is_set():
            try:
                mhz = nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM)
                rs = nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                self.samples.append((time.perf_counter(), mhz, rs))
            except Exception:
                pass
            time.sleep(0.002)

    def _run_smi(self):
        import subprocess
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        for line in self._proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            try:
                mhz, mx, rs = float(parts[0]), float(parts[1]), int(parts[2], 16)
            except (ValueError, IndexError):
                continue
            self.max_mhz = mx
            self.samples.append((time.perf_counter(), mhz, rs))
            if self._stop.is_set():
                break

    def __enter__(self):
        self.t = threading.Thread(target=self._run_nvml if self.source == "nvml" else self._run_smi,
                                  daemon=True)
        self.t.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
        self.t.join(timeout=5)

    def summary(self, t0, t1):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no_samples"],
                    "source": self.source}
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        note = "in_timed_region"
        if not inside:
            # the timed region was shorter than the sampling period: use the
            # samples closest to it
            inside = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            note = "nearest_to_timed_region"
        mask = 0
        for s in inside:
            mask |= s[2]
        reasons = [n for bit, n in self.REASONS.items() if mask & bit and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(inside), "window": note,
                "source": self.source}


KERNEL_OF_ALGO = {"tc": ("k_ssd_fused", "ssd_fused.cu"),
                  "tc2": ("k_chunk_state + k_chunk_output", "ssd_tc.cu"),
                  "simt": ("k1..k5 SIMT kernels", "ssd_simt.cu")}


def profiled_traffic(kernel_src: str, workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary (profiles/<kernel>_<workload>.md), or None when there is none or
    the kernel's source has changed since the counters were taken."""
    import hashlib
    src = os.path.join(ROOT, "mamba_ssd_layer_03_b300", "csrc", kernel_src)
    path = os.path.join(ROOT, "profiles", f"{kernel_src.split('.')[0]}_{workload}.md")
    try:
        with open(src, "rb") as f:
            sha = hashlib.sha1(f.read()).hexdigest()
        fields = {}
        with open(path) as f:
            for line in f:
                if ":" in line and line.startswith("- "):
                    k, v = line[2:].split(":", 1)
                    fields[k.strip()] = v.strip().strip("`")
        if fields.get("source_sha1") != sha:
            return None
        return int(fields["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def aggregate_over_ranks(local_ms: float, tokens_per_rank: int, steps: int, dist=None,
                         device=None):
    """Whole-job throughput of `steps` timed steps: every rank processed
    `tokens_per_rank` tokens per step; the job took as long as its slowest
    rank.  Returns (max over ranks of the timed milliseconds, tokens/s)."""
    world = 1
    if dist is not None and dist.is_initialized():
        world = dist.get_world_size()
        t = torch.tensor([local_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        local_ms = float(t.item())
    return local_ms, tokens_per_rank * world * steps / (local_ms / 1e3)


def time_oracle_sample(inp, budget_s: float):
    """Run the CPU oracle on (sequence, head) units of ``inp`` for about
    ``budget_s`` seconds, one unit per host thread at a time; return
    (tokens/s equivalent, units, seconds, threads)."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    H, nseq = inp["nheads"], inp["nseq"]
    threads = oracle.max_threads()
    cu = inp["cu_seqlens"]
    seq_len = ([int(cu[s + 1] - cu[s]) for s in range(nseq)] if cu is not None
               else [inp["seqlen"]] * nseq)
    order = [(s, h) for h in range(H) for s in range(nseq)]

    def one(u):
        oracle.recurrent_unit(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                              inp["initial_states"], cu, u[0], u[1])
        return seq_len[u[0]]

    done, tok_heads = 0, 0
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as pool:
        while time.perf_counter() - t0 < budget_s and done < len(order):
            batch = order[done:done + threads]
            tok_heads += sum(pool.map(one, batch))
            done += len(batch)
    elapsed = time.perf_counter() - t0
    return tok_heads / H / elapsed, done, elapsed, threads


def oracle_step_budget(steps: int, warmup: int) -> float:
    """Seconds of oracle work per sample: the reference arm spreads about
    150 s over its warm-up and timed steps, 1 to 20 s each."""
    return max(1.0, min(20.0, 150.0 / max(1, steps + warmup)))


def oracle_rate(inp, samples: int, warmup: int, budget_s: float):
    """The oracle's throughput as both arms report it: ``warmup`` untimed
    samples of ``budget_s`` seconds (the first one also starts the thread
    pool and touches the inputs), then the mean rate over ``samples`` timed
    samples of the same budget.  Returns (tokens/s, units, seconds, threads)."""
    for _ in range(warmup):
        time_oracle_sample(inp, budget_s)
    rates, units, secs, threads = [], 0, 0.0, 1
    for _ in range(max(1, samples)):
        rate, u, sec, threads = time_oracle_sample(inp, budget_s)
        rates.append(rate)
        units += u
        secs += sec
    return statistics.mean(rates), units, secs, threads


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--algo", default="auto", choices=["auto", "simt", "tc", "tc2"])
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="about this many seconds of timed oracle work for the cpu_baseline "
                         "leg (at least one sample of the reference arm's per-step budget)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=None,
                    help="seconds of oracle work per step of --impl reference (default: the "
                         "run's 150 s spread over its steps, 1 to 20 s each)")
    ap.add_argument("--seqlen", type=int, default=None,
                    help="override the workload's tokens per sequence (profiling captures)")
    ap.add_argument("--dt-softplus", action="store_true",
                    help="pass the raw step sizes and let the scan apply dt' = softplus(dt + "
                         "bias) (the step-size transform) as it reads them")
    ap.add_argument("--op", default="scan", choices=["scan", "step", "seqpar"])
    ap.add_argument("--shards", type=int, default=2,
                    help="shards per sequence (--op seqpar)")
    ap.add_argument("--step-batch", type=int, default=64,
                    help="sequences per decode step (--op step)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = ssd_synth.WORKLOADS[args.workload]

    if args.impl == "reference":
        return run_reference(args, w, rank, world)
    if args.op == "step":
        return run_step_bench(args, w, rank, world, local)
    if args.op == "seqpar":
        return run_seqpar_bench(args, w, rank, world, local)

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import mamba_ssd_layer_03_b300 as ssd

    inp = ssd_synth.make_inputs(w, seed=rank, seqlen=args.seqlen)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    shape = ssd.make_shape(inp["batch"], inp["seqlen"], inp["nheads"], inp["headdim"],
                           inp["dstate"], inp["ngroups"], inp["chunk"], inp["nseq"],
                           d["x"].dtype, args.algo)
    algo = ssd.resolve_algo(shape)
    # with --dt-softplus the scan reads the raw step sizes and the per-head
    # bias and applies the transform itself
    tfk = dict(dt_bias=d["dt_bias"], dt_softplus=True) if args.dt_softplus else {}
    dt_key = "dt_raw" if args.dt_softplus else "dt"
    ws = torch.empty(ssd.workspace_size(shape, ssd.make_dt_transform(**tfk)), dtype=torch.uint8,
                     device=dev)
    y = torch.empty_like(d["x"])
    fin = torch.empty(inp["nseq"], inp["nheads"], inp["headdim"], inp["dstate"],
                      dtype=torch.float32, device=dev)

    def step():
        ssd.ssd_scan(d["x"], d[dt_key], d["A"], d["B"], d["C"], d["D"], inp["chunk"],
                     d["initial_states"], d["cu_seqlens"], True, args.algo, out=y,
                     final_out=fin, workspace=ws, **tfk)

    stream = torch.cuda.current_stream(dev)
    # Warm-up (also checks the device status word once).
    for _ in range(max(args.warmup, 1)):
        step()
    rc = ssd.load_library().ssd_check_device_status(ssd._ptr(ws), ssd.ctypes.c_void_p(stream.cuda_stream))
    if rc != 0:
        raise ssd.SsdError(rc, "warm-up")

    nbytes, causal, dense = workload_cost(inp)
    peaks = load_peaks()

    # The K timed steps are captured once as a CUDA graph and replayed: the
    # device runs them back to back, with no host time between launches (a
    # small workload's kernel is shorter than the Python call that launches
    # it).  The end-to-end figure below keeps the host in the loop.
    # A workload that fits in L2 gets an L2 flush (a write over a buffer twice
    # the L2's size) before every step; the flushes alone are timed as a graph
    # of their own and subtracted.
    flush = None
    if nbytes < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(args.steps):
            if flush is not None:
                flush.fill_(1)
            step()
    flush_ms = 0.0
    if flush is not None:
        fgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(fgraph):
            for _ in range(args.steps):
                flush.fill_(1)
        fgraph.replay()
        torch.cuda.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        fgraph.replay()
        f1.record(stream)
        torch.cuda.synchronize()
        flush_ms = f0.elapsed_time(f1)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    with sampler:
        time.sleep(0.3)   # let the sampler start
        for _ in range(max(args.warmup, 1)):
            step()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        t_host0 = time.perf_counter()
        ev0.record(stream)
        graph.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        t_host1 = time.perf_counter()
        if dist:
            dist.barrier()
        time.sleep(0.15)
    total_ms = max(ev0.elapsed_time(ev1) - flush_ms, 1e-6)
    per_step = [total_ms / args.steps]
    tokens = inp["batch"] * inp["seqlen"]
    total_ms, value = aggregate_over_ranks(total_ms, tokens, args.steps, dist, dev)
    ms_per_step = total_ms / args.steps
    kernel_ms = statistics.mean(per_step)
    achieved_gbs = nbytes / (kernel_ms / 1e3) / 1e9
    tflops = causal / (ms_per_step / 1e3) / 1e12
    t_roof_ms = max(nbytes / (peaks["hbm_gbs"] * 1e9), causal / (peaks["bf16_tflops"] * 1e12)) * 1e3

    # End-to-end through the public API with host buffers: pinned host -> device
    # copies of the step's inputs, the scan, and the device -> host read of y.
    e2e = None
    if rank == 0 or world > 1:
        host = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        in_keys = ("x", dt_key, "A", "B", "C", "D", "initial_states", "cu_seqlens") + (
            ("dt_bias",) if tfk else ())
        h2d = sum(host[k].numel() * host[k].element_size() for k in in_keys if host[k] is not None)
        y_host = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
        fin_host = torch.empty(fin.shape, dtype=fin.dtype, pin_memory=True)
        d2h = y_host.numel() * y_host.element_size() + fin_host.numel() * fin_host.element_size()
        dbuf = {k: (torch.empty_like(d[k]) if d[k] is not None else None) for k in in_keys}

        def e2e_step():
            for k in in_keys:
                if host[k] is not None:
                    dbuf[k].copy_(host[k], non_blocking=True)
            tf_e2e = dict(dt_bias=dbuf["dt_bias"], dt_softplus=True) if tfk else {}
            ssd.ssd_scan(dbuf["x"], dbuf[dt_key], dbuf["A"], dbuf["B"], dbuf["C"], dbuf["D"],
                         inp["chunk"], dbuf["initial_states"], dbuf["cu_seqlens"], True,
                         args.algo, out=y, final_out=fin, workspace=ws, **tf_e2e)
            y_host.copy_(y, non_blocking=True)
            fin_host.copy_(fin, non_blocking=True)

        for _ in range(max(2, min(args.warmup, 3))):
            e2e_step()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        k_e2e = max(3, min(args.steps, 10))
        for _ in range(k_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / k_e2e
        e2e = {"value": tokens * world / (e2e_ms / 1e3), "unit": "tokens/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the reference arm's procedure and per-sample budget, fewer samples
        budget = oracle_step_budget(args.steps, args.warmup)
        nsamp = max(1, int(round(args.cpu_budget / budget)))
        rate, units, secs, threads = oracle_rate(inp, nsamp, 1, budget)
        cpu = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"1 warm-up + {nsamp} timed samples of {budget:.3g} s each (the "
                         f"reference arm's per-step budget for these --steps/--warmup): "
                         f"{units} (sequence, head) units of the same workload in total, full "
                         f"length, fp64 recurrence, {secs:.1f} s timed; mean of the samples' "
                         f"tokens/s = unit-tokens / nheads / seconds"}

    if rank == 0:
        clocks = sampler.summary(t_host0, t_host1)
        out = {
            "metric": "SSD fwd tokens/s (TFLOP/s and % of roofline alongside) on 1 B300",
            "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if inp["dtype"] == "bf16" else "f32",
            "data": "synthetic (seeded, the workload's distributions)",
            "config": {"workload": w.name, "batch": inp["batch"], "seqlen": inp["seqlen"],
                       "nheads": inp["nheads"], "headdim": inp["headdim"], "dstate": inp["dstate"],
                       "ngroups": inp["ngroups"], "chunk": inp["chunk"], "algo": algo,
                       "parallelism": f"replicas x{world} (independent problems)",
                       "launch": "cuda graph of the timed steps",
                       "l2": (f"inputs larger than L2: {nbytes / 1e6:.0f} MB streamed per step vs "
                              f"{L2_BYTES / 2**20:.0f} MiB L2, no flush") if flush is None else
                             (f"inputs ({nbytes / 1e6:.0f} MB) fit in L2: L2 flushed before every step "
                              f"(write of {2 * L2_BYTES / 2**20:.0f} MiB), flush time subtracted")},
            "tflops": tflops, "tflops_dense_equiv": dense / (ms_per_step / 1e3) / 1e12,
            "roofline_time_ms": t_roof_ms, "frac_of_roofline": t_roof_ms / ms_per_step,
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved_gbs / peaks["hbm_gbs"],
                         "traffic": profiled_traffic(KERNEL_OF_ALGO[algo][1], w.name)
                         if args.seqlen is None else None,
                         "peak_source": peaks["source"],
                         "kernel": KERNEL_OF_ALGO[algo][0] + " (timed as the whole ssd_scan call, "
                                   "mean over the graph's steps)",
                         "algorithmic_bytes": nbytes, "kernel_ms": kernel_ms},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": None,
            "clocks": clocks,
        }
        if args.seqlen is not None:
            out["config"]["seqlen_override"] = args.seqlen
        if tfk:
            out["config"]["dt_transform"] = "dt' = softplus(dt + bias), applied by the scan"
        out["gpu_launches"] = (launches_per_step(
            algo, inp, torch.cuda.get_device_properties(dev).multi_processor_count)
            + (1 if tfk and algo != "tc" else 0)) * args.steps
        print(json.dumps(out))
    if dist:
        dist.destroy_process_group()


def step_inputs(w, batch, seed):
    """One decode step's inputs for the shape of workload w: the token of each
    sequence drawn like the workload's tokens (seeded), the states ~ N(0, 0.1)."""
    inp = ssd_synth.make_inputs(w, seed=seed, batch=batch, seqlen=1)
    g = torch.Generator().manual_seed(seed + 1000)
    state = torch.randn(batch, inp["nheads"], inp["headdim"], inp["dstate"], generator=g) * 0.1
    return dict(x=inp["x"][:, 0].contiguous(), dt=inp["dt"][:, 0].contiguous(), A=inp["A"],
                B=inp["B"][:, 0].contiguous(), C=inp["C"][:, 0].contiguous(), D=inp["D"],
                state=state.contiguous(), dtype=inp["dtype"])


def step_cost(inp):
    """Algorithmic bytes of one decode step: the state read and written once,
    x, y, B, C, dt, A, D once."""
    nb = lambda t: t.numel() * t.element_size()
    return (2 * nb(inp["state"]) + 2 * nb(inp["x"]) + nb(inp["B"]) + nb(inp["C"]) + nb(inp["dt"])
            + nb(inp["A"]) + nb(inp["D"]))


def run_step_bench(args, w, rank, world, local):
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import mamba_ssd_layer_03_b300 as ssd

    inp = step_inputs(w, args.step_batch, seed=rank)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y = torch.empty_like(d["x"])
    stream = torch.cuda.current_stream(dev)

    def step():
        ssd.ssd_step(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["state"], out=y)

    nbytes = step_cost(inp)
    peaks = load_peaks()
    steps = max(args.steps, 1)
    # A decode loop replays its steps as a CUDA graph: one launch each, no
    # host time between them.  The K timed steps are one captured graph.
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(steps):
            step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    with sampler:
        time.sleep(0.3)
        for _ in range(max(args.warmup, 3)):
            graph.replay()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_host0 = time.perf_counter()
        ev0.record(stream)
        graph.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        t_host1 = time.perf_counter()
        if dist:
            dist.barrier()
        time.sleep(0.15)
    total_ms = ev0.elapsed_time(ev1)
    tokens = inp["x"].shape[0]
    total_ms, value = aggregate_over_ranks(total_ms, tokens, steps, dist, dev)
    ms = total_ms / steps
    achieved = nbytes / (ms / 1e3) / 1e9

    e2e = None
    if rank == 0 or world > 1:
        # a decode loop keeps the state on the device; each step's token
        # (x, dt, B, C) comes from the host and y goes back
        in_keys = ("x", "dt", "B", "C")
        host = {k: inp[k].pin_memory() for k in in_keys}
        dbuf = {k: torch.empty_like(d[k]) for k in in_keys}
        y_host = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
        h2d = sum(host[k].numel() * host[k].element_size() for k in in_keys)
        d2h = y_host.numel() * y_host.element_size()

        def e2e_step():
            for k in in_keys:
                dbuf[k].copy_(host[k], non_blocking=True)
            ssd.ssd_step(dbuf["x"], dbuf["dt"], d["A"], dbuf["B"], dbuf["C"], d["D"], d["state"],
                         out=y)
            y_host.copy_(y, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        k_e2e = max(3, min(steps, 50))
        for _ in range(k_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / k_e2e
        e2e = {"value": tokens * world / (e2e_ms / 1e3), "unit": "tokens/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        reps = 0
        t0 = time.perf_counter()
        while True:
            oracle.step(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"], inp["state"])
            reps += 1
            if time.perf_counter() - t0 > min(args.cpu_budget, 10.0):
                break
        secs = time.perf_counter() - t0
        cpu = {"value": reps * tokens / secs, "unit": "tokens/s", "cores": oracle.max_threads(),
               "kind": "oracle", "sample": f"{reps} full decode steps of the same batch, fp64, "
                                           f"{secs:.1f} s"}

    if rank == 0:
        b, H, P = inp["x"].shape
        N = inp["state"].shape[-1]
        wname = f"decode_h{H}_p{P}_n{N}_b{b}"
        out = {
            "metric": "SSD decode step tokens/s (one token per sequence, state in place) on 1 B300",
            "value": value, "unit": "tokens/s", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": inp["dtype"],
            "data": "synthetic (seeded, the workload's distributions)",
            "config": {"workload": wname, "batch": b, "nheads": H, "headdim": P,
                       "dstate": N, "ngroups": inp["B"].shape[1], "launch": "cuda graph of the timed steps",
                       "parallelism": f"replicas x{world} (independent problems)",
                       "l2": f"state larger than L2: {nbytes / 1e6:.0f} MB streamed per step vs "
                             f"{L2_BYTES / 2**20:.0f} MiB L2, no flush"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                         "traffic": profiled_traffic("ssd_step.cu", wname),
                         "peak_source": peaks["source"],
                         "kernel": "k_ssd_step (timed as the whole ssd_step call)",
                         "algorithmic_bytes": nbytes, "kernel_ms": ms},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": steps,
            "clocks": sampler.summary(t_host0, t_host1),
        }
        print(json.dumps(out))
    if dist:
        dist.destroy_process_group()


def run_seqpar_bench(args, w, rank, world, local):
    """Device work of one rank of the sequence-parallel scan (seqpar.py): the
    last of ``--shards`` consecutive shards of every sequence of workload w,
    which folds the most carries.  A step is the shard's state-only scan from
    a zero state, its log-decay, the fold of all shards' carries into its
    entry state and the final state, and the scan from the entry state.  The
    all_gather is not in the step (one GPU: there is no peer); the other
    shards' carries are stand-ins of the right size, and the rank's own carry
    is copied into its slot as the collective would place it."""
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from mamba_ssd_layer_03_b300 import seqpar
    R = max(1, args.shards)
    Ls = w.seqlen // R
    inp = ssd_synth.make_inputs(w, seed=rank, seqlen=Ls, init_states=True)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    b, H, P, N = inp["batch"], inp["nheads"], inp["headdim"], inp["dstate"]
    g = torch.Generator(device=dev).manual_seed(7)
    S_all = torch.randn(R, b, H, P, N, generator=g, device=dev) * 0.1
    ld_all = -torch.rand(R, b, H, generator=g, device=dev) * 4.0
    ops = seqpar.CudaOps(args.algo)
    y = torch.empty_like(d["x"])
    me = R - 1
    import mamba_ssd_layer_03_b300 as ssd
    algo = ssd.resolve_algo(ssd.make_shape(b, Ls, H, P, N, inp["ngroups"], inp["chunk"], b,
                                           d["x"].dtype, args.algo))
    launches = 2 * launches_per_step(algo, inp, torch.cuda.get_device_properties(dev)
                                     .multi_processor_count) + 2

    def step():
        S = ops.states(d["x"], d["dt"], d["A"], d["B"], d["C"], inp["chunk"])
        ld = ops.logdec(d["dt"], d["A"])
        S_all[me].copy_(S)
        ld_all[me].copy_(ld)
        entry, fin = ops.fold(S_all, ld_all, me, d["initial_states"])
        ops.scan(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], inp["chunk"], entry, out=y,
                 final=False)
        return fin

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    # the K timed steps as one CUDA graph, as in the scan bench: the four
    # library calls of a step are host work that would otherwise leave the
    # device idle between kernels
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(args.steps):
            step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(local)
    with sampler:
        time.sleep(0.3)
        graph.replay()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_host0 = time.perf_counter()
        ev0.record(stream)
        graph.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        t_host1 = time.perf_counter()
        time.sleep(0.15)
    ms = ev0.elapsed_time(ev1) / args.steps
    scan_bytes, _, _ = workload_cost(inp)
    state = b * H * P * N * 4
    # the state-only scan (x, B, dt read, states written), the full scan, the
    # log-decay's dt read, the fold's R carries read, initial states read,
    # entry and final states written
    esz = 2 if inp["dtype"] == "bf16" else 4
    first = b * Ls * (H * P * esz + inp["ngroups"] * N * esz + H * 4) + state
    nbytes = first + scan_bytes + b * Ls * H * 4 + R * (state + b * H * 4) + 3 * state
    peaks = load_peaks()
    if rank == 0:
        out = {
            "metric": "SSD sequence-parallel scan, one rank's device work, shard tokens/s on 1 B300",
            "value": b * Ls / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": inp["dtype"],
            "data": "synthetic (seeded, the workload's distributions)",
            "config": {"workload": f"{w.name}_shard{R - 1}of{R}", "batch": b, "shard_seqlen": Ls,
                       "nheads": H, "headdim": P, "dstate": N, "algo": algo,
                       "launch": "cuda graph of the timed steps (four library calls each)",
                       "collective": "not timed: one GPU, no peers; the other shards' carries "
                                     "are stand-ins"},
            "roofline": {"bound": "hbm", "achieved": nbytes / (ms / 1e3) / 1e9,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": nbytes / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                         "traffic": None, "peak_source": peaks["source"],
                         "kernel": "two scans + k_shard_logdec + k_carry_fold (whole step)",
                         "algorithmic_bytes": nbytes, "kernel_ms": ms},
            "cpu_baseline": None, "e2e": None,
            "gpu_launches": launches * args.steps,
            "clocks": sampler.summary(t_host0, t_host1),
        }
        print(json.dumps(out))


def fused_splits_lanes(inp, sms):
    """Whether the fused kernel splits lanes between CTAs (its two-run mode):
    at most half as many lanes as SMs, at least 16 blocks per lane, no
    packing."""
    if inp["cu_seqlens"] is not None:
        return False
    hpl = 1 if inp["dstate"] == 256 else 2
    hpg = inp["nheads"] // inp["ngroups"]
    lanes = inp["nseq"] * inp["ngroups"] * ((hpg + hpl - 1) // hpl)
    nb = (inp["seqlen"] + 127) // 128
    return lanes * 2 <= sms and nb >= 16


def launches_per_step(algo, inp, sms=148):
    """Kernels libssd launches per ssd_scan() (memset of the status word is
    a copy-engine op, not a kernel)."""
    varlen = inp["cu_seqlens"] is not None
    if algo == "simt":
        return 4 + (2 if varlen else 0)
    if algo == "tc":       # fused kernel (+ cu_seqlens check and set-up; + the pre run of split lanes)
        return 1 + (2 if varlen else 0) + (1 if fused_splits_lanes(inp, sms) else 0)
    return 2


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    import oracle
    inp = ssd_synth.make_inputs(w, seed=0)
    budget = args.ref_budget if args.ref_budget else oracle_step_budget(args.steps, args.warmup)
    value, _, _, threads = oracle_rate(inp, args.steps, args.warmup, budget)
    tokens = inp["batch"] * inp["seqlen"]
    sample = (f"each step: about {budget:.3g} s of (sequence, head) units of the same workload "
              f"(full length, fp64 recurrence); tokens/s = unit-tokens / nheads / seconds")
    out = {
        "impl": "reference", "metric": "SSD fwd tokens/s (TFLOP/s and % of roofline alongside) on 1 B300",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": tokens / value * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": inp["batch"], "seqlen": inp["seqlen"],
                   "nheads": inp["nheads"], "headdim": inp["headdim"], "dstate": inp["dstate"],
                   "ngroups": inp["ngroups"], "chunk": inp["chunk"]},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "kind": "oracle",
                         "cores": threads, "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))


if __name__ == "__main__":
    main()
