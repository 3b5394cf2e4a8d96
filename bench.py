#!/usr/bin/env python3
"""Benchmark of the grouped FP8 block-scaled GEMM on GB300.

One step = one call of the grouped GEMM over one batch of synthetic input
(the whole path: scale staging, tile scheduling, TMA operand loads,
block-scaled tcgen05 MMAs and the epilogue all run inside the one kernel the
call launches).  The default workload is the contiguous G=8 x 1024-row,
N=2048, K=7168 expert projection with transposed activation scales and bf16
output.  Metric: TFLOP/s = 2 * sum(valid rows) * N * K / time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle as the reference arm

Under torchrun (N > 1) every rank runs an independent replica (the path has
no exchange step), the timing is the max over ranks and `value` counts the
work of all ranks.  Only rank 0 prints the JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

DEFAULT_WORKLOAD = "c2_contig_g8_m1024_n2048_k7168"
METRIC = "grouped FP8 GEMM TFLOP/s (2*sum(m)*N*K/t)"
FP8_OVER_BF16 = 4.5 / 2.25   # nominal dense tensor-core ratios of GB300
FP4_OVER_BF16 = 13.5 / 2.25
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
CSRC = os.path.join(ROOT, "fp8_block_scaled_gb300", "csrc")


def _kernel_sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh")))


def _code_only(text: str) -> str:
    """Source text without comments and whitespace, so that the hash below
    changes with the code, not with its comments."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return re.sub(r"\s+", "", text)


def kernel_hash() -> str:
    h = hashlib.sha256()
    for p in _kernel_sources():
        with open(p, encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


# ----------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 100 ms while running."""

    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.device = device
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        bus = None
        try:
            props = torch.cuda.get_device_properties(self.device)
            bus = getattr(props, "pci_bus_id", None)
        except Exception:
            pass
        rows = []
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 10:
                continue
            rows.append(parts)
        if rows and len({r[0] for r in rows}) > 1:
            if bus is not None:
                sel = [r for r in rows if r[1].lower().endswith(f"{int(bus):02x}:00.0")
                       or f":{int(bus):02x}:" in r[1].lower()]
                rows = sel or rows
            idx = rows[0][0]
            rows = [r for r in rows if r[0] == idx]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        smax = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for name, val in zip(names, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def clocks_suspect(clk) -> bool:
    """True when a clock record shows a hardware or thermal slowdown, or a median SM
    clock below 80% of the maximum with no reason reported."""
    if not clk:
        return False
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    if bad & set(clk.get("reasons") or []):
        return True
    sm, smax = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    return bool(sm and smax and sm < 0.8 * smax and not clk.get("reasons"))


# ----------------------------------------------------------------- workloads
def make_inputs(name: str, device):
    import synth

    return synth.make_config(name, device=device)


def out_dtype_of(p):
    return torch.bfloat16 if p.out_dtype == 0 else torch.float16


def run_once(fb, p, a, sa, b, sb, rowinfo, d, stream=None):
    if p.is_mx:
        if p.variant == "contiguous":
            fb.gemm_grouped_contiguous_mxfp4(a, sa, b, sb, d, rowinfo, stream=stream)
        else:
            fb.gemm_grouped_masked_mxfp4(a, sa, b, sb, d, rowinfo, stream=stream)
    elif p.epilogue == "silu_mul_quant":
        q, qs = d
        if p.variant == "contiguous":
            fb.gemm_grouped_contiguous_silu_mul_quant(a, sa, b, sb, q, qs, rowinfo, stream=stream)
        else:
            fb.gemm_grouped_masked_silu_mul_quant(a, sa, b, sb, q, qs, rowinfo, stream=stream)
    elif p.scale_kind == "fp32":
        if p.variant == "contiguous":
            fb.gemm_grouped_contiguous_fp32_scales(a, sa, b, sb, d, rowinfo, stream=stream)
        else:
            fb.gemm_grouped_masked_fp32_scales(a, sa, b, sb, d, rowinfo, stream=stream)
    elif p.variant == "contiguous":
        fb.gemm_grouped_contiguous(a, sa, b, sb, d, rowinfo, stream=stream)
    else:
        fb.gemm_grouped_masked(a, sa, b, sb, d, rowinfo, stream=stream)


def alloc_out(p, dev, pinned=False, d_offset_bytes=0):
    """The step's output: D (bf16/f16), or for the fused epilogue the E4M3 codes and
    their fp32 scales in the activation-scale layout of the workload.  Returns the
    argument run_once takes and the list of underlying tensors (on the device, or
    in pinned host memory).  d_offset_bytes > 0 places D that many bytes into a
    larger buffer (a slice, as a caller's view of a bigger tensor would be)."""
    lead = (p.rows,) if p.variant == "contiguous" else (p.G, p.M_max)
    kw = {"pin_memory": True} if pinned else {"device": dev}
    if p.epilogue != "silu_mul_quant":
        if d_offset_bytes:
            numel = math.prod(lead) * p.N
            off = d_offset_bytes // 2
            buf = torch.empty(numel + off, dtype=out_dtype_of(p), **kw)
            d = buf[off:].view(lead + (p.N,))
            return d, [d]
        d = torch.empty(lead + (p.N,), dtype=out_dtype_of(p), **kw)
        return d, [d]
    q = torch.empty(lead + (p.N // 2,), dtype=torch.uint8, **kw)
    nblk = p.N // 256
    if p.sa_layout == 0:
        store = torch.empty(lead + (nblk,), dtype=torch.float32, **kw)
        view = store
    else:
        ld = (lead[-1] + 3) // 4 * 4
        if p.variant == "contiguous":
            store = torch.empty((nblk, ld), dtype=torch.float32, **kw)
            view = store[:, : lead[-1]].t()
        else:
            store = torch.empty((p.G, nblk, ld), dtype=torch.float32, **kw)
            view = store[:, :, : lead[-1]].transpose(1, 2)
    return (q, view), [q, store]


def describe(p, l2_note):
    cfg = {"workload": p.name, "variant": p.variant, "G": p.G, "N": p.N, "K": p.K,
           "valid_rows": p.valid_rows, "rows": p.rows,
           "out": "bf16" if p.out_dtype == 0 else "f16",
           "scale_a": ("E8M0 [M, K/32]" if p.is_mx else
                       "transposed [K/128, M]" if p.sa_layout == 1 else "[M, K/128]"),
           "scales": ("E8M0 per 32 elements of A and B rows (MXFP4)" if p.is_mx else
                      "UE8M0 (1,128) activation x (128,128) weight" if p.scale_kind == "ue8m0"
                      else "arbitrary fp32 (1,128) activation x (128,128) weight, promoted in "
                           "software"),
           "parallelism": "replicas (no exchange step)", "l2": l2_note}
    if p.variant == "masked":
        cfg["M_max"] = p.M_max
    if p.epilogue == "silu_mul_quant":
        cfg["epilogue"] = ("SiLU(gate) * up of the B halves [0, N/2) and [N/2, N), requantised "
                           "to E4M3 with (1,128) UE8M0 scales")
        cfg["out"] = "e4m3 [rows, N/2] + fp32 scales " + (
            "transposed [N/256, M]" if p.sa_layout == 1 else "[M, N/256]")
    return cfg


def bench_ours(args):
    import fp8_block_scaled_gb300 as fb

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    fb.load()
    p = make_inputs(args.workload, dev)
    sa_view = p.sa_mk_view()
    rowinfo = p.grouped_layout if p.variant == "contiguous" else p.masked_m
    in_bytes = sum(t.numel() * t.element_size() for t in (p.a, p.sa, p.b, p.sb, rowinfo))
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    sets = args.input_sets or max(2, math.ceil(3 * l2 / in_bytes))
    bufs = []
    for i in range(sets):
        if i == 0:
            a, sa, b, sb, ri = p.a, sa_view, p.b, p.sb, rowinfo
        else:
            a, b, sb, ri = p.a.clone(), p.b.clone(), p.sb.clone(), rowinfo.clone()
            sa_store = p.sa.clone()
            if p.sa_layout == 1:
                sa = (sa_store[:, : p.rows].t() if p.variant == "contiguous"
                      else sa_store[:, :, : p.M_max].transpose(1, 2))
            else:
                sa = sa_store
        d, _ = alloc_out(p, dev, d_offset_bytes=args.d_offset_bytes)
        bufs.append((a, sa, b, sb, ri, d))
    l2_note = (f"rotating {sets} input sets of {in_bytes / 1e6:.1f} MB "
               f"({sets * in_bytes / 1e6:.0f} MB > L2 {l2 / 1e6:.0f} MB)")
    stream = torch.cuda.current_stream(dev)

    for i in range(args.warmup):
        run_once(fb, p, *bufs[i % sets])
    torch.cuda.synchronize(dev)
    if fb.device_error(local):
        raise RuntimeError("device error word set during warm-up")

    def timed_region():
        clocks = ClockSampler(local)
        clocks.start()
        time.sleep(0.3)
        # A step is one call: one launch of the GEMM, preceded, for row-major
        # activation scales, by the library's scale pre-pass.  The GEMM's average
        # launch duration is taken as the timed region's event time over the step
        # count, which includes the pre-pass where there is one.  Events recorded
        # between the launches would stand between two kernels of the stream and
        # keep the next grid from being scheduled while the previous one finishes
        # (programmatic dependent launch), so there are none.
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        n0 = fb.kernel_launches()
        t0.record(stream)
        for i in range(args.steps):
            run_once(fb, p, *bufs[i % sets])
        t1.record(stream)
        launches = fb.kernel_launches() - n0
        torch.cuda.synchronize(dev)
        barrier(world)
        clk = clocks.stop()
        if fb.device_error(local):
            raise RuntimeError("device error word set during the timed region")
        return t0.elapsed_time(t1), clk, launches

    elapsed_ms, clk, launches = timed_region()
    # a run slowed by the hardware or a thermal limit, or with the SM clock stuck
    # well below its maximum for no reported reason (a clock lock left by someone
    # else), is not kept: it is measured once more (a power-cap slowdown is kept)
    if max_over_ranks(1.0 if clocks_suspect(clk) else 0.0, world, dev) > 0.0:
        elapsed_ms, clk, launches = timed_region()
        clk["remeasured"] = True
    ms_per_step = max_over_ranks(elapsed_ms / args.steps, world, dev)
    flops = p.flops()
    total_flops = sum_over_ranks(flops, world, dev)
    value = total_flops / (ms_per_step * 1e-3) / 1e12

    # roofline of the one kernel on the path
    peaks, peaks_kind = load_peaks()
    mean_launch_ms = elapsed_ms / args.steps  # with the scale pre-pass, if the step has one
    kernels_per_step = launches / args.steps
    achieved = flops / (mean_launch_ms * 1e-3) / 1e12
    # the contraction's own dtype: E4M3 (or E2M1 for the MXFP4 workloads)
    ratio, ratio_name = ((FP4_OVER_BF16, "fp4/bf16") if p.is_mx else (FP8_OVER_BF16, "fp8/bf16"))
    peak_fp8 = peaks["bf16_tflops"] * ratio
    alg_bytes = p.algorithmic_bytes(out_bytes=2)
    hbm_time = alg_bytes / (peaks["hbm_gbs"] * 1e9)
    tensor_time = flops / (peak_fp8 * 1e12)
    traffic = None
    if os.path.exists(TRAFFIC_FILE):
        with open(TRAFFIC_FILE) as f:
            tr = json.load(f)
        ent = tr.get(p.name)
        if ent and ent.get("kernel_hash") == kernel_hash():
            traffic = ent["dram_bytes_per_launch"]
    if tensor_time >= hbm_time:
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak_fp8, 1),
                "unit": "TFLOP/s", "frac": round(achieved / peak_fp8, 4), "traffic": traffic,
                "peak_source": f"{peaks_kind} bf16 burst {peaks['bf16_tflops']} TFLOP/s x "
                               f"{ratio:g} (nominal {ratio_name} ratio)",
                "algorithmic": {"flops_per_launch": flops, "bytes_per_launch": alg_bytes},
                "mean_launch_ms": round(mean_launch_ms, 5), "kernels_per_step": kernels_per_step}
    else:
        gbs = alg_bytes / (mean_launch_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": traffic,
                "peak_source": f"{peaks_kind} HBM copy",
                "algorithmic": {"flops_per_launch": flops, "bytes_per_launch": alg_bytes},
                "mean_launch_ms": round(mean_launch_ms, 5), "kernels_per_step": kernels_per_step}

    # end to end through the public API with host buffers
    def e2e_line(resident_weights):
        r = bench_e2e(fb, p, dev, args.e2e_steps, resident_weights)
        r_ms = max_over_ranks(r["ms_per_step"], world, dev)
        out = {"value": round(total_flops / (r_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
               "ms_per_step": round(r_ms, 4), "h2d_bytes_per_step": r["h2d"],
               "d2h_bytes_per_step": r["d2h"]}
        if resident_weights:
            out["weights"] = "B and scale_b resident in HBM (copied once before timing)"
        return out

    e2e = e2e_line(False) if args.e2e_steps > 0 else None
    e2e_resident = e2e_line(True) if args.e2e_steps > 0 else None

    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        cpu = cpu_baseline(p, args.cpu_seconds)

    line = {"metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e2m1" if p.is_mx else "e4m3",
            "data": ("synthetic (seeded N(0,1), MXFP4-quantised)" if p.is_mx else
                     "synthetic (seeded N(0,1), fp32 block scales)" if p.scale_kind == "fp32" else
                     "synthetic (seeded N(0,1), UE8M0 ceil-quantised)"),
            "config": dict(describe(p, l2_note),
                           **({"d_offset_bytes": args.d_offset_bytes} if args.d_offset_bytes else {})),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "e2e_resident_weights": e2e_resident,
            "gpu_launches": int(round(sum_over_ranks(launches, world, dev))), "clocks": clk,
            "roofline_time_ms": {"tensor_at_peak": tensor_time * 1e3, "hbm_at_peak": hbm_time * 1e3}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def bench_e2e(fb, p, dev, steps, resident_weights=False):
    """Same metric through the public API, inputs in pinned host memory: every
    step copies its inputs host->device, runs the GEMM and reads its result back.

    The steps are pipelined the way a serving loop would run them: two device
    copies of the inputs and of the result, the host->device copies of step i+1
    on one stream while step i computes on a second and its result returns on a
    third, so the two copy directions and the GEMM overlap.  Every step's copies
    are inside the timed region.

    resident_weights: the expert weights and their scales (B, scale_b) are model
    parameters held in HBM, copied once before the timed region; each step
    copies only the activations, their scales and the row map."""
    rowinfo = p.grouped_layout if p.variant == "contiguous" else p.masked_m
    host = [t.cpu().pin_memory() for t in (p.a, p.sa, p.b, p.sb, rowinfo)]
    sets = [[torch.empty_like(t, device=dev) for t in host] for _ in range(2)]
    per_step = [0, 1, 4] if resident_weights else [0, 1, 2, 3, 4]
    if resident_weights:
        for x in sets:
            for j in (2, 3):
                x[j].copy_(host[j])
    outs = [alloc_out(p, dev) for _ in range(2)]
    _, d_host = alloc_out(p, dev, pinned=True)
    s_in, s_gemm, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_gemm = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def sa_view(sa):
        if p.sa_layout == 0:
            return sa
        return sa[:, : p.rows].t() if p.variant == "contiguous" else sa[:, :, : p.M_max].transpose(1, 2)

    def step(i):
        b = i % 2
        s_in.wait_event(ev_gemm[b])          # the GEMM that last read input set b is done
        with torch.cuda.stream(s_in):
            for j in per_step:
                sets[b][j].copy_(host[j], non_blocking=True)
            ev_in[b].record(s_in)
        s_gemm.wait_event(ev_in[b])
        s_gemm.wait_event(ev_out[b])         # result buffer b has been read back
        with torch.cuda.stream(s_gemm):
            x = sets[b]
            run_once(fb, p, x[0], sa_view(x[1]), x[2], x[3], x[4], outs[b][0], stream=s_gemm)
            ev_gemm[b].record(s_gemm)
        s_out.wait_event(ev_gemm[b])
        with torch.cuda.stream(s_out):
            for h, g in zip(d_host, outs[b][1]):
                h.copy_(g, non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(2):
        step(i)
    torch.cuda.synchronize(dev)
    cur = torch.cuda.current_stream(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(cur)
    for s in (s_in, s_gemm, s_out):
        s.wait_stream(cur)
    for i in range(steps):
        step(i)
    for s in (s_in, s_gemm, s_out):
        cur.wait_stream(s)
    t1.record(cur)
    torch.cuda.synchronize(dev)
    h2d = sum(host[j].numel() * host[j].element_size() for j in per_step)
    return {"ms_per_step": t0.elapsed_time(t1) / steps, "h2d": h2d,
            "d2h": sum(t.numel() * t.element_size() for t in d_host)}


def _oracle_call(p, host, rows):
    import oracle

    a, sa, b, sb, ri = host
    if p.is_mx:
        if p.variant == "contiguous":
            return oracle.mxfp4_contiguous(a, sa, b, sb, ri, rows=rows)
        return oracle.mxfp4_masked(a, sa, b, sb, ri, rows=rows)
    if p.variant == "contiguous":
        res = oracle.grouped_contiguous(a, sa, p.sa_layout, b, sb, ri, rows=rows, ld_sa=p.ld_sa)
    else:
        res = oracle.grouped_masked(a, sa, p.sa_layout, b, sb, ri, rows=rows, ld_sa=p.ld_sa)
    if p.epilogue == "silu_mul_quant":
        oracle.silu_mul_quant(res[0])
    return res


def _host_inputs(p):
    rowinfo = p.grouped_layout if p.variant == "contiguous" else p.masked_m
    return [t.cpu().numpy() for t in (p.a, p.sa, p.b, p.sb, rowinfo)]


def _valid_row_list(p):
    """Every valid (computed) row of the problem, as flattened row indices."""
    rows = []
    for g, m in enumerate(p.group_sizes):
        base = p.row_offsets[g] if p.variant == "contiguous" else g * p.M_max
        rows.extend(range(base, base + m))
    return np.array(rows, dtype=np.int64)


def cpu_baseline(p, seconds: float):
    """The oracle as it stands, on the host cores, over a seeded row sample
    sized to take about `seconds` of CPU time."""
    import oracle

    host = _host_inputs(p)
    allrows = _valid_row_list(p)
    rng = np.random.default_rng(0)
    probe = np.sort(rng.choice(allrows, size=min(len(allrows), 2 * oracle.max_threads()),
                               replace=False))
    t = time.perf_counter()
    _oracle_call(p, host, probe)
    per_row = (time.perf_counter() - t) / len(probe)
    n = int(min(len(allrows), max(len(probe), seconds / max(per_row, 1e-9))))
    rows = np.sort(rng.choice(allrows, size=n, replace=False))
    t = time.perf_counter()
    _oracle_call(p, host, rows)
    dt = time.perf_counter() - t
    flops = 2.0 * n * p.N * p.K
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{n} of {len(allrows)} valid rows (seeded), all N={p.N} columns, "
                      f"{dt:.1f} s; fp64 C oracle, OpenMP over rows"}


def bench_reference(args):
    """Reference arm: the CPU oracle, timed as it stands, on the same workload
    (each step a bounded seeded sample of its rows)."""
    import oracle

    world, rank, _ = dist_env()
    if rank != 0:
        return
    p = make_inputs(args.workload, "cpu")
    host = _host_inputs(p)
    allrows = _valid_row_list(p)
    rng = np.random.default_rng(1)
    probe = np.sort(rng.choice(allrows, size=min(len(allrows), oracle.max_threads()), replace=False))
    t = time.perf_counter()
    _oracle_call(p, host, probe)
    per_row = (time.perf_counter() - t) / len(probe)
    budget = max(0.02, args.reference_seconds / max(1, args.steps + args.warmup))
    rows_per_step = int(max(1, min(len(allrows), budget / max(per_row, 1e-9))))
    samples = [np.sort(rng.choice(allrows, size=rows_per_step, replace=False))
               for _ in range(min(8, args.steps + args.warmup))]
    for i in range(args.warmup):
        _oracle_call(p, host, samples[i % len(samples)])
    t = time.perf_counter()
    for i in range(args.steps):
        _oracle_call(p, host, samples[i % len(samples)])
    dt = time.perf_counter() - t
    flops = 2.0 * rows_per_step * p.N * p.K * args.steps
    value = flops / dt / 1e12
    ms = dt * 1e3 / args.steps
    cpu = {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.max_threads(),
           "kind": "oracle",
           "sample": f"{rows_per_step} seeded valid rows x N={p.N} per step "
                     f"(of {len(allrows)}); fp64 C oracle, OpenMP over rows"}
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1), UE8M0)",
            "config": describe(p, "n/a (CPU)"), "cpu_baseline": cpu,
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--input-sets", type=int, default=0,
                    help="rotating input sets (default: enough to exceed 3x L2, at least 2)")
    ap.add_argument("--d-offset-bytes", type=int, default=0, choices=[0, 16],
                    help="place D 16 bytes into a larger buffer (16- but not 32-byte aligned)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=90.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
