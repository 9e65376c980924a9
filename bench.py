"""Benchmark: paged GQA verify-decode attention, B8 x 131072 keys, E4M3 K/V.

One step = one pa_decode_fp8 call (one kernel: split-KV attention, then the
log-sum-exp merge of the split partials into the output rows) over
one batch: 8 requests, 131072-token contexts, page 1648, 1 KV head, GQA 6,
q_len 8, head_dim 256, FP16 Q, E4M3 K/V with per-tensor FP32 scales.  Steps
rotate over 16 per-layer KV working sets (536,870,912 unique KV bytes each, so
every step's inputs are far larger than the 129 MB L2; no flush is needed).

Printed JSON (one line, rank 0):
  value      effective KV GB/s = unique KV bytes of all steps on all ranks / max
             wall time over ranks (CUDA events, inputs resident in HBM)
  roofline   decode-kernel achieved GB/s (algorithmic unique KV bytes / its own
             average launch time) vs the measured HBM copy bandwidth; the
             launch time comes from CUDA events around each kernel launch of a
             dedicated burst of --roofline-launches calls right after the timed
             region (the timed region itself carries no per-launch events)
  e2e        the same metric through the C ABI with pinned host buffers: each
             step copies its inputs host->device and reads the output back
  cpu_baseline  the FP64 oracle on a bounded sample, on this host's cores

--impl reference times the oracle itself as the comparison arm.

--workload prefill_q8192_kv262144 (or another name of workloads.PREFILL_SPECS)
times the causal prefill instead: one step = one pa_prefill_f16 call; value in
logical causal TFLOP/s; the tensor roofline of its attention kernel against the
measured sustained BF16 GEMM rate.
Multi-GPU (torchrun): independent replicas, one per rank (no data-path
collective); the barrier and the max over ranks use torch.distributed.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "b8_l128k"
METRIC = "µs per decode-attention call and effective KV GB/s (% of HBM peak) @B8/128K"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
NAMEPLATE_HBM_GBS = 8000.0  # GB300 HBM3e nameplate, for context next to the measured peak
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "split_kernel_b8_l128k_traffic.json")


def _progress(msg: str) -> None:
    """A progress note on stderr (the JSON line goes to stdout)."""
    print(f"[bench {time.strftime('%H:%M:%S')}] {msg}", file=sys.stderr, flush=True)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return None, 0, 1, 0
    import torch.distributed as dist

    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    dist.init_process_group("gloo")
    return dist, rank, ws, local


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C/C++/CUDA source with its comments removed and blank space collapsed,
    so that an edit to comments alone keeps the hash (the sources hold no
    comment markers inside string literals)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    """Hash of the code of every csrc/*.cu, *.cuh (comments excluded): the ncu
    traffic recorded under profiles/ is used only while it matches."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_gqa_decode_split_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def _traffic(workload: str):
    """DRAM bytes per split-kernel launch from the committed ncu capture, or
    None when absent or taken on a different kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        if t.get("kernel_source_hash") != kernel_source_hash() or t.get("workload") != workload:
            return None
        return float(t["dram_bytes_per_launch_full"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------- oracle --

def _oracle_rate(w, rows, threads=0):
    """Time the FP64 oracle on the given flat rows of workload w (host copy);
    returns (seconds, threads used)."""
    import numpy as np
    import torch

    import oracle

    lib = oracle.load()
    nthreads = threads or oracle.max_threads(lib)
    q_bits = w.q.contiguous().view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    oracle.paged_attn(w.spec.kind, q=q_bits, kv=w.kv.numpy(), k_offset=w.k_offset, v_offset=w.v_offset,
                      k_strides=w.k_strides, v_strides=w.v_strides, block_table=w.block_table.numpy(),
                      ctx_lens=w.ctx_lens.numpy(), num_kv_heads=w.spec.num_kv_heads, page_size=w.spec.page_size,
                      k_scale=w.k_scale, v_scale=w.v_scale, rows=np.asarray(rows, np.int32), num_threads=nthreads,
                      lib=lib)
    return time.perf_counter() - t0, nthreads


def cpu_baseline_sample(w_cpu, seconds_target=15.0):
    """Oracle on whole output rows (full contexts) of the benchmark call, as
    many rows as fit the time target (all of them if possible); returns the
    cpu_baseline dict."""
    spec = w_cpu.spec
    per_row = 2 * spec.head_dim * spec.elem_bytes * spec.num_kv_heads / (spec.num_q_heads * spec.q_len)
    import oracle

    nthreads = oracle.max_threads()
    rows_total = spec.batch * spec.q_len * spec.num_q_heads
    t1, _ = _oracle_rate(w_cpu, list(range(nthreads)), nthreads)  # calibration: one row per thread
    rounds = max(1, min(rows_total // nthreads, int(seconds_target / max(t1, 1e-3))))
    nrows = min(rows_total, rounds * nthreads)
    t, used = _oracle_rate(w_cpu, list(range(nrows)), nthreads)
    lens = w_cpu.ctx_lens.tolist()
    per_req = spec.q_len * spec.num_q_heads
    keys = sum(max(0, lens[r // per_req] - spec.q_len + ((r % per_req) // spec.num_q_heads) + 1)
               for r in range(nrows))
    value = keys * per_row / t / 1e9
    return {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"{nrows} of {rows_total} output rows of one call (full contexts), {t:.2f} s wall; "
                      f"GB/s counts {per_row:.3f} unique-KV bytes per (row, visible key)"}


# --------------------------------------------------------------------- arms --

def describe(spec) -> str:
    if spec.ctx_range is not None:
        lo, hi = spec.ctx_range
        ctx = f"B{spec.batch} slots, contexts uniform in [{lo}, {hi}] (drawn per working set)"
        extra = [f"{len(spec.zero_slots)} forced zero-length"] if spec.zero_slots else []
        extra += [f"{len(spec.padded_slots)} padded slots"] if spec.padded_slots else []
        if extra:
            ctx += " with " + " and ".join(extra)
    else:
        ctx = f"B{spec.batch} x {spec.max_ctx_len}-token contexts"
    layout = ""
    if spec.layout == "interleaved":
        layout = ", K/V interleaved per token and head" + (f" at base + {spec.base_pad} B" if spec.base_pad else "")
    return (f"{ctx}, page {spec.page_size}, Hkv {spec.num_kv_heads}, "
            f"Hq {spec.num_q_heads} (GQA {spec.num_q_heads // spec.num_kv_heads}), q_len {spec.q_len}, "
            f"D {spec.head_dim}, " + KIND_TEXT[spec.kind] + layout + ", random block table")


KIND_TEXT = {"fp8": "FP16 Q, E4M3 K/V per-tensor scales", "e5m2": "FP16 Q, E5M2 K/V per-tensor scales",
             "f16": "FP16 Q/K/V", "bf16": "BF16 Q/K/V"}
DTYPE_TEXT = {"fp8": "f16xe4m3->f32", "e5m2": "f16xe5m2->f32", "f16": "f16->f32", "bf16": "bf16->f32"}


def entry_point(spec) -> str:
    return {"fp8": "pa_decode_fp8", "e5m2": "pa_decode_e5m2", "f16": "pa_decode_f16",
            "bf16": f"pa_decode_bf16_d{spec.head_dim}"}[spec.kind]


def reduce_max(values, dist):
    """Element-wise max of a list of floats over all ranks (no-op on one rank)."""
    import torch

    t = torch.tensor(values, dtype=torch.float64)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def run_reference(args, rank, world):
    """The comparison arm: the FP64 oracle itself, on host cores."""
    from paged_gqa_decode_split_gb300 import workloads as wl

    if rank != 0:
        return
    import oracle

    oracle.build()
    spec = wl.SPECS[args.workload]
    w = wl.generate(spec, wl.working_set_seed(args.workload, 0), device="cpu")
    nthreads = oracle.max_threads()
    per_row = 2 * spec.head_dim * spec.elem_bytes * spec.num_kv_heads / (spec.num_q_heads * spec.q_len)
    # each step: one row per thread over a prefix of request 0, sized so the run fits ~2 minutes
    budget = 120.0 / (args.steps + args.warmup)
    t_full, _ = _oracle_rate(w, list(range(nthreads)), nthreads)
    L = int(w.ctx_lens[0])
    n_keys = int(min(L, max(256, L * budget / max(t_full, 1e-6))))
    w_s = wl.Workload(**{**w.__dict__, "ctx_lens": w.ctx_lens.clone().fill_(n_keys)})
    rows = list(range(nthreads))
    for _ in range(args.warmup):
        _oracle_rate(w_s, rows, nthreads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_rate(w_s, rows, nthreads)
    dt = time.perf_counter() - t0
    keys = sum(max(0, n_keys - spec.q_len + (r // spec.num_q_heads) + 1) for r in rows)
    value = keys * per_row * args.steps / dt / 1e9
    sample = (f"per step {len(rows)} output rows of request 0 over its first {n_keys} keys; GB/s counts "
              f"{per_row:.3f} unique-KV bytes per (row, visible key)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe(spec), "global_batch": spec.batch, "seq_len": spec.max_ctx_len,
                       "parallelism": "none (host cores)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nthreads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_gpu(args, dist, rank, world, local):
    import torch

    from paged_gqa_decode_split_gb300 import binding as B
    from paged_gqa_decode_split_gb300 import build as pa_build
    from paged_gqa_decode_split_gb300 import decode as D
    from paged_gqa_decode_split_gb300 import workloads as wl

    if rank == 0 or not pa_build.up_to_date():
        pa_build.build()
    if dist is not None:
        dist.barrier()
    B.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    name = args.workload
    spec = wl.SPECS[name]
    nsets = args.working_sets
    sets = [wl.generate(spec, wl.working_set_seed(name, w) + 1000 * rank, device=dev) for w in range(nsets)]
    decs = [D.Decoder(w) for w in sets]
    uniq = [w.unique_kv_bytes() for w in sets]  # per working set (lengths may differ per set)
    unique = uniq[0]
    stream = torch.cuda.current_stream(dev)
    for i in range(args.warmup):
        B.check(decs[i % nsets](stream), "warm-up call")
    torch.cuda.synchronize(dev)
    for d in decs:
        if d.status() != 0:
            raise RuntimeError(f"status flags {d.status():#x} after warm-up")

    # the timed steps replay one CUDA graph holding a pass over the working
    # sets (calls in rotation), as a decode step is deployed; a remainder of
    # steps runs as direct calls, so exactly args.steps calls are timed
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for i in range(nsets):
            B.check(decs[i](side), "graph warm-up call")
    stream.wait_stream(side)
    pass_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(pass_graph):
        for i in range(nsets):
            B.check(decs[i](torch.cuda.current_stream(dev)), "captured call")
    pass_graph.replay()
    torch.cuda.synchronize(dev)

    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "") or "")
    sampler = ClockSampler(("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else (uuid or str(local)))
    sampler.start()
    time.sleep(0.3)  # let the sampler take its first readings
    B.pa_timing_collect(0)
    B.pa_timing_collect(1)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps // nsets):
        pass_graph.replay()
    for i in range(args.steps % nsets):
        B.check(decs[i](stream), "timed call")
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    ms = ev0.elapsed_time(ev1)
    timed_bytes = sum(uniq[i % nsets] for i in range(args.steps))
    del pass_graph
    # the same calls launched one by one from the host (no graph), for reference
    n_direct = min(args.steps, 512)
    ed0, ed1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ed0.record(stream)
    for i in range(n_direct):
        B.check(decs[i % nsets](stream), "direct call")
    ed1.record(stream)
    torch.cuda.synchronize(dev)
    direct_us = ed0.elapsed_time(ed1) * 1e3 / n_direct
    # roofline burst: the same calls back to back, CUDA events around every
    # kernel launch; a whole number of passes over the sets
    n_roof = max(16, -(-args.roofline_launches // nsets) * nsets)
    B.pa_timing_enable(True)
    for i in range(n_roof):
        B.check(decs[i % nsets](stream), "roofline call")
    B.pa_timing_enable(False)
    torch.cuda.synchronize(dev)
    st0, split_ms, split_n = B.pa_timing_collect(0)
    roof_bytes = sum(uniq[i % nsets] for i in range(n_roof))
    # the operator measurement protocol of "DFlash2 concurrent long-context
    # attention": one CUDA graph of 16 calls (the working sets in rotation),
    # replayed 8 times per sample; per call, the median of 5 samples
    g_calls, g_reps, g_samples = 16, 8, 5
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for i in range(g_calls):
            B.check(decs[i % nsets](side), "graph warm-up call")
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(g_calls):
            B.check(decs[i % nsets](torch.cuda.current_stream(dev)), "captured call")
    graph.replay()
    torch.cuda.synchronize(dev)
    g_us = []
    for _ in range(g_samples):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(g_reps):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        g_us.append(e0.elapsed_time(e1) * 1e3 / (g_calls * g_reps))
    g_bytes = sum(uniq[i % nsets] for i in range(g_calls)) / g_calls
    del graph
    clocks = sampler.stop()
    for d in decs:
        if d.status() != 0:
            raise RuntimeError(f"status flags {d.status():#x} after the timed region")

    # e2e through the C ABI with pinned host buffers
    host = wl.generate(spec, wl.working_set_seed(name, 0) + 1000 * rank, device=dev).to("cpu")
    hq, hkv = host.q.pin_memory(), host.kv.pin_memory()
    hbt, hcl = host.block_table.pin_memory(), host.ctx_lens.pin_memory()
    hsc = torch.tensor([host.k_scale, host.v_scale], dtype=torch.float32).pin_memory()
    hout = torch.empty_like(host.q).pin_memory()
    dw = wl.Workload(**{**host.__dict__, "q": torch.empty_like(hq, device=dev), "kv": torch.empty_like(hkv, device=dev),
                        "block_table": torch.empty_like(hbt, device=dev), "ctx_lens": torch.empty_like(hcl, device=dev)})
    e2e_dec = D.Decoder(dw)
    h2d = hq.nbytes + hkv.nbytes + hbt.nbytes + hcl.nbytes + hsc.nbytes
    d2h = hout.nbytes

    def e2e_step():
        dw.q.copy_(hq, non_blocking=True)
        dw.kv.copy_(hkv, non_blocking=True)
        dw.block_table.copy_(hbt, non_blocking=True)
        dw.ctx_lens.copy_(hcl, non_blocking=True)
        e2e_dec.scales.copy_(hsc, non_blocking=True)
        B.check(e2e_dec(stream), "e2e call")
        hout.copy_(e2e_dec.out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    e_steps = args.e2e_steps
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e_steps):
        e2e_step()
        stream.synchronize()
    e2e_s = time.perf_counter() - t0
    ref_out = D.Decoder(wl.generate(spec, wl.working_set_seed(name, 0) + 1000 * rank, device=dev)).run()
    torch.cuda.synchronize(dev)
    if not torch.equal(hout.to(dev).view(torch.int16), ref_out.view(torch.int16)):
        raise RuntimeError("e2e output differs from the device-resident call")

    ms, e2e_s = reduce_max([ms, e2e_s], dist)
    if rank != 0:
        return

    peak, peak_kind = _peaks()
    total_bytes = timed_bytes * world
    value = total_bytes / (ms / 1e3) / 1e9
    split_avg_s = split_ms / max(split_n, 1) / 1e3
    # every launch in the timed region is this kernel (one per call), so its
    # average launch duration is the region's time per call (it includes the
    # gaps between consecutive graph nodes: a slight underestimate of the rate)
    kernel_avg_s = ms / 1e3 / args.steps
    achieved = timed_bytes / args.steps / kernel_avg_s / 1e9
    traffic = _traffic(name)
    rotated = sum(uniq)
    l2_note = (f"no flush: every step's KV ({min(uniq) / 1e6:.0f} MB or more) exceeds the 129 MB L2"
               if min(uniq) > 129e6 else
               f"no flush: {nsets} working sets of {min(uniq) / 1e6:.1f}-{max(uniq) / 1e6:.1f} MB rotated per call "
               f"({rotated / 1e6:.0f} MB in all)" + ("" if rotated > 129e6 else ", L2-resident: latency only"))
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_sample(host)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "us_per_call": ms / args.steps * 1e3,
        "pct_of_hbm_peak": 100.0 * value / world / peak,
        "pct_of_nameplate_8tbs": 100.0 * value / world / NAMEPLATE_HBM_GBS,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_TEXT[spec.kind],
        "data": "synthetic",
        "config": {"workload": describe(spec),
                   "global_batch": spec.batch * world, "seq_len": spec.max_ctx_len,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "working_sets": nsets, "l2": l2_note,
                   "unique_kv_bytes_per_call": timed_bytes / args.steps,
                   "l2_bytes": int(getattr(props, "L2_cache_size", 0) or 0)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_source": f"{peak_kind} hbm_gbs",
                     "kernel": f"split-KV kernel with its merge phase (the one kernel of {entry_point(spec)})",
                     "kernel_avg_us": kernel_avg_s * 1e6,
                     "timed_launches": args.steps,
                     "algorithmic_bytes_per_launch": timed_bytes / args.steps,
                     "timing": "CUDA events on the launching stream around the timed region, which holds "
                               "only this kernel's launches (one per call)",
                     "per_launch_events_us": split_avg_s * 1e6,
                     "per_launch_events": f"CUDA events around each of {split_n} kernel launches of a burst of "
                                          f"{n_roof} calls after the timed region (the events hold back "
                                          f"back-to-back launches)",
                     "per_launch_events_bytes_per_launch": roof_bytes / max(split_n, 1)},
        "gpu_launches": args.steps,
        "timing": f"{args.steps // nsets} replays of a CUDA graph of {nsets} calls (one per working set)"
                  + (f" + {args.steps % nsets} direct calls" if args.steps % nsets else "")
                  + ", CUDA events on the launching stream",
        "direct": {"us_per_call": direct_us, "calls": n_direct,
                   "note": "the same calls launched one by one from the host, after the timed region"},
        "graph": {"us_per_call": statistics.median(g_us), "GBps": g_bytes / statistics.median(g_us) / 1e3,
                  "pct_of_hbm_peak": 100.0 * g_bytes / statistics.median(g_us) / 1e3 / peak,
                  "samples_us": g_us, "calls_per_graph": g_calls, "replays_per_sample": g_reps,
                  "note": "one CUDA graph of 16 calls (working sets in rotation), 8 replays per sample, "
                          "median of 5 samples per call; this GPU's calls"},
        "clocks": clocks,
        "e2e": {"value": unique * e_steps * world / e2e_s / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e_steps,
                "note": "pinned host -> device copy of Q, K/V pages, block table, lengths and scales, the call, "
                        "and a device -> host read of the output, synchronised every step"},
        "cpu_baseline": cpu,
        "kernel_source_hash": kernel_source_hash(),
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ prefill --
PREFILL_METRIC = "logical causal TFLOP/s of the Q8192 x KV262144 causal prefill (FP16 in, FP32 accumulate)"


def describe_prefill(spec) -> str:
    return (f"causal prefill B{spec.batch}, {spec.q_len} queries (the last positions of a {spec.kv_len}-key "
            f"context), Hq {spec.num_q_heads}, Hkv {spec.num_kv_heads} (GQA {spec.num_q_heads // spec.num_kv_heads}), "
            f"D {spec.head_dim}, FP16 Q/K/V dense per request, FP32 accumulation")


def _prefill_oracle_seconds(w_cpu, rows, nthreads):
    import numpy as np
    import torch

    import oracle

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    s = w_cpu.spec
    t0 = time.perf_counter()
    oracle.prefill_attn(q=bits(w_cpu.q), k=bits(w_cpu.k_buf), v=bits(w_cpu.v_buf), k_strides=w_cpu.k_strides,
                        v_strides=w_cpu.v_strides, kv_len=s.kv_len, num_kv_heads=s.num_kv_heads,
                        rows=np.asarray(rows, np.int32), num_threads=nthreads)
    return time.perf_counter() - t0


def _prefill_row_flops(spec, rows):
    """Logical causal FLOPs of the listed flat rows (4 D per visible key)."""
    total = 0
    for r in rows:
        i = (r // spec.num_q_heads) % spec.q_len
        total += 4 * spec.head_dim * max(0, min(spec.kv_len, spec.kv_len - spec.q_len + i + 1))
    return total


def prefill_cpu_baseline(w_cpu, seconds_target=15.0):
    import oracle

    spec = w_cpu.spec
    nthreads = oracle.max_threads()
    # the last queries of every head (full contexts), one row per thread per round
    rows_all = [((spec.q_len - 1 - k) * spec.num_q_heads + h) for k in range(spec.q_len) for h in range(spec.num_q_heads)]
    t1 = _prefill_oracle_seconds(w_cpu, rows_all[:nthreads], nthreads)
    rounds = max(1, min(len(rows_all) // nthreads, int(seconds_target / max(t1, 1e-3))))
    _progress(f"oracle: {t1:.2f} s for {nthreads} rows on {nthreads} threads; sampling {rounds} rounds")
    rows = rows_all[:rounds * nthreads]
    t = _prefill_oracle_seconds(w_cpu, rows, nthreads)
    return {"value": _prefill_row_flops(spec, rows) / t / 1e12, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{len(rows)} of {spec.batch * spec.q_len * spec.num_q_heads} output rows (the last queries of "
                      f"each head, full contexts), {t:.2f} s wall"}


def run_reference_prefill(args, rank, world):
    from paged_gqa_decode_split_gb300 import workloads as wl

    if rank != 0:
        return
    import oracle

    oracle.build()
    spec = wl.PREFILL_SPECS[args.workload]
    w = wl.generate_prefill(spec, wl.PREFILL_SEED[args.workload], device="cpu")
    nthreads = oracle.max_threads()
    rows = [((spec.q_len - 1) * spec.num_q_heads + h) % (spec.q_len * spec.num_q_heads) for h in range(nthreads)]
    for _ in range(args.warmup):
        _prefill_oracle_seconds(w, rows, nthreads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _prefill_oracle_seconds(w, rows, nthreads)
    dt = time.perf_counter() - t0
    value = _prefill_row_flops(spec, rows) * args.steps / dt / 1e12
    line = {"impl": "reference", "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe_prefill(spec), "global_batch": spec.batch, "seq_len": spec.kv_len,
                       "parallelism": "none (host cores)"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
                             "sample": f"per step {len(rows)} output rows (last query of each head, full context)"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _tensor_peak():
    """(TFLOP/s, source): the measured sustained BF16 GEMM rate (FP16 has the
    same nominal dense rate on this part), else the fallback figure."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        for k in ("bf16_tflops_sustained", "bf16_tflops"):
            if d.get(k):
                return float(d[k]), f"measured {k} (FP16 dense rate = BF16 nominal)"
    except Exception:
        pass
    return 1700.0, "fallback sustained BF16 (FP16 dense rate = BF16 nominal)"


def run_gpu_prefill(args, dist, rank, world, local):
    import torch

    from paged_gqa_decode_split_gb300 import binding as B
    from paged_gqa_decode_split_gb300 import build as pa_build
    from paged_gqa_decode_split_gb300 import workloads as wl
    from paged_gqa_decode_split_gb300.prefill import Prefill, logical_causal_flops

    if rank == 0 or not pa_build.up_to_date():
        pa_build.build()
    if dist is not None:
        dist.barrier()
    B.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    name = args.workload
    spec = wl.PREFILL_SPECS[name]
    seed = wl.PREFILL_SEED[name] + 1000 * rank
    w = wl.generate_prefill(spec, seed, device=dev)
    pf = Prefill(w)
    flops = logical_causal_flops(spec.batch, spec.q_len, spec.kv_len, spec.num_q_heads, spec.head_dim)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        B.check(pf(stream), "warm-up call")
    torch.cuda.synchronize(dev)
    if pf.status() != 0:
        raise RuntimeError(f"status flags {pf.status():#x} after warm-up")
    _progress("warm-up done")
    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "") or "")
    sampler = ClockSampler(("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else (uuid or str(local)))
    sampler.start()
    time.sleep(0.3)
    B.pa_timing_collect(0)
    B.pa_timing_collect(1)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # attention-kernel events on every call (each call is milliseconds long)
    B.pa_timing_enable(True)
    ev0.record(stream)
    for _ in range(args.steps):
        B.check(pf(stream), "timed call")
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    B.pa_timing_enable(False)
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    ms = ev0.elapsed_time(ev1)
    st, k_ms, k_n = B.pa_timing_collect(1)
    if pf.status() != 0:
        raise RuntimeError(f"status flags {pf.status():#x} after the timed region")
    _progress(f"timed region done: {ms / args.steps:.3f} ms per call")

    # e2e: pinned host Q, K, V in; output and LSE out, every step
    hq, hk, hv = w.q.cpu().pin_memory(), w.k_buf.cpu().pin_memory(), w.v_buf.cpu().pin_memory()
    _progress("e2e host buffers pinned")
    hout = torch.empty_like(hq).pin_memory()
    hlse = torch.empty(tuple(hq.shape[:3]), dtype=torch.float32).pin_memory()
    dw = wl.PrefillWorkload(spec=spec, q=torch.empty_like(w.q), k_buf=torch.empty_like(w.k_buf),
                            v_buf=torch.empty_like(w.v_buf), k_strides=w.k_strides, v_strides=w.v_strides)
    e2e_pf = Prefill(dw)
    h2d = hq.nbytes + hk.nbytes + hv.nbytes
    d2h = hout.nbytes + hlse.nbytes

    def e2e_step():
        dw.q.copy_(hq, non_blocking=True)
        dw.k_buf.copy_(hk, non_blocking=True)
        dw.v_buf.copy_(hv, non_blocking=True)
        B.check(e2e_pf(stream), "e2e call")
        hout.copy_(e2e_pf.out, non_blocking=True)
        hlse.copy_(e2e_pf.lse, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    _progress("e2e warm-up step done")
    e_steps = max(3, min(args.e2e_steps, 10))
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e_steps):
        e2e_step()
        stream.synchronize()
    e2e_s = time.perf_counter() - t0
    if not torch.equal(hout.to(dev).view(torch.int16), pf.out.view(torch.int16)):
        raise RuntimeError("e2e output differs from the device-resident call")
    _progress(f"e2e done: {e2e_s / e_steps * 1e3:.1f} ms per step")
    del dw, e2e_pf
    ms, e2e_s = reduce_max([ms, e2e_s], dist)
    if rank != 0:
        return
    peak, peak_src = _tensor_peak()
    kv_bytes = hk.nbytes + hv.nbytes
    l2_note = (f"no flush: K and V ({kv_bytes / 1e6:.0f} MB) exceed the 129 MB L2" if kv_bytes > 129e6 else
               f"K and V ({kv_bytes / 1e6:.0f} MB) fit in L2")
    value = flops * args.steps * world / (ms / 1e3) / 1e12
    k_avg_s = k_ms / max(k_n, 1) / 1e3
    achieved = flops / k_avg_s / 1e12
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        del w, pf
        torch.cuda.empty_cache()
        cpu = prefill_cpu_baseline(wl.generate_prefill(spec, seed, device=dev).to("cpu"))
    line = {
        "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16->f32", "data": "synthetic",
        "config": {"workload": describe_prefill(spec), "global_batch": spec.batch * world, "seq_len": spec.kv_len,
                   "q_len": spec.q_len, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "logical_causal_flops_per_call": flops,
                   "l2": l2_note},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "traffic": None, "peak_source": peak_src,
                     "kernel": "prefill attention kernel (tcgen05, FP32 accumulate), without its merge kernel",
                     "kernel_avg_us": k_avg_s * 1e6, "timed_launches": k_n,
                     "algorithmic_flops_per_launch": flops,
                     "timing": "CUDA events around the attention kernel of every timed call"},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "e2e": {"value": flops * e_steps * world / e2e_s / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e_steps,
                "note": "pinned host -> device copy of Q, K and V, the call, and a device -> host read of the "
                        "output and LSE, synchronised every step"},
        "cpu_baseline": cpu,
        "kernel_source_hash": kernel_source_hash(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, help="workload name (default: the B8/128K metric config)")
    ap.add_argument("--working-sets", type=int, default=16)
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--roofline-launches", type=int, default=64,
                    help="calls in the roofline burst after the timed region (at least 16; CUDA events around "
                         "each kernel launch)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    dist, rank, world, local = _dist()
    prefill = args.workload.startswith("prefill_")
    if args.impl == "reference":
        (run_reference_prefill if prefill else run_reference)(args, rank, world)
    else:
        (run_gpu_prefill if prefill else run_gpu)(args, dist, rank, world, local)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
