"""Benchmark of one paged decode step (slot lookup + K/V write + copy-on-write
copies + split-context decode + combine) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload gqa]
    python bench.py --impl reference ...     # the CPU oracle, timed the same way

Prints one JSON line.  ``value`` is logical K/V bytes read by decode per second
over the whole job (inputs resident in HBM, device-timed with CUDA events);
``e2e`` is the same metric through the public API with the step's inputs
copied from pinned host memory and the output copied back inside the timed
region.  The step reads 1 GiB of K/V on the default workload, far more than
the 129 MB L2, so no L2 flush is needed between steps; a workload whose
distinct K/V is under 4x the L2 (the shared-prefix one) gets a 512 MiB buffer
written and read back between steps, outside the timed intervals.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import signal
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

NOMINAL_HBM_GBS = 8000.0
KERNEL_SOURCES = ["paged_kv_cache_170_gb300/csrc/pa_decode_mma.cuh", "paged_kv_cache_170_gb300/csrc/pa_sched.cuh",
                  "paged_kv_cache_170_gb300/csrc/pa_mma_tile.cuh",
                  "paged_kv_cache_170_gb300/csrc/pa_common.cuh"]  # the tensor-core decode kernel
SHARED_SOURCES = KERNEL_SOURCES + ["paged_kv_cache_170_gb300/csrc/pa_decode_shared.cuh",
                                   "paged_kv_cache_170_gb300/csrc/pa_share.cu",
                                   "paged_kv_cache_170_gb300/csrc/pa_share_plan.h",
                                   "paged_kv_cache_170_gb300/csrc/pa_prefill.cuh"]  # the shared-block decode's kernels
PREFILL_SOURCES = ["paged_kv_cache_170_gb300/csrc/pa_prefill.cuh", "paged_kv_cache_170_gb300/csrc/pa_sched.cuh",
                   "paged_kv_cache_170_gb300/csrc/pa_common.cuh"]  # the tcgen05 prefill kernel


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    """Hash of the kernel's code with comments, blank space and trace-build
    blocks (`#ifdef PA_TRACE`, not compiled in a product build) removed: an
    edit of those alone leaves a profiled kernel the same kernel."""
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("\n".join(_product_lines(text.splitlines())).encode())
    return h.hexdigest()[:16]


def _product_lines(lines):
    """The stripped, non-blank lines a build without PA_TRACE compiles: the
    body of each `#ifdef PA_TRACE` is dropped up to its `#else` or `#endif`."""
    out, depth, skipping = [], 0, False
    for raw in lines:
        line = raw.strip()
        if not line:
            continue
        directive = line.split()[0] if line.startswith("#") else ""
        if skipping:
            if directive in ("#if", "#ifdef", "#ifndef"):
                depth += 1
            elif directive == "#endif":
                if depth == 0:
                    skipping = False
                else:
                    depth -= 1
            elif directive == "#else" and depth == 0:
                skipping = False
                out.append("#ifndef PA_TRACE")
            continue
        if line == "#ifdef PA_TRACE":
            skipping, depth = True, 0
            continue
        out.append(line)
    return out


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d.get("bf16_tflops", 1900.0)),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def profiled_traffic(workload: str, kernel: str = "decode_partition", sources=KERNEL_SOURCES):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path, encoding="utf-8").read()
    m_hash = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash(sources):
        return None
    return float(m_bytes.group(1))


def workload_inputs(name: str, seed: int, device, num_seqs=None, placement: str = "random"):
    """Inputs of a named workload; ``num_seqs`` shrinks the plain workloads (and
    their pools) to fewer sequences of the same shape, for profiler captures;
    ``placement`` "contiguous" gives each sequence of a plain workload one run
    of consecutive physical blocks instead of random ones."""
    from paged_kv_cache_170_gb300 import scenarios, workloads

    if name == "prefix":
        return scenarios.shared_prefix_inputs(seed, device=device)
    if name == "longctx":
        return scenarios.long_context_inputs(seed, device=device)
    w = workloads.scaled(workloads.WORKLOADS[name], placement=placement)
    if num_seqs is not None and name != "tiny":
        w = workloads.scaled(w, num_seqs=num_seqs, num_blocks=num_seqs * w.max_blocks_per_seq + 64)
    return workloads.make_inputs(w, seed, device=device)


def kv_bytes(inp) -> int:
    """Logical K+V bytes one decode reads: every valid token of every sequence,
    for every kv head (partial tail blocks count only their valid slots)."""
    _, Hkv, _, D = inp.k_cache.shape
    e = inp.k_cache.element_size()
    return int(inp.context_lens.to(torch.int64).sum().item()) * Hkv * D * e * 2


def unique_kv_bytes(inp) -> int:
    """K+V bytes of the distinct physical tiles one decode touches: a block that
    several sequences share counts once, with the most valid rows any sharer
    reads from it.  This is the least DRAM traffic a decode can have."""
    B = inp.k_cache.shape[2]
    _, Hkv, _, D = inp.k_cache.shape
    lens = inp.context_lens.to(torch.int64).cpu()
    tables = inp.block_tables.to(torch.int64).cpu()
    nb = (lens + B - 1) // B
    idx = torch.arange(tables.shape[1], dtype=torch.int64)
    used = idx[None, :] < nb[:, None]
    rows = torch.clamp(lens[:, None] - idx[None, :] * B, 0, B)
    pid, r = tables[used], rows[used]
    if pid.numel() == 0:
        return 0
    best = torch.zeros(int(pid.max()) + 1, dtype=torch.int64).scatter_reduce(0, pid, r, reduce="amax")
    return int(best.sum()) * Hkv * D * inp.k_cache.element_size() * 2


L2_BYTES = 129 * 1024 * 1024
FLUSH_BYTES = 512 * 1024 * 1024  # written between timed steps when a step's distinct K/V would sit in L2


def flush_l2(buf: torch.Tensor, k: int) -> None:
    """Evict the step's K/V from L2 between timed steps: write ``buf`` (4x
    the L2), then read it back.  The read leaves L2 holding clean lines of
    the flush buffer; after the write alone up to 129 MB of dirty flush lines
    stay in L2, and the next decode would pay for writing them back to DRAM
    (traffic of the harness, not of the kernel)."""
    buf.fill_(k & 255)
    torch.amax(buf.view(torch.int32))


def needs_l2_flush(inp, mode: str = "auto") -> bool:
    """auto: flush when a step's distinct K/V is under 4x the L2; "flush" /
    "warm" force it on / off ("warm" numbers are for analysis, not the line's
    headline)."""
    if mode != "auto":
        return mode == "flush"
    return unique_kv_bytes(inp) < 4 * L2_BYTES


def decode_kernel_name(inp, shared: bool, fused: bool = False, shared_kernels=None) -> str:
    """The kernel(s) the timed decode call runs: the tensor-core kernel takes
    fp16 / bf16 caches whose block size is a multiple of 16; pa_write_decode
    runs the write kernel first; the shared decode runs the kernels its plan
    needs."""
    if shared and shared_kernels:
        return " + ".join(shared_kernels)
    name = "decode_partition_mma_kernel" if inp.k_cache.dtype != torch.float32 and inp.k_cache.shape[2] % 16 == 0 \
        else "decode_partition_kernel"
    return "append_last_kernel + " + name + " (pa_write_decode, timed as one call)" if fused else name


def algorithmic_bytes(inp, with_write: bool = False) -> int:
    """Bytes the decode kernel must move: K/V + q + out + the table entries it
    reads + lengths; with_write (pa_write_decode, timed as one call) adds its
    write kernel's: the new K/V rows read and stored, one table entry and one
    length per sequence."""
    B = inp.k_cache.shape[2]
    lens = inp.context_lens.to(torch.int64)
    entries = int(((lens + B - 1) // B).sum().item())
    Hkv = inp.k_cache.shape[1]
    write = 2 * (inp.new_key.numel() + inp.new_value.numel()) * inp.new_key.element_size() + 8 * lens.numel() \
        if with_write else 0
    return kv_bytes(inp) + 2 * inp.q.numel() * inp.q.element_size() + entries * 4 * Hkv + lens.numel() * 4 + write


def memory_report(inp) -> dict:
    """The pages' memory figures (waste ratio, its half-block estimate, memory
    saved by sharing, use against a contiguous max-length reservation) for
    this step's block tables."""
    from paged_kv_cache_170_gb300.block_manager import pool_report

    _, Hkv, B, D = inp.k_cache.shape
    rep = pool_report(inp.block_tables.cpu().numpy(), inp.context_lens.cpu().numpy(), B,
                      2 * Hkv * D * inp.k_cache.element_size(), max_len=inp.block_tables.shape[1] * B)
    return {k: round(v, 6) if isinstance(v, float) else v for k, v in rep.items()}


def workload_config(name: str, inp, l2_mode: str = "auto") -> dict:
    w = inp.workload
    lens = inp.context_lens.to(torch.int64)
    if l2_mode == "warm":
        l2 = "warm: no flush between steps (forced for analysis; the step's distinct K/V is %.2f GB)" % (
            unique_kv_bytes(inp) / 1e9)
    elif needs_l2_flush(inp, l2_mode):
        l2 = ("flush: %d MiB written then read between timed steps (outside the timed intervals); the step's "
              "distinct K/V is %.2f GB" % (FLUSH_BYTES >> 20, unique_kv_bytes(inp) / 1e9))
    else:
        l2 = "no flush: each step reads %.2f GB of distinct K/V, larger than the 129 MB L2" % (
            unique_kv_bytes(inp) / 1e9)
    return {"workload": f"{name}: {w.note}", "num_seqs": int(inp.q.shape[0]), "block_size": int(inp.k_cache.shape[2]),
            "num_heads": int(inp.q.shape[1]), "num_kv_heads": int(inp.k_cache.shape[1]),
            "head_dim": int(inp.q.shape[2]), "pool_blocks": int(inp.k_cache.shape[0]),
            "context_min": int(lens.min()), "context_max": int(lens.max()), "context_sum": int(lens.sum()),
            "cow_pairs": int(inp.copy_pairs.shape[0]), "new_tokens": int(inp.new_seq.numel()),
            "l2_policy": l2, "placement": w.placement, "memory": memory_report(inp)}


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the loaded phase and the timed
    loop run (the caller keeps the GPU busy for ``LOAD_SECONDS`` first, so
    that the record covers the workload's own clocks, not an idle GPU)."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,utilization.gpu")
    LOAD_SECONDS = 1.2
    BUSY_PCT = 50.0  # a sample counts as under load at this GPU utilisation or more

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.5)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.send_signal(signal.SIGTERM)
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self) -> dict:
        """Median SM clock over the samples taken under load (GPU utilisation
        >= BUSY_PCT; the upper half of all samples if none reports it), the
        throttle reasons seen in any sample, and the sample counts."""
        sm, loaded, mx, reasons = [], [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz = float(f[1])
                mx = float(f[2])
            except ValueError:
                continue
            sm.append(mhz)
            try:
                if len(f) > 9 and float(f[9]) >= self.BUSY_PCT:
                    loaded.append(mhz)
            except ValueError:
                pass
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0,
                    "samples_under_load": 0}
        busy = loaded if loaded else sorted(sm)[len(sm) // 2:]
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "samples_under_load": len(loaded)}


def keep_busy(step, seconds: float, device, flush=None) -> int:
    """Replay ``step`` (and the L2 flush between steps, when given) untimed
    for about ``seconds``; returns the steps run."""
    n, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for _ in range(64):
            if flush is not None:
                flush(n)
            step()
            n += 1
        torch.cuda.synchronize(device)
    return n


def time_cpu_oracle(inp_cpu, max_seconds: float, nthreads: int = 0):
    """The C oracle on whole sequences of the workload, cycling over them until
    the time budget is spent (at least one).  Returns (GB/s of logical K/V,
    seconds, sequence decodes, threads)."""
    from oracle import native

    S = inp_cpu.q.shape[0]
    tables = inp_cpu.block_tables.numpy()
    lens = inp_cpu.context_lens.numpy()
    Hkv, D = inp_cpu.k_cache.shape[1], inp_cpu.k_cache.shape[3]
    e = inp_cpu.k_cache.element_size()
    done, t_total = 0, 0.0
    nbytes = 0
    while done == 0 or t_total < max_seconds:
        s = done % S
        t0 = time.perf_counter()
        native.decode(inp_cpu.q[s:s + 1], inp_cpu.k_cache, inp_cpu.v_cache, tables[s:s + 1], lens[s:s + 1],
                      inp_cpu.scale, nthreads=nthreads)
        t_total += time.perf_counter() - t0
        nbytes += int(lens[s]) * Hkv * D * e * 2
        done += 1
    threads = nthreads if nthreads > 0 else native.max_threads()
    return nbytes / t_total / 1e9, t_total, done, threads


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return rank, world, local, dist
    return 0, 1, 0, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x: float, dist) -> float:
    if dist is None:
        return x
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, dist) -> float:
    if dist is None:
        return x
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def run_gpu(args) -> dict:
    from paged_kv_cache_170_gb300 import ops

    rank, world, local, dist = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    # every rank runs its own replica of the workload on different data (weak scaling)
    inp = workload_inputs(args.workload, args.seed + rank, dev, args.num_seqs, args.placement)
    S, Hq, D = inp.q.shape
    stream = torch.cuda.current_stream(dev)
    from paged_kv_cache_170_gb300.step import DecodeStep, StepPipeline

    runner = DecodeStep(inp, graphs=not args.no_graph, shared=args.shared, fused=not args.unfused)
    out, err = runner.out, runner.err
    step = runner.run
    launches_per_step = runner.launches_per_step

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert int(err.item()) == 0, ops.error_names(int(err.item()))

    # -- device-timed step loop (inputs resident)
    flush = needs_l2_flush(inp, args.l2)
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)] \
        if flush else None
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        # the same step, untimed, so that the clock record covers this load
        load_steps = keep_busy(step, args.load_seconds, dev, (lambda k: flush_l2(flush_buf, k)) if flush else None)
        torch.cuda.synchronize(dev)
        start.record(stream)
        for k in range(args.steps):
            if flush:
                flush_l2(flush_buf, k)
                sev[k][0].record(stream)
            step(*kev[k])
            if flush:
                sev[k][1].record(stream)
        end.record(stream)
        torch.cuda.synchronize(dev)
    barrier(dist)
    if flush:
        step_ms = sum(a.elapsed_time(b) for a, b in sev) / args.steps
    else:
        step_ms = start.elapsed_time(end) / args.steps
    kernel_times = [a.elapsed_time(b) for a, b in kev]
    kernel_ms = sum(kernel_times) / args.steps
    step_ms_max = max_over_ranks(step_ms, dist)

    # -- end to end through the public API: pinned host inputs in, output out,
    # every step; two step slots pipelined so that one slot's copies overlap
    # the other slot's kernels
    pipe = StepPipeline(inp, graphs=not args.no_graph, shared=args.shared, fused=not args.unfused)
    h2d, d2h = pipe.h2d_bytes, pipe.d2h_bytes
    e2e_steps = max(1, min(args.steps, 2000))
    for _ in range(3):
        pipe.step()
    pipe.drain()
    torch.cuda.synchronize(dev)
    barrier(dist)
    # each step's inputs are staged anew on the host: written (one copy, in
    # the packed layout) into the pinned buffer the step uploads from, as a
    # serving loop hands over a new batch
    host_src = pipe.slots[0].packed.host.clone()  # pageable memory, the same layout
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        pipe.next_host_buffer().copy_(host_src)
        pipe.step()
    pipe.drain()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist)
    for sl in pipe.slots:
        assert int(sl.runner.err.item()) == 0, ops.error_names(int(sl.runner.err.item()))
    assert int(err.item()) == 0, ops.error_names(int(err.item()))

    kvb = kv_bytes(inp)
    total_kv = sum_over_ranks(float(kvb), dist)
    alg = algorithmic_bytes(inp, with_write=runner.fused)
    uniq = unique_kv_bytes(inp) + (alg - kvb)
    peaks = measured_peaks()
    achieved = alg / (kernel_ms * 1e-3) / 1e9
    value = total_kv / (step_ms_max * 1e-3) / 1e9
    line = {
        "metric": "pa_decode achieved KV GB/s (logical K+V bytes / decode-step time)",
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms_max, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}[inp.q.dtype],
        "data": "synthetic: seeded N(0,1) q/K/V, random physical placement",
        "config": dict(workload_config(args.workload, inp, args.l2),
                       step_launch="%s: %s%s (%d launch%s per step)" % (
                           "eager, kernel by kernel" if args.no_graph else "CUDA graphs",
                           "copy-on-write copies, then " if inp.copy_pairs.numel() else "",
                           "pa_write_decode: slot lookup + K/V write in one kernel, the decode launched early "
                           "(programmatic dependent launch)" if runner.fused
                           else "slot lookup, K/V write, then decode", runner.launches_per_step,
                           "" if runner.launches_per_step == 1 else "es"),
                       decode="pa_decode_shared (plan: %d shared and %d own groups, %d pieces, %d tensor-core "
                              "items)" % (
                           runner.plan_info["num_shared_groups"],
                           runner.plan_info["num_groups"] - runner.plan_info["num_shared_groups"],
                           runner.plan_info["num_pieces"], runner.plan_info["num_tc_items"]) if args.shared
                       else "pa_decode"),
        "tokens_per_s": round(sum_over_ranks(float(S), dist) / (step_ms_max * 1e-3), 0),
        "pct_of_nominal_8000_gbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_hbm": round(100 * value / world / peaks["hbm_gbs"], 2),
        "decode_kernel_us": round(kernel_ms * 1e3, 2),
        "decode_kernel_us_median": round(statistics.median(kernel_times) * 1e3, 2),
        "roofline": {"kernel": decode_kernel_name(inp, args.shared, runner.fused, runner.shared_kernels), "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)",
                     "frac_of_nominal_8000": round(achieved / NOMINAL_HBM_GBS, 4),
                     "algorithmic_bytes_per_launch": alg,
                     "distinct_bytes_per_launch": uniq,
                     "frac_distinct": round(uniq / (kernel_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                     "traffic": profiled_traffic(args.workload, "decode_shared", SHARED_SOURCES) if args.shared
                     else profiled_traffic(args.workload)},
        "e2e": {"value": round(total_kv / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "host_staging": "each step's inputs written into the pinned upload buffer by the host (one copy "
                                "of the packed inputs), one upload, the output read back; two steps in flight"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": dict(clocks.summary(), untimed_load_steps=load_steps,
                       load_note="the same step replayed untimed for %.1f s inside the sampling window before the "
                                 "timed loop" % args.load_seconds),
    }
    if rank == 0 and not args.no_cpu_baseline:
        cpu = inp.to("cpu")
        gbs, secs, nseq, threads = time_cpu_oracle(cpu, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(gbs, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
                                "sample": f"{nseq} sequence decodes ({nseq / S:.1f} passes over the {S} sequences), "
                                          f"all {Hq} heads, C float64 oracle, {secs:.1f} s"}
    if dist is not None:
        dist.destroy_process_group()
    return line if rank == 0 else None


def prefill_flops(inp) -> int:
    """Causal attention flops of a prompt step: 4 * D per (query row, head,
    visible token); the row at position p sees p + 1 tokens."""
    lens = inp.context_lens.to(torch.int64).cpu()
    qs = inp.q_start.to(torch.int64).cpu()
    n = qs[1:] - qs[:-1]
    # sum over rows of (p + 1), p = L - n + i, i = 0 .. n-1
    visible = int((n * (lens - n) + n * (n + 1) // 2).sum())
    return 4 * inp.q.shape[2] * inp.q.shape[1] * visible


def prefill_config(name: str, inp, l2: str) -> dict:
    w = inp.workload
    lens = inp.context_lens.to(torch.int64)
    n = (inp.q_start[1:] - inp.q_start[:-1]).to(torch.int64)
    return {"workload": f"{name}: {w.note}", "num_seqs": int(lens.numel()), "block_size": int(inp.k_cache.shape[2]),
            "num_heads": int(inp.q.shape[1]), "num_kv_heads": int(inp.k_cache.shape[1]),
            "head_dim": int(inp.q.shape[2]), "pool_blocks": int(inp.k_cache.shape[0]),
            "context_sum": int(lens.sum()), "prompt_tokens": int(n.sum()), "placement": w.placement, "l2_policy": l2}


def run_prefill_gpu(args) -> dict:
    """The prompt step: pa_prefill over every sequence's prompt (its K/V
    already in the cache), timed with CUDA events around each launch."""
    from paged_kv_cache_170_gb300 import ops, workloads

    rank, world, local, dist = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    inp = workloads.make_prefill_inputs(workloads.WORKLOADS[args.workload], args.seed + rank, device=dev)
    # the prompt's inputs in one device buffer with a pinned host mirror (one upload per step)
    from paged_kv_cache_170_gb300.step import PackedInputs
    packed = PackedInputs(inp, names=("q", "block_tables", "context_lens", "q_start"))
    out = torch.empty_like(inp.q)
    err = ops.new_error_word(dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev_a=None, ev_b=None):
        if ev_a is not None:
            ev_a.record(stream)
        ops.pa_prefill(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.q_start,
                       inp.max_q_len, inp.scale, out, err)
        if ev_b is not None:
            ev_b.record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert int(err.item()) == 0, ops.error_names(int(err.item()))
    _, Hkv, _, D = inp.k_cache.shape
    distinct = int(inp.context_lens.to(torch.int64).sum()) * Hkv * D * inp.k_cache.element_size() * 2
    flush = args.l2 == "flush" or (args.l2 == "auto" and distinct < 4 * L2_BYTES)
    l2 = ("flush: %d MiB written then read between timed steps (outside the timed intervals); the step's K/V "
          "is %.3f GB"
          % (FLUSH_BYTES >> 20, distinct / 1e9)) if flush else "no flush (%s)" % args.l2
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        load_steps = keep_busy(step, args.load_seconds, dev, (lambda k: flush_l2(flush_buf, k)) if flush else None)
        for k in range(args.steps):
            if flush:
                flush_l2(flush_buf, k)
            step(*kev[k])
        torch.cuda.synchronize(dev)
    barrier(dist)
    times = [a.elapsed_time(b) for a, b in kev]
    step_ms = max_over_ranks(sum(times) / args.steps, dist)
    flops = prefill_flops(inp)
    total_flops = sum_over_ranks(float(flops), dist)
    peaks = measured_peaks()
    tflops = total_flops / (step_ms * 1e-3) / 1e12
    # end to end: the prompts' queries in from pinned host memory, the outputs back
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = packed.nbytes
    d2h = out_host.numel() * out_host.element_size()
    e2e_steps = max(1, min(args.steps, 200))
    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        packed.upload()
        step()
        out_host.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist)
    assert int(err.item()) == 0, ops.error_names(int(err.item()))
    bf16 = float(peaks.get("bf16_tflops", 1900.0))
    line = {
        "metric": "pa_prefill causal attention TFLOP/s (4*D flops per query row, head and visible token)",
        "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {torch.bfloat16: "bf16", torch.float16: "f16"}[inp.q.dtype],
        "data": "synthetic: seeded N(0,1) q/K/V, random physical placement",
        "config": prefill_config(args.workload, inp, l2),
        "tokens_per_s": round(sum_over_ranks(float(inp.q.shape[0]), dist) / (step_ms * 1e-3), 0),
        "prefill_kernel_us": round(step_ms * 1e3, 2),
        "roofline": {"kernel": "prefill_tc_kernel", "bound": "tensor", "achieved": round(tflops / world, 2),
                     "peak": bf16, "unit": "TFLOP/s", "frac": round(tflops / world / bf16, 4),
                     "peak_source": peaks["source"] + " (MEASURED_PEAKS.json bf16_tflops, cuBLAS bf16 GEMM burst)",
                     "algorithmic_flops_per_launch": flops,
                     "traffic": profiled_traffic(args.workload, "prefill_tc", PREFILL_SOURCES)},
        "e2e": {"value": round(total_flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": dict(clocks.summary(), untimed_load_steps=load_steps),
    }
    if rank == 0 and not args.no_cpu_baseline:
        cpu = inp.to("cpu")
        v, secs, rows, threads = time_cpu_prefill(cpu, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(v, 4), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                                "sample": f"{rows} query rows (all heads) of the workload's prompts, C float64 "
                                          f"oracle, {secs:.1f} s"}
    if dist is not None:
        dist.destroy_process_group()
    return line if rank == 0 else None


def time_cpu_prefill(inp_cpu, max_seconds: float):
    """The C oracle on one-row prompts cut from the workload (row i of a prompt
    is position p of its sequence: a one-token prompt on the context cut
    after p), cycling until the time budget is spent.  Returns (TFLOP/s,
    seconds, rows, threads)."""
    from oracle import native

    lens = inp_cpu.context_lens.numpy()
    qs = inp_cpu.q_start.numpy()
    tables = inp_cpu.block_tables.numpy()
    D, Hq = inp_cpu.q.shape[2], inp_cpu.q.shape[1]
    order = [(s, r) for s in range(len(lens)) for r in range(int(qs[s]), int(qs[s + 1]))]
    step = max(1, len(order) // 97)
    picks = order[::step]
    t_total, flops, done = 0.0, 0, 0
    while done == 0 or t_total < max_seconds:
        s, r = picks[done % len(picks)]
        p = int(lens[s]) - int(qs[s + 1] - qs[s]) + (r - int(qs[s]))
        t0 = time.perf_counter()
        native.prefill(inp_cpu.q[r:r + 1], inp_cpu.k_cache, inp_cpu.v_cache, tables[s:s + 1],
                       np.array([p + 1], np.int32), np.array([0, 1], np.int32), inp_cpu.scale)
        t_total += time.perf_counter() - t0
        flops += 4 * D * Hq * (p + 1)
        done += 1
    return flops / t_total / 1e12, t_total, done, native.max_threads()


def run_reference(args) -> dict:
    """The CPU oracle as the reference arm: each step decodes a bounded sample
    of whole sequences of the same workload on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    from oracle import native

    if args.workload.startswith("prefill"):
        return run_prefill_reference(args)
    inp = workload_inputs(args.workload, args.seed, "cuda" if torch.cuda.is_available() else "cpu").to("cpu")
    S, Hq, D = inp.q.shape
    Hkv = inp.k_cache.shape[1]
    e = inp.k_cache.element_size()
    tables, lens = inp.block_tables.numpy(), inp.context_lens.numpy()
    # calibrate: seconds per sequence, then size each step for ~90 s over all steps
    t0 = time.perf_counter()
    native.decode(inp.q[:1], inp.k_cache, inp.v_cache, tables[:1], lens[:1], inp.scale)
    per_seq = max(time.perf_counter() - t0, 1e-6)
    total_steps = args.steps + args.warmup
    nseq = max(1, min(S, int(90.0 / total_steps / per_seq)))
    heads_note = "all heads"
    sample_q = inp.q[:nseq]
    for _ in range(args.warmup):
        native.decode(sample_q, inp.k_cache, inp.v_cache, tables[:nseq], lens[:nseq], inp.scale)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        native.decode(sample_q, inp.k_cache, inp.v_cache, tables[:nseq], lens[:nseq], inp.scale)
    secs = time.perf_counter() - t0
    nbytes = int(lens[:nseq].astype("int64").sum()) * Hkv * D * e * 2 * args.steps
    value = nbytes / secs / 1e9
    threads = native.max_threads()
    sample = f"{nseq} of {S} sequences per step, {heads_note}, C float64 oracle"
    return {
        "impl": "reference",
        "metric": "pa_decode achieved KV GB/s (logical K+V bytes / decode-step time)",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload, inp),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_prefill_reference(args) -> dict:
    """The CPU oracle as the reference arm of a prompt workload: each step a
    bounded sample of one-row prompts cut from the workload."""
    from paged_kv_cache_170_gb300 import workloads

    inp = workloads.make_prefill_inputs(workloads.WORKLOADS[args.workload], args.seed, device="cpu")
    budget = max(0.5, 90.0 / (args.steps + args.warmup))
    for _ in range(args.warmup):
        time_cpu_prefill(inp, budget)
    vals, secs, rows, threads = [], 0.0, 0, 1
    for _ in range(args.steps):
        v, t, r, threads = time_cpu_prefill(inp, budget)
        vals.append(v)
        secs += t
        rows += r
    value = sum(vals) / len(vals)
    sample = f"{rows} one-row prompts cut from the workload over {args.steps} steps, C float64 oracle"
    return {
        "impl": "reference",
        "metric": "pa_prefill causal attention TFLOP/s (4*D flops per query row, head and visible token)",
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": prefill_config(args.workload, inp, "n/a (CPU)"),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=6000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", choices=["tiny", "mha", "gqa", "prefix", "longctx", "prefill", "prefill_hist"],
                    default="gqa")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--num-seqs", type=int, default=None, help="fewer sequences (profiling captures only)")
    ap.add_argument("--no-graph", action="store_true", help="launch the step's kernels one by one")
    ap.add_argument("--unfused", action="store_true",
                    help="slot lookup and K/V write as their own kernels before the decode (default: one "
                         "pa_write_decode call when every sequence appends one token)")
    ap.add_argument("--l2", choices=["auto", "flush", "warm"], default="auto",
                    help="L2 between timed steps: auto (flush when the distinct K/V is under 4x L2), "
                         "flush, or warm (no flush; analysis only)")
    ap.add_argument("--placement", choices=["random", "contiguous"], default="random",
                    help="physical placement of the plain workloads' blocks")
    ap.add_argument("--load-seconds", type=float, default=ClockSampler.LOAD_SECONDS,
                    help="untimed replay of the step inside the clock-sampling window before the timed loop")
    ap.add_argument("--shared", action="store_true",
                    help="decode with pa_decode_shared (each shared block read once per group of sharers)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        line = run_reference(args)
    elif args.workload.startswith("prefill"):
        line = run_prefill_gpu(args)
    else:
        line = run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
