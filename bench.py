"""Benchmark of MLA decode over a paged latent KV cache on GB300.

One step = the whole hot path once: the split-KV schedule (mla_get_metadata),
the split-KV decode kernel and the log-sum-exp combine, over one batch of the
workload.  Default workload: b=128, s_q=1, h_q=128, h_kv=1, d=576, dv=512,
64-token pages, every sequence 4096 tokens, 576-element entries, pages in
order (the shape of FlashMLA's benchmark in the PAI tutorial, section 4).

Metric (the benchmark's own formula, compare_a in that section):
  bytes = (sum(seqlens)*h_kv*576 + b*s_q*h_q*576 + b*s_q*h_q*512) * 2
  flops = 2 * s_q * sum(seqlens) * h_q * (576 + 512)
  GB/s  = bytes / 1e6 / ms        TFLOPS = flops / 1e9 / ms

`--impl reference` times the fp64 CPU oracle on the host cores instead, on a
bounded sample of the same workload (whole sequences, all heads).

Prints one JSON line.  Run with no flags for N=1; under torchrun each rank runs
its own replica of the workload (no data-path collective) and rank 0 prints.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from mla_decode_attention_03_gb300 import workloads as W  # noqa: E402

L2_FLUSH_BYTES = 512 << 20
BREAKDOWN_EVERY = 8  # every 8th timed pass also times each kernel on its own
MIN_TIMED_S = 1.0    # the timed loop lasts at least this long, so that clock samples fall inside it

# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the decode
# kernel a workload runs on, taken from one ncu capture, keyed by a digest of
# that kernel's sources (comments and whitespace ignored) and by the workload
# (name, entry stride).  A kernel whose code changed since the capture reports
# null traffic.  Tiles of at most 16 rows (s_q x heads per KV head) run on the
# 16-row kernel, all others on the 128-row one.
KERNEL_SOURCES = {
    "mla_decode_kernel": ("mla_decode.cu", "mla_walk.cuh", "sm103_ptx.cuh", "mla_sched.cu", "mla_internal.h"),
    "mla_decode_small_kernel": ("mla_decode_small.cu", "mla_walk.cuh", "sm103_ptx.cuh", "mla_sched.cu",
                                "mla_internal.h"),
}
MEASURED_TRAFFIC = {
    ("304f7b3be80d2291", "bench", 576): 626847744,
    ("9c7e7b29035142a4", "v2lite", 640): 53639168,
}


def decode_kernel(s_q: int, h_q: int, h_kv: int) -> str:
    """Name of the decode kernel that runs this shape."""
    return "mla_decode_small_kernel" if s_q * (h_q // h_kv) <= 16 else "mla_decode_kernel"


def breakdown_steps(steps: int):
    """Indices of the timed passes that also carry events between the kernels
    (every BREAKDOWN_EVERY-th, at least one) and of the plain passes `value`
    is taken from (all passes if there are no others)."""
    inner = [k for k in range(steps) if k % BREAKDOWN_EVERY == BREAKDOWN_EVERY - 1] or [steps - 1]
    plain = [k for k in range(steps) if k not in set(inner)] or list(range(steps))
    return inner, plain


def passes_per_step(steps: int, seconds_per_pass: float, min_seconds: float = MIN_TIMED_S) -> int:
    """Passes of the hot path per timed step, so that `steps` steps last at
    least `min_seconds` (one pass per step when they already do)."""
    need = min_seconds / max(steps * seconds_per_pass, 1e-9)
    return max(1, int(np.ceil(need)))


def kernel_digest(kernel: str = "mla_decode_kernel") -> str:
    """Hash of a decode kernel's sources with // comments and whitespace
    removed: a comment edit keeps the measured traffic, a code edit drops it."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "mla_decode_attention_03_gb300", "csrc", name), encoding="utf-8") as f:
            code = re.sub(r"//[^\n]*", "", f.read())
        h.update("".join(code.split()).encode())
    return h.hexdigest()[:16]


def metric_bytes_flops(w) -> tuple[int, int]:
    S = int(w.cache_seqlens.sum())
    b, s_q, h_q = w.b, w.s_q, w.h_q
    nbytes = (S * w.h_kv * 576 + b * s_q * h_q * 576 + b * s_q * h_q * 512) * 2
    flops = 2 * s_q * S * h_q * (576 + 512)
    return nbytes, flops


def describe(w) -> str:
    sl = w.cache_seqlens.numpy()
    lens = f"L={int(sl[0])} for all" if (sl == sl[0]).all() else \
        f"L in [{int(sl.min())},{int(sl.max())}] sum {int(sl.sum())}"
    return (f"{w.name}: MLA decode b={w.b} s_q={w.s_q} h_q={w.h_q} h_kv={w.h_kv} d=576 dv=512 "
            f"page=64 {lens} entry stride {w.stride} causal={int(w.causal)}")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1900.0)), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed loop runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def window(self, t0: float, t1: float):
        """Keep only the samples taken between t0 and t1 (perf_counter seconds)."""
        self.lines = [(t, ln) for t, ln in self.lines if t0 <= t <= t1]

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 6:
                continue
            try:
                mhz.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for name, v in zip(names, f[2:6]):
                if v.lower() in ("active", "1"):
                    reasons.add(name)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    from mla_decode_attention_03_gb300 import ops

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = W.named(args.workload, stride=args.stride)
    nbytes, flops = metric_bytes_flops(w)
    q = w.q.to(dev)
    kc_alloc = w.kcache_alloc.to(dev)
    kc = kc_alloc[..., :576]
    bt = w.block_table.to(dev)
    sl = w.cache_seqlens.to(dev)
    parts = ops.num_parts(w.s_q, w.h_q, w.h_kv, dev)
    dec = ops.MLADecoder(w.b, w.s_q, w.h_q, w.h_kv, device=dev, parts=parts)
    out = torch.empty((w.b, w.s_q, w.h_q, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.b, w.h_q, w.s_q), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    # A timed step is R passes of the hot path over the batch, R chosen so the
    # K timed steps last at least MIN_TIMED_S (clock samples then fall inside
    # the loop).  Every pass is bracketed by two events (ev[0], ev[3]) with the
    # L2 flush outside them; the three kernels run back to back, each starting
    # its set-up while the one before it finishes (programmatic dependent
    # launch).  Every BREAKDOWN_EVERY-th pass also records events between the
    # kernels (which serialises them) for the per-kernel breakdown and the
    # decode kernel's own duration; `value` comes from the other passes.
    def step(ev=None, inner=False):
        if ev is not None:
            ev[0].record(stream)
        meta, nsplit = ops.get_mla_metadata(sl, parts, dec.status)
        if inner:
            ev[1].record(stream)
        ops.mla_decode_with_kvcache(q, kc, bt, sl, meta, nsplit, w.softmax_scale, w.causal, out=out,
                                    lse=lse, workspace=dec.workspace, status=dec.status, combine=False)
        if inner:
            ev[2].record(stream)
        ops.combine_splits(nsplit, dec.workspace, parts, out, lse)
        if ev is not None:
            ev[3].record(stream)

    # the clock sampler starts before the warm-up so that its own start-up falls
    # outside the timed loop; only samples taken during the loop are kept
    with ClockSampler(local) as clk:
        for _ in range(args.warmup):
            flush.fill_(1)
            step()
        torch.cuda.synchronize()
        ops.check_status(dec.status)
        # wall time of one pass with its flush, for the passes per step
        tp0 = time.perf_counter()
        for k in range(5):
            flush.fill_(k)
            step()
        torch.cuda.synchronize()
        reps = passes_per_step(args.steps, (time.perf_counter() - tp0) / 5)
        reps = int(max_over_ranks(float(reps), world))
        total = args.steps * reps
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(total)]
        inner_passes, plain = breakdown_steps(total)
        inner_set = set(inner_passes)
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for k in range(total):
            flush.fill_(k & 0xFF)  # L2 flush: a 512 MB write between passes, outside the events
            step(evs[k], inner=(k in inner_set))
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        wall = t1 - t0
    clk.window(t0, t1)
    barrier(world)
    ops.check_status(dec.status)
    t_meta = [evs[k][0].elapsed_time(evs[k][1]) for k in inner_passes]
    t_dec = [evs[k][1].elapsed_time(evs[k][2]) for k in inner_passes]
    t_comb = [evs[k][2].elapsed_time(evs[k][3]) for k in inner_passes]
    t_pass = [evs[k][0].elapsed_time(evs[k][3]) for k in plain]
    ms_pass = max_over_ranks(float(np.mean(t_pass)), world)
    ms_step = ms_pass * reps
    ms_dec = float(np.mean(t_dec))

    # end to end through the public API: pinned host q / block_table / seqlens in,
    # out / lse back, the cache resident in HBM
    e2e = run_e2e(args, w, dev, kc, parts, dec, flush, nbytes)
    e2e_runs = None
    if args.e2e_runs:
        e2e_runs = []
        for c in (int(x) for x in args.e2e_runs.split(",")):
            r = run_e2e(args, w, dev, kc, parts, dec, flush, nbytes, chunks=c)
            e2e_runs.append({"runs": r["runs"], "ms_per_step": r["ms_per_step"], "value": r["value"]})

    hbm_peak, tf_peak, peak_src = peaks()
    achieved = nbytes / 1e9 / (ms_dec / 1e3)
    kname = decode_kernel(w.s_q, w.h_q, w.h_kv)
    value = world * nbytes / 1e6 / ms_pass
    clocks = clk.summary()
    line = {
        "metric": "MLA decode achieved GB/s (pages' bandwidth formula), whole step",
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) bf16 q and cache (numpy PCG64), no weights",
        "config": {
            "workload": describe(w),
            "b": w.b, "s_q": w.s_q, "h_q": w.h_q, "h_kv": w.h_kv, "stride": w.stride,
            "sum_seqlens": int(w.cache_seqlens.sum()),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "num_parts": parts,
            "l2": "flushed between passes by a 512 MB write outside the timed events",
            "step": f"{reps} pass(es) of metadata + split-KV decode + combine over the batch",
            "passes_per_step": reps,
            "timing": f"{args.steps} steps x {reps} passes = {total} passes in {wall:.2f} s; value from the "
                      f"{len(plain)} passes timed with two events each; breakdown and roofline from the "
                      f"{len(inner_passes)} passes (every {BREAKDOWN_EVERY}th) with events between the kernels",
            "bytes_per_pass": nbytes, "flops_per_pass": flops,
        },
        "ms_per_pass": round(ms_pass, 5),
        "tflops": round(world * flops / 1e9 / ms_pass, 1),
        "breakdown_us": {"metadata": round(1e3 * float(np.mean(t_meta)), 2),
                         "decode": round(1e3 * ms_dec, 2),
                         "combine": round(1e3 * float(np.mean(t_comb)), 2),
                         "decode_median": round(1e3 * float(np.median(t_dec)), 2)},
        "wall_s_timed_loop": round(wall, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "traffic": MEASURED_TRAFFIC.get((kernel_digest(kname), w.name, w.stride)),
                     "kernel": kname, "peak_source": peak_src,
                     "tensor_tflops_achieved": round(flops / 1e9 / ms_dec, 1),
                     "tensor_frac": round(flops / 1e9 / ms_dec / tf_peak, 4)},
        "e2e": e2e,
        **({"e2e_runs": e2e_runs} if e2e_runs else {}),
        "gpu_launches": 3 * total,
        "clocks": clocks,
    }
    if clocks.get("sm_mhz"):
        # the pass time in SM cycles at the median clock under load
        line["clock_normalised"] = {"sm_cycles_per_pass": round(ms_pass * 1e-3 * clocks["sm_mhz"] * 1e6),
                                    "decode_sm_cycles": round(ms_dec * 1e-3 * clocks["sm_mhz"] * 1e6)}
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(args, w, dev, kc, parts, dec, flush, nbytes, chunks=0):
    """The same step through the host-buffer entry point (mla_decode_host):
    q, block_table and cache_seqlens copied in from pinned host memory and
    out and lse copied back, every step, with the copies of one run of
    sequences overlapping the decode of its neighbours."""
    from mla_decode_attention_03_gb300 import ops

    q_h = w.q.pin_memory()
    bt_h = w.block_table.pin_memory()
    sl_h = w.cache_seqlens.pin_memory()
    out_h = torch.empty((w.b, w.s_q, w.h_q, 512), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty((w.b, w.h_q, w.s_q), dtype=torch.float32).pin_memory()
    hd = ops.HostDecoder(w.b, w.s_q, w.h_q, bt_h.shape[1], w.h_kv, device=dev, parts=parts)
    stream = torch.cuda.current_stream()
    h2d = q_h.numel() * 2 + bt_h.numel() * 4 + sl_h.numel() * 4
    d2h = out_h.numel() * 2 + lse_h.numel() * 4
    runs = len(ops.host_chunks(sl_h, chunks)) - 1

    def step():
        hd(q_h, kc, bt_h, sl_h, w.softmax_scale, w.causal, out=out_h, lse=lse_h, chunks=chunks)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    n = max(10, min(args.steps, 200))
    times = []
    for k in range(n):
        flush.fill_(k & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    ops.check_status(hd.status)
    hd.close()
    ms = float(np.mean([a.elapsed_time(b) for a, b in times]))
    link = host_link(dev, h2d, d2h, stream)
    link["copies_fraction_of_step"] = round(link["copies_ms"] / ms, 3)
    return {"value": round(nbytes / 1e6 / ms, 1), "unit": "GB/s", "ms_per_step": round(ms, 5), "runs": runs,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "host_link": link,
            "note": f"mla_decode_host: pinned host q/block_table/seqlens in, out/lse out, {runs} run(s) of "
                    "sequences with copies overlapping the decode; the KV cache stays resident"}


def host_link(dev, h2d: int, d2h: int, stream, reps: int = 20) -> dict:
    """The host link's own rate for the step's copy sizes: one plain
    cudaMemcpyAsync of h2d bytes from pinned host memory to the device, and one
    of d2h bytes back, each timed alone with CUDA events (median of `reps`)."""
    def timed(dst, src):
        for _ in range(3):
            dst.copy_(src, non_blocking=True)
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dst.copy_(src, non_blocking=True)
            b.record(stream)
            ts.append((a, b))
        torch.cuda.synchronize()
        return float(np.median([a.elapsed_time(b) for a, b in ts]))
    h_in = torch.empty(h2d, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(h2d, dtype=torch.uint8, device=dev)
    d_out = torch.empty(d2h, dtype=torch.uint8, device=dev)
    h_out = torch.empty(d2h, dtype=torch.uint8).pin_memory()
    ms_in = timed(d_in, h_in)
    ms_out = timed(h_out, d_out)
    return {"h2d_gbs": round(h2d / 1e6 / ms_in, 1), "d2h_gbs": round(d2h / 1e6 / ms_out, 1),
            "copies_ms": round(ms_in + ms_out, 5),
            "note": "plain pinned cudaMemcpyAsync of the step's copy sizes, each direction alone"}


# ----------------------------------------------------------- CPU baseline
def sample_rows(w, n_rows: int, offset: int = 0) -> np.ndarray:
    """A bounded sample of the workload's output rows: whole sequences (all
    query positions and heads) taken in order from `offset`, or a leading run
    of one sequence's rows when n_rows is below one sequence."""
    per_seq = w.s_q * w.h_q
    rows = []
    i = offset % w.b
    while len(rows) < n_rows:
        take = min(per_seq, n_rows - len(rows))
        for r in range(take):
            rows.append((i, r // w.h_q, r % w.h_q))
        i = (i + 1) % w.b
    return np.asarray(rows, dtype=np.int32)


def sample_bytes(w, rows) -> float:
    """The metric's bytes attributable to a row sample: each sequence's cache
    bytes in proportion to the share of its rows sampled, plus the q and out
    bytes of the sampled rows (for whole sequences this is the formula itself)."""
    per_seq = w.s_q * w.h_q
    seqs, counts = np.unique(rows[:, 0], return_counts=True)
    L = w.cache_seqlens.numpy()[seqs].astype(np.float64)
    cache = float((L * w.h_kv * 576 * 2 * counts / per_seq).sum())
    return cache + len(rows) * (576 + 512) * 2


def time_oracle(w, rows, bits):
    import oracle
    qb, kb = bits
    t0 = time.perf_counter()
    oracle.decode_rows(qb, kb, w.block_table.numpy(), w.cache_seqlens.numpy(), rows,
                       softmax_scale=w.softmax_scale, causal=w.causal)
    return time.perf_counter() - t0


def cpu_baseline(w, target_s: float = 10.0):
    """The oracle, as it stands, on the host cores: a probe of 2 sequences sets
    the sample size to about `target_s` seconds of work (capped at the whole batch)."""
    import oracle
    bits = w.numpy_bits()
    per_seq = w.s_q * w.h_q
    probe = sample_rows(w, 2 * per_seq)
    dt = time_oracle(w, probe, bits)
    n_seqs = int(max(2, min(w.b, round(2 * target_s / max(dt, 1e-3)))))
    rows = sample_rows(w, n_seqs * per_seq)
    dt = time_oracle(w, rows, bits)
    nbytes = sample_bytes(w, rows)
    return {"value": round(nbytes / 1e6 / (dt * 1e3), 4), "unit": "GB/s",
            "cores": oracle.host_threads(), "kind": "oracle",
            "sample": f"{n_seqs} of {w.b} sequences, every query position and head "
                      f"({len(rows)} rows), {dt:.1f} s of fp64 C on the host cores"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = W.named(args.workload, stride=args.stride)
    bits = w.numpy_bits()
    # about two minutes of oracle work in total, whatever --steps is
    n_rows = int(max(16, min(16 * w.s_q * w.h_q, 150000 // max(1, args.steps + args.warmup))))
    for k in range(args.warmup):
        time_oracle(w, sample_rows(w, n_rows, k), bits)
    times, total_bytes = [], 0
    for k in range(args.steps):
        rows = sample_rows(w, n_rows, args.warmup + k)
        times.append(time_oracle(w, rows, bits))
        total_bytes += sample_bytes(w, rows)
    ms = 1e3 * sum(times) / len(times)
    value = total_bytes / 1e6 / (1e3 * sum(times))
    sample = f"{n_rows} output rows per step (whole sequences in order when >= {w.s_q * w.h_q})"
    line = {
        "impl": "reference",
        "metric": "MLA decode achieved GB/s (pages' bandwidth formula), whole step",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(w), "sample_per_step": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.host_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_sweep(args):
    """Bandwidth against mean sequence length at b=128, h_q=128 (the shape of the
    seqlen sweep plotted in the PAI tutorial, section 4; `--sweep-heads` sets
    another head count, e.g. 16 for the 16-row kernel), for the 576- and
    640-element entry layouts.  Inputs are drawn on the device (a seeded
    torch generator): this mode times only, it compares nothing."""
    from mla_decode_attention_03_gb300 import ops

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    b, h_q = 128, args.sweep_heads
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    parts = ops.num_parts(1, h_q, 1, dev)
    dec = ops.MLADecoder(b, 1, h_q, 1, device=dev, parts=parts)
    q = torch.randn((b, 1, h_q, 576), generator=gen, device=dev).to(torch.bfloat16)
    for L in [int(x) for x in args.sweep.split(",")]:
        n_pages = -(-L // 64)
        for stride in (576, 640):
            kc_alloc = torch.zeros((b * n_pages, 64, 1, stride), dtype=torch.bfloat16, device=dev)
            kc_alloc[..., :576] = torch.randn((b * n_pages, 64, 1, 576), generator=gen, device=dev)
            kc = kc_alloc[..., :576]
            bt = torch.arange(b * n_pages, dtype=torch.int32, device=dev).view(b, n_pages)
            sl = torch.full((b,), L, dtype=torch.int32, device=dev)
            out = torch.empty((b, 1, h_q, 512), dtype=torch.bfloat16, device=dev)
            lse = torch.empty((b, h_q, 1), dtype=torch.float32, device=dev)
            nbytes = (b * L * 576 + b * h_q * 576 + b * h_q * 512) * 2

            def step():
                meta, nsplit = ops.get_mla_metadata(sl, parts, dec.status)
                ops.mla_decode_with_kvcache(q, kc, bt, sl, meta, nsplit, 576 ** -0.5, False, out=out,
                                            lse=lse, workspace=dec.workspace, status=dec.status)
            for _ in range(5):
                flush.fill_(1)
                step()
            evs = []
            for k in range(args.steps):
                flush.fill_(k & 0xFF)
                a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                step()
                e.record()
                evs.append((a, e))
            torch.cuda.synchronize()
            ops.check_status(dec.status)
            ms = float(np.mean([a.elapsed_time(e) for a, e in evs]))
            print(json.dumps({"mode": "sweep", "mean_seqlen": L, "stride": stride, "b": b, "h_q": h_q,
                              "ms": round(ms, 5), "GB/s": round(nbytes / 1e6 / ms, 1),
                              "TFLOPS": round(2 * b * L * h_q * 1088 / 1e9 / ms, 1)}), flush=True)
            del kc_alloc, kc


def run_cache_ops(args):
    """Throughput of the cache maintenance next to the decode (mla_write_cache,
    mla_copy_blocks) on 640-element entries: one decode step's new tokens
    (b=128), a prefill-sized write (65536 tokens), and copy_blocks_mla over 2048
    page pairs of 4 layer caches.  GB/s counts bytes read + written; L2 is
    flushed between iterations.  Timing only, it compares nothing."""
    from mla_decode_attention_03_gb300 import ops

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    status = ops.new_status(dev)

    def timed(fn):
        for _ in range(5):
            flush.fill_(1)
            fn()
        evs = []
        for k in range(args.steps):
            flush.fill_(k & 0xFF)
            a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            e.record()
            evs.append((a, e))
        torch.cuda.synchronize()
        ops.check_status(status)
        return float(np.median([a.elapsed_time(e) for a, e in evs]))

    num_blocks = 4096
    kc_alloc = torch.zeros((num_blocks, 64, 1, 640), dtype=torch.bfloat16, device=dev)
    kc = kc_alloc[..., :576]
    for tokens, label in ((128, "write_cache: one decode step, b=128"), (65536, "write_cache: 65536 tokens")):
        kv_c = torch.randn((tokens, 512), generator=gen, device=dev).to(torch.bfloat16)
        k_pe = torch.randn((tokens, 64), generator=gen, device=dev).to(torch.bfloat16)
        slots = torch.randperm(num_blocks * 64, generator=gen, device=dev)[:tokens].to(torch.int64)
        ms = timed(lambda: ops.write_cache(kv_c, k_pe, slots, kc, status))
        nbytes = tokens * (576 * 2) * 2 + tokens * 8
        print(json.dumps({"mode": "cache_ops", "op": label, "ms": round(ms, 5),
                          "GB/s": round(nbytes / 1e6 / ms, 1), "bytes": nbytes}), flush=True)
    layers = [torch.zeros((num_blocks, 64, 1, 640), dtype=torch.bfloat16, device=dev) for _ in range(4)]
    perm = torch.randperm(num_blocks, generator=gen, device=dev)
    mapping = torch.stack([perm[:2048], perm[2048:4096]], dim=1).to(torch.int64)
    ptrs = torch.tensor([c.data_ptr() for c in layers], dtype=torch.int64, device=dev)
    mapping = mapping.to(dev)
    lib = ops.load_library()
    stream = torch.cuda.current_stream(dev).cuda_stream

    def copy_step():
        # the C ABI call with the layer-pointer array already on the device
        rc = lib.mla_copy_blocks(ptrs.data_ptr(), len(layers), mapping.data_ptr(), mapping.shape[0],
                                 num_blocks, 64, 640, status.data_ptr(), stream)
        if rc != 0:
            raise RuntimeError(f"mla_copy_blocks failed: {rc}")

    ms = timed(copy_step)
    nbytes = 2 * 4 * 2048 * 64 * 640 * 2
    print(json.dumps({"mode": "cache_ops", "op": "copy_blocks: 2048 pairs x 4 layers, 640-element entries",
                      "ms": round(ms, 5), "GB/s": round(nbytes / 1e6 / ms, 1), "bytes": nbytes}), flush=True)


# Small cases of each workload for ncu captures with many passes: larger than
# L2 (129 MB) so that DRAM counters mean something, a few hundred MB at most.
NCU_CASES = {
    "bench_full": lambda: W.named("bench"),
    "bench32": lambda: W.make(32, 1, 128, 1, [4096] * 32, stride=576, seed=0, permute=False, name="bench32"),
    "mtp32": lambda: W.make(32, 2, 128, 1,
                            lambda r: np.clip(np.round(r.normal(4096.0, 1024.0, size=32)), 256, 8192),
                            stride=640, causal=True, seed=0, name="mtp32"),
    "skewed_s": lambda: W.make(64, 1, 128, 1,
                               lambda r: np.concatenate([[49152, 49152], r.integers(64, 1024, size=62, endpoint=True)]),
                               stride=640, seed=0, peaky_frac=0.01, name="skewed_s"),
    "v2lite": lambda: W.named("v2lite"),
}


def run_ncu_case(args):
    """Three L2-flushed passes of the hot path on one small case, for ncu
    (capture the third decode launch with -k regex:mla_decode_kernel -s 2 -c 1)."""
    from mla_decode_attention_03_gb300 import ops

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = NCU_CASES[args.ncu_case]()
    q, kc = w.q.to(dev), w.kcache_alloc.to(dev)[..., :576]
    bt, sl = w.block_table.to(dev), w.cache_seqlens.to(dev)
    parts = ops.num_parts(w.s_q, w.h_q, w.h_kv, dev)
    dec = ops.MLADecoder(w.b, w.s_q, w.h_q, w.h_kv, device=dev, parts=parts)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for k in range(3):
        flush.fill_(k)
        dec.plan(sl)
        dec(q, kc, bt, sl, w.softmax_scale, w.causal)
    torch.cuda.synchronize()
    ops.check_status(dec.status)
    nbytes, flops = metric_bytes_flops(w)
    print(json.dumps({"mode": "ncu_case", "case": args.ncu_case, "workload": describe(w),
                      "bytes_per_pass": nbytes, "flops_per_pass": flops}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="bench", choices=sorted(W.WORKLOADS))
    ap.add_argument("--stride", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", default=None,
                    help="comma-separated mean sequence lengths: print one line per (length, stride)")
    ap.add_argument("--sweep-heads", type=int, default=128, help="query heads (h_kv = 1) of the --sweep batch")
    ap.add_argument("--cache-ops", action="store_true",
                    help="time the cache write and copy_blocks kernels instead of the decode step")
    ap.add_argument("--e2e-runs", default=None,
                    help="comma-separated run counts: also time the host-buffer step with each "
                         "(1 = copies in, decode, copies out one after another) and add them as e2e_runs")
    ap.add_argument("--ncu-case", default=None, choices=sorted(NCU_CASES),
                    help="run three passes of one small case for an ncu capture and exit")
    args = ap.parse_args()
    if args.ncu_case:
        run_ncu_case(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.cache_ops:
        run_cache_ops(args)
        return
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
