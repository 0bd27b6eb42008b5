#!/usr/bin/env python3
"""Benchmark of single-token paged GQA decode attention on GB300.

Metric: effective KV-read bandwidth, i.e. the algorithmic K/V bytes of the attended tokens
divided by the device time of one call (and the same time as microseconds per call).
One step = one pass of the whole hot path over the batch: [codebook format: query
rotation] -> split-K partition kernel -> float reduce, through the C-ABI library.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line. ``--impl reference`` times the fp64 CPU oracle (the only reference
this method has here) on bounded samples of the same workload.
Multi-GPU (torchrun, N > 1): every rank runs an independent replica of the batch (the path
has no cross-GPU exchange), times are maxed over ranks and value sums all ranks' bytes.
"""
from __future__ import annotations

import argparse
import csv
import datetime as _dt
import glob
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention effective KV-read GB/s (% of GB300 HBM peak); µs/call"
UNIT = "GB/s"
DEFAULT_WORKLOAD = "llama3_8b_bf16"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20
# device-side hold ahead of a timed loop: SM cycles per second (the maximum SM clock, so the
# hold lasts at least as long at lower clocks), margin over the host's enqueue time, minimum
HOLD_CYCLES_PER_S = 2.07e9
HOLD_MARGIN = 2.0
HOLD_MIN_S = 0.5e-3


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true", help="skip the nvidia-smi clock sampling and its soak")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="time only the chosen workload (skip the FP8, Gemma-style, 4-bit and tiny entries)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- ranks
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- peaks / clocks
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 measurement)"


class ClockSampler:
    """nvidia-smi samples (every 200 ms) over a window that contains the timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.dev), "-lms", "200"], stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark_begin(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for r in csv.reader(f):
                if len(r) < 10:
                    continue
                try:
                    ts = _dt.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(r[2]), float(r[3]), float(r[4]), [x.strip() for x in r[5:]]))
                except ValueError:
                    continue
        os.unlink(self.path)
        win = [x for x in rows if self.t0 - 0.25 <= x[0] <= self.t1 + 0.25] or rows
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for x in win for i in range(4) if x[4][1 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(x[1] for x in win), "sm_max_mhz": max(x[2] for x in win),
                "power_w_max": max(x[3] for x in win), "samples": len(win), "reasons": reasons}


# ----------------------------------------------------------------------------- inputs
def build_inputs(spec, encode_on_gpu=True, writer_times=None):
    """Seeded inputs on the host for the chosen workload. BF16 caches come straight from the
    generator; FP8 and codebook caches are written on the GPU by the library's own encoders
    from the seeded fp32 source (and copied back to the host for the end-to-end leg).
    writer_times: a dict that receives, per cache side, the cache writer's device time
    (CUDA events around its launches) and the vectors (rows of D) it wrote.
    Returns (layout, host tensors, fp32 sources or None)."""
    import math

    import torch

    import decode_attention_paged_gqa_gb300 as da
    from decode_attention_paged_gqa_gb300 import workloads as wl

    lay = wl.make_layout(spec)
    host = {"q": wl.make_query(spec), "bt": torch.from_numpy(lay.block_tables),
            "lens": torch.from_numpy(lay.context_lens), "k_scales": None, "v_scales": None, "codebook": None,
            "sign": None}
    if spec.kv_format == "bf16":
        host["k"] = wl.kv_bf16(spec, "k", lay.num_blocks)
        host["v"] = wl.kv_bf16(spec, "v", lay.num_blocks)
        return lay, host, None
    sides = {"fp8": ("fp8", "fp8"), "cb4": ("cb4", "cb4"), "fp8k_cb4v": ("fp8", "cb4"),
             "cb3k_cb4v": ("cb3", "cb4")}[spec.kv_format]
    src = {w: wl.kv_source(spec, w, lay.num_blocks) for w in ("k", "v")}
    D = spec.head_dim
    if "cb3" in sides or "cb4" in sides:
        host["sign"] = wl.sign_pattern(spec)
    if not encode_on_gpu:  # the CPU reference arm encodes with the oracle from `src`
        return lay, host, src
    cbs = {}
    if "cb3" in sides or "cb4" in sides:
        cbs = {b: torch.tensor(da.decode_attn_codebook_lloyd_max(1 << b, 1.0 / math.sqrt(D))) for b in (3, 4)}
        host["codebook"] = torch.cat([cbs[3], cbs[4]]) if sides[0] == "cb3" else cbs[4]
        sg_d = host["sign"].cuda()
    for w, side in zip(("k", "v"), sides):
        x = src[w].cuda()
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        if side == "fp8":
            codes = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
            sc = torch.empty(1, dtype=torch.float32, device="cuda")
            torch.cuda.synchronize()
            ev[0].record()
            da.decode_attn_encode_fp8(x, x.numel(), codes, sc)
            ev[1].record()
        else:
            bits = 3 if side == "cb3" else 4
            codes = torch.empty(x.shape[:-1] + (D * bits // 8,), dtype=torch.uint8, device="cuda")
            sc = torch.empty(x.shape[:-1], dtype=torch.float32, device="cuda")
            cb_d = cbs[bits].cuda()
            torch.cuda.synchronize()
            ev[0].record()
            da.decode_attn_encode_codebook(x, x.numel() // D, D, bits, sg_d, cb_d, codes, sc)
            ev[1].record()
        torch.cuda.synchronize()
        if writer_times is not None:
            ms = ev[0].elapsed_time(ev[1])
            nvec = x.numel() // D
            writer_times[w] = {"format": side, "vectors": nvec, "ms": ms, "ns_per_vector": ms * 1e6 / nvec,
                               "input_gbs": x.numel() * 4 / (ms * 1e-3) / 1e9}
        host[w], host[w + "_scales"] = codes.cpu(), sc.cpu()
        del x
    return lay, host, src


# the sources each partition kernel is compiled from (a recorded DRAM traffic figure is only
# reported while the kernel's sources still hash to the profiled build)
PARTITION_SOURCES = {
    "partition_tc_kernel": ("partition_tc.cu", "page_softmax.cuh", "page_walk.cuh", "ptx.cuh", "da_internal.cuh"),
    "partition_cb_kernel": ("partition_cb.cuh", "item_walk.cuh", "page_softmax.cuh", "page_walk.cuh", "ptx.cuh",
                            "da_internal.cuh", "kv_formats.cuh"),
}


def partition_kernel(kv_format: str) -> str:
    return "partition_tc_kernel" if kv_format in ("bf16", "fp8") else "partition_cb_kernel"


def source_hash(kernel: str) -> str:
    h = hashlib.sha1()
    for name in PARTITION_SOURCES[kernel]:
        with open(os.path.join(ROOT, "decode_attention_paged_gqa_gb300", "csrc", name), "rb") as fh:
            h.update(name.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summaries, if taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entries = json.load(f)["entries"]
    except (OSError, KeyError, ValueError):
        return None
    for t in entries:
        if t.get("kernel") == kernel and t.get("workload") == workload and t.get("source_hash") == source_hash(kernel):
            return t.get("dram_bytes_per_launch")
    return None


# ----------------------------------------------------------------------------- CPU oracle
def oracle_inputs(spec, host, src, nseq):
    """The oracle's inputs for the first nseq sequences: a compact cache holding only their
    blocks (renumbered), encoded by the oracle's own encoders for FP8 and the codebook."""
    import numpy as np

    import oracle

    bt, lens = host["bt"].numpy()[:nseq], host["lens"].numpy()[:nseq]
    pages = -(-lens // spec.block_size)
    used = np.unique(np.concatenate([bt[b, :pages[b]] for b in range(nseq)] + [np.zeros(0, np.int32)]))
    remap = np.full(max(int(host["bt"].max()) + 1, 1), -1, np.int64)
    remap[used] = np.arange(len(used))
    sub_bt = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
    q = host["q"][:nseq].contiguous().view(__import__("torch").int16).numpy().view(np.uint16)
    kw = {}
    if spec.kv_format == "bf16":
        k = host["k"].view(__import__("torch").int16).numpy().view(np.uint16)[used]
        v = host["v"].view(__import__("torch").int16).numpy().view(np.uint16)[used]
    else:
        sides = oracle.SIDES[spec.kv_format]
        D = spec.head_dim
        cb = {b: oracle.lloyd_max(1 << b, 1.0 / np.sqrt(D))[1] for b in (3, 4)}
        sg = host["sign"].numpy() if host["sign"] is not None else None
        enc = {}
        for w, side in zip(("k", "v"), sides):
            if side == "fp8":
                codes, sc = oracle.fp8_quantize(src[w].numpy())
                enc[w] = (codes[used], sc)
            else:
                bits = 3 if side == "cb3" else 4
                enc[w] = oracle.cb_encode(bits, src[w].numpy()[used], sg, cb[bits])
        k, v = enc["k"][0], enc["v"][0]
        kw = dict(k_scales=enc["k"][1], v_scales=enc["v"][1])
        if sg is not None:
            kw["codebook"] = np.concatenate([cb[3], cb[4]]) if sides[0] == "cb3" else cb[4]
            kw["sign_pattern"] = sg
    return q, k, v, sub_bt, lens, kw


def oracle_sample(spec, host, src, target_s: float, max_seqs=None, threads: int = 0):
    """Time the fp64 oracle on the first n sequences (all heads) of the workload, n chosen so
    that the timed sample takes about target_s; when the whole batch takes less than that,
    the batch is repeated until target_s has passed. threads: 0 = every host core, else that
    many. Returns (GB/s, seconds, n, threads, reps)."""
    import oracle
    from decode_attention_paged_gqa_gb300.metrics import algorithmic_kv_bytes

    def run(nseq):
        q, k, v, bt, lens, kw = oracle_inputs(spec, host, src, nseq)
        t0 = time.perf_counter()
        _, thr = oracle.decode_attention(q, k, v, bt, lens, kv_format=spec.kv_format, num_kv_heads=spec.num_kv_heads,
                                         softmax_scale=spec.scale, softcap=spec.softcap, window=spec.window,
                                         partition_size=spec.partition_size, split_threshold=spec.split_threshold,
                                         threads=threads, return_threads=True, **kw)
        return time.perf_counter() - t0, thr, lens

    t1, _, _ = run(1)
    n = max(1, min(spec.batch, int(target_s / max(t1, 1e-3))))
    if max_seqs:
        n = min(n, max_seqs)
    dt, thr, lens = run(n)
    reps = 1
    while dt < target_s and not max_seqs:
        more, thr, _ = run(n)
        dt += more
        reps += 1
    nbytes = reps * algorithmic_kv_bytes(lens, spec.window, spec.num_kv_heads, spec.kv_format, spec.head_dim)
    return nbytes / dt / 1e9, dt, n, thr, reps


def reference_arm(args, spec, rank, world):
    if rank != 0:
        return
    import oracle

    oracle.build()
    lay, host, src = build_inputs(spec, encode_on_gpu=False)
    per_step = max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(spec, host, src, per_step / 4, max_seqs=1)
    vals, secs, nseq, thr = [], 0.0, 0, 0
    for _ in range(args.steps):
        gbs, dt, n, thr, _ = oracle_sample(spec, host, src, per_step)
        vals.append(gbs)
        secs += dt
        nseq = n
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * secs / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": spec.name, "sample_sequences_per_step": nseq},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle",
                             "sample": f"first {nseq} of {spec.batch} sequences, all {spec.num_q_heads} heads, "
                                       f"per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm
# workloads timed beside the headline in the same process (one entry each in "per_workload"):
# the FP8 long-context batch, the Gemma-style windowed batch, the 4-bit codebook batch, and the
# tiny batch (L2-resident, latency-bound; its oracle is timed on every core and on one)
EXTRA_WORKLOADS = ("fp8_long_32k", "gemma_window_softcap", "cb4_long_32k", "tiny_bf16")
# kernels per call: the partition kernel and the reduce, plus the query rotation for formats
# whose keys are stored on the rotated basis
KERNELS_PER_CALL = {"bf16": 2, "fp8": 2, "cb4": 3, "fp8k_cb4v": 2, "cb3k_cb4v": 3}


class Prepared:
    """One workload resident on the device: inputs, params, workspace and output."""

    def __init__(self, spec):
        import torch

        import decode_attention_paged_gqa_gb300 as da
        from decode_attention_paged_gqa_gb300.metrics import algorithmic_kv_bytes

        self.spec = spec
        self.writer_times = {}
        self.lay, self.host, self.src = build_inputs(spec, writer_times=self.writer_times)
        self.dev = {k: (None if t is None else t.cuda()) for k, t in self.host.items()}
        self.kv_bytes = algorithmic_kv_bytes(self.lay.context_lens, spec.window, spec.num_kv_heads, spec.kv_format,
                                             spec.head_dim)
        self.cache_bytes = sum(self.host[w].numel() * self.host[w].element_size() for w in ("k", "v"))
        self.p = da.make_params(batch=spec.batch, num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                                head_dim=spec.head_dim, num_blocks=self.lay.num_blocks,
                                max_blocks_per_seq=self.lay.block_tables.shape[1], max_context_len=spec.ctx_max,
                                kv_format=spec.kv_format, softmax_scale=spec.scale, softcap=spec.softcap,
                                window=spec.window, partition_size=spec.partition_size,
                                split_threshold=spec.split_threshold, query_len=spec.query_len)
        self.ws = torch.empty(da.decode_attn_workspace_bytes(self.p), dtype=torch.uint8, device="cuda")
        da.attach_workspace(self.p, self.ws)
        da.decode_attn_workspace_init(self.p)
        self.out = torch.empty(tuple(self.host["q"].shape), dtype=torch.float32, device="cuda")  # [B, (T,) Hq, D]
        self.stream = torch.cuda.current_stream()
        d = self.dev
        self.call = (d["q"], d["k"], d["v"], d["k_scales"], d["v_scales"], d["codebook"], d["sign"], d["bt"],
                     d["lens"], self.out, self.p)

    def step(self):
        """One call of the public entry point: query rotation (codebook keys), partition kernel, reduce."""
        import decode_attention_paged_gqa_gb300 as da

        da.decode_attn_paged(*self.call, stream=self.stream)

    def partition_only(self):
        """The partition phase alone, through its own entry point (its inputs -- the rotated query
        for codebook keys -- left in place by an earlier call)."""
        import decode_attention_paged_gqa_gb300 as da

        da.decode_attn_partition(*self.call, stream=self.stream)

    def device_error(self):
        import decode_attention_paged_gqa_gb300 as da

        return da.decode_attn_get_device_error(self.p)

    def host_seconds(self, fn, n=8):
        """Host time to enqueue one fn() (the device is not waited for)."""
        import torch

        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        t1 = time.perf_counter()
        torch.cuda.synchronize()
        return (t1 - t0) / n

    def hold(self, seconds):
        """Queues a device-side busy wait of at least `seconds` on the stream. The timed launches
        are enqueued behind it, so the device runs them back to back and the events around them
        time the device's work, not the host's launch rate (which, for calls of a few tens of
        microseconds through the Python binding, can be the slower of the two)."""
        import torch

        with torch.cuda.stream(self.stream):
            torch.cuda._sleep(int(seconds * HOLD_CYCLES_PER_S))

    def time_calls(self, K, world=1):
        """Device time of K back-to-back calls (CUDA events on the launching stream, barrier and
        synchronize on both sides, the calls queued behind a hold); ms per call, maxed over ranks."""
        import torch

        host_s = self.host_seconds(self.step)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        self.hold(HOLD_MARGIN * K * host_s + HOLD_MIN_S)
        a.record(self.stream)
        for _ in range(K):
            self.step()
        b.record(self.stream)
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(a.elapsed_time(b) / K, world)

    def time_partition(self, K):
        """Device time per launch of the partition kernel (ms): K launches back to back between two
        events on the launching stream, queued behind a hold, after one full call that leaves the
        phase's inputs in place. Each launch is scheduled during the previous one's last CTAs and
        waits in-kernel for it to finish, as in a stream of calls, so the launch latency that an
        event pair around a single launch would add is not counted."""
        import torch

        self.step()
        host_s = self.host_seconds(self.partition_only)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        self.hold(HOLD_MARGIN * K * host_s + HOLD_MIN_S)
        a.record(self.stream)
        for _ in range(K):
            self.partition_only()
        b.record(self.stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / K


def soak(prep, seconds):
    """Untimed load so the clock samples bracket the timed region."""
    import torch

    end = time.time() + seconds
    while time.time() < end:
        for _ in range(20):
            prep.step()
        torch.cuda.synchronize()


def cpu_baseline_entry(spec, prep, seconds, threads=0):
    gbs, dt, n, thr, reps = oracle_sample(spec, prep.host, prep.src, seconds, threads=threads)
    return {"value": gbs, "unit": UNIT, "cores": thr, "kind": "oracle",
            "sample": f"first {n} of {spec.batch} sequences, all {spec.num_q_heads} heads, {reps} pass(es), "
                      f"{dt:.1f} s"}


def per_workload_entries(names, K, warmup, peak, local, with_cpu, cpu_seconds):
    """The partition kernel and the whole call of each named workload, timed like the headline
    (same K, warm-up, events), inside one clock-sampling window."""
    import gc

    import torch

    import oracle
    from decode_attention_paged_gqa_gb300 import workloads as wl

    entries = {}
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.6)
    clocks.mark_begin()
    for name in names:
        spec = wl.WORKLOADS[name]
        prep = Prepared(spec)
        for _ in range(max(3, warmup)):
            prep.step()
        torch.cuda.synchronize()
        soak(prep, 0.3)
        call_ms = prep.time_calls(K)
        part_ms = prep.time_partition(K)
        if prep.device_error():
            raise SystemExit(f"device reported bad input on {name}")
        kernel = partition_kernel(spec.kv_format)
        gbs, part_gbs = prep.kv_bytes / (call_ms * 1e-3) / 1e9, prep.kv_bytes / (part_ms * 1e-3) / 1e9
        e = {"kv_format": spec.kv_format, "us_per_call": call_ms * 1000, "value": gbs, "unit": UNIT,
             "pct_of_hbm_peak": 100 * gbs / peak, "algorithmic_kv_bytes": prep.kv_bytes,
             "roofline": {"bound": "hbm", "kernel": kernel, "achieved": part_gbs, "peak": peak, "unit": "GB/s",
                          "frac": part_gbs / peak, "partition_us": part_ms * 1000,
                          "traffic": recorded_traffic(kernel, spec.name)},
             "gpu_launches": K * KERNELS_PER_CALL[spec.kv_format]}
        if prep.cache_bytes <= L2_BYTES:
            e["note"] = "L2-resident and latency-bound: not compared with the HBM peak"
        if prep.writer_times:  # the cache writers that filled this workload's quantised caches
            e["cache_writers"] = prep.writer_times
        if with_cpu and spec.name == "tiny_bf16":
            oracle.build()
            e["cpu_baseline"] = {"all_cores": cpu_baseline_entry(spec, prep, cpu_seconds),
                                 "one_core": cpu_baseline_entry(spec, prep, cpu_seconds, threads=1)}
        entries[name] = e
        del prep
        gc.collect()
        torch.cuda.empty_cache()
    clocks.mark_end()
    clk = clocks.stop()
    for e in entries.values():
        e["clocks"] = clk
    return entries


def main():
    args = parse_args()
    from decode_attention_paged_gqa_gb300 import workloads as wl

    spec = wl.WORKLOADS[args.workload]
    rank, world, local = dist_setup()
    if args.impl == "reference":
        reference_arm(args, spec, rank, world)
        return

    import torch

    import decode_attention_paged_gqa_gb300 as da
    from decode_attention_paged_gqa_gb300 import build as lib_build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the product path has no CPU fallback)")
    lib_build.build()
    torch.cuda.set_device(local)
    prep = Prepared(spec)
    for _ in range(max(3, args.warmup)):
        prep.step()
    torch.cuda.synchronize()
    if prep.device_error():
        raise SystemExit("device reported bad input during warm-up")

    clocks = None if args.no_clocks else ClockSampler(local)
    if clocks:
        clocks.start()
        time.sleep(0.6)  # nvidia-smi start-up
        clocks.mark_begin()
        soak(prep, 1.0)
    K = args.steps
    step_ms = prep.time_calls(K, world)
    # the partition kernel's duration: a second pass of K steps, right after the timed one
    part_ms = prep.time_partition(K)
    clk = None
    if clocks:
        time.sleep(0.3)
        clocks.mark_end()
        clk = clocks.stop()
    if prep.device_error():
        raise SystemExit("device reported bad input during the timed steps")

    # end to end through decode_attn_paged with host buffers: every step copies all inputs
    # from pinned host memory and reads the output back
    e2e = None
    if not args.no_e2e:
        pin = {k: (None if t is None else t.pin_memory()) for k, t in prep.host.items()}
        out_h = torch.empty(prep.out.shape, dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in pin.values() if t is not None)
        d2h = out_h.numel() * 4

        def e2e_step():
            for k2, t in pin.items():
                if t is not None:
                    prep.dev[k2].copy_(t, non_blocking=True)
            da.decode_attn_paged(*prep.call, stream=prep.stream)
            out_h.copy_(prep.out, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        Ke = max(3, min(K, 20))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        a.record(prep.stream)
        for _ in range(Ke):
            e2e_step()
        b.record(prep.stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b) / Ke, world)
        e2e = {"value": world * prep.kv_bytes / (e2e_ms * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    peak, peak_src = hbm_peak()
    kv_bytes, cache_bytes = prep.kv_bytes, prep.cache_bytes
    gbs = world * kv_bytes / (step_ms * 1e-3) / 1e9
    part_gbs = kv_bytes / (part_ms * 1e-3) / 1e9
    kernel = partition_kernel(spec.kv_format)
    traffic = recorded_traffic(kernel, spec.name)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        oracle.build()
        cpu = cpu_baseline_entry(spec, prep, args.cpu_seconds)
        if spec.name == "tiny_bf16":  # the tiny batch is also timed on one core
            cpu["one_core"] = cpu_baseline_entry(spec, prep, args.cpu_seconds, threads=1)
    per_workload = None
    if world == 1 and not args.no_per_workload:
        names = [n for n in EXTRA_WORKLOADS if n != spec.name]
        del prep
        torch.cuda.empty_cache()
        per_workload = per_workload_entries(names, K, args.warmup, peak, local, not args.no_cpu_baseline,
                                            min(args.cpu_seconds, 3.0))
    line = {
        "metric": METRIC, "value": gbs, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms, "us_per_call": step_ms * 1000, "pct_of_hbm_peak": 100 * gbs / world / peak,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": spec.kv_format, "data": "synthetic",
        "config": {"workload": spec.name, "batch": spec.batch, "num_q_heads": spec.num_q_heads,
                   "num_kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim, "kv_format": spec.kv_format,
                   "context": [spec.ctx_min, spec.ctx_max], "window": spec.window, "softcap": spec.softcap,
                   "block_size": spec.block_size, "partition_size": spec.partition_size,
                   "query_len": spec.query_len, "algorithmic_kv_bytes": kv_bytes, "cache_bytes": cache_bytes,
                   "l2": "inputs larger than L2 (KV cache %.2f GB vs 129 MB L2), no flush" % (cache_bytes / 1e9)
                   if cache_bytes > L2_BYTES else "inputs smaller than L2",
                   "timing": "CUDA events on the launching stream around K calls queued behind a device-side hold",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": kernel, "achieved": part_gbs, "peak": peak, "unit": "GB/s",
                     "frac": part_gbs / peak, "peak_source": peak_src, "traffic": traffic,
                     "partition_us": part_ms * 1000, "bytes_per_launch": kv_bytes},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": K * KERNELS_PER_CALL[spec.kv_format],
        "clocks": clk,
        "per_workload": per_workload,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
