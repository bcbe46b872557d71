#!/usr/bin/env python3
"""Decode-attention benchmark: one JSON line on rank 0.

A step is one pass of the whole hot path over one decode batch of the
70B-class layer workload (B=64, Hq=64, Hkv=8, D=128, bf16, 16-token blocks,
lognormal lengths with median 2,400 / p95 ~18,000): the slot-mapped cache
write of the step's new K/V (pa_reshape_and_cache), split-KV paged decode
attention into caller-visible partials (pa_decode_splitkv) and their
log-sum-exp merge (pa_merge_lse).  Inputs are resident in HBM when the timed
region starts; the KV read per step (~1.3 GB) is far larger than L2, so no
flush is needed.  The line also carries "per_config": the prefix-sharing,
long-context, FP8 and 4-bit workloads timed the same way in the same process.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

With N > 1 it runs under torch.distributed.run, one rank per GPU; each rank
decodes its own batch (weak scaling, no collective on the data path) and the
time is the max over ranks.  --impl reference times the CPU oracle (plain fp64
C) on this host's cores instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import threading
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode-attn tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
FALLBACK_HBM_GBS = 6800.0

# DRAM traffic per decode launch from ncu (dram__bytes_read.sum + dram__bytes_write.sum), by
# workload and kernel, with the hash of the kernel sources it was measured on; reported only
# while they still match.
TRAFFIC = {
    ("llama70b_layer", "decode_segment_kernel"): {"bytes": 1_338_623_488 + 2_550_528, "kernel_hash": "e2f9552a00f0b381"},
    ("llama70b_layer", "decode_pair_kernel"): {"bytes": 1_337_551_104 + 1_244_928, "kernel_hash": "e2f9552a00f0b381"},
    ("prefix_sharing", "decode_segment_kernel"): {"bytes": 2_545_307_392 + 3_103_232, "kernel_hash": "e2f9552a00f0b381"},
    ("prefix_sharing", "decode_persist_kernel"): {"bytes": 2_551_124_992 + 1_275_648, "kernel_hash": "e2f9552a00f0b381"},
    ("long_context", "decode_segment_kernel"): {"bytes": 4_296_252_928 + 2_440_192, "kernel_hash": "e2f9552a00f0b381"},
    ("fp8_mixed", "decode_pair_kernel"): {"bytes": 2_216_397_056 + 12_930_816, "kernel_hash": "e2f9552a00f0b381"},
    ("fp8_mixed", "decode_segment_kernel"): {"bytes": 2_248_222_464 + 17_221_120, "kernel_hash": "e2f9552a00f0b381"},
    ("int4_mixed", "decode_segment_kernel"): {"bytes": 1_125_001_984 + 16_473_856, "kernel_hash": "e2f9552a00f0b381"},
}



# ----------------------------------------------------------------------------
# distributed helpers (one process per GPU; no collective on the data path)
# ----------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank decodes its own batch drawn with its own seed (weak scaling)."""
    return base_seed + 1009 * rank


def reduce_max(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling the SM clocks and throttle reasons every 100 ms.  start() waits
    for its first sample, so that its start-up (driver queries) is over before a timed
    region begins; mark() at the region's start drops the samples taken before it."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.first = 0
        self.reader = None

    def _pump(self):
        for ln in self.proc.stdout:
            if ln.strip():
                self.lines.append(ln)

    def start(self, wait_s: float = 3.0):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={CLOCK_QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._pump, daemon=True)
        self.reader.start()
        t0 = time.perf_counter()
        while not self.lines and time.perf_counter() - t0 < wait_s:
            time.sleep(0.005)

    def mark(self):
        self.first = len(self.lines)

    def stop(self) -> dict:
        lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            self.reader.join(timeout=5)
            lines = self.lines[self.first:]
        if not lines:     # the timed region was shorter than one sample: take one now
            try:
                lines = subprocess.run(
                    ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={CLOCK_QUERY}",
                     "--format=csv,noheader,nounits"], capture_output=True, text=True,
                    timeout=10).stdout.splitlines()
            except (OSError, subprocess.TimeoutExpired):
                lines = []
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

# the sources the decode kernel is compiled from
DECODE_SOURCES = ("pa_common.cuh", "pa_decode.cu", "pa_internal.h")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_28_gb300", "csrc")
    for name in DECODE_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


L2_BYTES = 128 << 20                 # GB300 L2 (~129 MB)
L2_FLUSH_BELOW = 4 * L2_BYTES        # steps reading less KV than this are timed flushed


def step_kv_tokens(batch, args, selected=None) -> int:
    """KV tokens one decode step reads once each (averaged over the KV heads): the
    unique tokens, only the window's, or only the chosen pages' (pages of 16 tokens,
    a sequence's last page may be short); selected: [B, Hkv, topk] page indices."""
    if args.quest_topk > 0:
        L = batch.seq_lens.astype(np.int64)[:, None, None]
        pages = np.asarray(selected, dtype=np.int64)
        rows = np.where(pages >= 0, np.minimum(16, L - 16 * pages), 0)
        return int(rows.sum()) // batch.Hkv
    return batch.unique_kv_tokens(args.window)


def step_kv_bytes(batch, args, selected=None) -> int:
    """Algorithmic bytes of one decode launch: KV rows (+ per-block scales of a
    quantised pool)."""
    n = step_kv_tokens(batch, args, selected) * batch.kv_bytes_per_token()
    if batch.quantized:
        n += sum(int(x) for x in (batch.seq_lens + batch.block_size - 1)
                 // batch.block_size) * batch.scale_bytes_per_block()
    return n


def measured_peak_hbm():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def cpu_baseline(batch, cores: int) -> dict:
    """The oracle, as it stands, on this host's cores: cache write + decode of the
    whole batch, once."""
    import oracle
    t0 = time.perf_counter()
    kp, vp = batch.k_pool.copy(), batch.v_pool.copy()
    if batch.quantized:
        ks, vs = batch.k_scale.copy(), batch.v_scale.copy()
        write = (oracle.reshape_and_cache_fp8 if batch.kv_dtype == "fp8_e4m3"
                 else oracle.reshape_and_cache_int4)
        write(batch.k_new, batch.v_new, kp, vp, ks, vs, batch.slot_mapping, batch.block_size)
    else:
        ks = vs = None
        oracle.reshape_and_cache_bf16(batch.k_new, batch.v_new, kp, vp, batch.slot_mapping,
                                      batch.block_size)
    oracle.paged_decode(batch.q, kp, vp, batch.block_tables, batch.seq_lens, batch.sm_scale,
                        Hkv=batch.Hkv, block_size=batch.block_size, k_scale=ks, v_scale=vs,
                        nthreads=cores)
    dt = time.perf_counter() - t0
    return {"value": batch.B / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"one full step of the same batch (write + decode of all {batch.B} "
                      f"sequences x {batch.Hq} heads), fp64 C with OpenMP, {dt:.2f} s wall"}


# The decode kernel's mean time over the timed steps, from events around some of its calls
# (an event between two kernels of the launch chain stops the next one from starting
# early: bracketing every call slowed the 70B step by 4 %).  A stratified sample: the
# first timed step, which follows the synchronisation and runs 5-8 % slower than the rest,
# is always timed and counts once; the others are represented by the middle step of
# each later block of EVENT_EVERY steps.
EVENT_EVERY = 8


def sampled_steps(steps: int) -> list:
    """Timed steps whose decode call is bracketed by events: step 0, then the middle of
    every block of EVENT_EVERY steps after the first step."""
    return [0] + [i for i in range(1, steps) if i % EVENT_EVERY == EVENT_EVERY // 2]


def mean_decode_ms(times: dict, steps: int) -> float:
    """Mean over all timed steps from the stratified sample: step 0 once, the mean of the
    other samples for the remaining steps (step 0's own time when there are none)."""
    rest = [t for i, t in times.items() if i != 0]
    other = statistics.mean(rest) if rest else times[0]
    return (times[0] + (steps - 1) * other) / steps


def resolve_call(config: str, call: str, window: int, quest_topk: int, cascade: bool) -> str:
    """The decode entry point of a step: "splitkv" (pa_decode_splitkv + pa_merge_lse),
    "segments" (pa_decode given a workspace: the same split kernel and a merge, with the
    options pa_decode_splitkv does not take) or "decode" (pa_decode, no workspace)."""
    if call != "auto":
        if call == "splitkv" and cascade:
            raise SystemExit("the cascade goes through --call segments (pa_decode with a "
                             "workspace)")
        if call == "decode" and cascade:
            raise SystemExit("--cascade needs a workspace (--call segments)")
        return call
    if config == "fp8_mixed":          # that workload's description names pa_decode
        return "decode"
    return "segments" if cascade else "splitkv"


def device_pools(batch, seed: int, device):
    """Seeded random pools generated on the GPU (for the per-workload lines, whose host
    pools would take a minute to draw): the value distributions of workload.py --
    N(0,1) bf16; E4M3 codes of N(0,1) * 112; 4-bit codes rint(N(0,1) * 7/3) clipped to
    +-7; scales base * U(0.8, 1.2).  Timing does not depend on the values."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    shape = (batch.nblocks, batch.block_size, batch.Hkv, batch.D)

    def pool():
        if batch.kv_dtype == "bf16":
            return torch.randn(shape, generator=g, device=device, dtype=torch.bfloat16)
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if batch.kv_dtype == "fp8_e4m3":
            return (x * 112.0).clamp_(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        c = (x * (7.0 / 3.0)).round_().clamp_(-7, 7).to(torch.int16) + 8
        return (c[..., 0::2] | (c[..., 1::2] << 4)).to(torch.uint8).contiguous()

    def scale(base):
        u = torch.rand((batch.nblocks, batch.Hkv), generator=g, device=device)
        return (base * (0.8 + 0.4 * u)).to(torch.float32).contiguous()

    kp, vp = pool(), pool()
    if batch.kv_dtype == "bf16":
        return kp, vp, None, None
    base = 4.0 / 448.0 if batch.kv_dtype == "fp8_e4m3" else 3.0 / 7.0
    return kp, vp, scale(base), scale(base)


class StepRunner:
    """One decode step of a workload on the GPU -- the cache write, (Quest's summary and
    selection,) the decode call -- with the decode call bracketed by events on demand."""

    def __init__(self, dev, batch, call, args, ns_segments, ns_splits, stream):
        from paged_kv_cache_28_gb300 import _lib
        self._lib = _lib
        self.dev, self.batch, self.call, self.args = dev, batch, call, args
        self.ns_segments, self.ns_splits, self.stream = ns_segments, ns_splits, stream
        self.quest = args.quest_topk > 0
        if call == "segments":
            dev.ensure_workspace(ns_segments)
        if call == "splitkv":
            dev.ensure_parts(ns_splits)
        if args.cascade:        # shared prefixes attended once per group (prefix-aware decode)
            if not batch.prefix_groups:
                raise SystemExit("--cascade needs a workload with prefix groups (prefix_sharing)")
            dev.enable_cascade()
        if self.quest:          # summaries of the whole cache, then per step: summarise the
            dev.quest_build_summaries(stream)       # new token's page, select, sparse decode
            dev.quest_buffers(args.quest_topk)

    def __call__(self, ev=None, st=None):
        dev, b, args, _lib = self.dev, self.batch, self.args, self._lib
        st = self.stream if st is None else st
        dev.reshape_and_cache(st)
        if self.quest:
            _lib.pa_quest_summarize(dev.shape, dev.k_pool, dev.k_scale, dev.key_summaries,
                                    dev.slot_mapping, dev.err, st)
            _lib.pa_quest_select(dev.shape, dev.q, dev.key_summaries, dev.block_tables,
                                 dev.seq_lens, args.quest_topk, dev.page_scores,
                                 dev.selected_pages, dev.err, st)
        if ev is not None:
            ev[0].record(st)
        sel = dev.selected_pages if self.quest else None
        if self.call == "splitkv":
            _lib.pa_decode_splitkv(dev.shape, dev.o_part, dev.lse, self.ns_splits, dev.q,
                                   dev.k_pool, dev.v_pool, dev.k_scale, dev.v_scale,
                                   dev.block_tables, dev.seq_lens, b.sm_scale, dev.err, st,
                                   args.window, sel, dev.shared_prefix_lens)
            if ev is not None:
                ev[1].record(st)
            _lib.pa_merge_lse(dev.shape, dev.out, dev.o_part, dev.lse, self.ns_splits, st)
            return
        ws = dev.workspace if self.call == "segments" else None
        _lib.pa_decode(dev.shape, dev.out, dev.q, dev.k_pool, dev.v_pool, dev.k_scale,
                       dev.v_scale, dev.block_tables, dev.seq_lens, b.sm_scale, dev.err, st,
                       args.window, sel, ws, self.ns_segments if ws is not None else 0,
                       shared_prefix_lens=dev.shared_prefix_lens,
                       cascade=dev.cascade if args.cascade else None)
        if ev is not None:
            ev[1].record(st)

    def kernel_name(self):
        if self.call == "decode":
            return decode_kernel(self.batch, self.args.window, self.quest, self.dev.device)
        return "decode_segment_kernel"

    def kernel_label(self):
        if self.call == "splitkv":
            return "decode_segment_kernel (the pa_decode_splitkv call)"
        if self.call == "decode":
            return self.kernel_name() + " (the pa_decode call, no workspace)"
        return ("pa_decode call with a workspace: "
                + ("cascade_kernel + " if self.args.cascade else "")
                + "decode_segment_kernel + merge_kernel")

    def step_label(self):
        quest = "pa_quest_summarize + pa_quest_select + " if self.quest else ""
        if self.call == "splitkv":
            return "pa_reshape_and_cache + " + quest + "pa_decode_splitkv + pa_merge_lse"
        if self.call == "decode":
            return ("pa_reshape_and_cache + " + quest + "pa_decode (no workspace: persistent "
                    "CTAs, or one CTA or a cluster of CTAs per sequence and KV head)")
        return ("pa_reshape_and_cache + " + quest + "pa_decode with a workspace ("
                + ("cascade + " if self.args.cascade else "") + "split kernel + merge)")

    def launches(self):
        # our kernels per step: the cache write; Quest's summary, scores and top-k; then
        # the pair kernel, or the split kernel and a merge (with the cascade also its plan
        # and its two launches, beside and after the split kernel)
        return (1 + (3 if self.quest else 0) +
                (1 if self.call == "decode" else 2 + (3 if self.args.cascade else 0)))


def time_steps(run, steps: int, warmup: int, kv_bytes: int, device, world: int, clocks=None):
    """Warm up, then time `steps` steps with CUDA events (max over ranks): returns
    (ms per step, mean ms of the bracketed decode call, clock record or None)."""
    import torch
    stream = run.stream
    ev = {i: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for i in sampled_steps(steps)}
    if clocks is not None:
        clocks.start()       # before the warm-up: its start-up is over by the timed region
    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    if run.dev.read_err():
        raise RuntimeError("device error flag set during warm-up")
    # a step that reads less than L2_FLUSH_BELOW bytes of KV would find part of it in
    # L2 from the step before: read a buffer twice the L2 size between such steps (a
    # read leaves L2 clean, as the weight reads of a model's other kernels would; a
    # written buffer would leave dirty lines for the next step to write back) and time
    # each step alone with events (the flush is not timed)
    flush = None
    if kv_bytes < L2_FLUSH_BELOW:
        flush = torch.ones(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
        flush_sink = torch.empty((), dtype=torch.float32, device=device)
        st_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.mark()        # samples from here on
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(steps):
        if flush is not None:
            torch.sum(flush, dim=0, out=flush_sink)
            st_ev[i][0].record(stream)
        run(ev.get(i))
        if flush is not None:
            st_ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clock_info = clocks.stop() if clocks is not None else None
    barrier(world)
    if flush is None:
        ms_total = t_start.elapsed_time(t_end)
    else:
        ms_total = sum(a.elapsed_time(b) for a, b in st_ev)
    ms_per_step = reduce_max(ms_total, world, device) / steps
    decode_ms = reduce_max(mean_decode_ms({i: a.elapsed_time(b) for i, (a, b) in ev.items()},
                                          steps), world, device)
    if run.dev.read_err():
        raise RuntimeError("device error flag set during the timed steps")
    return ms_per_step, decode_ms, clock_info


def decode_kernel(batch, window: int, quest: bool, device) -> str:
    """The kernel pa_decode without a workspace runs (the library's choice): persistent
    CTAs for bf16 batches of up to 8 query heads per KV head with more (sequence, KV head)
    units than two per resident CTA, at most 4,096, and no window or page selection; one
    CTA (or a cluster of CTAs) per unit otherwise."""
    import torch
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    units, g = batch.B * batch.Hkv, batch.Hq // batch.Hkv
    per_sm = {128: 2, 64: 4}.get(batch.D, 0)     # resident CTAs of the per-unit kernel
    if (batch.kv_dtype == "bf16" and g <= 8 and per_sm and window == 0 and not quest
            and 2 * sms * per_sm < units <= 4096):
        return "decode_persist_kernel"
    return "decode_pair_kernel"


def traffic_for(config: str, kernel: str):
    tr = TRAFFIC.get((config, kernel))
    return tr["bytes"] if tr and tr.get("kernel_hash") == kernel_source_hash() else None


# The per-workload lines: the other workloads of the measurement plan, each timed in
# the same process as the headline, through the call named (the cross-sequence prefix
# batch and the FP8 batch through both the split decode and pa_decode without a
# workspace).
PER_CONFIG = (("prefix_sharing", "splitkv"), ("prefix_sharing", "decode"),
              ("long_context", "splitkv"), ("fp8_mixed", "decode"), ("fp8_mixed", "splitkv"),
              ("int4_mixed", "splitkv"))


def per_config_lines(args, device, world, rank):
    import torch

    from paged_kv_cache_28_gb300 import workload as wl
    from paged_kv_cache_28_gb300.device import (DeviceBatch, default_num_segments,
                                                default_num_splits)
    peak, _ = measured_peak_hbm()
    out = {}
    for config, call in PER_CONFIG:
        seed = rank_seed(wl.DEFAULT_SEEDS[config], rank)
        batch = wl.make(config, seed=seed, with_pools=False)
        dev = DeviceBatch(batch, device=device, pools=device_pools(batch, seed, device))
        sub = argparse.Namespace(window=0, quest_topk=0, cascade=False)
        run = StepRunner(dev, batch, call, sub, default_num_segments(dev.shape, device),
                         default_num_splits(dev.shape, device), torch.cuda.current_stream(device))
        kv_bytes = step_kv_bytes(batch, sub)
        steps = max(EVENT_EVERY, args.steps)
        ms, kms, _ = time_steps(run, steps, args.warmup, kv_bytes, device, world)
        achieved = kv_bytes / (kms * 1e-3) / 1e9
        kernel = run.kernel_name()
        out[f"{config}/{call}"] = {
            "call": run.step_label(), "kernel": run.kernel_label(),
            "tokens_per_s": world * batch.B / (ms * 1e-3), "ms_per_step": ms, "kernel_ms": kms,
            "algorithmic_bytes": kv_bytes, "achieved_gbs": achieved, "frac": achieved / peak,
            "traffic": traffic_for(config, kernel),
            "num_splits": run.ns_splits if call == "splitkv" else None,
            "steps": steps, "pools": "seeded on the GPU (torch.Generator), values as workload.py"}
        del run, dev
        torch.cuda.empty_cache()
    return out


def end_to_end(args, run, dev, batch, stream, dev_id, world):
    """Steps timed on the host clock from pinned host buffers: every step copies its
    inputs in, runs the step's C-ABI calls and reads its output back.

    Default (pipelined): two sets of input and output buffers, as a serving loop keeps
    them; step i's upload and step i-1's read-back run on copy streams beside step i-1's
    and step i's kernels, and the host waits for each step's output one step later.
    --e2e-serial: one set, copy in -> step -> copy out -> wait, per step (a CUDA graph
    replay, or eager launches with --e2e-eager)."""
    import torch

    # the step's inputs packed into one pinned host buffer and one device buffer (each
    # input 256-byte aligned); the device batch's inputs become views of the latter, so
    # one copy in and one copy out carry the whole step
    inputs = {name: getattr(dev, name) for name in
              ("q", "k_new", "v_new", "slot_mapping", "seq_lens", "block_tables")}
    if dev.shared_prefix_lens is not None:
        inputs["shared_prefix_lens"] = dev.shared_prefix_lens
    if args.cascade:                          # the prefix groups (not the workspace)
        for k, t in zip(("group_offsets", "group_seqs", "group_prefix_len"), dev.cascade):
            inputs[k] = t
    parts, off = {}, 0
    for name, t in inputs.items():
        n = t.numel() * t.element_size()
        parts[name] = (off, n, t.dtype, t.shape)
        off = (off + n + 255) // 256 * 256
    host_inputs = {name: t.reshape(-1).cpu() for name, t in inputs.items()}
    cascade_tail = tuple(dev.cascade[3:]) if args.cascade else ()

    def make_set():
        host_in = torch.empty(off, dtype=torch.uint8).pin_memory()
        dev_in = torch.empty(off, dtype=torch.uint8, device=dev_id)
        views = {}
        for name, (o, n, dt, shp) in parts.items():
            host_in[o:o + n].view(dt).copy_(host_inputs[name])
            views[name] = dev_in[o:o + n].view(dt).view(shp)
        out = torch.empty_like(dev.out)
        out_host = torch.empty(dev.out.shape, dtype=dev.out.dtype).pin_memory()
        return {"host_in": host_in, "dev_in": dev_in, "views": views, "out": out,
                "out_host": out_host}

    def bind(st):
        views = st["views"]
        for name in ("q", "k_new", "v_new", "slot_mapping", "seq_lens", "block_tables",
                     "shared_prefix_lens"):
            if name in views:
                setattr(dev, name, views[name])
        if args.cascade:
            dev.cascade = (views["group_offsets"], views["group_seqs"],
                           views["group_prefix_len"]) + cascade_tail
        dev.out = st["out"]

    sets = [make_set() for _ in range(1 if args.e2e_serial else 2)]
    h2d = sum(n for _, n, _, _ in parts.values())
    d2h = sets[0]["out_host"].numel() * sets[0]["out_host"].element_size()

    if args.e2e_serial:
        st0 = sets[0]
        bind(st0)

        def e2e_body(s):
            st0["dev_in"].copy_(st0["host_in"], non_blocking=True)
            run(st=s)
            st0["out_host"].copy_(st0["out"], non_blocking=True)

        if args.e2e_eager:
            def e2e_step(i):
                e2e_body(stream)
                stream.synchronize()
        else:
            # the whole step -- input copies from pinned host memory, the launch chain,
            # the read-back -- captured once into a CUDA graph and replayed per step
            side = torch.cuda.Stream(dev_id)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                for _ in range(3):
                    e2e_body(side)
            stream.wait_stream(side)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                e2e_body(torch.cuda.current_stream(dev_id))

            def e2e_step(i):
                graph.replay()
                torch.cuda.current_stream(dev_id).synchronize()

        def e2e_finish():
            pass
    else:
        copy_in, copy_out = torch.cuda.Stream(dev_id), torch.cuda.Stream(dev_id)
        ev = {k: [torch.cuda.Event() for _ in sets] for k in ("in", "comp", "out")}
        for k in ev:                              # every event starts out recorded
            for e in ev[k]:
                e.record(stream)
        torch.cuda.synchronize()

        def e2e_step(i):
            j = i % 2
            st = sets[j]
            copy_in.wait_event(ev["comp"][j])     # step i-2 has read this input set
            with torch.cuda.stream(copy_in):
                st["dev_in"].copy_(st["host_in"], non_blocking=True)
            ev["in"][j].record(copy_in)
            stream.wait_event(ev["in"][j])
            stream.wait_event(ev["out"][j])       # step i-2's output has been read back
            bind(st)
            run(st=stream)
            ev["comp"][j].record(stream)
            copy_out.wait_event(ev["comp"][j])
            with torch.cuda.stream(copy_out):
                st["out_host"].copy_(st["out"], non_blocking=True)
            ev["out"][j].record(copy_out)
            ev["out"][1 - j].synchronize()        # the host has step i-1's output

        def e2e_finish():
            torch.cuda.synchronize()

    for i in range(max(3, args.warmup)):
        e2e_step(i)
    e2e_finish()
    barrier(world)
    t0 = time.perf_counter()
    n_e2e = max(3, min(args.steps, 200))
    for i in range(n_e2e):
        e2e_step(i)
    e2e_finish()
    e2e_s = reduce_max((time.perf_counter() - t0) / n_e2e, world, dev_id)
    if dev.read_err():
        raise RuntimeError("device error flag set during the end-to-end steps")
    for st in sets:                                # each set's output is the decode's
        if not torch.equal(st["out"], sets[0]["out"]):
            raise RuntimeError("end-to-end output sets differ")
    return {"value": world * batch.B / e2e_s, "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "mode": ("serial: copy in, step, copy out, wait"
                     + (" (eager launches)" if args.e2e_eager else " (CUDA graph replay)"))
            if args.e2e_serial else
            "pipelined: two input/output sets; uploads and read-backs on copy streams "
            "beside the neighbouring steps' kernels, each output waited for one step later"}


def run_ours(args):
    import torch

    from paged_kv_cache_28_gb300 import _lib
    from paged_kv_cache_28_gb300 import workload as wl
    from paged_kv_cache_28_gb300.device import (DeviceBatch, default_num_segments,
                                                default_num_splits)

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev_id = torch.device("cuda", local)
    if not os.path.exists(_lib.LIB_PATH):
        from paged_kv_cache_28_gb300 import build
        build.build()
    _lib.load()

    seed = rank_seed(wl.DEFAULT_SEEDS[args.config], rank)
    batch = wl.make(args.config, seed=seed)
    dev = DeviceBatch(batch, device=dev_id)
    call = resolve_call(args.config, args.call, args.window, args.quest_topk, args.cascade)
    stream = torch.cuda.current_stream(dev_id)
    run = StepRunner(dev, batch, call, args,
                     args.num_segments or default_num_segments(dev.shape, dev_id),
                     args.num_splits or default_num_splits(dev.shape, dev_id), stream)
    selected = None
    if args.quest_topk > 0:
        run()                                   # one step so the selection exists
        torch.cuda.synchronize()
        selected = dev.selected_pages.cpu().numpy()
    kv_bytes = step_kv_bytes(batch, args, selected)
    clocks = ClockSampler(local)
    ms_per_step, decode_ms, clock_info = time_steps(run, args.steps, args.warmup, kv_bytes,
                                                    dev_id, world, clocks)

    # ---- end to end through the C ABI from pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(args, run, dev, batch, stream, dev_id, world)

    unique_tokens = step_kv_tokens(batch, args, selected)
    peak, peak_kind = measured_peak_hbm()
    achieved = kv_bytes / (decode_ms * 1e-3) / 1e9
    kernel = run.kernel_name()
    plain = args.window == 0 and args.quest_topk == 0 and not args.cascade
    traffic = traffic_for(args.config, kernel) if plain and call != "segments" else None
    result = {
        "metric": METRIC,
        "value": world * batch.B / (ms_per_step * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": batch.kv_dtype,
        "data": "synthetic",
        "config": {
            "workload": args.config,
            "B": batch.B, "Hq": batch.Hq, "Hkv": batch.Hkv, "D": batch.D,
            "block_size": batch.block_size, "seq_len_sum": batch.logical_tokens,
            "seq_len_max": int(batch.seq_lens.max()),
            "unique_kv_tokens": unique_tokens,
            "num_splits": run.ns_splits if call == "splitkv" else None,
            "num_segments": run.ns_segments if call == "segments" else None,
            "window": args.window,
            "quest_topk": args.quest_topk,
            "cascade": bool(args.cascade),
            "l2": (f"no flush: {kv_bytes / 1e9:.2f} GB of KV read per step >> 129 MB L2"
                   if kv_bytes >= L2_FLUSH_BELOW else
                   f"flushed: {kv_bytes / 1e9:.3f} GB of KV per step, a {2 * L2_BYTES >> 20} MB "
                   "buffer read between steps, each step timed alone with events"),
            "parallelism": f"replicas x{world}" if world > 1 else "single",
            "step": run.step_label(),
        },
        "roofline": {
            "bound": "hbm",
            "achieved": achieved,
            "peak": peak,
            "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": traffic,
            "kernel": run.kernel_label(),
            "kernel_ms": decode_ms,
            "algorithmic_bytes": kv_bytes,
            "peak_kind": peak_kind,
        },
        "gpu_launches": run.launches() * args.steps,
        "clocks": clock_info,
    }
    if e2e is not None:
        result["e2e"] = e2e
    del run, dev
    torch.cuda.empty_cache()
    if not args.no_per_config and plain and args.config == "llama70b_layer":
        result["per_config"] = per_config_lines(args, dev_id, world, rank)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(batch, os.cpu_count() or 1)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ----------------------------------------------------------------------------
# reference arm: the CPU oracle on this host's cores
# ----------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from paged_kv_cache_28_gb300 import workload as wl
    oracle.build()
    batch = wl.make(args.config)
    cores = os.cpu_count() or 1
    # each step decodes a bounded sample of (sequence, head) rows, sized so that the
    # whole --steps/--warmup run takes about REF_BUDGET_S; the time is scaled to the
    # whole batch by the KV tokens the sample reads
    REF_BUDGET_S = 90.0
    rng = np.random.default_rng(0)
    all_rows = np.array([(b, h) for b in range(batch.B) for h in range(batch.Hq)], np.int32)
    rng.shuffle(all_rows)
    row_tokens = batch.seq_lens[all_rows[:, 0]].astype(np.int64)
    total_token_heads = int(batch.seq_lens.astype(np.int64).sum()) * batch.Hq

    def time_rows(rows):
        t0 = time.perf_counter()
        oracle.paged_decode(batch.q, batch.k_pool, batch.v_pool, batch.block_tables,
                            batch.seq_lens, batch.sm_scale, Hkv=batch.Hkv,
                            block_size=batch.block_size, k_scale=batch.k_scale,
                            v_scale=batch.v_scale, rows=rows, nthreads=cores)
        return time.perf_counter() - t0

    calib = all_rows[:4 * cores]
    s_per_token_head = time_rows(calib) / max(1, int(row_tokens[:len(calib)].sum()))
    per_step = REF_BUDGET_S / (args.steps + args.warmup)
    want = per_step / max(s_per_token_head, 1e-12)
    n = int(np.searchsorted(np.cumsum(row_tokens), want)) + 1
    n = max(cores, min(n, len(all_rows)))
    rows = np.ascontiguousarray(all_rows[:n])
    sample_token_heads = int(row_tokens[:n].sum())
    frac = sample_token_heads / total_token_heads
    idx = np.unique(rows[:, 0])

    def ref_step():
        # the cache write touches only this step's B rows; the sample's decode reads them
        time_rows(rows)

    for _ in range(args.warmup):
        ref_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ref_step()
    dt = (time.perf_counter() - t0) / args.steps
    full_step_s = dt / frac
    value = batch.B / full_step_s
    result = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": full_step_s * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.config, "B": batch.B, "Hq": batch.Hq, "Hkv": batch.Hkv,
                   "D": batch.D, "block_size": batch.block_size,
                   "seq_len_sum": batch.logical_tokens},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} random (sequence, head) rows of {batch.B * batch.Hq} "
                                   f"({frac:.2%} of the KV token-heads) per step, decoded by "
                                   f"the fp64 oracle; time scaled to the whole batch by "
                                   f"KV token-heads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="llama70b_layer",
                    choices=["tiny", "llama70b_layer", "prefix_sharing", "long_context",
                             "fp8_mixed", "int4_mixed", "code_assistant_turns"])
    ap.add_argument("--num-splits", type=int, default=0,
                    help="pa_decode_splitkv's partial slots per head (0: pa_default_num_splits)")
    ap.add_argument("--num-segments", type=int, default=0,
                    help="segments of pa_decode's split decode (0: pa_default_num_segments)")
    ap.add_argument("--call", choices=["auto", "splitkv", "segments", "decode"], default="auto",
                    help="the decode entry point of each step: pa_decode_splitkv + pa_merge_lse, "
                         "pa_decode with a workspace (the same split kernel and its own merge; "
                         "the cascade goes this way), or pa_decode without a workspace (a CTA "
                         "or a cluster of CTAs per sequence and KV head); auto: pa_decode for "
                         "fp8_mixed, whose workload names that call, the workspace form with "
                         "the cascade, pa_decode_splitkv otherwise")
    ap.add_argument("--e2e-serial", action="store_true",
                    help="e2e leg: one buffer set, copy in -> step -> copy out -> wait per step")
    ap.add_argument("--e2e-eager", action="store_true",
                    help="with --e2e-serial: launch each call eagerly instead of replaying "
                         "a CUDA graph")
    ap.add_argument("--cascade", action="store_true",
                    help="prefix-aware decode: each prefix group's shared tokens attended once")
    ap.add_argument("--quest-topk", type=int, default=0,
                    help="query-aware sparse decode over the K best 16-token pages (0 = off)")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding-window layer: attend over the last W positions (0 = all)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload lines (prefix sharing, long context, FP8, "
                         "4-bit) added to the default 70B line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
