#!/usr/bin/env python3
"""Benchmark of the split-KV paged decode/verify path on GB300.

One step = one pass of the whole hot path over one batch: plan (the cache is
reset first, as at the start of a forward), split-KV attention, LSE merge.
The default workload is the uniform MTP verify batch: 16 sequences x 119000
tokens, 4 query tokens each, 32 query / 2 KV heads, head_dim 128, bf16 pages
of 16 tokens behind a random block table (1.95 GB of K/V per call, larger
than L2, so no flush is needed between steps).

Metric: effective KV-read TB/s = K/V bytes of the batch / time per step
(higher is better); the JSON line also carries microseconds per call.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--config I]

Besides the contract's keys the line carries e2e_serving: the same step as a
server runs it (cache resident in HBM, the step's new K/V written by
sk_reshape_and_cache, inputs copied from pinned host memory, one CUDA graph);
per_config: every other workload (1 and 3-8) timed the same way on the same
box, one at a time, with its per-kernel split, KV TB/s, roofline fraction and
clocks (no CPU or e2e legs; --no-per-config skips them); and skew_vs_uniform:
the agentic batch's KV TB/s over the uniform batch's, for attention + merge and
for the whole step.
Other modes print a line of their own:

  python bench.py --config I --forward-layers 15   # one plan + 15 layers, CUDA graph
  python bench.py --kv-write bf16|fp8               # the KV write, 65536 tokens x 8 heads
  python bench.py --shuffle bf16|fp8                # standard -> shuffled pages, a whole cache

Under torchrun (N > 1) every rank runs its own copy of the batch on its own
GPU (weak scaling: work items are independent, no collective on the data
path); the timed region is bracketed by barriers and the max over ranks is
reported.  ``--impl reference`` times the fp64 CPU oracle on the host cores
on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import sk_inputs as si  # noqa: E402

METRIC = "decode-attention us/call and effective KV-read TB/s vs GB300 HBM peak"
FALLBACK_HBM_GBS = 6800.0


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="sk", choices=["sk", "reference"])
    ap.add_argument("--config", type=int, default=2, help="workload 1..8 (default 2)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--forward-layers", type=int, default=0,
                    help="time a CUDA-graph forward: one plan + this many layers of attention + merge")
    ap.add_argument("--shuffle", choices=["bf16", "fp8"], default=None,
                    help="time the standard -> shuffled page conversion of a whole cache "
                         "(config 2's for bf16, config 4's for fp8)")
    ap.add_argument("--kv-write", choices=["bf16", "fp8"], default=None,
                    help="time the KV write step (65536 tokens x 8 KV heads) instead of the path")
    ap.add_argument("--eager", action="store_true",
                    help="launch every step from Python instead of replaying the steps as one CUDA graph")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other workloads' per_config summaries in the default line")
    ap.add_argument("--fixed-split", action="store_true",
                    help="time the fixed split even when bs > 1 (bs == 1 always uses it, as the method does)")
    return ap.parse_args()


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, world_size: int, device=None) -> float:
    """Largest `value` over all ranks (the slowest rank sets the job time)."""
    if world_size == 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_tbps(bytes_per_rank_per_step: int, steps: int, world_size: int, max_ms: float) -> float:
    """Whole-job throughput: every rank processed its own batch each step."""
    return world_size * bytes_per_rank_per_step * steps / (max_ms * 1e-3) / 1e12


def _config_json(w, extra=None):
    cfg = {"workload": w.name, "batch": w.bs, "seq_lens_total": int(w.seq_lens.sum()),
           "q_len": int(w.max_q_len), "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
           "head_dim": w.head_dim, "page": w.page, "kv_dtype": "fp8_e4m3" if w.kv_dtype else "bf16",
           "kv_bytes_per_call": w.kv_bytes, "num_sms_plan": w.num_sms, "seg_max": w.seg_max,
           "l2": "inputs larger than L2 (K/V %.2f GB per call), no flush" % (w.kv_bytes / 1e9)
           if w.kv_bytes > 129e6 else ("L2 flushed before every step, outside the timed sum: a 256 MB write, "
                                       "then a 256 MB read of another buffer so that the write-backs of "
                                       "the dirty lines happen before the step")}
    if extra:
        cfg.update(extra)
    return cfg


# ----------------------------------------------------------------------------- CPU oracle

def _oracle_units(w, q_host_bits, kv_gather, rng, seconds):
    """Times the fp64 oracle on whole (sequence, KV head) units of ``w`` until
    ``seconds`` of CPU time have passed.  kv_gather(s) -> host page bits of sequence s."""
    from oracle import oracle
    units = [(s, h) for s in range(w.bs) if w.seq_lens[s] > 0 and w.q_lens[s] > 0
             for h in range(w.num_kv_heads)]
    order = rng.permutation(len(units))
    cu = w.cu_q
    done_bytes, elapsed, n = 0, 0.0, 0
    cache = {}
    for k in order:
        s, h = units[k]
        L, qs = int(w.seq_lens[s]), int(w.q_lens[s])
        if s not in cache:
            cache.clear()
            cache[s] = kv_gather(s)
        kv_bits = cache[s]
        npg = (L + w.page - 1) // w.page
        bt = np.arange(npg, dtype=np.int32)[None, :]
        rows = np.array([j * w.num_q_heads + h * w.group + i for j in range(qs) for i in range(w.group)],
                        dtype=np.int64)
        qb = q_host_bits[cu[s]:cu[s] + qs]
        t0 = time.perf_counter()
        oracle.attention(qb, kv_bits, w.kv_dtype, w.k_scale, w.v_scale, bt, w.page,
                         np.array([L], np.int32), np.array([0, qs], np.int32), w.num_q_heads,
                         w.num_kv_heads, w.head_dim, w.sm_scale, w.causal, rows=rows)
        elapsed += time.perf_counter() - t0
        done_bytes += L * 2 * w.head_dim * w.elem_bytes
        n += 1
        if elapsed >= seconds:
            break
    return done_bytes, elapsed, n


def _host_inputs(w):
    """Host copies of the workload's inputs, generated on the CPU with the same seeds."""
    import torch
    q = si.make_q(w, "cpu")
    q_bits = q.view(torch.int16).numpy().view(np.uint16)

    def gather(s):
        L = int(w.seq_lens[s])
        npg = (L + w.page - 1) // w.page
        return _kv_pages_cpu(w, w.block_table[s, :npg])
    return q_bits, gather


_KV_CPU = {}


def _kv_pages_cpu(w, blocks):
    import torch
    key = w.name
    if key not in _KV_CPU:
        _KV_CPU.clear()
        _KV_CPU[key] = si.make_kv(w, "cpu")
    kv = _KV_CPU[key][torch.as_tensor(blocks.astype(np.int64))]
    return kv.numpy() if w.kv_dtype == si.KV_FP8 else kv.view(torch.int16).numpy().view(np.uint16)


def _cpu_baseline(w, seconds, seed=0, from_device=None):
    from oracle import oracle
    rng = np.random.default_rng(seed)
    if from_device is not None:
        q_bits, gather = from_device
    else:
        q_bits, gather = _host_inputs(w)
    nbytes, el, n = _oracle_units(w, q_bits, gather, rng, seconds)
    cores = oracle.num_threads()
    # the same oracle on one core, for a few seconds
    oracle.set_num_threads(1)
    try:
        b1, el1, n1 = _oracle_units(w, q_bits, gather, rng, max(1.0, seconds / 4))
    finally:
        oracle.set_num_threads(cores)
    return {"value": nbytes / el / 1e12, "unit": "TB/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} (sequence, KV head) units of {w.name}: all G*q query rows over the whole "
                      f"sequence, {nbytes / 1e6:.1f} MB of K/V in {el:.2f} s, fp64 C oracle, OpenMP",
            "single_core": {"value": b1 / el1 / 1e12, "unit": "TB/s", "cores": 1,
                            "sample": f"{n1} units, {b1 / 1e6:.1f} MB of K/V in {el1:.2f} s"}}


def run_reference(a, w, rank):
    if rank != 0:
        return 0
    from oracle import oracle
    oracle.build()
    q_bits, gather = _host_inputs(w)
    rng = np.random.default_rng(7)
    per_step = max(1.0, min(6.0, 150.0 / max(1, a.steps + a.warmup)))
    for _ in range(a.warmup):
        _oracle_units(w, q_bits, gather, rng, per_step / 4)
    tot_b, tot_t, tot_n = 0, 0.0, 0
    for _ in range(a.steps):
        b, t, n = _oracle_units(w, q_bits, gather, rng, per_step)
        tot_b += b
        tot_t += t
        tot_n += n
    val = tot_b / tot_t / 1e12
    sample = (f"each step: (sequence, KV head) units of {w.name} for ~{per_step:.1f} s of oracle time; "
              f"{tot_n} units, {tot_b / 1e6:.1f} MB of K/V over {a.steps} steps")
    line = {"metric": METRIC, "value": val, "unit": "TB/s", "n_gpus": a.gpus, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": 1e3 * tot_t / a.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference", "config": _config_json(w),
            "cpu_baseline": {"value": val, "unit": "TB/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        busy = [s for s, p in zip(sm, pw) if p > 1.15 * min(pw)] if pw else sm
        return {"sm_mhz": statistics.median(busy or sm), "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ----------------------------------------------------------------------------- roofline helpers

def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "of measured"
    return FALLBACK_HBM_GBS, "of fallback"


ATTN_SOURCES = ("sk_attn_tc.cu", "sk_sm100.cuh", "sk_internal.cuh")


def _strip_comments(src: str) -> str:
    """C/C++ source without comments and blank lines (string literals are left alone)."""
    out, i, n = [], 0, len(src)
    while i < n:
        if src.startswith("//", i):
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif src[i] == '"':
            j = i + 1
            while j < n and src[j] != '"':
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            out.append(src[i])
            i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def _kernel_sources_sha():
    """Short hash of the attention kernel's code (comments and blank lines do not
    count): an ncu traffic figure is only reported while it was taken on this code."""
    h = hashlib.sha256()
    for name in ATTN_SOURCES:
        with open(os.path.join(ROOT, "paged_split_kv_gb300", "csrc", name)) as fh:
            h.update(name.encode())
            h.update(_strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def _ncu_traffic(workload, sha):
    """DRAM bytes per attention launch from the committed ncu summary, if it was
    taken on the current kernel sources (else None)."""
    for f in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        text = open(f).read()
        if f"workload: {workload}" not in text or f"source_sha: {sha}" not in text:
            continue
        for line in text.splitlines():
            if line.strip().startswith("dram_bytes_per_launch:"):
                try:
                    return int(float(line.split(":", 1)[1].strip()))
                except ValueError:
                    return None
    return None


# ----------------------------------------------------------------------------- GPU arm

class PathBench:
    """Device buffers of one workload and the timed replay of its steps.

    One step = plan-cache reset, plan (unless the fixed split runs), attention,
    merge.  The timed steps (and the warm-up) are captured once as a CUDA graph
    (every call is capture safe) and replayed once: the device runs exactly the
    kernels of K eager steps, but the timing does not depend on how fast the
    host issues the calls.  Inputs larger than L2 run the K steps back to back
    between one event pair (an event between two steps would cut the overlap of
    one step's last kernel with the next step's first launch, ~5 us per step);
    smaller inputs get an L2 flush before every step and an event pair around
    each step, so the flushes stay out of the sum.  A second graph of the same
    steps, with events around each kernel, gives the per-kernel split.
    ``eager`` keeps Python-launched loops instead."""

    def __init__(self, sk, torch, w, dev, fixed_split=False, eager=False):
        self.sk, self.torch, self.w, self.dev = sk, torch, w, dev
        self.use_plan = w.bs > 1 and not fixed_split
        nt, hq, d = w.num_tokens, w.num_q_heads, w.head_dim
        self.q = si.make_q(w, dev)
        self.kv = si.make_kv(w, dev)
        self.bt = torch.as_tensor(w.block_table, device=dev)
        self.lens = torch.as_tensor(w.seq_lens, device=dev)
        self.cu = torch.as_tensor(w.cu_q, device=dev)
        cap = sk.plan_capacity(w.bs, w.num_kv_heads, w.num_sms)
        self.plan = torch.empty(cap, dtype=torch.int32, device=dev) if self.use_plan else None
        self.tok = torch.empty(nt, dtype=torch.int32, device=dev) if self.use_plan else None
        self.part_o = torch.empty((nt, w.seg_max, hq, d), dtype=torch.float32, device=dev)
        self.part_m = torch.empty((nt, w.seg_max, hq), dtype=torch.float32, device=dev)
        self.part_l = torch.empty((nt, w.seg_max, hq), dtype=torch.float32, device=dev)
        self.out = torch.empty((nt, hq, d), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((nt, hq), dtype=torch.float32, device=dev)
        self.fixed = 0 if self.use_plan else sk.sk_fixed_nseg(w.bs, w.num_kv_heads, w.num_sms, w.seg_max)
        # L2 flush for inputs that fit in L2: a write larger than L2, then a read of another buffer
        # larger than L2, which evicts the written (dirty) lines, so that their write-backs to HBM
        # happen in the flush and not inside the timed step
        small = w.kv_bytes <= 129e6
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if small else None
        self.flush_rd = torch.ones(256 << 20, dtype=torch.uint8, device=dev) if small else None
        self.flush_sink = torch.zeros(1, dtype=torch.int64, device=dev) if small else None
        try:
            self.graphs = not eager and torch.cuda.Event(enable_timing=True, external=True) is not None
        except TypeError:                  # a PyTorch without graph-recorded events
            self.graphs = False
        self.stream = torch.cuda.Stream(device=dev) if self.graphs else torch.cuda.current_stream()

    def step(self, ev=None):
        # ev: None, [start, end] of the step, or [start, after plan, after attention, end].  Events
        # between kernels cut the launch overlap of dependent kernels, so the timed steps carry the
        # pair only and a second replay of the same steps gives the per-kernel split.
        sk, w, st = self.sk, self.w, self.stream
        parts = ev is not None and len(ev) == 4
        if self.flush is not None:
            self.flush.fill_(1)
            self.torch.sum(self.flush_rd.view(self.torch.int64), dim=0, keepdim=True, out=self.flush_sink)
        if ev is not None and ev[0] is not None:
            ev[0].record(st)
        if self.use_plan:
            sk.sk_plan_cache_reset()
            sk.sk_build_plan(self.lens, self.cu, w.num_kv_heads, self.plan, self.tok, w.num_sms, w.seg_max, st)
        if parts:
            ev[1].record(st)
        sk.sk_paged_decode_attn(self.q, self.kv, self.bt, self.lens, self.cu, self.plan, self.part_o,
                                self.part_m, self.part_l, max_q_len=w.max_q_len, sm_scale=w.sm_scale,
                                num_sms=w.num_sms, k_scale=w.k_scale, v_scale=w.v_scale,
                                causal=bool(w.causal), stream=st)
        if parts:
            ev[2].record(st)
        sk.sk_merge_segments(self.part_o, self.part_m, self.part_l, self.tok, self.out, self.lse,
                             fixed_nseg=self.fixed, stream=st)
        if ev is not None and ev[-1] is not None:
            ev[-1].record(st)

    def run(self, steps, warmup, ws=1, sampler=None):
        """Warm-up, K timed steps, then K steps with events around each kernel.  Returns
        {local_ms, plan_ms, attn_ms, merge_ms, clocks}."""
        torch = self.torch
        flushed = self.flush is not None
        if sampler:
            sampler.start()
        self.stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(self.stream):
            for _ in range(3):
                self.step()
        torch.cuda.synchronize()
        ext = {"external": True} if self.graphs else {}
        evs = [[torch.cuda.Event(enable_timing=True, **ext) for _ in range(2)] for _ in range(steps)]
        evp = [[torch.cuda.Event(enable_timing=True, **ext) for _ in range(4)] for _ in range(steps)]

        def timed_events(i):
            # the events step i of the timed run records: its own pair with the flush, else only
            # the first step's start and the last step's end
            if flushed:
                return evs[i]
            return [evs[0][0] if i == 0 else None, evs[-1][1] if i == steps - 1 else None]

        if self.graphs:
            g_warm, g_timed, g_parts = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            with torch.cuda.stream(self.stream):
                with torch.cuda.graph(g_warm, stream=self.stream):
                    for _ in range(max(3, warmup)):
                        self.step()
                with torch.cuda.graph(g_timed, stream=self.stream):
                    for i in range(steps):
                        self.step(timed_events(i))
                with torch.cuda.graph(g_parts, stream=self.stream):
                    for i in range(steps):
                        self.step(evp[i])
            g_warm.replay()
        else:
            for _ in range(max(3, warmup)):
                self.step()
        torch.cuda.synchronize()
        status = self.sk.sk_get_device_status(clear=True)
        if status:
            raise RuntimeError(f"device status {status:#x} after warm-up ({self.w.name})")
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        if self.graphs:
            g_timed.replay()
        else:
            for i in range(steps):
                self.step(timed_events(i))
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        # the per-kernel split: the same steps again, with an event pair around each kernel
        if self.graphs:
            g_parts.replay()
        else:
            for i in range(steps):
                self.step(evp[i])
        torch.cuda.synchronize()
        clocks = sampler.stop() if sampler else None
        if self.sk.sk_get_device_status(clear=True):
            raise RuntimeError(f"device status set during the timed steps ({self.w.name})")
        local_ms = (sum(e[0].elapsed_time(e[1]) for e in evs) if flushed
                    else evs[0][0].elapsed_time(evs[-1][1]))
        return {"local_ms": local_ms, "plan_ms": [e[0].elapsed_time(e[1]) for e in evp],
                "attn_ms": [e[1].elapsed_time(e[2]) for e in evp],
                "merge_ms": [e[2].elapsed_time(e[3]) for e in evp], "clocks": clocks}

    def attention_bytes(self):
        """Algorithmic bytes of one attention launch: K/V once, Q once, partials written;
        and the number of work items (planned split)."""
        w = self.w
        q_bytes = w.num_tokens * w.num_q_heads * w.head_dim * 2
        items = None
        if self.use_plan:
            p_np = self.plan.cpu().numpy()
            items = int((p_np[1:] >= 0).sum())
            seg_rows = int(self.tok.cpu().numpy().astype(np.int64).sum())
        else:
            seg_rows = w.num_tokens * self.fixed
        part_bytes = seg_rows * w.num_q_heads * (w.head_dim + 2) * 4
        return w.kv_bytes + q_bytes + part_bytes, items

    def launch_mode(self):
        if self.graphs:
            return ("timed steps replayed as one CUDA graph (one event pair around the back-to-back steps, "
                    "or around each step when L2 is flushed between steps; the per-kernel split comes from a "
                    "second replay with events around each kernel)")
        return "eager, one Python call per kernel"


def _kernel_summary(t, steps, kv_bytes):
    """Per-kernel means (us) and KV TB/s of a PathBench.run result."""
    am = [x + y for x, y in zip(t["attn_ms"], t["merge_ms"])]
    ms = t["local_ms"] / steps
    return {"ms_per_step": round(ms, 5), "us_attention": round(1e3 * statistics.mean(t["attn_ms"]), 2),
            "us_merge": round(1e3 * statistics.mean(t["merge_ms"]), 2),
            "us_plan": round(1e3 * statistics.mean(t["plan_ms"]), 2),
            "us_per_call": round(1e3 * statistics.mean(am), 2),
            "kv_tbps_step": round(kv_bytes / (ms * 1e-3) / 1e12, 4),
            "kv_tbps_attention_plus_merge": round(kv_bytes / (1e-3 * statistics.mean(am)) / 1e12, 4)}


PER_CONFIG = (1, 3, 4, 5, 6, 7, 8)


def run_per_config(a, sk, torch, dev, local, main=None):
    """Every other workload on the same box, timed as the headline one (same graph
    replay, steps and warm-up; no CPU or e2e legs), one workload in memory at a
    time.  Returns {config index: summary}; ``main`` is the headline's own summary,
    used for the skew-vs-uniform ratios."""
    peak, peak_kind = _peaks()
    res = {}
    for idx in PER_CONFIG:
        if idx == a.config:
            continue
        w = si.config(idx)
        pb = PathBench(sk, torch, w, dev, eager=a.eager)
        t = pb.run(a.steps, a.warmup, 1, ClockSampler(local))
        attn_bytes, items = pb.attention_bytes()
        summ = _kernel_summary(t, a.steps, w.kv_bytes)
        achieved = attn_bytes / (statistics.mean(t["attn_ms"]) * 1e-3) / 1e9
        summ.update({"workload": w.name, "split": "plan" if pb.use_plan else "fixed", "work_items": items,
                     "kv_dtype": "fp8_e4m3" if w.kv_dtype else "bf16", "kv_bytes_per_call": w.kv_bytes,
                     "l2": "flushed before every step" if pb.flush is not None else "inputs larger than L2",
                     "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                                  "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                                  "frac_of_8tbps_nominal": round(achieved / 8000.0, 4),
                                  "algorithmic_bytes_per_launch": int(attn_bytes)},
                     "clocks": t["clocks"], "gpu_launches": a.steps * (3 if pb.use_plan else 2)})
        res[str(idx)] = summ
        del pb
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return res


def run_sk(a, w, ws, rank, local):
    import torch
    import paged_split_kv_gb300 as sk
    if not os.path.exists(sk.LIB_PATH):
        from paged_split_kv_gb300 import build as b
        b.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    pb = PathBench(sk, torch, w, dev, fixed_split=a.fixed_split, eager=a.eager)
    use_plan, nsm = pb.use_plan, w.num_sms
    q, kv, bt, lens, cu, out, lse = pb.q, pb.kv, pb.bt, pb.lens, pb.cu, pb.out, pb.lse
    t = pb.run(a.steps, a.warmup, ws, ClockSampler(local) if rank == 0 else None)
    clocks = t["clocks"]
    plan_ms, attn_ms, merge_ms = t["plan_ms"], t["attn_ms"], t["merge_ms"]
    total_ms = max_over_ranks(t["local_ms"], ws, dev)
    ms_per_step = total_ms / a.steps
    value = weak_scaling_tbps(w.kv_bytes, a.steps, ws, total_ms)

    # end to end through the public call with host inputs (pinned), copies inside the region
    e2e = None
    e2e_serving = None
    if a.e2e_steps > 0:
        host = {"q": q.cpu().pin_memory(), "kv": kv.cpu().pin_memory(), "bt": bt.cpu().pin_memory(),
                "lens": lens.cpu().pin_memory(), "cu": cu.cpu().pin_memory()}
        dq, dkv = torch.empty_like(q), torch.empty_like(kv)
        dbt, dlens, dcu = torch.empty_like(bt), torch.empty_like(lens), torch.empty_like(cu)
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        wsp = {}
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()

        def e2e_step():
            dq.copy_(host["q"], non_blocking=True)
            dkv.copy_(host["kv"], non_blocking=True)
            dbt.copy_(host["bt"], non_blocking=True)
            dlens.copy_(host["lens"], non_blocking=True)
            dcu.copy_(host["cu"], non_blocking=True)
            sk.sk_plan_cache_reset()
            o, l = sk.paged_decode_attention(dq, dkv, dbt, dlens, dcu, max_q_len=w.max_q_len,
                                             sm_scale=w.sm_scale, num_sms=nsm, k_scale=w.k_scale,
                                             v_scale=w.v_scale, causal=bool(w.causal),
                                             seg_max=w.seg_max, use_plan=use_plan, workspace=wsp)
            out_h.copy_(o, non_blocking=True)
            lse_h.copy_(l, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if ws > 1:
            torch.distributed.barrier()
        e0.record()
        for _ in range(a.e2e_steps):
            e2e_step()
        e1.record()
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws, dev)
        assert torch.equal(out_h, out.cpu()), "end-to-end output differs from the device-resident run"
        e2e = {"value": weak_scaling_tbps(w.kv_bytes, a.e2e_steps, ws, e2e_ms), "unit": "TB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_ms / a.e2e_steps}
        e2e_serving = _e2e_serving(a, w, sk, torch, dev, q, kv, bt, lens, cu, use_plan, nsm, ws, out)
        del host, dq, dkv

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return 0

    attn_avg = statistics.mean(attn_ms)
    peak, peak_kind = _peaks()
    attn_bytes, nseg_items = pb.attention_bytes()
    achieved = attn_bytes / (attn_avg * 1e-3) / 1e9
    sha = _kernel_sources_sha()
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_kind": peak_kind + " (a copy: every byte read and written)",
                "frac_of_8tbps_nominal": round(achieved / 8000.0, 4),
                "traffic": _ncu_traffic(w.name, sha), "kernel": "sk attention (split-KV, paged)",
                "algorithmic_bytes_per_launch": int(attn_bytes), "source_sha": sha}

    cpu = None
    gather = None
    if not a.no_cpu_baseline and ws == 1:
        q_bits = q.view(torch.int16).cpu().numpy().view(np.uint16)

        def gather(s):
            L = int(w.seq_lens[s])
            npg = (L + w.page - 1) // w.page
            idx = torch.as_tensor(w.block_table[s, :npg].astype(np.int64), device=dev)
            sub = kv.index_select(0, idx).cpu()
            return sub.numpy() if w.kv_dtype == si.KV_FP8 else sub.view(torch.int16).numpy().view(np.uint16)
        cpu = _cpu_baseline(w, a.cpu_seconds, from_device=(q_bits, gather))

    launch = pb.launch_mode()
    per_config, skew = None, None
    if ws == 1 and not a.no_per_config:
        main = _kernel_summary(t, a.steps, w.kv_bytes)
        # free this workload's device memory before the next one is generated
        pb = q = kv = bt = lens = cu = out = lse = gather = None
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        per_config = run_per_config(a, sk, torch, dev, local)
        pair = {2: main} if a.config == 2 else ({3: main} if a.config == 3 else {})
        uni = pair.get(2) or per_config.get("2")
        sk3 = pair.get(3) or per_config.get("3")
        if uni and sk3:
            skew = {"attention_plus_merge": round(sk3["kv_tbps_attention_plus_merge"]
                                                  / uni["kv_tbps_attention_plus_merge"], 4),
                    "step": round(sk3["kv_tbps_step"] / uni["kv_tbps_step"], 4),
                    "definition": "KV TB/s of the agentic skew batch / KV TB/s of the uniform batch"}
    line = {"metric": METRIC, "value": round(value, 4), "unit": "TB/s", "n_gpus": ws, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.kv_dtype == si.KV_BF16 else "fp8_e4m3",
            "data": "synthetic (seeded N(0,1) Q/K/V, random-permuted block table)",
            "config": _config_json(w, {"split": "plan" if use_plan else "fixed",
                                       "work_items": nseg_items}),
            "us_per_call": round(1e3 * statistics.mean([x + y for x, y in zip(attn_ms, merge_ms)]), 2),
            "us_attention": round(1e3 * attn_avg, 2), "us_merge": round(1e3 * statistics.mean(merge_ms), 2),
            "us_plan": round(1e3 * statistics.mean(plan_ms), 2),
            "kv_tbps_attention_plus_merge": round(w.kv_bytes / (1e-3 * statistics.mean(
                [x + y for x, y in zip(attn_ms, merge_ms)])) / 1e12, 4),
            "frac_of_8tbps_nominal": round(value / 8.0, 4),
            "per_config": per_config, "skew_vs_uniform": skew,
            "roofline": roofline, "clocks": clocks, "e2e": e2e, "e2e_serving": e2e_serving, "cpu_baseline": cpu,
            "gpu_launches": a.steps * (3 if use_plan else 2),
            "launch": launch}
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def _e2e_serving(a, w, sk, torch, dev, q, kv, bt, lens, cu, use_plan, nsm, ws, ref_out):
    """A serving step through the public calls with the K/V cache resident in HBM
    (model state, as in a server): every step copies this step's inputs from pinned
    host memory -- Q, the new tokens' K and V, their cache slots, seq_lens,
    cu_seqlens_q and the block table, packed in one staging buffer, so one copy --
    writes the new K/V into the cache (sk_reshape_and_cache), runs plan + attention
    + merge into one output buffer, and copies out and lse back in one copy.  The new
    tokens' K/V are the cache's own rows, so the cache is unchanged.  The step runs as
    one captured CUDA graph."""
    nt, hkv = w.num_tokens, w.num_kv_heads
    slots = np.concatenate([
        w.block_table[s, np.arange(int(w.seq_lens[s]) - int(w.q_lens[s]), int(w.seq_lens[s])) // w.page]
        .astype(np.int64) * w.page + np.arange(int(w.seq_lens[s]) - int(w.q_lens[s]), int(w.seq_lens[s])) % w.page
        for s in range(w.bs)]) if nt else np.zeros(0, np.int64)
    st = torch.as_tensor(slots, device=dev)
    blk, off = st // w.page, st % w.page
    d = w.head_dim
    k_new = kv[blk, :, off, :d].contiguous()
    v_new = kv[blk, :, off, d:].contiguous()
    if w.kv_dtype == si.KV_FP8:      # the step's K/V arrive in bf16 and are quantised by the write
        k_new = (k_new.view(torch.float8_e4m3fn).float() * w.k_scale).to(torch.bfloat16)
        v_new = (v_new.view(torch.float8_e4m3fn).float() * w.v_scale).to(torch.bfloat16)
    inputs = {"q": q, "k": k_new, "v": v_new, "slots": st, "lens": lens, "cu": cu, "bt": bt}

    def packed(tensors, pinned):
        """One byte buffer holding every tensor (256-byte aligned) and typed views into it."""
        offs, total = {}, 0
        for k, t in tensors.items():
            offs[k] = total
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.empty(max(total, 256), dtype=torch.uint8, device="cpu" if pinned else dev)
        if pinned:
            buf = buf.pin_memory()
        views = {k: buf[offs[k]:offs[k] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                 for k, t in tensors.items()}
        return buf, views
    host_buf, host_in = packed(inputs, True)
    for k, t in inputs.items():
        host_in[k].copy_(t.cpu())
    dev_buf, dev_in = packed(inputs, False)
    outs = {"out": torch.empty((nt, w.num_q_heads, d), dtype=torch.bfloat16, device=dev),
            "lse": torch.empty((nt, w.num_q_heads), dtype=torch.float32, device=dev)}
    out_dbuf, out_d = packed(outs, False)
    out_hbuf, out_h = packed(outs, True)
    wsp = {}
    h2d = host_buf.numel()
    d2h = out_hbuf.numel()

    def step():
        dev_buf.copy_(host_buf, non_blocking=True)
        sk.sk_reshape_and_cache(dev_in["k"], dev_in["v"], dev_in["slots"], kv, k_scale=w.k_scale, v_scale=w.v_scale)
        sk.sk_plan_cache_reset()
        sk.paged_decode_attention(dev_in["q"], kv, dev_in["bt"], dev_in["lens"], dev_in["cu"],
                                  max_q_len=w.max_q_len, sm_scale=w.sm_scale, num_sms=nsm,
                                  k_scale=w.k_scale, v_scale=w.v_scale, causal=bool(w.causal),
                                  seg_max=w.seg_max, use_plan=use_plan, workspace=wsp,
                                  out=out_d["out"], lse=out_d["lse"])
        out_hbuf.copy_(out_dbuf, non_blocking=True)

    # the step is captured once as a CUDA graph (the calls are capture safe) and replayed,
    # as a server would run it: no per-call host work inside the timed region
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            step()
        side.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            step()
    torch.cuda.synchronize()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    steps = max(a.e2e_steps, 20)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    e0.record()
    for _ in range(steps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), ws, dev)
    if sk.sk_get_device_status(clear=True):
        raise RuntimeError("device status set during the serving-step run")
    assert torch.equal(out_h["out"], ref_out.cpu()), "serving-step output differs from the device-resident run"
    return {"value": weak_scaling_tbps(w.kv_bytes, steps, ws, ms), "unit": "TB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": ms / steps,
            "cache": "resident in HBM; each step writes its new tokens' K/V with sk_reshape_and_cache",
            "launch": ("one CUDA graph per step: one H2D copy of the packed inputs, KV write, plan, attention, "
                       "merge, one D2H copy of out and lse")}


def _back_to_back_ms(torch, f, steps):
    """Mean ms per call of `steps` calls of f issued back to back on the current stream
    between one event pair (inputs larger than L2, so no flush between calls)."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(steps):
        f()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_kv_write(a, local):
    """The KV write step on a prefill-sized chunk: 65536 new tokens x 8 KV heads
    written into standard pages at randomly permuted slots (256 MB of bf16 K/V in,
    larger than L2)."""
    import torch
    import paged_split_kv_gb300 as sk
    if not os.path.exists(sk.LIB_PATH):
        from paged_split_kv_gb300 import build as b
        b.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    nt, hkv, d, page = 65536, 8, 128, 16
    fp8 = a.kv_write == "fp8"
    g = torch.Generator(device=dev).manual_seed(77)
    key = torch.randn((nt, hkv, d), generator=g, device=dev).to(torch.bfloat16)
    val = torch.randn((nt, hkv, d), generator=g, device=dev).to(torch.bfloat16)
    nb = nt // page + 64
    slots = torch.randperm(nb * page, generator=g, device=dev)[:nt].to(torch.int64)
    pages = torch.empty((nb, hkv, page, 2 * d), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
    ks, vs = (0.5, 0.25) if fp8 else (1.0, 1.0)
    f = lambda: sk.sk_reshape_and_cache(key, val, slots, pages, k_scale=ks, v_scale=vs)
    for _ in range(max(3, a.warmup)):
        f()
    torch.cuda.synchronize()
    if sk.sk_get_device_status(clear=True):
        raise RuntimeError("device status set by the KV write")
    sampler = ClockSampler(local)
    sampler.start()
    ms = _back_to_back_ms(torch, f, a.steps)
    clocks = sampler.stop()
    moved = nt * hkv * (2 * d * 2 + 2 * d * (1 if fp8 else 2)) + nt * 8   # K/V in, page rows out, slots
    gbs = moved / (ms * 1e-3) / 1e9
    peak, kind = _peaks()
    line = {"metric": "KV write GB/s (reshape_and_cache into standard pages)", "value": round(gbs, 1),
            "unit": "GB/s", "n_gpus": 1, "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "dtype": "fp8_e4m3" if fp8 else "bf16", "data": "synthetic",
            "config": {"workload": f"kv_write_{nt}x{hkv}_{a.kv_write}", "tokens": nt, "num_kv_heads": hkv,
                       "head_dim": d, "page": page, "l2": "inputs larger than L2, no flush"},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "peak_kind": kind, "traffic": None,
                         "algorithmic_bytes_per_launch": int(moved)},
            "clocks": clocks, "gpu_launches": a.steps}
    print(json.dumps(line), flush=True)
    return 0


def run_forward(a, w, local):
    """One forward as a CUDA graph: the plan once, then `layers` x (attention +
    merge), replayed.  A second graph without the plan gives the plan's share.
    Every layer reads the same K/V cache; it is larger than L2, so each layer
    streams it from HBM as a layer of its own would."""
    import torch
    import paged_split_kv_gb300 as sk
    if not os.path.exists(sk.LIB_PATH):
        from paged_split_kv_gb300 import build as b
        b.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    L = a.forward_layers
    if w.kv_bytes <= 129e6:
        raise SystemExit("--forward-layers needs a workload larger than L2")
    q = si.make_q(w, dev)
    kv = si.make_kv(w, dev)
    bt = torch.as_tensor(w.block_table, device=dev)
    lens = torch.as_tensor(w.seq_lens, device=dev)
    cu = torch.as_tensor(w.cu_q, device=dev)
    nt, hkv, nsm = w.num_tokens, w.num_kv_heads, w.num_sms
    use_plan = w.bs > 1
    plan = torch.empty(sk.plan_capacity(w.bs, hkv, nsm), dtype=torch.int32, device=dev) if use_plan else None
    tok = torch.empty(nt, dtype=torch.int32, device=dev) if use_plan else None
    part_o = torch.empty((nt, w.seg_max, w.num_q_heads, w.head_dim), dtype=torch.float32, device=dev)
    part_m = torch.empty((nt, w.seg_max, w.num_q_heads), dtype=torch.float32, device=dev)
    part_l = torch.empty_like(part_m)
    outs = [torch.empty((nt, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=dev) for _ in range(L)]
    fixed = 0 if use_plan else sk.sk_fixed_nseg(w.bs, hkv, nsm, w.seg_max)
    side = torch.cuda.Stream()

    def layers(stream, with_plan):
        if with_plan and use_plan:
            sk.sk_build_plan(lens, cu, hkv, plan, tok, nsm, w.seg_max, stream)
        for i in range(L):
            sk.sk_paged_decode_attn(q, kv, bt, lens, cu, plan, part_o, part_m, part_l, max_q_len=w.max_q_len,
                                    sm_scale=w.sm_scale, num_sms=nsm, k_scale=w.k_scale, v_scale=w.v_scale,
                                    causal=bool(w.causal), stream=stream)
            sk.sk_merge_segments(part_o, part_m, part_l, tok, outs[i], None, fixed_nseg=fixed, stream=stream)

    graphs = {}
    with torch.cuda.stream(side):
        for with_plan in (True, False):
            sk.sk_plan_cache_reset()
            layers(side, with_plan)          # warm (and plan) outside capture
            side.synchronize()
            sk.sk_plan_cache_reset()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                layers(side, with_plan)
            graphs[with_plan] = g
    torch.cuda.synchronize()
    res = {}
    sampler = ClockSampler(local)
    sampler.start()
    for with_plan in (True, False):
        g = graphs[with_plan]
        for _ in range(max(3, a.warmup)):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(a.steps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        res[with_plan] = e0.elapsed_time(e1) / a.steps
    clocks = sampler.stop()
    if sk.sk_get_device_status(clear=True):
        raise RuntimeError("device status set during the forward")
    ms = res[True]
    tbps = L * w.kv_bytes / (ms * 1e-3) / 1e12
    line = {"metric": METRIC + f" (graph-captured forward, {L} layers)", "value": round(tbps, 4), "unit": "TB/s",
            "n_gpus": 1, "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.kv_dtype == si.KV_BF16 else "fp8_e4m3",
            "data": "synthetic; one K/V cache read by every layer (larger than L2)",
            "config": _config_json(w, {"layers": L, "split": "plan" if use_plan else "fixed",
                                       "graph": "one plan + layers x (attention + merge) per replay"}),
            "us_per_layer": round(1e3 * res[False] / L, 2),
            "us_plan_per_forward": round(1e3 * (res[True] - res[False]), 2),
            "clocks": clocks, "gpu_launches": a.steps * (2 * L + (1 if use_plan else 0))}
    print(json.dumps(line), flush=True)
    return 0


def run_shuffle(a, local):
    """The standard -> shuffled conversion of every block of a workload's cache
    (K/V larger than L2): bytes read plus bytes written per call."""
    import torch
    import paged_split_kv_gb300 as sk
    if not os.path.exists(sk.LIB_PATH):
        from paged_split_kv_gb300 import build as b
        b.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = si.config(2 if a.shuffle == "bf16" else 4)
    kv = si.make_kv(w, dev, poison_tail=False)
    nb, hkv, page, d2 = kv.shape
    x = 16 // kv.element_size()
    k_shuf = torch.empty((nb, hkv, d2 // 2 // x, page, x), dtype=kv.dtype, device=dev)
    v_shuf = torch.empty((nb, hkv, page // x, d2 // 2, x), dtype=kv.dtype, device=dev)
    f = lambda: sk.sk_std_to_shuffled(kv, k_shuf, v_shuf)
    for _ in range(max(3, a.warmup)):
        f()
    torch.cuda.synchronize()
    if sk.sk_get_device_status(clear=True):
        raise RuntimeError("device status set by the conversion")
    sampler = ClockSampler(local)
    sampler.start()
    ms = _back_to_back_ms(torch, f, a.steps)
    clocks = sampler.stop()
    moved = 2 * kv.numel() * kv.element_size()
    gbs = moved / (ms * 1e-3) / 1e9
    peak, kind = _peaks()
    line = {"metric": "standard -> shuffled page conversion GB/s", "value": round(gbs, 1), "unit": "GB/s",
            "n_gpus": 1, "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "dtype": a.shuffle if a.shuffle == "bf16" else "fp8_e4m3",
            "data": "synthetic", "config": {"workload": f"shuffle_all_blocks_{w.name}", "num_blocks": nb,
                                            "num_kv_heads": hkv, "bytes_per_call": moved,
                                            "l2": "inputs larger than L2, no flush"},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "peak_kind": kind, "traffic": None,
                         "algorithmic_bytes_per_launch": int(moved)},
            "clocks": clocks, "gpu_launches": a.steps}
    print(json.dumps(line), flush=True)
    return 0


def main():
    a = _args()
    if a.shuffle:
        return run_shuffle(a, int(os.environ.get("LOCAL_RANK", 0)))
    if a.forward_layers > 0:
        return run_forward(a, si.config(a.config), int(os.environ.get("LOCAL_RANK", 0)))
    if a.kv_write:
        return run_kv_write(a, int(os.environ.get("LOCAL_RANK", 0)))
    ws, rank, local = _dist()
    w = si.config(a.config)
    if a.impl == "reference":
        return run_reference(a, w, rank)
    return run_sk(a, w, ws, rank, local)


if __name__ == "__main__":
    sys.exit(main())
