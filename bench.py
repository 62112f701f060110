#!/usr/bin/env python3
"""Benchmark of the MXFP4 DSA lightning indexer on GB300.

One step = one decode step of the hot path on the long-context workload (16 sequences x
131072 cached keys, 64 index heads, head_dim 128, top-2048, MXFP4 paged cache with block 64):
the writer quantises the step's new key and query heads, the schedule is rebuilt, and the
decode kernel scores every cached key and selects each sequence's top-k. Writer + schedule and
the decode call are each captured in a CUDA graph and replayed; between timed steps a buffer
twice the L2 size is written and then read, so each step starts with none of its inputs in L2
and no dirty lines left to write back.

The same line carries, as sub-objects: the other decode workloads (batch 1 x 4096, batch 8 x
96K..128K, batch 8 x 262144), graph replay across changing context sets, the writer and the
schedule on their own, decode with two verify rows per sequence (next_n 2) through the decode
and the prefill calls, causal prefill (4 prompts of 2634..4295 tokens in 512-row steps) and
prefill over a staged flat cache, and the oracle on the host cores (all cores, and one core).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0). With --gpus N under torchrun every rank runs its own copy of
the workload (weak scaling, no collective on the data path); the value is all ranks' keys over
the slowest rank's time. --impl reference times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode indexer µs/layer & keys scored/s, % HBM roofline; prefill % FP4 peak"
UNIT = "keys/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense ratio of the FP4 and bf16 tensor rates
# the decode kernel's sources; the committed ncu traffic figure holds while their code is unchanged
DECODE_SOURCES = ["decode_kernel.cuh", "block.cuh", "decode_sched.cuh", "ptx.cuh", "common.cuh", "decode.cu",
                  "decode_n1.cu"]
DECODE_PROFILE = "decode_kernel_b16_ctx131072.txt"
L2_NOTE = ("inputs (142.6 MB of keys) larger than L2, and a 2x-L2 buffer written then read between timed "
           "calls (no step input left in L2, no dirty line left to write back); graph-replayed calls")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--profile", action="store_true",
                    help="only set up the decode workload and run warmup+steps direct launches (for ncu)")
    ap.add_argument("--profile-prefill", action="store_true",
                    help="only set up the prefill workload and run warmup+steps direct passes (for ncu)")
    ap.add_argument("--no-extras", action="store_true", help="skip the CPU baseline, e2e and prefill legs")
    return ap.parse_args(argv)


# ---- multi-process plumbing ------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(backend: str):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def aggregate(dist, units_local: float, seconds_local: float, device=None):
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    import torch
    t = torch.tensor([seconds_local, units_local], dtype=torch.float64, device=device)
    if dist is not None:
        mx = t.clone()
        dist.all_reduce(mx[0:1], op=dist.ReduceOp.MAX)
        sm = t.clone()
        dist.all_reduce(sm[1:2], op=dist.ReduceOp.SUM)
        seconds, units = float(mx[0]), float(sm[1])
    else:
        seconds, units = float(t[0]), float(t[1])
    return units / seconds if seconds > 0 else 0.0, seconds


# ---- measured peaks and clocks ----------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), \
            "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.gpu_index, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.1)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_index_for_smi(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v.strip() for v in vis.split(",") if v.strip()]
    if ids:
        return ids[local_rank] if local_rank < len(ids) else ids[0]
    return str(local_rank)


_CODE_TOKENS = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\])*"|\'(?:\\.|[^\'\\])*\'', re.S)


def _code_only(text: str) -> str:
    """C++ source without comments and with whitespace collapsed (string literals kept)."""
    text = _CODE_TOKENS.sub(lambda m: " " if m.group(0).startswith("/") else m.group(0), text)
    return " ".join(text.split())


def decode_source_hash() -> str:
    """Hash of the decode kernel's code (comments and layout ignored)."""
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(ROOT, "fp4_sparse_attention_mxfp4_gb300", "csrc", name)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, if it still matches the source."""
    path = os.path.join(ROOT, "profiles", DECODE_PROFILE)
    try:
        kv = {}
        with open(path) as f:
            for ln in f:
                if "=" in ln and not ln.startswith("#"):
                    k, v = ln.strip().split("=", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("source_hash") == decode_source_hash():
            return float(kv["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ---- workloads ---------------------------------------------------------------------------

def decode_alg_bytes(ctx_lens, heads: int, topk: int, next_n: int = 1) -> int:
    """Algorithmic bytes of one decode call: 68 B per key (64 packed + 4 scale) read once for all
    next_n rows, 4 B per page-table entry, and per query row 72 B per head (64 + 4 packed/scales,
    4 weight) and 8 B per output slot."""
    tot = 0
    for c in ctx_lens:
        c = int(c)
        tot += 68 * c + 4 * (-(-c // 64)) + next_n * (heads * (68 + 4) + topk * 8)
    return tot


class L2Flush:
    """Between timed calls: write a buffer of twice the L2 size, then read it back, so the next
    call finds none of its inputs in L2 and no dirty lines to write back."""

    def __init__(self, torch):
        props = torch.cuda.get_device_properties(torch.cuda.current_device())
        l2 = getattr(props, "L2_cache_size", 128 << 20)
        self.buf = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.int32, device="cuda")

    def __call__(self):
        self.buf.fill_(1)
        self.buf.sum()


class DecodeBench:
    """One decode workload resident on the device: cache filled once (setup), per-step inputs, and
    the writer + schedule and decode calls, each capturable in a graph. Works for a DecodeCase
    (one row per sequence) and an MtpCase (next_n verify rows per sequence, decode-shaped call)."""

    def __init__(self, case):
        import numpy as np
        import torch

        import fp4_sparse_attention_mxfp4_gb300 as fx
        self.fx, self.torch, self.np, self.case = fx, torch, np, case
        self.next_n = n = int(getattr(case, "next_n", 1))
        B, H, k = case.batch, case.heads, case.topk
        R = B * n
        d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
        self.d = d
        self.kv_p = torch.full((case.layout.num_pages, 4, 64, 16), 0x77, dtype=torch.uint8, device="cuda")
        self.kv_s = torch.full((case.layout.num_pages, 4, 64), 0xFF, dtype=torch.uint8, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        slots = case.all_slots()
        # fill the cache with every sequence's context (setup, not timed), in chunks
        chunk = 1 << 20
        for a in range(0, slots.size, chunk):
            fx.idx_fp4_quant_and_cache(d(case.k_bf16[a:a + chunk].view(np.int16)), d(slots[a:a + chunk]),
                                       self.kv_p, self.kv_s, status=self.status)
        # per-step inputs: each sequence's newest next_n keys and the query heads
        ends = np.cumsum(case.ctx_lens)
        new = np.concatenate([np.arange(e - n, e) for e in ends])
        self.k_new = d(case.k_bf16[new].view(np.int16))
        self.slots_new = d(slots[new])
        self.q_bf16 = d(case.q_bf16.view(np.int16))
        self.q_packed = torch.empty((R, H, 64), dtype=torch.uint8, device="cuda")
        self.q_scale = torch.empty((R, H, 4), dtype=torch.uint8, device="cuda")
        self.w = d(case.w)
        self.bt = d(case.layout.block_tables)
        self.ctx = d(case.ctx_lens)
        self.max_ctx = int(case.ctx_lens.max())
        self.sched = torch.zeros(fx.idx_fp4_decode_schedule_bytes(B, self.max_ctx), dtype=torch.uint8, device="cuda")
        ws = fx.idx_fp4_decode_mtp_workspace_bytes(B, self.max_ctx, k, n)
        self.ws = torch.zeros(ws, dtype=torch.uint8, device="cuda")
        self.topk_idx = torch.empty((R, k), dtype=torch.int32, device="cuda")
        self.topk_val = torch.empty((R, k), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()

    def set_contexts(self, ctx_lens):
        """A new context-length set in the same device buffers (between graph replays): the
        sequences' lengths, and the keys and slots of their newest positions (each sequence's keys
        are a prefix of its full context, so the cache stays consistent)."""
        np, case, n = self.np, self.case, self.next_n
        ctx_lens = np.asarray(ctx_lens, np.int32)
        assert np.all(ctx_lens >= n) and np.all(ctx_lens <= case.ctx_lens)
        starts = np.cumsum(case.ctx_lens) - case.ctx_lens
        new = np.concatenate([np.arange(s + c - n, s + c) for s, c in zip(starts, ctx_lens)])
        slots = np.concatenate([case.layout.slots(b, int(c) - n, int(c)) for b, c in enumerate(ctx_lens)])
        self.ctx.copy_(self.d(ctx_lens))
        self.k_new.copy_(self.d(case.k_bf16[new].view(np.int16)))
        self.slots_new.copy_(self.d(slots.astype(np.int32)))
        self.torch.cuda.synchronize()

    def write(self):
        self.fx.idx_fp4_quant_and_cache(self.k_new, self.slots_new, self.kv_p, self.kv_s, q_bf16=self.q_bf16,
                                        q_packed=self.q_packed, q_scale=self.q_scale, status=self.status)

    def schedule(self):
        if self.next_n == 1:
            self.fx.idx_fp4_build_decode_schedule(self.ctx, self.case.batch, self.max_ctx, self.sched,
                                                  status=self.status)
        else:
            self.fx.idx_fp4_build_decode_schedule_mtp(self.ctx, self.next_n, self.case.batch, self.max_ctx,
                                                      self.sched, status=self.status)

    def prep(self):
        self.write()
        self.schedule()

    def decode(self):
        fx = self.fx
        if self.next_n == 1:
            fx.idx_fp4_decode_logits_topk(self.q_packed, self.q_scale, self.w, self.kv_p, self.kv_s, self.bt,
                                          self.ctx, self.case.topk, self.sched, self.ws, self.topk_idx,
                                          self.topk_val, status=self.status)
        else:
            fx.idx_fp4_decode_mtp_logits_topk(self.q_packed, self.q_scale, self.w, self.kv_p, self.kv_s, self.bt,
                                              self.ctx, self.next_n, self.case.topk, self.sched, self.ws,
                                              self.topk_idx, self.topk_val, status=self.status)

    def capture(self):
        torch = self.torch
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(2):
                self.prep()
                self.decode()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.g_prep, self.g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        self.g_write, self.g_sched = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        self.g_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_step):
            self.prep()
            self.decode()
        with torch.cuda.graph(self.g_prep):
            self.prep()
        with torch.cuda.graph(self.g_dec):
            self.decode()
        with torch.cuda.graph(self.g_write):
            self.write()
        with torch.cuda.graph(self.g_sched):
            self.schedule()
        torch.cuda.synchronize()

    def ok(self):
        return int(self.status.item()) == 0


def time_decode(bench: DecodeBench, steps: int, warmup: int, flush: L2Flush, dist=None, clock=None):
    """Replays the whole step (writer, schedule and decode call, one graph: each kernel may begin
    while the one before it finishes) `steps` times after `warmup` untimed steps, with events around
    each replay on the launching stream and an L2 flush between steps; then, as many times, the
    writer and schedule graph followed by the decode call's own graph, with events around the
    decode call alone. Returns per-step milliseconds of the whole step and of the decode call, and
    the clock record (sampled over both passes)."""
    torch = bench.torch
    for _ in range(warmup):
        bench.g_step.replay()
        flush()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    ev_dec = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    barrier(dist)
    if clock is not None:
        clock.start()
    torch.cuda.synchronize()
    for e0, e1 in ev:
        e0.record()
        bench.g_step.replay()
        e1.record()
        flush()
    torch.cuda.synchronize()
    barrier(dist)
    for e0, e1 in ev_dec:
        bench.g_prep.replay()
        e0.record()
        bench.g_dec.replay()
        e1.record()
        flush()
    torch.cuda.synchronize()
    clocks = clock.stop() if clock is not None else None
    step_ms = [a.elapsed_time(b) for a, b in ev]
    dec_ms = [a.elapsed_time(b) for a, b in ev_dec]
    return step_ms, dec_ms, clocks


def time_graph(torch, graph, steps: int, warmup: int, flush: L2Flush, before=None):
    """Mean milliseconds of one graph replay, L2 flushed between replays."""
    for _ in range(warmup):
        if before is not None:
            before()
        graph.replay()
        flush()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record()
        graph.replay()
        b.record()
        flush()
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


def shape_line(name, case, dec_ms, hbm, next_n=1, extra=None):
    alg = decode_alg_bytes(case.ctx_lens, case.heads, case.topk, next_n)
    dec_s = statistics.mean(dec_ms) / 1e3
    keys = int(case.ctx_lens.sum())
    out = {"workload": name, "batch": int(case.batch), "keys": keys, "us_per_call": dec_s * 1e6,
           "us_min": min(dec_ms) * 1e3, "keys_per_s": keys / dec_s, "alg_bytes": alg,
           "hbm_frac": alg / dec_s / 1e9 / hbm}
    if extra:
        out.update(extra)
    return out


def run_decode_shapes(steps: int, warmup: int, flush: L2Flush, hbm: float, single_row_us: float):
    """The other decode workloads, each at its own size, plus decode with two verify rows."""
    import synth
    import torch
    shapes = []
    for n, name in [(2, "batch 1 x 4096 keys (latency-bound)"), (3, "batch 8 x 96K..128K keys"),
                    (5, "batch 8 x 262144 keys")]:
        case = synth.decode_config(n)
        b = DecodeBench(case)
        b.capture()
        _, dec_ms, _ = time_decode(b, steps, warmup, flush)
        shapes.append(shape_line(name, case, dec_ms, hbm, extra={"status_ok": b.ok()}))
        del b
        torch.cuda.empty_cache()
    case = synth.mtp_config()
    b = DecodeBench(case)
    b.capture()
    _, dec_ms, _ = time_decode(b, steps, warmup, flush)
    mtp = shape_line("decode, next_n 2 verify rows per sequence, decode-shaped call: 16 x 131072 keys, 64 heads, "
                     "top-2048 per row", case, dec_ms, hbm, next_n=2,
                     extra={"row_key_pairs_per_s": int(case.row_ends().astype("int64").sum()) /
                            (statistics.mean(dec_ms) / 1e3),
                            "vs_single_row_call": statistics.mean(dec_ms) * 1e3 / single_row_us,
                            "status_ok": b.ok()})
    del b
    torch.cuda.empty_cache()
    return shapes, mtp


def run_replay_sets(bench: DecodeBench, steps: int, warmup: int, flush: L2Flush, hbm: float):
    """One captured writer + schedule + decode graph pair replayed across changing context-length
    sets (the buffers' contents change, the graphs do not): decode time per set."""
    import synth
    case = bench.case
    sets = synth.replay_ctx_sets(3, case.batch, bench.max_ctx)
    names = ["all 131072", "U[65536, 131072]", "U[1, 131072], first below k", "all 131072 again"]
    out = []
    ok = True
    for name, ctx in zip(names, sets):
        bench.set_contexts(ctx)
        _, dec_ms, _ = time_decode(bench, steps, warmup, flush)
        ok = ok and bench.ok()
        sub = type("C", (), {})()
        sub.ctx_lens, sub.heads, sub.topk, sub.batch = ctx, case.heads, case.topk, case.batch
        out.append(shape_line(name, sub, dec_ms, hbm))
    bench.set_contexts(case.ctx_lens)
    return {"sets": out, "status_ok": ok}


def run_decode_e2e(bench: DecodeBench, steps: int, warmup: int):
    """Same step through the public API with host buffers: the step's inputs copied from pinned
    host memory, the three calls, and a device -> host read of the step's top-k. The caller
    keeps its inputs side by side in one pinned buffer (and the outputs in one device buffer),
    so each direction is one copy."""
    import numpy as np
    torch, fx, case = bench.torch, bench.fx, bench.case
    last = np.cumsum(case.ctx_lens) - 1
    arrays = {
        "k_new": case.k_bf16[last].view(np.int16), "slots": case.all_slots()[last],
        "q": case.q_bf16.view(np.int16), "w": case.w, "ctx": case.ctx_lens, "bt": case.layout.block_tables,
    }
    offs, size = {}, 0
    for name, a in arrays.items():
        offs[name] = size
        size += (a.nbytes + 255) // 256 * 256
    h_in = torch.zeros(size, dtype=torch.uint8).pin_memory()
    d_buf = torch.empty(size, dtype=torch.uint8, device="cuda")
    d_in = {}
    for name, a in arrays.items():
        a = np.ascontiguousarray(a)
        h_in.numpy()[offs[name]:offs[name] + a.nbytes] = a.reshape(-1).view(np.uint8)
        dt = torch.from_numpy(a[:0]).dtype
        d_in[name] = d_buf[offs[name]:offs[name] + a.nbytes].view(dt).view(a.shape)
    B, k = bench.topk_idx.shape
    d_out = torch.empty(B * k * 8, dtype=torch.uint8, device="cuda")
    h_out = torch.empty(B * k * 8, dtype=torch.uint8).pin_memory()
    out_idx = d_out[:B * k * 4].view(torch.int32).view(B, k)
    out_val = d_out[B * k * 4:].view(torch.float32).view(B, k)
    h2d = size
    d2h = d_out.numel()

    def step():
        d_buf.copy_(h_in, non_blocking=True)
        fx.idx_fp4_quant_and_cache(d_in["k_new"], d_in["slots"], bench.kv_p, bench.kv_s, q_bf16=d_in["q"],
                                   q_packed=bench.q_packed, q_scale=bench.q_scale, status=bench.status)
        fx.idx_fp4_build_decode_schedule(d_in["ctx"], case.batch, bench.max_ctx, bench.sched, status=bench.status)
        fx.idx_fp4_decode_logits_topk(bench.q_packed, bench.q_scale, d_in["w"], bench.kv_p, bench.kv_s, d_in["bt"],
                                      d_in["ctx"], case.topk, bench.sched, bench.ws, out_idx, out_val,
                                      status=bench.status)
        h_out.copy_(d_out, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(warmup):
        step()
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    # the read-back is the step's result: the same top-k as the device-resident run
    got = h_out[:B * k * 4].view(torch.int32).view(B, k)
    if not torch.equal(got, bench.topk_idx.cpu()):
        raise RuntimeError("end-to-end top-k differs from the device-resident step")
    return statistics.mean(times), h2d, d2h


def run_prefill(steps: int, warmup: int, flush: L2Flush, case=None, direct_passes: int = 0):
    """Causal prefill of a PrefillCase (default: 4 prompts of 2634..4295 tokens) in 512-row steps,
    all steps captured in one graph; returns seconds per full prefill pass and the algorithmic
    FLOPs of a pass."""
    import numpy as np
    import torch

    import synth
    import fp4_sparse_attention_mxfp4_gb300 as fx
    if case is None:
        case = synth.prefill_config("pad8")
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    H, k = case.heads, case.topk
    kv_p = torch.full((case.layout.num_pages, 4, 64, 16), 0x77, dtype=torch.uint8, device="cuda")
    kv_s = torch.full((case.layout.num_pages, 4, 64), 0xFF, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots_all = case.token_slots()
    per = []
    flops = 0
    for st in case.steps:
        q = np.zeros((st.rows, H, 128), np.uint16)
        q[:st.real_rows] = case.q_bf16[st.token_ids]
        w = np.zeros((st.rows, H), np.float32)
        w[:st.real_rows] = case.w[st.token_ids]
        flops += 2 * H * 128 * int(st.row_ends.astype(np.int64).sum())
        per.append(dict(
            k=d(case.k_bf16[st.token_ids].view(np.int16)), slots=d(slots_all[st.token_ids]), q=d(q.view(np.int16)),
            w=d(w), qp=torch.empty((st.rows, H, 64), dtype=torch.uint8, device="cuda"),
            qs=torch.empty((st.rows, H, 4), dtype=torch.uint8, device="cuda"),
            bt=d(case.layout.block_tables[st.requests]), ctx=d(st.ctx_lens), cu=d(st.cu_seqlens),
            re=d(st.row_ends),
            mc=max(int(st.ctx_lens.max()), 1),
            ws=torch.zeros(fx.idx_fp4_prefill_workspace_bytes(len(st.requests), st.rows, H, max(int(st.ctx_lens.max()), 1), k),
                           dtype=torch.uint8, device="cuda"),
            idx=torch.empty((st.rows, k), dtype=torch.int32, device="cuda"),
            val=torch.empty((st.rows, k), dtype=torch.float32, device="cuda")))

    def one_pass():
        for p in per:
            fx.idx_fp4_quant_and_cache(p["k"], p["slots"], kv_p, kv_s, q_bf16=p["q"], q_packed=p["qp"],
                                       q_scale=p["qs"], status=status)
            fx.idx_fp4_prefill_logits_topk(p["qp"], p["qs"], p["w"], kv_p, kv_s, p["bt"], p["ctx"], p["cu"], p["re"],
                                           k, p["mc"], p["ws"], p["idx"], p["val"], status=status)

    if direct_passes > 0:
        for _ in range(direct_passes):
            one_pass()
        torch.cuda.synchronize()
        return 0.0, flops, len(case.steps), int(status.item()) == 0
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        one_pass()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        one_pass()
    for _ in range(warmup):
        g.replay()
        flush()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record()
        g.replay()
        b.record()
        flush()
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in ev]
    ok = int(status.item()) == 0
    return statistics.mean(ms) / 1e3, flops, len(case.steps), ok


def run_mtp_prefill_form(steps: int, warmup: int, flush: L2Flush):
    """Decode with two verify rows per sequence (16 x 131072 keys, next_n 2) through the prefill
    call, captured in a graph and replayed with an L2 flush between calls. Returns seconds per
    call, (query row, key) pairs scored per call, algorithmic bytes per call and the status."""
    import numpy as np
    import torch

    import synth
    import fp4_sparse_attention_mxfp4_gb300 as fx
    case = synth.mtp_config()
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    B, H, k, n = case.batch, case.heads, case.topk, case.next_n
    R = B * n
    kv_p = torch.full((case.layout.num_pages, 4, 64, 16), 0x77, dtype=torch.uint8, device="cuda")
    kv_s = torch.full((case.layout.num_pages, 4, 64), 0xFF, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = case.all_slots()
    chunk = 1 << 20
    for a in range(0, slots.size, chunk):
        fx.idx_fp4_quant_and_cache(d(case.k_bf16[a:a + chunk].view(np.int16)), d(slots[a:a + chunk]), kv_p, kv_s,
                                   status=status)
    qp = torch.empty((R, H, 64), dtype=torch.uint8, device="cuda")
    qs = torch.empty((R, H, 4), dtype=torch.uint8, device="cuda")
    fx.idx_fp4_quant_and_cache(d(case.k_bf16[:0].view(np.int16)), d(slots[:0]), kv_p, kv_s,
                               q_bf16=d(case.q_bf16.view(np.int16)), q_packed=qp, q_scale=qs, status=status)
    w, bt, ctx = d(case.w), d(case.layout.block_tables), d(case.ctx_lens)
    cu, re = d(case.cu_seqlens()), d(case.row_ends())
    max_ctx = int(case.ctx_lens.max())
    ws = torch.zeros(fx.idx_fp4_prefill_workspace_bytes(B, R, H, max_ctx, k), dtype=torch.uint8, device="cuda")
    idx = torch.empty((R, k), dtype=torch.int32, device="cuda")
    val = torch.empty((R, k), dtype=torch.float32, device="cuda")

    def call():
        fx.idx_fp4_prefill_logits_topk(qp, qs, w, kv_p, kv_s, bt, ctx, cu, re, k, max_ctx, ws, idx, val,
                                       status=status)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for _ in range(warmup):
        g.replay()
        flush()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record()
        g.replay()
        b.record()
        flush()
    torch.cuda.synchronize()
    sec = statistics.mean(a.elapsed_time(b) for a, b in ev) / 1e3
    pairs = int(case.row_ends().astype(np.int64).sum())
    alg = decode_alg_bytes(case.ctx_lens, H, k, n)  # keys once; n query rows' operands and outputs
    return sec, pairs, alg, int(status.item()) == 0


def run_mxf4_probe(iters: int = 2048, reps: int = 5):
    """The MXFP4 tensor-core rate at the scorers' MMA shape (the library's probe kernel, one CTA per
    SM issuing back-to-back block-scaled MMAs from shared memory): TFLOP/s over `reps` launches."""
    import torch

    import fp4_sparse_attention_mxfp4_gb300 as fx
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        fx.idx_fp4_mxf4_probe(iters, status)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        a.record()
        fx.idx_fp4_mxf4_probe(iters, status)
        b.record()
    torch.cuda.synchronize()
    sec = statistics.median(a.elapsed_time(b) for a, b in ev) / 1e3
    return fx.idx_fp4_mxf4_probe_flops(iters) / sec / 1e12, int(status.item()) == 0


def oracle_decode_rate(case, threads: int, min_seconds: float, max_reps: int = 5):
    """The oracle (fp64 scoring + exact sort top-k) on the given decode workload, host cores:
    keys per second over whole repetitions."""
    import numpy as np

    import oracle
    kv_p = np.full((case.layout.num_pages, 4, 64, 16), 0x77, np.uint8)
    kv_s = np.full((case.layout.num_pages, 4, 64), 0xFF, np.uint8)
    oracle.quant_and_cache(case.k_bf16, case.all_slots(), kv_p, kv_s)
    qp, qs = oracle.quantize_plain(case.q_bf16)
    keys = int(case.ctx_lens.sum())
    reps, t_total = 0, 0.0
    while reps < 1 or (t_total < min_seconds and reps < max_reps):
        t0 = time.perf_counter()
        oracle.decode_topk(qp, qs, case.w, kv_p, kv_s, case.layout.block_tables, case.ctx_lens, case.topk,
                           threads=threads)
        t_total += time.perf_counter() - t0
        reps += 1
    return keys * reps / t_total, reps, keys


# ---- arms ----------------------------------------------------------------------------------

def workload_config(case):
    return {"workload": "decode: 16 sequences x 131072 cached keys, 64 index heads, head_dim 128, top-2048, "
                        "MXFP4 paged index cache (page 64, swizzled scale plane), random page tables",
            "batch": int(case.batch), "ctx_len": int(case.ctx_lens[0]), "heads": int(case.heads),
            "topk": int(case.topk), "cache_bytes_per_key": 68, "l2": L2_NOTE, "seed": 3}


def run_reference(args):
    """The oracle as the reference arm: each step scores a bounded sample of the workload (the 16
    sequences' first 8192 keys) on the host cores."""
    rank, world, _ = dist_env()
    if world > 1 and rank != 0:
        return 0
    import synth
    threads = os.cpu_count() or 1
    sample = synth.decode_case("decode sample 16 x 8192", 3, [8192] * 16, 64, 2048)
    import numpy as np

    import oracle
    kv_p = np.full((sample.layout.num_pages, 4, 64, 16), 0x77, np.uint8)
    kv_s = np.full((sample.layout.num_pages, 4, 64), 0xFF, np.uint8)
    oracle.quant_and_cache(sample.k_bf16, sample.all_slots(), kv_p, kv_s)
    qp, qs = oracle.quantize_plain(sample.q_bf16)

    def step():
        oracle.decode_topk(qp, qs, sample.w, kv_p, kv_s, sample.layout.block_tables, sample.ctx_lens, 2048,
                           threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    keys = int(sample.ctx_lens.sum()) * args.steps
    value = keys / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "decode: 16 sequences x 131072 cached keys, 64 index heads, head_dim 128, top-2048, "
                               "MXFP4 paged index cache", "batch": 16, "ctx_len": 131072, "heads": 64, "topk": 2048,
                   "reference_sample": "each step: the 16 sequences' first 8192 keys (131072 keys)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "16 sequences x 8192 keys per step, fp64 scoring + exact sort top-k"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_profile(args):
    """Direct launches of the decode step (no graphs, no flush) for an ncu capture: writer,
    schedule and decode kernel per step, on the 16 x 131072 workload."""
    import synth
    import torch
    bench = DecodeBench(synth.decode_config(4))
    for _ in range(args.warmup + args.steps):
        bench.prep()
        bench.decode()
    torch.cuda.synchronize()
    print(json.dumps({"profile_run": "decode b16 x 131072", "launches_per_step": 3,
                      "status": int(bench.status.item())}), flush=True)
    return 0 if bench.ok() else 1


def cpu_baselines(case):
    """The oracle as it stands on the host cores: all cores on the full workload, and one core on
    a bounded sample of it (the 16 sequences' first 16384 keys)."""
    import synth
    threads = os.cpu_count() or 1
    rate, reps, keys = oracle_decode_rate(case, threads, min_seconds=6.0)
    sample = synth.decode_case("decode sample 16 x 16384", 3, [16384] * 16, case.heads, case.topk)
    rate1, reps1, keys1 = oracle_decode_rate(sample, 1, min_seconds=6.0)
    return {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"the full workload ({keys} keys) scored and selected {reps}x, fp64 oracle, {threads} threads",
            "single_core": {"value": rate1, "unit": UNIT, "cores": 1,
                            "sample": f"16 sequences x 16384 keys ({keys1} keys) scored and selected {reps1}x"}}


def run_ours(args):
    import torch

    import synth
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = dist_init("nccl") if world > 1 else None
    import fp4_sparse_attention_mxfp4_gb300 as fx
    fx.lib()
    hbm, bf16, bf16_sus, peak_kind = measured_peaks()
    case = synth.decode_config(4)
    bench = DecodeBench(case)
    bench.capture()
    flush = L2Flush(torch)
    clock = ClockSampler(gpu_index_for_smi(local))
    step_ms, dec_ms, clocks = time_decode(bench, args.steps, args.warmup, flush, dist, clock)
    keys_per_step = int(case.ctx_lens.sum())
    local_seconds = sum(step_ms) / 1e3
    value, seconds_max = aggregate(dist, keys_per_step * args.steps, local_seconds, device="cuda")
    ms_per_step = seconds_max / args.steps * 1e3
    dec_mean_s = statistics.mean(dec_ms) / 1e3
    alg = decode_alg_bytes(case.ctx_lens, case.heads, case.topk)
    achieved = alg / dec_mean_s / 1e9
    ok = bench.ok()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "mxfp4->f32", "data": "synthetic",
        "config": workload_config(case) | {"parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "decode_us_per_layer": dec_mean_s * 1e6,
        "decode_us_min": min(dec_ms) * 1e3,
        "step_us": {"writer+schedule": statistics.mean(s - d for s, d in zip(step_ms, dec_ms)) * 1e3,
                    "decode": dec_mean_s * 1e6},
        "roofline": {"bound": "hbm", "kernel": "decode_kernel (idx_fp4_decode_logits_topk: one cooperative launch, "
                                               "scoring and exact top-k)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "peak_source": f"{peak_kind} hbm_gbs (burst copy)", "alg_bytes_per_launch": alg,
                     "traffic": profiled_traffic()},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "status_ok": ok,
    }
    if not args.no_extras:
        n_small = max(10, min(args.steps, 50))
        e2e_s, h2d, d2h = run_decode_e2e(bench, max(10, min(args.steps, 100)), 3)
        e2e_val, _ = aggregate(dist, keys_per_step, e2e_s, device="cuda")
        line["e2e"] = {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        line["writer_schedule_alone_us"] = {
            "writer (16 keys + 16 x 64 query heads)": time_graph(torch, bench.g_write, n_small, 3, flush) * 1e3,
            "schedule": time_graph(torch, bench.g_sched, n_small, 3, flush) * 1e3}
        line["graph_replay_ctx_sets"] = run_replay_sets(bench, n_small, 3, flush, hbm)
        single_row_us = dec_mean_s * 1e6
        del bench
        torch.cuda.empty_cache()
        shapes, mtp = run_decode_shapes(n_small, 3, flush, hbm, single_row_us)
        line["decode_shapes"] = shapes
        line["decode_mtp"] = mtp
        mt_s, mt_pairs, mt_alg, mt_ok = run_mtp_prefill_form(n_small, 3, flush)
        line["decode_mtp_prefill_form"] = {
            "workload": "the same next_n 2 rows through the prefill call", "us_per_layer": mt_s * 1e6,
            "row_key_pairs_per_s": mt_pairs / mt_s, "alg_bytes_per_call": mt_alg,
            "hbm_frac": mt_alg / mt_s / 1e9 / hbm, "status_ok": mt_ok}
        fp4_peak = bf16 * FP4_OVER_BF16
        probe_tflops, probe_ok = run_mxf4_probe()
        line["fp4_mma_probe"] = {
            "what": "tcgen05.mma kind::mxf4 block_scale, M128 N128 K64 (the scorers' instruction), one CTA per "
                    "SM, 8 issuing warps, shared-memory operands", "tflops": probe_tflops, "status_ok": probe_ok}
        pf_s, pf_flops, pf_steps, pf_ok = run_prefill(max(5, min(args.steps, 50)), 3, flush)
        line["prefill"] = {
            "workload": "causal prefill: 4 prompts (2634..4295 tokens), 512-row steps with padding rows, "
                        "64 heads, top-2048", "steps_per_pass": pf_steps, "ms_per_pass": pf_s * 1e3,
            "alg_flop_per_pass": pf_flops, "tflops": pf_flops / pf_s / 1e12,
            "peak_tflops": fp4_peak, "peak_source": f"{peak_kind} bf16_tflops x {FP4_OVER_BF16:g} (nominal FP4/bf16)",
            "frac_fp4_peak": pf_flops / pf_s / 1e12 / fp4_peak,
            "frac_of_mxf4_probe": pf_flops / pf_s / 1e12 / probe_tflops, "status_ok": pf_ok}
        pf_s, pf_flops, pf_steps, pf_ok = run_prefill(max(5, min(args.steps, 20)), 3, flush,
                                                      synth.prefill_flat_config())
        line["prefill_flat"] = {
            "workload": "causal prefill over a staged flat cache (identity page table): one 16384-token prompt, "
                        "512-row steps with padding rows, 64 heads, top-2048; rows past 8192 keys merged from "
                        "key chunks", "steps_per_pass": pf_steps, "ms_per_pass": pf_s * 1e3,
            "alg_flop_per_pass": pf_flops, "tflops": pf_flops / pf_s / 1e12, "peak_tflops": fp4_peak,
            "frac_fp4_peak": pf_flops / pf_s / 1e12 / fp4_peak, "status_ok": pf_ok}
        ok = ok and all(s["status_ok"] for s in shapes) and mtp["status_ok"] and pf_ok
        if rank == 0 and world == 1:
            line["cpu_baseline"] = cpu_baselines(case)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0 if ok else 1


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        return run_profile(args)
    if args.profile_prefill:
        _, _, steps, ok = run_prefill(0, 0, None, direct_passes=args.warmup + args.steps)
        print(json.dumps({"profile_run": "causal prefill, 4 prompts", "steps_per_pass": steps, "status_ok": ok}),
              flush=True)
        return 0 if ok else 1
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
