"""Benchmark of the reuse-time MLA KV reconstruction path on GB300.

Default (no flags): N=1, the DeepSeek-V2-Lite-shaped decode workload (16 heads, batch 8,
context 8192, 75% reused chunks with delta-rotation), reported as logical KV GB/s, plus
the other workloads (V3-shaped decode, chunked prefill, rotate+gather) in "workloads".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one pass of the whole hot path over one batch: chunk-table walk, per-chunk
rotation angles, gather of [cKV | k_r] rows, delta-rotation in shared memory, Q.K^T,
online softmax, P.cKV (and the split-KV merge for decode) -- one call of the C ABI.
Steps are timed with CUDA events on the launching stream, each step replayed from a CUDA
graph, with L2 flushed (256 MiB write then 256 MiB read, untimed) between steps.  The oracle arm
(--impl reference) times the fp64 CPU oracle on a bounded sample of the same workload.
Under torchrun every rank runs its own replica (weak scaling); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("δ-rotated MLA attn: decode KV GB/s & prefill TFLOP/s (% roofline); "
          "rotate-gather tok/s")
ROW_BYTES = 1152
PAIR_FLOPS = 2176
L2_FLUSH_BYTES = 256 << 20


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# --------------------------------------------------------------------------- distributed

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    from mla_position_independent_gb300.replicas import max_over_ranks as _m
    return _m(x, world, device="cuda" if torch.cuda.is_available() else "cpu")


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples during the timed region (clock, limit reasons)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "20"]
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            cmd += ["-i", uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"]
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"], samples=0)
        time.sleep(0.1)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return dict(sm_mhz=statistics.median(sm) if sm else None,
                    sm_max_mhz=max(mx) if mx else None, reasons=sorted(reasons),
                    samples=len(sm))


# --------------------------------------------------------------------------- workloads

def _prep_case(name, seed):
    from mla_position_independent_gb300 import synth
    if name == "v2lite_decode":
        return synth.v2lite_decode(seed, device="cuda")
    if name == "v3_decode":
        return synth.v3_decode(seed, device="cuda")
    if name == "chunked_prefill":
        return synth.chunked_prefill(seed, device="cuda")
    if name == "chunked_prefill_256":
        return synth.chunked_prefill(seed, device="cuda", n_q=256)
    if name.startswith("rotate_gather_"):
        n = int(name.split("_")[-1].rstrip("M")) << 20
        return synth.rotate_gather_case(n, seed, device="cuda", fill_kv=False)
    if name.startswith("cdc_"):
        S, per = CDC_SHAPES[name]
        return synth.cdc_streams(S, per, seed=seed)
    raise ValueError(name)


# content-defined chunking workloads: (streams, tokens per stream)
CDC_SHAPES = {"cdc_4M": (64, 1 << 16), "cdc_16M": (256, 1 << 16)}
CDC_VOCAB = 102400


DESCR = {
    "v2lite_decode": "DeepSeek-V2-Lite-shaped decode: 16 heads, batch 8, ctx 8192, 1 query/request, "
                     "chunks geometric mean 128 in [32,512], 75% reused, delta ~ U[-4096,4096]",
    "v3_decode": "DeepSeek-V3-shaped decode: 128 heads, batch 64, ctx 32768, 256 shared pool "
                 "chunks in shuffled order (~80% of tokens), delta ~ U[-16384,16384]",
    "chunked_prefill": "chunked prefill: 128 heads, 4 requests, 2048 causal queries over a "
                       "16384-token prefix (4096 exact-prefix delta=0, 12288 moved delta ~ U[-8192,8192])",
    "chunked_prefill_256": "profiling-size slice of the chunked prefill: the same prefix, 256 new "
                           "causal queries per request",
    "cdc_4M": "content-defined chunking of 64 token streams x 65536 tokens (shared documents at "
              "shifting offsets, vocab 102400): Gear hash (SplitMix64 Gear words), [32,512] "
              "chunks, xxHash64 fingerprints",
    "cdc_16M": "content-defined chunking of 256 token streams x 65536 tokens (as cdc_4M)",
}


def _fill_large(kv, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed + 101)
    step = 1 << 20
    for i in range(0, kv.shape[0], step):
        kv[i:i + step] = torch.randn(kv[i:i + step].shape, generator=g, device="cuda").to(torch.bfloat16)


class Workload:
    """Device-resident inputs and the C-ABI call of one step."""

    def __init__(self, name, seed=0):
        import mla_position_independent_gb300 as irm
        self.irm = irm
        self.name = name
        if name.startswith("cdc_"):
            from mla_position_independent_gb300 import synth
            tokens, offsets = _prep_case(name, seed)
            self.kind = "cdc"
            self.tokens = torch.from_numpy(tokens).cuda()
            self.offsets = offsets
            self.offsets_dev = torch.from_numpy(offsets.copy()).cuda()
            self.gear = None  # Gear words generated from SplitMix64 (no table lookups)
            nbytes, slots = irm.cdc_sizes(offsets)
            self.ws = irm.new_workspace(nbytes)
            S = offsets.shape[0] - 1
            self.cdc_out = (torch.empty(S, dtype=torch.int32, device="cuda"),
                            torch.empty(slots, dtype=torch.int32, device="cuda"),
                            torch.empty(slots, dtype=torch.int32, device="cuda"),
                            torch.empty(slots, dtype=torch.int64, device="cuda"))
            self.ctx_total = int(offsets[-1])
            self.n_tokens = self.ctx_total
            # algorithmic bytes: every token id read once (4 B); the chunk records written
            # (start, len, fingerprint: 16 B) for ~n/156 chunks
            self.bytes = 4 * self.n_tokens + 16 * (self.n_tokens // 156)
            self.flops = 0.0
            self.table = None
            return
        case = _prep_case(name, seed)
        if name.startswith("rotate_gather_"):
            _fill_large(case.kv_rows, seed)
        self.case = case
        self.table = irm.ChunkTable(case.chunks, case.indptr)
        ctx = case.ctx
        self.ctx_total = int(ctx.sum())
        self.kind = ("gather" if name.startswith("rotate_gather_") else
                     "prefill" if case.n_q > 1 else "decode")
        if self.kind == "decode":
            self.q_lat = case.q_lat[:, 0].contiguous()
            self.q_rope = case.q_rope[:, 0].contiguous()
            B, H = self.q_lat.shape[:2]
            self.H = H
            self.out = torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda")
            self.lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
            self.ws = irm.new_workspace(irm.decode_workspace_size(self.table, H))
            self.S_split = None
            self.bytes = self.ctx_total * ROW_BYTES
            self.flops = float(self.ctx_total) * H * PAIR_FLOPS
        elif self.kind == "prefill":
            self.q_lat, self.q_rope = case.q_lat, case.q_rope
            B, n_q, H = self.q_lat.shape[:3]
            self.out = torch.empty((B, n_q, H, 512), dtype=torch.bfloat16, device="cuda")
            self.lse = torch.empty((B, n_q, H), dtype=torch.float32, device="cuda")
            self.ws = irm.new_workspace(irm.prefill_workspace_size(B, n_q, H))
            # causal pairs: query i at ctx-n_q+i sees ctx-n_q+i+1 keys
            pairs = sum(H * (n_q * (c - n_q) + n_q * (n_q + 1) // 2) for c in ctx)
            self.flops = float(pairs) * PAIR_FLOPS
            self.bytes = self.ctx_total * ROW_BYTES
        else:
            self.paged = torch.empty((case.n_pages, 64, 576), dtype=torch.bfloat16, device="cuda")
            self.page_table = torch.from_numpy(case.page_table).cuda()
            self.ws = irm.new_workspace(irm.assemble_kv_workspace_size(self.table.B))
            self.bytes = 2 * self.ctx_total * ROW_BYTES
            self.flops = 0.0

    def step(self, stream=None):
        irm = self.irm
        if self.kind == "cdc":
            irm.irm_cdc_chunk(self.tokens, self.offsets, self.gear, out=self.cdc_out,
                              workspace=self.ws, stream=stream, offsets_dev=self.offsets_dev,
                              vocab=CDC_VOCAB)
            return
        if self.kind == "decode":
            irm.irm_mla_attn_decode(self.q_lat, self.q_rope, self.table, self.case.kv_rows,
                                    out=self.out, lse=self.lse, workspace=self.ws, stream=stream)
        elif self.kind == "prefill":
            irm.irm_mla_attn_prefill(self.q_lat, self.q_rope, self.table, self.case.kv_rows,
                                     out=self.out, lse=self.lse, workspace=self.ws, stream=stream)
        else:
            irm.irm_assemble_kv(self.table, self.case.kv_rows, self.paged, self.page_table,
                                workspace=self.ws, stream=stream)

    def launches_per_step(self):
        if self.kind == "cdc":
            return 5  # base scans, hash + candidate bits, speculative walks, fix-up, fingerprints
        return 1  # one fused kernel per call (the split-KV merge runs inside it)

    def kernel_name(self):
        if self.kind == "cdc":
            return "cdc (5 kernels: base, hash, spec walk, fix-up, fingerprint)"
        if self.kind == "gather":
            return "rotate_gather_kernel"
        if self.kind == "decode" and self.H in (16, 32):
            return "mla_decode_kernel"  # split-KV decode for a few heads
        return "mla_attn_kernel"

    def check_status(self):
        self.irm.device_status(self.ws)


class L2Flush:
    """Untimed L2 flush between steps: write a buffer twice the size of L2, then read another
    one.  The read evicts the written (dirty) lines, so the timed step starts with an L2 that
    holds neither its inputs nor write-backs owed by the flush itself (the cold-cache state
    that ncu's cache control also gives a kernel)."""

    def __init__(self):
        self.wr = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.rd = torch.ones(L2_FLUSH_BYTES // 8, dtype=torch.int64, device="cuda")
        self.acc = torch.empty((), dtype=torch.int64, device="cuda")

    def __call__(self, i):
        self.wr.fill_(i & 0xff)
        torch.sum(self.rd, dim=0, out=self.acc)


L2_NOTE = ("flushed between steps (untimed): 256 MiB write, then 256 MiB read so that no "
           "dirty flush lines are written back inside the timed step")


def time_steps(wl: Workload, steps: int, warmup: int, use_graph=True):
    """Per-step CUDA-event time (ms) of `steps` steps, L2 flushed before each (untimed)."""
    stream = torch.cuda.current_stream()
    flush = L2Flush()
    for _ in range(max(warmup, 1)):
        wl.step()
    torch.cuda.synchronize()
    wl.check_status()
    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                wl.step(stream=side)
        stream.wait_stream(side)
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush(i)
        starts[i].record(stream)
        if graph is not None:
            graph.replay()
        else:
            wl.step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    wl.check_status()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def e2e_decode(wl: Workload, steps: int):
    """Decode through the public API from pinned host buffers: per step H2D of the queries
    and the chunk table, the call, D2H of the output; wall clock per step."""
    assert wl.kind == "decode"
    irm = wl.irm
    ql_h = wl.q_lat.cpu().pin_memory()
    qr_h = wl.q_rope.cpu().pin_memory()
    ch_h = torch.from_numpy(wl.table.chunks_host.view(np.uint8).copy()).pin_memory()
    out_h = torch.empty(wl.out.shape, dtype=torch.bfloat16).pin_memory()
    flush = L2Flush()
    times = []
    for i in range(steps + 3):
        flush(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        wl.q_lat.copy_(ql_h, non_blocking=True)
        wl.q_rope.copy_(qr_h, non_blocking=True)
        wl.table.chunks_dev.copy_(ch_h, non_blocking=True)
        irm.irm_mla_attn_decode(wl.q_lat, wl.q_rope, wl.table, wl.case.kv_rows, out=wl.out,
                                lse=wl.lse, workspace=wl.ws)
        out_h.copy_(wl.out, non_blocking=True)
        torch.cuda.synchronize()
        if i >= 3:
            times.append(time.perf_counter() - t0)
    h2d = ql_h.numel() * 2 + qr_h.numel() * 2 + ch_h.numel()
    d2h = out_h.numel() * 2
    return statistics.mean(times) * 1e3, h2d, d2h


def assemble_host(wl: Workload, rounds: int = 3):
    """Host-side chunk-table assembly (irm_registry_assemble) of the CDC workload's streams as
    requests, twice over (the second pass reuses the first one's chunks): requests and
    segments per second on one host thread."""
    irm = wl.irm
    wl.step()
    torch.cuda.synchronize()
    n_chunks, c_start, c_len, c_hash = (t.cpu().numpy() for t in wl.cdc_out)
    base = irm.cdc_slot_base(wl.offsets)
    tokens = wl.tokens.cpu().numpy()
    S = len(wl.offsets) - 1
    reqs = []
    for s in range(S):
        k = int(n_chunks[s])
        b0 = int(base[s])
        reqs.append((tokens[wl.offsets[s]:wl.offsets[s + 1]], c_start[b0:b0 + k], c_len[b0:b0 + k],
                     c_hash[b0:b0 + k].view(np.uint64)))
    best = None
    for _ in range(rounds):
        reg = irm.Registry(pool_rows=int(wl.offsets[-1]) + 1024, capacity=1 << 16)
        t0 = time.perf_counter()
        reused = 0
        for _pass in range(2):
            for tok, st, ln, hs in reqs:
                table, _ = reg.assemble(tok, 0, 0, st, ln, hs)
                reused += int(table["len"][table["reused"] == 1].sum())
        dt = time.perf_counter() - t0
        reg.close()
        best = dt if best is None else min(best, dt)
    segs = 2 * sum(len(r[1]) for r in reqs)
    return dict(requests_per_s=round(2 * S / best, 1), segments_per_s=round(segs / best, 1),
                ms_per_pass=round(best / 2 * 1e3, 3), reused_tokens_second_pass=reused // rounds,
                note="host, one thread, ctypes call per request included")


def roofline(wl: Workload, ms: float, pk):
    if wl.kind == "prefill":
        ach = wl.flops / (ms * 1e-3) / 1e12
        return dict(bound="tensor", achieved=round(ach, 2), peak=pk["bf16"], unit="TFLOP/s",
                    frac=round(ach / pk["bf16"], 4))
    ach = wl.bytes / (ms * 1e-3) / 1e9
    return dict(bound="hbm", achieved=round(ach, 1), peak=pk["hbm"], unit="GB/s",
                frac=round(ach / pk["hbm"], 4))


KERNEL_SOURCES = {
    "mla_decode_kernel": ["irm_decode.cu", "irm_pipeline.cuh", "irm_common.cuh", "ptx.cuh", "irm_internal.h"],
    "mla_attn_kernel": ["irm_attn.cu", "irm_pipeline.cuh", "irm_common.cuh", "ptx.cuh", "irm_internal.h"],
    "rotate_gather_kernel": ["irm_gather.cu", "irm_common.cuh", "ptx.cuh", "irm_internal.h"],
}


def kernel_digest(kernel=None):
    """Digest of the sources a kernel is built from (all of csrc/ when kernel is None)."""
    csrc = os.path.join(ROOT, "mla_position_independent_gb300", "csrc")
    files = KERNEL_SOURCES.get(kernel) or sorted(os.listdir(csrc))
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(name):
    """DRAM bytes per launch from the committed ncu summary, if its kernel's sources have not
    changed since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(name)
    if not ent or ent.get("kernel_digest") != kernel_digest(ent.get("kernel")):
        return None
    return ent.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------- oracle arm

def oracle_sample(name, budget_s=None, steps=None, warmup=0):
    """Times the fp64 oracle on (request, head) units of the workload; each unit assembles
    the request's rows and computes one head's attention.  Returns (GB/s-equivalent,
    seconds, units, threads) where one unit counts ctx*1152/H bytes (the GPU reads the KV
    once for all H heads)."""
    import oracle
    from mla_position_independent_gb300 import synth
    case = {"v2lite_decode": synth.v2lite_decode, "v3_decode": synth.v3_decode,
            "chunked_prefill": synth.chunked_prefill,
            "chunked_prefill_256": lambda seed: synth.chunked_prefill(seed, n_q=256)}[name](0)
    kv = synth.bits(case.kv_rows)
    ql, qr = synth.bits(case.q_lat), synth.bits(case.q_rope)
    B, n_q, H = ql.shape[:3]
    ctx = case.ctx
    rng = np.random.default_rng(0)
    units = [(b, n_q - 1, h) for b in range(B) for h in range(H)]
    rng.shuffle(units)
    done_bytes, t_total, n = 0.0, 0.0, 0
    i = 0
    while True:
        b, qi, h = units[i % len(units)]
        t0 = time.perf_counter()
        oracle.mla_attention(ql, qr, case.chunks, case.indptr, kv, 1 / math.sqrt(192),
                             select=np.array([[b, qi, h]]))
        dt = time.perf_counter() - t0
        if i >= warmup:
            t_total += dt
            done_bytes += ctx[b] * ROW_BYTES / H
            n += 1
        i += 1
        if steps is not None and n >= steps:
            break
        if budget_s is not None and t_total >= budget_s:
            break
    return done_bytes / t_total / 1e9, t_total, n, oracle.num_threads()


# --------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="v2lite_decode")
    ap.add_argument("--no-extras", action="store_true",
                    help="report only the selected workload")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing (profiling runs)")
    args = ap.parse_args()
    rank, world, local = dist_init()
    pk = peaks()

    if args.impl == "reference":
        if rank != 0:
            return
        steps = max(1, min(args.steps, 200))
        value, secs, n, thr = oracle_sample(args.workload, steps=steps, warmup=min(args.warmup, 2))
        line = dict(metric=METRIC, value=round(value, 4), unit="GB/s", n_gpus=args.gpus,
                    steps=args.steps, warmup=args.warmup, impl="reference",
                    ms_per_step=round(secs / n * 1e3, 3), higher_is_better=True,
                    scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
                    config=dict(workload=args.workload, description=DESCR.get(args.workload)),
                    cpu_baseline=dict(value=round(value, 4), unit="GB/s", cores=thr, kind="oracle",
                                      sample=f"{n} (request, head) units of {args.workload}, "
                                             f"each assembling the request's rows in fp64 and "
                                             f"computing one head's attention; bytes counted as "
                                             f"ctx*1152/H per unit"),
                    e2e=dict(value=round(value, 4), unit="GB/s", h2d_bytes_per_step=0,
                             d2h_bytes_per_step=0))
        print(json.dumps(line), flush=True)
        return

    import mla_position_independent_gb300 as irm
    irm.lib()
    wl = Workload(args.workload, seed=rank)
    barrier(world)
    torch.cuda.synchronize()
    clk = ClockSampler(local)
    per_step = time_steps(wl, args.steps, args.warmup)
    clocks = clk.stop()
    torch.cuda.synchronize()
    barrier(world)
    ms = statistics.mean(per_step)
    ms = max_over_ranks(ms, world)
    unit_val = wl.bytes if wl.kind != "prefill" else wl.flops
    if wl.kind == "prefill":
        value = world * wl.flops / (ms * 1e-3) / 1e12
        unit = "TFLOP/s"
    else:
        value = world * wl.bytes / (ms * 1e-3) / 1e9
        unit = "GB/s"
    rf = roofline(wl, ms, pk)
    rf["peak_source"] = pk["src"]
    rf["kernel"] = wl.kernel_name()
    rf["traffic"] = traffic_for(args.workload)
    e2e = None
    if wl.kind == "decode":
        e2e_ms, h2d, d2h = e2e_decode(wl, min(args.steps, 200))
        e2e = dict(value=round(world * wl.bytes / (e2e_ms * 1e-3) / 1e9, 2), unit=unit,
                   h2d_bytes_per_step=int(h2d), d2h_bytes_per_step=int(d2h),
                   ms_per_step=round(e2e_ms, 4),
                   note="wall clock per step: H2D of queries and chunk table from pinned host "
                        "memory, the C-ABI call, D2H of the output, synchronize")
    line = dict(metric=METRIC, value=round(value, 2), unit=unit, n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=round(ms, 5), higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="bf16", data="synthetic",
                config=dict(workload=args.workload, description=DESCR.get(args.workload),
                            requests=(wl.table.B if wl.table is not None else len(wl.offsets) - 1),
                            ctx_total=wl.ctx_total,
                            l2=L2_NOTE,
                            parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
                roofline=rf, e2e=e2e, gpu_launches=args.steps * wl.launches_per_step(),
                clocks=dict(sm_mhz=clocks["sm_mhz"], sm_max_mhz=clocks["sm_max_mhz"],
                            reasons=clocks["reasons"], samples=clocks["samples"]))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, secs, n, thr = oracle_sample("v2lite_decode" if wl.kind != "prefill" else args.workload,
                                        budget_s=12.0)
        line["cpu_baseline"] = dict(value=round(v, 4), unit="GB/s", cores=thr, kind="oracle",
                                    sample=f"{n} (request, head) units of v2lite_decode in "
                                           f"{secs:.1f} s; bytes counted as ctx*1152/H per unit")
    if not args.no_extras and world == 1:
        extras = {}
        steps_of = {"v3_decode": 50, "chunked_prefill": 5, "rotate_gather_1M": 50,
                    "rotate_gather_4M": 50, "rotate_gather_16M": 20, "rotate_gather_64M": 10,
                    "cdc_4M": 50}
        for name, st in steps_of.items():
            if name == args.workload:
                continue
            del wl
            wl = None
            torch.cuda.empty_cache()
            if name.startswith("rotate_gather_"):
                # row store + pages (2 x 1152 B per row), plus room for the L2 flush buffers
                n = int(name.split("_")[-1].rstrip("M")) << 20
                need = 2 * n * ROW_BYTES + (2 << 30)
                if torch.cuda.mem_get_info()[0] < need:
                    extras[name] = dict(skipped=f"needs {need / 1e9:.1f} GB of free device memory")
                    continue
            wl = Workload(name, seed=rank)
            t = statistics.mean(time_steps(wl, st, 3))
            r = roofline(wl, t, pk)
            r["kernel"] = wl.kernel_name()
            ent = dict(ms_per_step=round(t, 4), roofline=r, steps=st)
            if wl.kind == "gather":
                ent["rows_per_s"] = round(wl.ctx_total / (t * 1e-3), 1)
                ent["GB_per_s_moved"] = r["achieved"]
            elif wl.kind == "cdc":
                ent["tokens_per_s"] = round(wl.n_tokens / (t * 1e-3), 1)
            elif wl.kind == "decode":
                ent["logical_KV_GB_per_s"] = r["achieved"]
            else:
                ent["TFLOP_per_s"] = r["achieved"]
            ent["traffic"] = traffic_for(name)
            extras[name] = ent
            if wl.kind == "cdc":
                extras["assemble_host"] = assemble_host(wl)
        line["workloads"] = extras
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
