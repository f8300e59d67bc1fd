"""Benchmark of the reuse-time MLA KV reconstruction path on GB300.

Default (no flags): N=1, the DeepSeek-V2-Lite-shaped decode workload (16 heads, batch 8,
context 8192, 75% reused chunks with delta-rotation), reported as logical KV GB/s, plus
the other workloads (V3-shaped decode, chunked prefill, rotate+gather) in "workloads".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one pass of the whole hot path over one batch -- one call of the C ABI: the
copy of the validated host chunk table into the workspace, then the fused kernel
(chunk-table walk, per-chunk rotation angles, gather of [cKV | k_r] rows, delta-rotation
in shared memory, Q.K^T, online softmax, P.cKV, and the split-KV merge for decode).
Steps are timed with CUDA events on the launching stream, each step replayed from a CUDA
graph, with L2 flushed (256 MiB write then 256 MiB read, untimed) between steps.  Every
workload also gets an end-to-end figure (host buffers in, result back), its own clock
record, and the fp64 oracle timed on the host cores on a bounded sample of it.  The oracle
arm (--impl reference) times the oracle alone on the selected workload.
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
    if name == "tiny":
        return synth.tiny_case(seed, device="cuda")
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
# table sizes that the library passes in the kernel launch parameters (larger ones are copied
# into the workspace by one more kernel): chunk records and requests of an attention call,
# streams of a chunking call
INLINE_CHUNKS, INLINE_REQUESTS, CDC_INLINE_STREAMS = 1024, 256, 1024


DESCR = {
    "tiny": "tiny correctness case: 1 request, ctx 512 (carve-out + 4 reused chunks of 64/96/128/192 "
            "from a pool of 8), 16 causal queries x 16 heads",
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
for _n in ("1M", "4M", "16M", "64M"):
    DESCR[f"rotate_gather_{_n}"] = (f"rotate+gather of {_n} rows of [cKV 512 | k_r 64] bf16 from a chunk "
                                    "pool (geometric chunks, mean 128, [32,512]) into 64-row pages in "
                                    "random physical order, delta ~ U[-65536,65536] per chunk")


def _fill_large(kv, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed + 101)
    step = 1 << 20
    for i in range(0, kv.shape[0], step):
        kv[i:i + step] = torch.randn(kv[i:i + step].shape, generator=g, device="cuda").to(torch.bfloat16)


class Workload:
    """Device-resident inputs and the C-ABI call of one step.  The chunk table is the
    library's input in page-locked host memory: every call validates it and copies it into
    the workspace (inside the timed step)."""

    def __init__(self, name, seed=0):
        import mla_position_independent_gb300 as irm
        self.irm = irm
        self.name = name
        if name.startswith("cdc_"):
            tokens, offsets = _prep_case(name, seed)
            self.kind = "cdc"
            self.tokens = torch.from_numpy(tokens).cuda()
            # page-locked, so the library's copy of the offsets can be captured into the graph
            self._offsets_pinned = torch.from_numpy(offsets.copy()).pin_memory()
            self.offsets = self._offsets_pinned.numpy()
            self.gear = None  # Gear words generated from SplitMix64 (no table lookups)
            nbytes, slots = irm.cdc_sizes(self.offsets)
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
            self.bytes = self.ctx_total * ROW_BYTES
            self.flops = float(self.ctx_total) * H * PAIR_FLOPS
        elif self.kind == "prefill":
            self.q_lat, self.q_rope = case.q_lat, case.q_rope
            B, n_q, H = self.q_lat.shape[:3]
            self.H = H
            self.out = torch.empty((B, n_q, H, 512), dtype=torch.bfloat16, device="cuda")
            self.lse = torch.empty((B, n_q, H), dtype=torch.float32, device="cuda")
            self.ws = irm.new_workspace(irm.prefill_workspace_size(self.table, n_q, H))
            # causal pairs: query i at ctx-n_q+i sees ctx-n_q+i+1 keys
            pairs = sum(H * (n_q * (c - n_q) + n_q * (n_q + 1) // 2) for c in ctx)
            self.flops = float(pairs) * PAIR_FLOPS
            self.bytes = self.ctx_total * ROW_BYTES
        else:
            self.paged = torch.empty((case.n_pages, 64, 576), dtype=torch.bfloat16, device="cuda")
            self.page_table = torch.from_numpy(case.page_table).cuda()
            self.ws = irm.new_workspace(irm.assemble_kv_workspace_size(self.table))
            self.bytes = 2 * self.ctx_total * ROW_BYTES
            self.flops = 0.0
        self.table_bytes = int(self.table._buf.numel())

    def step(self, stream=None):
        irm = self.irm
        if self.kind == "cdc":
            irm.irm_cdc_chunk(self.tokens, self.offsets, self.gear, out=self.cdc_out,
                              workspace=self.ws, stream=stream, vocab=CDC_VOCAB)
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
        """Kernels of this library that one step launches."""
        if self.kind == "cdc":
            # segment hashing + speculative walks, resolve; a batch of more than 1024 streams
            # adds the kernel that scans the stream offsets on the device
            return 2 + (len(self.offsets) - 1 > CDC_INLINE_STREAMS)
        if self.kind == "gather":
            return 2  # the table copy into the workspace, the rotate+gather kernel
        # one fused kernel (the split-KV merge runs inside it); a table of more than 1024
        # records or 256 requests is copied into the workspace by one more kernel
        inline = self.table.n_chunks <= INLINE_CHUNKS and self.table.B <= INLINE_REQUESTS
        return 1 if inline else 2

    def kernel_name(self):
        if self.kind == "cdc":
            return "cdc_segment_kernel + cdc_resolve_kernel"
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
    """Per-step CUDA-event time (ms) of `steps` steps, L2 flushed before each (untimed).  A
    step (the C-ABI call: the chunk-table copy into the workspace and the kernel launch) is
    captured once into a CUDA graph and replayed."""
    stream = torch.cuda.current_stream()
    flush = L2Flush()
    for _ in range(max(warmup, 3)):
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


def timed(wl: Workload, steps: int, warmup: int, device_index: int):
    """time_steps with nvidia-smi clock samples taken during the timed region."""
    clk = ClockSampler(device_index)
    per_step = time_steps(wl, steps, warmup)
    clocks = clk.stop()
    return per_step, dict(sm_mhz=clocks["sm_mhz"], sm_max_mhz=clocks["sm_max_mhz"],
                          reasons=clocks["reasons"], samples=clocks["samples"])


def _cudart():
    """The CUDA runtime already loaded by torch (for plain cudaMemcpyAsync calls in the
    end-to-end loop, which avoid torch's per-copy dispatch), or None."""
    import ctypes
    for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
        except OSError:
            continue
        rt.cudaMemcpyAsync.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                                       ctypes.c_void_p]
        rt.cudaMemcpyAsync.restype = ctypes.c_int
        return rt
    return None


def e2e(wl: Workload, steps: int):
    """The step end to end through the C ABI with host buffers, wall clock per step: H2D of
    the step's inputs from page-locked host memory (queries; the page table for
    rotate+gather), the C-ABI call (which validates the host chunk table and copies it into
    the workspace), and the read-back of the step's result (the attention output; for
    rotate+gather, whose output stays on the device as the paged cache, its status word),
    then a synchronize.  L2 is flushed (untimed) before each step.  Returns (ms per step,
    H2D bytes, D2H bytes)."""
    import ctypes
    irm = wl.irm
    L = irm.lib()
    stream = torch.cuda.current_stream()
    sp = ctypes.c_void_p(stream.cuda_stream)
    t = wl.table
    ch, ip = t.chunks_host.ctypes.data, t.indptr_host.ctypes.data
    ws = wl.ws
    if wl.kind in ("decode", "prefill"):
        nl, nr = wl.q_lat.numel(), wl.q_rope.numel()
        dq = torch.empty(nl + nr, dtype=torch.bfloat16, device="cuda")  # [q_lat | q_rope]
        hq = torch.empty(nl + nr, dtype=torch.bfloat16).pin_memory()
        hq[:nl].copy_(wl.q_lat.reshape(-1).cpu())
        hq[nl:].copy_(wl.q_rope.reshape(-1).cpu())
        hout = torch.empty(wl.out.shape, dtype=torch.bfloat16).pin_memory()
        ql, qr = dq.data_ptr(), dq.data_ptr() + 2 * nl
        scale = ctypes.c_float(1.0 / math.sqrt(192.0))
        kv, n_rows = wl.case.kv_rows.data_ptr(), int(wl.case.kv_rows.shape[0])
        if wl.kind == "decode":
            B, H = wl.q_lat.shape[:2]
            args = (ql, qr, B, H, ch, ip, kv, n_rows, scale, wl.out.data_ptr(), None, ws.data_ptr(),
                    ws.numel(), sp)
            call = L.irm_mla_attn_decode
        else:
            B, n_q, H = wl.q_lat.shape[:3]
            args = (ql, qr, B, n_q, H, ch, ip, kv, n_rows, scale, wl.out.data_ptr(), None,
                    ws.data_ptr(), ws.numel(), sp)
            call = L.irm_mla_attn_prefill

        args = tuple(ctypes.c_void_p(x) if isinstance(x, int) and x > (1 << 32) else x for x in args)
        rt = _cudart()
        qb, ob = hq.numel() * 2, hout.numel() * 2
        cp_args = (ctypes.c_void_p(dq.data_ptr()), ctypes.c_void_p(hq.data_ptr()), ctypes.c_size_t(qb), 1, sp)
        back_args = (ctypes.c_void_p(hout.data_ptr()), ctypes.c_void_p(wl.out.data_ptr()), ctypes.c_size_t(ob), 2, sp)

        def one():
            if rt is not None:
                rt.cudaMemcpyAsync(*cp_args)
            else:
                dq.copy_(hq, non_blocking=True)
            st = call(*args)
            if st != 0:
                raise RuntimeError(L.irm_last_error().decode())
            if rt is not None:
                rt.cudaMemcpyAsync(*back_args)
            else:
                hout.copy_(wl.out, non_blocking=True)
            stream.synchronize()
        h2d = hq.numel() * 2 + wl.table_bytes
        d2h = hout.numel() * 2
    else:
        hpt = torch.from_numpy(wl.case.page_table.copy()).pin_memory()
        kv = wl.case.kv_rows
        args = (ch, ip, t.B, kv.data_ptr(), int(kv.shape[0]), wl.paged.data_ptr(),
                int(wl.paged.shape[0]), wl.page_table.data_ptr(), int(wl.page_table.shape[1]),
                None, None, None, ws.data_ptr(), ws.numel(), sp)

        def one():
            wl.page_table.copy_(hpt, non_blocking=True)
            st = L.irm_assemble_kv(*args)
            if st != 0:
                raise RuntimeError(L.irm_last_error().decode())
            if L.irm_device_status(ws.data_ptr(), sp) != 0:  # reads the status word, synchronizes
                raise RuntimeError(L.irm_last_error().decode())
        h2d = hpt.numel() * 4 + wl.table_bytes
        d2h = 4
    flush = L2Flush()
    times = []
    for i in range(steps + 3):
        flush(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        one()
        if i >= 3:
            times.append(time.perf_counter() - t0)
    wl.check_status()
    if wl.kind in ("decode", "prefill") and not torch.equal(hout, wl.out.cpu()):
        raise RuntimeError("end-to-end loop: the output read back differs from the device output")
    return statistics.median(times) * 1e3, int(h2d), int(d2h)


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


# Content-defined chunking is integer arithmetic.  Its algorithmic work, in 32-bit integer
# operations per token: the SplitMix64 Gear word (a 64 x 32-bit multiply-add 2, the seed add 2,
# three 64-bit xor-shifts 4 each, two 64 x 64-bit multiplies 3 each: 22), the Gear step
# h = 2 h + G (shift 2, add 2), the boundary test (2), and an eighth of an xxHash64 stripe
# (four lanes of multiply 3, add 2, rotate 2, multiply 3 per 32 bytes: 5 per token): 33.
CDC_INT_OPS_PER_TOKEN = 33
# Its peak: every scheduler issuing one 32-bit integer instruction for 32 lanes each clock,
# 152 SMs x 4 schedulers x 32 lanes x 2070 MHz (the maximum SM clock).
ALU_PEAK_GOPS = 152 * 4 * 32 * 2.07
ALU_PEAK_NOTE = "derived: 152 SMs x 4 schedulers x 32 lanes x 2070 MHz, one 32-bit integer op per lane per clock"


def roofline(wl: Workload, ms: float, pk):
    if wl.kind == "cdc":
        ach = CDC_INT_OPS_PER_TOKEN * wl.n_tokens / (ms * 1e-3) / 1e9
        return dict(bound="alu", achieved=round(ach, 1), peak=round(ALU_PEAK_GOPS, 1), unit="Gop/s",
                    frac=round(ach / ALU_PEAK_GOPS, 4), peak_source=ALU_PEAK_NOTE,
                    ops_per_token=CDC_INT_OPS_PER_TOKEN)
    if wl.kind == "prefill":
        ach = wl.flops / (ms * 1e-3) / 1e12
        return dict(bound="tensor", achieved=round(ach, 2), peak=pk["bf16"], unit="TFLOP/s",
                    frac=round(ach / pk["bf16"], 4))
    ach = wl.bytes / (ms * 1e-3) / 1e9
    r = dict(bound="hbm", achieved=round(ach, 1), peak=pk["hbm"], unit="GB/s",
             frac=round(ach / pk["hbm"], 4))
    if wl.kind == "decode":
        # decode also runs the two contractions on the tensor cores (2176 flop per (head, key));
        # with shared pool chunks served from L2 (V3-shaped decode) that can be the tighter bound
        tf = wl.flops / (ms * 1e-3) / 1e12
        r["tensor"] = dict(achieved=round(tf, 2), peak=pk["bf16"], unit="TFLOP/s",
                           frac=round(tf / pk["bf16"], 4))
    return r


KERNEL_SOURCES = {
    "mla_decode_kernel": ["irm_decode.cu", "irm_pipeline.cuh", "irm_common.cuh", "ptx.cuh", "irm_internal.h"],
    "mla_attn_kernel": ["irm_attn.cu", "irm_pipeline.cuh", "irm_common.cuh", "ptx.cuh", "irm_internal.h"],
    "rotate_gather_kernel": ["irm_gather.cu", "irm_common.cuh", "ptx.cuh", "irm_internal.h"],
    "cdc_segment_kernel + cdc_resolve_kernel": ["irm_cdc.cu", "irm_common.cuh", "irm_internal.h"],
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

def _host_cores():
    try:
        aff = len(os.sched_getaffinity(0))
    except AttributeError:
        aff = os.cpu_count()
    return os.cpu_count(), aff


_ORACLE_CASES = {}


def _oracle_case(name):
    """Inputs of a workload on the host (generated once per process)."""
    key = "rotate_gather" if name.startswith("rotate_gather_") else name
    if key not in _ORACLE_CASES:
        _ORACLE_CASES.clear()
        _ORACLE_CASES[key] = _make_oracle_case(name)
    return _ORACLE_CASES[key]


def _make_oracle_case(name):
    from mla_position_independent_gb300 import synth
    import oracle
    if name == "tiny":
        case = synth.tiny_case(0)
        enc = oracle.rotate(case.rope_content, case.rope_pos)
        case.kv_rows[torch.as_tensor(case.rope_rows), 512:] = torch.from_numpy(enc).to(torch.bfloat16)
    elif name.startswith("rotate_gather_"):
        case = synth.rotate_gather_case(1 << 20, 0)
    else:
        case = {"v2lite_decode": synth.v2lite_decode, "v3_decode": synth.v3_decode,
                "chunked_prefill": synth.chunked_prefill,
                "chunked_prefill_256": lambda seed: synth.chunked_prefill(seed, n_q=256)}[name](0)
    kv = synth.bits(case.kv_rows)
    ql = qr = None
    if case.q_lat is not None:
        ql, qr = synth.bits(case.q_lat), synth.bits(case.q_rope)
    return case, kv, ql, qr


def _oracle_units(name, case):
    """The oracle's units of work on a workload and the algorithmic amount each stands for
    (the GPU metric's unit: KV bytes for decode, flops for prefill, bytes moved for
    rotate+gather).  Decode: one request with all its heads in one call (the oracle
    assembles the request once and runs its H query rows in parallel).  Prefill: one
    request with 8 query positions (always the first and the last) x 16 heads.  Tiny: the
    whole case.  Rotate+gather: the whole 1M-row table."""
    rng = np.random.default_rng(0)
    if name.startswith("rotate_gather_"):
        return [("gather", None, 2.0 * int(case.ctx.sum()) * ROW_BYTES)], "GB/s", 1e9
    B, n_q, H = case.q_lat.shape[:3]
    ctx = case.ctx
    if name == "tiny":
        sel = np.stack(np.meshgrid([0], np.arange(n_q), np.arange(H), indexing="ij"), -1).reshape(-1, 3)
        return [("attn", sel, _attn_amount(case, sel))], "TFLOP/s", 1e12
    if n_q == 1:
        units = []
        for b in rng.permutation(B):
            sel = np.array([[b, 0, h] for h in range(H)])
            units.append(("attn", sel, _attn_amount(case, sel)))
        return units, "GB/s", 1e9
    units = []
    for b in rng.permutation(B):
        qs = np.unique(np.concatenate([[0, n_q - 1], rng.choice(n_q, 6, replace=False)]))
        hs = rng.choice(H, 16, replace=False)
        sel = np.array([[b, i, h] for i in qs for h in hs])
        units.append(("attn", sel, _attn_amount(case, sel)))
    return units, "TFLOP/s", 1e12


def _attn_amount(case, sel):
    """What the selected (b, i, h) rows stand for in the GPU metric: decode reads each KV row
    once for all H heads, so a row counts ctx_b * 1152 / H bytes; prefill counts the flops of
    its visible keys."""
    B, n_q, H = case.q_lat.shape[:3]
    ctx = case.ctx
    if n_q == 1:
        return float(sum(ctx[b] for b in sel[:, 0])) * ROW_BYTES / H
    return float(sum(ctx[b] - n_q + i + 1 for b, i in sel[:, :2])) * PAIR_FLOPS


def oracle_sample(name, budget_s=10.0, max_units=None, threads=None):
    """Times the fp64 oracle, as it stands, on units of a workload (see _oracle_units), until
    `budget_s` seconds or `max_units` units.  Returns dict(value, unit, seconds, units,
    threads, sample)."""
    import oracle
    from mla_position_independent_gb300 import synth
    oracle.build()
    if threads is not None:
        oracle.set_num_threads(threads)
    case, kv, ql, qr = _oracle_case(name)
    units, unit, div = _oracle_units(name, case)
    if threads == 1:
        if name.startswith("rotate_gather_"):
            # one thread: the first 65536 target rows (the whole table would take minutes)
            rows = np.stack([np.zeros(1 << 16, np.int64), np.arange(1 << 16)], 1)
            units = [("gather_rows", rows, 2.0 * (1 << 16) * ROW_BYTES)]
        elif name != "tiny":
            # one thread: 16 rows of the first unit
            sel = units[0][1][:16]
            units = [("attn", sel, _attn_amount(case, sel))]
    done, secs, n, i = 0.0, 0.0, 0, 0
    while True:
        kind, sel, amount = units[i % len(units)]
        t0 = time.perf_counter()
        if kind == "gather":
            oracle.rotate_gather(kv, case.chunks, case.indptr, case.page_table)
        elif kind == "gather_rows":
            oracle.rotate_gather(kv, case.chunks, case.indptr, case.page_table, rows=sel)
        else:
            oracle.mla_attention(ql, qr, case.chunks, case.indptr, kv, 1 / math.sqrt(192), select=sel)
        secs += time.perf_counter() - t0
        done += amount
        n += 1
        i += 1
        if max_units is not None and n >= max_units:
            break
        if secs >= budget_s or (name == "tiny" and n >= 1) or kind.startswith("gather"):
            break
    thr = oracle.num_threads()
    return dict(value=done / secs / div, unit=unit, seconds=secs, units=n, threads=thr)


def cpu_baseline(name, budget_s=8.0, one_thread_budget_s=3.0):
    """The oracle on the host cores (all of them, then one thread) on a bounded sample of a
    workload; the figures are per unit of the GPU metric, extrapolated where the sample is
    a subset."""
    import oracle
    ncpu, aff = _host_cores()
    full = oracle_sample(name, budget_s=budget_s, threads=aff)
    one = oracle_sample(name, budget_s=one_thread_budget_s, max_units=1, threads=1)
    oracle.set_num_threads(aff)
    what = {"tiny": "the whole case (16 queries x 16 heads)",
            "v2lite_decode": "whole requests (all 16 heads each)",
            "v3_decode": "whole requests (all 128 heads each) of the 64; extrapolated to the batch",
            "chunked_prefill": "(request, 8 query positions incl. the first and last, 16 heads) "
                               "units; extrapolated per flop to the whole prefill"}
    if name.startswith("rotate_gather_"):
        samp = "the whole 1M-row rotate+gather" + ("" if name == "rotate_gather_1M" else
                                                   f"; extrapolated per row to {name[14:]} rows")
    else:
        samp = f"{full['units']} units: {what.get(name, name)}"
    return dict(value=round(full["value"], 6), unit=full["unit"], cores=full["threads"],
                threads_used=full["threads"], host_cpus=ncpu, affinity=aff, kind="oracle",
                sample=f"{samp}; {full['seconds']:.1f} s of oracle time",
                one_thread=dict(value=round(one["value"], 6), unit=one["unit"],
                                seconds=round(one["seconds"], 2), units=one["units"]),
                extrapolated=name not in ("tiny", "v2lite_decode", "rotate_gather_1M"))


# --------------------------------------------------------------------------- main

# extra workloads reported beside the headline: timed steps each
EXTRA_STEPS = {"tiny": 200, "v3_decode": 100, "chunked_prefill": 20, "rotate_gather_1M": 100,
               "rotate_gather_4M": 50, "rotate_gather_16M": 20, "rotate_gather_64M": 20,
               "cdc_4M": 100}
E2E_STEPS = {"decode": 200, "prefill": 5, "gather": 20}


def _value_unit(wl, ms):
    if wl.kind == "prefill":
        return wl.flops / (ms * 1e-3) / 1e12, "TFLOP/s"
    return wl.bytes / (ms * 1e-3) / 1e9, "GB/s"


def measure(name, steps, warmup, pk, device_index, rank, want_cpu, want_e2e=True):
    """One workload: device-timed steps with their clock record, the roofline of its kernel,
    the end-to-end figure through the C ABI, and the oracle on the host cores."""
    wl = Workload(name, seed=rank)
    per_step, clocks = timed(wl, steps, warmup, device_index)
    ms = statistics.mean(per_step)
    val, unit = _value_unit(wl, ms)
    ent = dict(value=round(val, 4), unit=unit, ms_per_step=round(ms, 5), steps=steps,
               clocks=clocks, description=DESCR.get(name))
    r = roofline(wl, ms, pk)
    r["kernel"] = wl.kernel_name()
    r["traffic"] = traffic_for(name)
    ent["roofline"] = r
    if wl.kind != "cdc":
        ent["table_bytes"] = wl.table_bytes
    if wl.kind == "gather":
        ent["rows_per_s"] = round(wl.ctx_total / (ms * 1e-3), 1)
    elif wl.kind == "cdc":
        ent["tokens_per_s"] = round(wl.n_tokens / (ms * 1e-3), 1)
        ent["hbm_frac"] = round(wl.bytes / (ms * 1e-3) / 1e9 / pk["hbm"], 4)
        ent["assemble_host"] = assemble_host(wl)
    if want_e2e and wl.kind in E2E_STEPS:
        e_ms, h2d, d2h = e2e(wl, E2E_STEPS[wl.kind])
        ev, _ = _value_unit(wl, e_ms)
        ent["e2e"] = dict(value=round(ev, 4), unit=unit, h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h,
                          ms_per_step=round(e_ms, 4), ratio_to_device_step=round(e_ms / ms, 3),
                          note="median wall clock per step: H2D of the step's inputs from "
                               "page-locked host memory, the C-ABI call (host chunk table "
                               "validated and copied into the workspace), read-back of the "
                               "result, synchronize")
    lp = wl.launches_per_step()
    del wl
    torch.cuda.empty_cache()
    if want_cpu and not name.startswith("cdc_"):
        ent["cpu_baseline"] = cpu_baseline(name)
    return ent, lp


def run_config(name, world):
    """The `config` of the JSON line (the same for the GPU arm and the oracle arm)."""
    return dict(workload=name, description=DESCR.get(name),
                step="one C-ABI call: chunk-table copy into the workspace + the fused kernel(s), "
                     "replayed from a CUDA graph",
                l2=L2_NOTE, parallelism=f"replicas x{world}" if world > 1 else "single GPU")


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
        import oracle
        ncpu, aff = _host_cores()
        oracle.build()
        oracle.set_num_threads(aff)
        # a step is one oracle unit of the workload (a whole request for decode); K steps, or
        # as many as fit in about two minutes (the line reports how many ran)
        steps = max(1, args.steps)
        if args.warmup > 0:
            oracle_sample(args.workload, budget_s=5.0, max_units=min(args.warmup, 2))
        r = oracle_sample(args.workload, budget_s=120.0, max_units=steps)
        line = dict(metric=METRIC, value=round(r["value"], 6), unit=r["unit"], n_gpus=args.gpus,
                    steps=r["units"], warmup=min(args.warmup, 2), impl="reference",
                    ms_per_step=round(r["seconds"] / r["units"] * 1e3, 3), higher_is_better=True,
                    scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
                    config=run_config(args.workload, world=1),
                    cpu_baseline=dict(value=round(r["value"], 6), unit=r["unit"], cores=r["threads"],
                                      host_cpus=ncpu, affinity=aff, kind="oracle",
                                      sample=f"{r['units']} oracle units of {args.workload} "
                                             f"({r['seconds']:.1f} s); a unit is a whole request "
                                             f"with all its heads for decode, (request, 8 query "
                                             f"positions, 16 heads) for prefill"),
                    e2e=dict(value=round(r["value"], 6), unit=r["unit"], h2d_bytes_per_step=0,
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
    val, unit = _value_unit(wl, ms)
    value = world * val
    rf = roofline(wl, ms, pk)
    rf.setdefault("peak_source", pk["src"])
    rf["kernel"] = wl.kernel_name()
    rf["traffic"] = traffic_for(args.workload)
    e2e_d = None
    if wl.kind in E2E_STEPS:
        e_ms, h2d, d2h = e2e(wl, min(args.steps, E2E_STEPS[wl.kind]))
        e_ms = max_over_ranks(e_ms, world)
        ev, _ = _value_unit(wl, e_ms)
        e2e_d = dict(value=round(world * ev, 2), unit=unit, h2d_bytes_per_step=h2d,
                     d2h_bytes_per_step=d2h, ms_per_step=round(e_ms, 4),
                     ratio_to_device_step=round(e_ms / ms, 3),
                     note="median wall clock per step: H2D of the queries from page-locked host "
                          "memory, the C-ABI call (host chunk table validated and copied into "
                          "the workspace, kernel launch), D2H of the output, synchronize")
    line = dict(metric=METRIC, value=round(value, 2), unit=unit, n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=round(ms, 5), higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="bf16", data="synthetic",
                config=run_config(args.workload, world),
                roofline=rf, e2e=e2e_d, gpu_launches=args.steps * wl.launches_per_step(),
                clocks=dict(sm_mhz=clocks["sm_mhz"], sm_max_mhz=clocks["sm_max_mhz"],
                            reasons=clocks["reasons"], samples=clocks["samples"]))
    del wl
    torch.cuda.empty_cache()
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    if want_cpu:
        line["cpu_baseline"] = cpu_baseline(args.workload)
    if not args.no_extras and world == 1:
        extras = {}
        for name, st in EXTRA_STEPS.items():
            if name == args.workload:
                continue
            if name.startswith("rotate_gather_"):
                # row store + pages (2 x 1152 B per row), plus room for the L2 flush buffers
                n = int(name.split("_")[-1].rstrip("M")) << 20
                need = 2 * n * ROW_BYTES + (2 << 30)
                if torch.cuda.mem_get_info()[0] < need:
                    extras[name] = dict(skipped=f"needs {need / 1e9:.1f} GB of free device memory")
                    continue
            ent, _ = measure(name, st, 3, pk, local, rank, want_cpu)
            extras[name] = ent
        line["workloads"] = extras
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
