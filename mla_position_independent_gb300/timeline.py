"""Where the time of a split-KV decode step goes: launch, ramp, steady state and merge.

    python -m mla_position_independent_gb300.timeline [--reps 9]

Runs the DeepSeek-V2-Lite-shaped decode (16 heads, batch 8, context 8192) on cuda:0 with the
timeline build of the library (libirm_timeline.so: the product kernels plus %globaltimer
stamps from the CTAs of request 0) and prints, as medians over the repetitions:
  - the event-timed step (CUDA graph replay after an untimed L2 flush, as bench.py times it)
    and the same for a graph holding one trivial kernel: the launch floor of any one-kernel
    step;
  - the kernel span (first CTA entry to last CTA end) and its phases: set-up, first tile's
    data landed, its scores issued, the steady-state period per tile, the pipeline end,
    the in-cluster merge and the end (after the cross-cluster merge);
  - the set-up's steps, each from its CTA's own entry: the split's chunk range known (launch
    arguments read), TMEM allocated, tile 0's row map built, its copies issued.
The stamps cost a few global stores per phase; the step times come from the same build.
"""
from __future__ import annotations

import argparse
import ctypes
import statistics

import numpy as np
import torch

from . import binding, build, synth

N_CTAS, N_TILES, N_EV = 64, 64, 11
EV = ["entry", "setup", "pipe_end", "parked", "cluster_barrier", "cluster_merged", "end",
      "split_known", "tmem_allocated", "tile0_map_built", "tile0_copies_issued"]


def _graph(fn, stream):
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            fn(side)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    return g


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--reps", type=int, default=9)
    args = ap.parse_args()
    binding._LIB_PATH = build.build(timeline=True)
    binding._lib = None
    L = binding.lib()
    L.irm_timeline_read.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    L.irm_timeline_read.restype = ctypes.c_int
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    case = synth.v2lite_decode(0, device="cuda")
    table = binding.ChunkTable(case.chunks, case.indptr)
    ql, qr = case.q_lat[:, 0].contiguous(), case.q_rope[:, 0].contiguous()
    B, H = ql.shape[:2]
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda")
    ws = binding.new_workspace(binding.decode_workspace_size(table, H))

    def step(s=None):
        binding.irm_mla_attn_decode(ql, qr, table, case.kv_rows, out=out, workspace=ws, stream=s)

    wr = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    rd = torch.ones(32 << 20, dtype=torch.int64, device="cuda")
    acc = torch.empty((), dtype=torch.int64, device="cuda")

    def flush(i):
        wr.fill_(i & 0xff)
        torch.sum(rd, dim=0, out=acc)

    for _ in range(5):
        step()
    torch.cuda.synchronize()
    tiny = torch.zeros(1024, device="cuda")
    g_dec = _graph(lambda s: step(s), stream)
    g_tiny = _graph(lambda s: tiny.add_(1), stream)

    def event_time(g, n=200):
        ts = []
        for i in range(n):
            flush(i)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            ts.append((a, b))
        torch.cuda.synchronize()
        return statistics.median(x.elapsed_time(y) * 1e3 for x, y in ts)

    t_step, t_floor = event_time(g_dec), event_time(g_tiny)
    cta = np.zeros((N_CTAS, N_EV), np.uint64)
    tile = np.zeros((N_CTAS, N_TILES, 3), np.uint64)
    binding._check(L.irm_timeline_read(cta.ctypes.data, tile.ctypes.data))  # clear
    rows = []
    for r in range(args.reps):
        flush(r)
        torch.cuda.synchronize()
        g_dec.replay()
        torch.cuda.synchronize()
        binding._check(L.irm_timeline_read(cta.ctypes.data, tile.ctypes.data))
        n = int((cta[:, 0] > 0).sum())
        c = cta[:n].astype(np.int64)
        t = tile[:n].astype(np.int64)
        t0 = c[:, 0].min()
        us = lambda x: (x - t0) / 1e3
        nt = int((t[0, :, 1] > 0).sum())
        s_issue = np.median(us(t[:, :nt, 1]), axis=0)  # per tile, median over CTAs
        period = float(np.median(np.diff(s_issue[1:]))) if nt > 2 else float("nan")
        own = lambda j: float(np.median((c[:, j] - c[:, 0]) / 1e3))  # from each CTA's own entry
        rows.append(dict(split_known=own(7), tmem=own(8), map=own(9), issued=own(10), setup_own=own(1),
                         entry_skew=float(np.median(us(c[:, 0]))),
                         span=us(c[:, 6].max()), setup=np.median(us(c[:, 1])),
                         first_landed=np.median(us(t[:, 0, 0])), first_scores=s_issue[0],
                         period=period, tiles=nt, pipe_end=np.median(us(c[:, 2])),
                         pipe_end_max=us(c[:, 2].max()), cluster=np.median(us(c[:, 4])),
                         merged=np.median(us(c[:, 5])), end=us(c[:, 6].max()), ctas=n))
    med = {k: statistics.median(r[k] for r in rows) for k in rows[0]}
    print(f"V2-Lite decode (B={B}, H={H}, ctx 8192), {args.reps} traced steps, medians (us)")
    print(f"  event-timed step (graph, L2 flushed)      {t_step:8.2f}")
    print(f"  one-kernel graph step floor (trivial)     {t_floor:8.2f}")
    print(f"  kernel span: first CTA entry -> last end  {med['span']:8.2f}")
    print(f"  phases of request 0's {int(med['ctas'])} CTAs, from the first entry:")
    for k, lab in (("setup", "set-up done"), ("first_landed", "tile 0 data landed"),
                   ("first_scores", "tile 0 scores issued"), ("pipe_end", "pipeline end (median CTA)"),
                   ("pipe_end_max", "pipeline end (slowest CTA)"), ("cluster", "cluster barrier passed"),
                   ("merged", "in-cluster merge done"), ("end", "end (after cross-cluster merge)")):
        print(f"    {lab:<38}{med[k]:8.2f}")
    print(f"  steady state: {med['period']:.2f} us per 64-row tile over {int(med['tiles'])} tiles per CTA")
    print(f"  set-up, from each CTA's own entry (median CTA entry {med['entry_skew']:.2f} after the first):")
    for k, lab in (("split_known", "split's chunk range and tiles known"), ("tmem", "TMEM allocated"),
                   ("map", "tile 0's row map built"), ("issued", "tile 0's copies issued"),
                   ("setup_own", "block-wide set-up barrier passed")):
        print(f"    {lab:<38}{med[k]:8.2f}")


if __name__ == "__main__":
    main()
