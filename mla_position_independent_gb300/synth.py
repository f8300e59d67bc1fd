"""Seeded synthetic inputs for the reuse-time MLA KV reconstruction workloads.

This module only draws random numbers and lays out chunk tables; it performs none of the
method's arithmetic (no rotation, no attention).  Where a workload wants cached k_r rows
that were RoPE-encoded at their source position (the tiny correctness case), it returns
the content vectors and positions and leaves the encoding to the caller.

Chunk records follow the layout of ``irm_chunk`` in include/irm.h (24 bytes):
pool_offset (int64, first row of the chunk in the row store), len, p_src, p_tgt (int32),
reused (uint8), 3 padding bytes.  Requests list their chunks in target order, and
``indptr`` (int32, B+1) delimits each request's chunks.

Workloads (the shapes, sizes and distributions of the serving scenario described in
"Irminsul: MLA-Native Position-Independent Caching for Agentic LLM Serving"; see the
design notes for the recipe):
  tiny_case          1 request, ctx 512, carve-out + 4 reused chunks of 64/96/128/192
  v2lite_decode      DeepSeek-V2-Lite-shaped decode, 16 heads, batch 8, ctx 8192
  v3_decode          DeepSeek-V3-shaped decode, 128 heads, batch 64, ctx 32768, shared pool
  chunked_prefill    128 heads, 4 requests, 2048 causal queries over a 16384-token prefix
  rotate_gather_case N rows scattered from a chunk pool into 64-row pages
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

CHUNK_DTYPE = np.dtype([("pool_offset", "<i8"), ("len", "<i4"), ("p_src", "<i4"),
                        ("p_tgt", "<i4"), ("reused", "u1"), ("pad", "u1", (3,))])
assert CHUNK_DTYPE.itemsize == 24

D_LAT, D_ROPE, D_ROW = 512, 64, 576
PAGE = 64
CARVE_OUT = 32
Q_STD = 1.0 / np.sqrt(192.0)


@dataclass
class Case:
    name: str
    chunks: np.ndarray            # CHUNK_DTYPE, all requests concatenated
    indptr: np.ndarray            # int32 [B+1]
    kv_rows: torch.Tensor         # bf16 [n_rows, 576]
    n_q: int = 0
    H: int = 0
    q_lat: Optional[torch.Tensor] = None   # bf16 [B, n_q, H, 512]
    q_rope: Optional[torch.Tensor] = None  # bf16 [B, n_q, H, 64]
    page_table: Optional[np.ndarray] = None  # int32 [B, max_pages]
    n_pages: int = 0
    rope_rows: Optional[np.ndarray] = None   # rows whose k_r the caller must RoPE-encode
    rope_pos: Optional[np.ndarray] = None    # position of each such row
    rope_content: Optional[np.ndarray] = None  # fp64 [len(rope_rows), 64] content vectors
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return int(self.indptr.shape[0] - 1)

    @property
    def ctx(self) -> np.ndarray:
        out = np.zeros(self.B, np.int64)
        for b in range(self.B):
            c = self.chunks[self.indptr[b]:self.indptr[b + 1]]
            out[b] = int(c["len"].astype(np.int64).sum())
        return out


def _rngs(seed: int, n: int):
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def _torch_gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, seed: int, std: float = 1.0, device="cpu") -> torch.Tensor:
    """N(0, std^2) samples rounded to bf16 (round to nearest even), seeded."""
    g = _torch_gen(seed, device)
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits(b: np.ndarray, device="cpu") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(device)


def geometric_lengths(rng, total: int, mean: int = 128, lo: int = 32, hi: int = 512):
    """Chunk lengths ~ Geometric(1/mean) clipped to [lo, hi]; the last one is cut to fit."""
    out, acc = [], 0
    while acc < total:
        n = int(np.clip(rng.geometric(1.0 / mean), lo, hi))
        n = min(n, total - acc)
        out.append(n)
        acc += n
    return out


def make_table(reqs):
    """reqs: list (per request) of lists of (pool_offset, len, p_src, reused) in target order.

    p_tgt is the running sum of lengths (concatenation).  Returns (chunks, indptr).
    """
    rows, indptr = [], [0]
    for req in reqs:
        p = 0
        for (off, n, p_src, reused) in req:
            rows.append((int(off), int(n), int(p_src), int(p), int(bool(reused))))
            p += int(n)
        indptr.append(len(rows))
    chunks = np.zeros(len(rows), CHUNK_DTYPE)
    if rows:
        a = np.array(rows, dtype=np.int64)
        chunks["pool_offset"] = a[:, 0]
        chunks["len"] = a[:, 1]
        chunks["p_src"] = a[:, 2]
        chunks["p_tgt"] = a[:, 3]
        chunks["reused"] = a[:, 4]
    return chunks, np.asarray(indptr, np.int32)


def _queries(B, n_q, H, seed, std, device):
    q_lat = normal_bf16((B, n_q, H, D_LAT), seed, std, device)
    q_rope = normal_bf16((B, n_q, H, D_ROPE), seed + 1, std, device)
    return q_lat, q_rope


def tiny_case(seed: int = 0, q_std: float = Q_STD, device="cpu", H: int = 16) -> Case:
    """1 request, ctx 512: fresh carve-out [0, 32), then 4 reused chunks of 64/96/128/192
    drawn from a pool of 8 chunks with p_src ~ U{32..4096}; 16 causal queries at the tail,
    H heads (16 in the configured workload).  k_r of every row is RoPE(position) of a N(0,1)
    content vector; the caller encodes it (see rope_rows / rope_pos / rope_content)."""
    r_tab, r_v = _rngs(seed, 2)
    used = [64, 96, 128, 192]
    pool_lens = used + list(r_tab.choice(used, size=4))
    order = r_tab.permutation(8)          # storage order of the 8 pool chunks
    p_src = r_tab.integers(32, 4096, size=8, endpoint=True)
    offs = np.zeros(8, np.int64)
    cur = CARVE_OUT                       # rows 0..31 hold the fresh carve-out
    for slot in order:
        offs[slot] = cur
        cur += pool_lens[slot]
    n_rows = cur
    req = [(0, CARVE_OUT, 0, 0)] + [(offs[k], used[k], p_src[k], 1) for k in range(4)]
    chunks, indptr = make_table([req])
    kv = normal_bf16((n_rows, D_ROW), seed + 101, 1.0, device)
    rope_rows = np.arange(n_rows, dtype=np.int64)
    rope_pos = np.empty(n_rows, np.int64)
    rope_pos[:CARVE_OUT] = np.arange(CARVE_OUT)
    for k in range(8):
        rope_pos[offs[k]:offs[k] + pool_lens[k]] = p_src[k] + np.arange(pool_lens[k])
    content = r_v.standard_normal((n_rows, D_ROPE))
    q_lat, q_rope = _queries(1, 16, H, seed + 202, q_std, device)
    return Case("tiny", chunks, indptr, kv, n_q=16, H=H, q_lat=q_lat, q_rope=q_rope,
                rope_rows=rope_rows, rope_pos=rope_pos, rope_content=content,
                meta=dict(pool_lens=pool_lens, p_src=p_src))


def _shuffle_place(rng, reqs_rows, base: int = 0):
    """Give every (request, chunk) of reqs_rows=[[len, ...], ...] a row-store offset; the
    chunks are laid out in one global random order starting at `base`."""
    flat = [(b, k) for b, req in enumerate(reqs_rows) for k in range(len(req))]
    perm = rng.permutation(len(flat))
    offs = [[0] * len(req) for req in reqs_rows]
    cur = base
    for i in perm:
        b, k = flat[i]
        offs[b][k] = cur
        cur += reqs_rows[b][k]
    return offs, cur


def v2lite_decode(seed: int = 0, B: int = 8, ctx: int = 8192, H: int = 16, reuse_p: float = 0.75,
                  delta_max: int = 4096, q_std: float = Q_STD, device="cpu") -> Case:
    """DeepSeek-V2-Lite-shaped decode: carve-out, then geometric chunks (mean 128, [32, 512]),
    each reused with probability 0.75 and delta ~ U{-4096..4096}; rows private per request;
    one query token per request."""
    r_len, r_reuse, r_delta, r_place = _rngs(seed, 4)
    lens = [[CARVE_OUT] + geometric_lengths(r_len, ctx - CARVE_OUT) for _ in range(B)]
    offs, n_rows = _shuffle_place(r_place, lens)
    reqs = []
    for b in range(B):
        p, req = 0, []
        for k, n in enumerate(lens[b]):
            reused = k > 0 and r_reuse.random() < reuse_p
            d = int(r_delta.integers(-delta_max, delta_max, endpoint=True)) if reused else 0
            req.append((offs[b][k], n, p - d if reused else 0, reused))
            p += n
        reqs.append(req)
    chunks, indptr = make_table(reqs)
    kv = normal_bf16((n_rows, D_ROW), seed + 101, 1.0, device)
    q_lat, q_rope = _queries(B, 1, H, seed + 202, q_std, device)
    return Case("v2lite_decode", chunks, indptr, kv, n_q=1, H=H, q_lat=q_lat, q_rope=q_rope)


def v3_decode(seed: int = 0, B: int = 64, ctx: int = 32768, H: int = 128, n_pool: int = 256,
              reuse_p: float = 0.8, delta_max: int = 16384, q_std: float = Q_STD,
              device="cpu") -> Case:
    """DeepSeek-V3-shaped decode: a pool of 256 shared chunks; each request walks its own
    shuffled order of the pool for ~80% of its tokens, with fresh geometric chunks
    interleaved at seeded places, after the fresh carve-out; delta ~ U{-16384..16384} is
    drawn per (request, chunk use) and p_src := p_tgt - delta."""
    r_pool, r_mix, r_len, r_delta, r_perm, r_place = _rngs(seed, 6)
    pool_lens = [int(np.clip(r_pool.geometric(1.0 / 128), 32, 512)) for _ in range(n_pool)]
    pool_offs = np.concatenate([[0], np.cumsum(pool_lens)[:-1]]).astype(np.int64)
    n_pool_rows = int(sum(pool_lens))
    plans, fresh_lens = [], []
    for b in range(B):
        perm, pi = r_perm.permutation(n_pool), 0
        p, items, fl = CARVE_OUT, [("fresh", CARVE_OUT)], [CARVE_OUT]
        while p < ctx:
            if r_mix.random() < reuse_p:
                if pi == n_pool:
                    perm, pi = r_perm.permutation(n_pool), 0
                k = int(perm[pi]); pi += 1
                n = min(pool_lens[k], ctx - p)
                items.append(("pool", k, n))
            else:
                n = min(int(np.clip(r_len.geometric(1.0 / 128), 32, 512)), ctx - p)
                items.append(("fresh", n))
                fl.append(n)
            p += n
        plans.append(items)
        fresh_lens.append(fl)
    fresh_offs, n_rows = _shuffle_place(r_place, fresh_lens, base=n_pool_rows)
    reqs = []
    for b in range(B):
        p, fi, req = 0, 0, []
        for it in plans[b]:
            if it[0] == "fresh":
                req.append((fresh_offs[b][fi], it[1], 0, 0)); fi += 1
                p += it[1]
            else:
                _, k, n = it
                d = int(r_delta.integers(-delta_max, delta_max, endpoint=True))
                req.append((pool_offs[k], n, p - d, 1))
                p += n
        reqs.append(req)
    chunks, indptr = make_table(reqs)
    kv = normal_bf16((n_rows, D_ROW), seed + 101, 1.0, device)
    q_lat, q_rope = _queries(B, 1, H, seed + 202, q_std, device)
    return Case("v3_decode", chunks, indptr, kv, n_q=1, H=H, q_lat=q_lat, q_rope=q_rope,
                meta=dict(n_pool_rows=n_pool_rows))


def chunked_prefill(seed: int = 0, B: int = 4, H: int = 128, n_q: int = 2048,
                    exact_prefix: int = 4096, reused_rows: int = 12288, delta_max: int = 8192,
                    q_std: float = Q_STD, device="cpu") -> Case:
    """Chunked prefill: per request a fresh carve-out [0, 32), an exact-prefix region
    [32, exact_prefix) of reused chunks with delta = 0, reused_rows rows of reused CDC-like
    chunks with delta ~ U{-8192..8192}, then the n_q new tokens (fresh) whose queries
    attend causally.  Row stores are private per request; ctx = exact_prefix + reused_rows
    + n_q."""
    r_len, r_delta, r_place = _rngs(seed, 3)
    kinds, lens = [], []
    for b in range(B):
        k_b = [("fresh", CARVE_OUT)]
        k_b += [("exact", n) for n in geometric_lengths(r_len, exact_prefix - CARVE_OUT)]
        k_b += [("moved", n) for n in geometric_lengths(r_len, reused_rows)]
        k_b += [("fresh", n_q)]
        kinds.append(k_b)
        lens.append([n for _, n in k_b])
    offs, n_rows = _shuffle_place(r_place, lens)
    reqs = []
    for b in range(B):
        p, req = 0, []
        for k, (kind, n) in enumerate(kinds[b]):
            if kind == "fresh":
                req.append((offs[b][k], n, 0, 0))
            elif kind == "exact":
                req.append((offs[b][k], n, p, 1))
            else:
                d = int(r_delta.integers(-delta_max, delta_max, endpoint=True))
                req.append((offs[b][k], n, p - d, 1))
            p += n
        reqs.append(req)
    chunks, indptr = make_table(reqs)
    kv = normal_bf16((n_rows, D_ROW), seed + 101, 1.0, device)
    q_lat, q_rope = _queries(B, n_q, H, seed + 202, q_std, device)
    return Case("chunked_prefill", chunks, indptr, kv, n_q=n_q, H=H, q_lat=q_lat, q_rope=q_rope)


def rotate_gather_case(n_rows: int, seed: int = 0, delta_max: int = 65536, device="cpu",
                       fill_kv: bool = True) -> Case:
    """n_rows rows of a chunk pool (geometric chunks) permuted onto one logical sequence and
    scattered into 64-row pages in a random physical order; delta ~ U{-65536..65536} per
    chunk.  Chunks that start inside the carve-out stay fresh."""
    r_len, r_perm, r_delta, r_page = _rngs(seed, 4)
    pool_lens = np.asarray(geometric_lengths(r_len, n_rows), np.int64)
    pool_offs = np.concatenate([[0], np.cumsum(pool_lens)[:-1]]).astype(np.int64)
    perm = r_perm.permutation(pool_lens.shape[0])
    lens_t = pool_lens[perm]
    p_tgt = np.concatenate([[0], np.cumsum(lens_t)[:-1]]).astype(np.int64)
    reused = p_tgt >= CARVE_OUT
    delta = r_delta.integers(-delta_max, delta_max, size=perm.shape[0], endpoint=True)
    delta = np.where(reused, delta, 0)
    chunks = np.zeros(perm.shape[0], CHUNK_DTYPE)
    chunks["pool_offset"] = pool_offs[perm]
    chunks["len"] = lens_t
    chunks["p_tgt"] = p_tgt
    chunks["p_src"] = np.where(reused, p_tgt - delta, 0)
    chunks["reused"] = reused
    indptr = np.asarray([0, perm.shape[0]], np.int32)
    n_pages = (n_rows + PAGE - 1) // PAGE
    page_table = r_page.permutation(n_pages).astype(np.int32)[None, :]
    if fill_kv:
        kv = normal_bf16((n_rows, D_ROW), seed + 101, 1.0, device)
    else:
        kv = torch.empty((n_rows, D_ROW), dtype=torch.bfloat16, device=device)
    return Case("rotate_gather", chunks, indptr, kv, page_table=page_table, n_pages=n_pages)


def custom_case(reqs, n_rows: int, seed: int = 0, n_q: int = 1, H: int = 16,
                q_std: float = Q_STD, device="cpu", pages: bool = False) -> Case:
    """Hand-written tables for edge cases: reqs as in make_table."""
    chunks, indptr = make_table(reqs)
    kv = normal_bf16((n_rows, D_ROW), seed + 101, 1.0, device)
    B = indptr.shape[0] - 1
    q_lat = q_rope = None
    if n_q > 0:
        q_lat, q_rope = _queries(B, n_q, H, seed + 202, q_std, device)
    case = Case("custom", chunks, indptr, kv, n_q=n_q, H=H, q_lat=q_lat, q_rope=q_rope)
    if pages:
        ctx = case.ctx
        max_pages = int(max(1, ((ctx + PAGE - 1) // PAGE).max()))
        n_pages = int(((ctx + PAGE - 1) // PAGE).sum())
        rng = _rngs(seed + 7, 1)[0]
        perm = rng.permutation(n_pages).astype(np.int32)
        pt = np.full((B, max_pages), -1, np.int32)
        cur = 0
        for b in range(B):
            k = int((ctx[b] + PAGE - 1) // PAGE)
            pt[b, :k] = perm[cur:cur + k]
            cur += k
        case.page_table, case.n_pages = pt, n_pages
    return case


def gear_table(vocab: int, seed: int = 0) -> np.ndarray:
    """A seeded 64-bit Gear table for content-defined chunking (one random word per token id;
    the pages do not publish theirs, so it is an input of our own choosing)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0x6EA2])))
    return rng.integers(0, 2**64, size=vocab, dtype=np.uint64)


def cdc_streams(n_streams: int, tokens_per_stream: int, vocab: int = 102400, seed: int = 0,
                doc_len: int = 4096, n_docs: int = 16):
    """Token streams for content-defined chunking: each stream interleaves random tokens with
    documents drawn from a shared set, placed at random offsets (agentic prompts that reorder
    the same documents).  Returns (tokens int32 [sum], offsets int64 [n_streams + 1])."""
    r_doc, r_mix = _rngs(seed, 2)
    docs = r_doc.integers(0, vocab, size=(n_docs, doc_len)).astype(np.int32)
    parts, offs = [], [0]
    for _ in range(n_streams):
        cur, stream = 0, []
        while cur < tokens_per_stream:
            if r_mix.random() < 0.6:
                piece = docs[r_mix.integers(0, n_docs)]
            else:
                piece = r_mix.integers(0, vocab, size=int(r_mix.integers(16, 1024))).astype(np.int32)
            piece = piece[: tokens_per_stream - cur]
            stream.append(piece)
            cur += piece.shape[0]
        parts.append(np.concatenate(stream))
        offs.append(offs[-1] + tokens_per_stream)
    return np.concatenate(parts).astype(np.int32), np.asarray(offs, np.int64)
