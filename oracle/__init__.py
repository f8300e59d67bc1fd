"""Reference oracle for delta-rotated MLA KV reconstruction (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  It shares no code with the CUDA path: the arithmetic lives in
``irm_oracle.c`` (fp64, plain loops), and this module only marshals numpy arrays into it
and composes its steps per request.

Pages cited:
  [walkthrough] "Irminsul论文详解：面向Agentic LLM Serving的MLA原生位置无关缓存" (gentlecold.top)
  [summary]     "Irminsul: MLA-Native Position-Independent Caching for Agentic LLM Serving"
                (gist.science technical summary)

Functions and the passages they follow:
  rope_theta   NeoX frequencies theta_j = 10000^(-2j/64)   (convention fixed for this build;
               the pages warn the rotary class must match the model, [walkthrough §11])
  rotate       R(steps) on 64-d rows                        [walkthrough §4, §15]
               (rope=(theta[32], pairing) selects a RoPE variant: any frequency table, NeoX
               half split (pairing 0) or interleaved pairs (pairing 1) [walkthrough §11])
  plan         chunk table -> per-row src_row, delta, pos_src [walkthrough §5 pseudo-code]
  assemble     [cKV | R(delta) k_r] in fp64                 [walkthrough §4], [summary §2.2]
  attn         absorbed MLA softmax attention in fp64       [walkthrough §4]
  mla_attention  plan + assemble + attn per request, all or sampled (b, i, h) rows
  rotate_gather  expected paged rows for a set of target rows
  gear_hash    64-token-window Gear hash of a token stream   [summary §2.2], [walkthrough §6]
  cdc          content-defined chunks (7-bit test, [32, 512] clip) of a token stream
  xxh64, chunk_fingerprint   xxHash64 of bytes / of a chunk's token ids [summary §2.2]
  splitmix_gear  Gear words from SplitMix64 (G[t] = its (t+1)-th output), instead of a table

Pins (tests/test_oracle.py): composition R(delta)R(p_src) = R(p_tgt), the worked example of
[walkthrough §15] (tests/golden/worked_example.json), delta = 0 identity, norm preservation,
inverse, NeoX pairing and frequency special cases, brute-force plan enumeration,
closed-form attention cases, causal masking, shift invariance, full-recompute equivalence,
and the bf16 rotation error bound of [summary §3].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "irm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

D_LAT, D_ROPE, D_ROW = 512, 64, 576


def build(force: bool = False) -> str:
    """Compile irm_oracle.c into liboracle.so (gcc, fp64, OpenMP) if it is missing or stale."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int64
            lib.oracle_rope_theta.argtypes = [P]
            lib.oracle_rotate.argtypes = [P, I, P, P]
            lib.oracle_rotate_ex.argtypes = [P, I, P, P, ctypes.c_int, P]
            lib.oracle_assemble_ex.argtypes = [P, I, P, P, P, ctypes.c_int, P]
            lib.oracle_plan.argtypes = [I, P, P, P, P, P, P, P, P, P, P]
            lib.oracle_plan.restype = ctypes.c_int
            lib.oracle_assemble.argtypes = [P, I, P, P, P]
            lib.oracle_attn.argtypes = [P, P, I, P, I, ctypes.c_double, P, P]
            lib.oracle_widen.argtypes = [P, I, P]
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            lib.oracle_set_num_threads.restype = None
            lib.oracle_gear_hash.argtypes = [P, I, P, P]
            lib.oracle_cdc.argtypes = [P, I, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, P, P]
            lib.oracle_cdc.restype = I
            lib.oracle_xxh64.argtypes = [P, I, ctypes.c_uint64]
            lib.oracle_xxh64.restype = ctypes.c_uint64
            lib.oracle_chunk_fingerprint.argtypes = [P, I, I, ctypes.c_uint64]
            lib.oracle_chunk_fingerprint.restype = ctypes.c_uint64
            lib.oracle_splitmix_gear.argtypes = [I, ctypes.c_uint64, P]
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of later oracle calls (for timing only; results do not depend on it)."""
    _load().oracle_set_num_threads(int(n))


def rope_theta() -> np.ndarray:
    out = np.empty(32, np.float64)
    _load().oracle_rope_theta(_p(out))
    return out


def _rope(rope):
    """(theta[32] fp64, pairing) of a RoPE spec; None is the default convention."""
    if rope is None:
        return None
    theta, pairing = rope
    theta = _c(np.asarray(theta, np.float64).reshape(32), np.float64)
    if int(pairing) not in (0, 1):
        raise ValueError("pairing must be 0 (NeoX half split) or 1 (interleaved)")
    return theta, int(pairing)


def rotate(k, steps, rope=None) -> np.ndarray:
    """R(steps[r]) k[r] for rows of 64 values (fp64); rope=(theta[32], pairing) or None."""
    k = _c(np.atleast_2d(k), np.float64)
    steps = _c(np.broadcast_to(np.asarray(steps, np.int64), (k.shape[0],)), np.int64)
    out = np.empty_like(k)
    rp = _rope(rope)
    if rp is None:
        _load().oracle_rotate(_p(k), k.shape[0], _p(steps), _p(out))
    else:
        _load().oracle_rotate_ex(_p(k), k.shape[0], _p(steps), _p(rp[0]), rp[1], _p(out))
    return out


def widen(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp64, exactly."""
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float64)
    _load().oracle_widen(_p(bits), bits.size, _p(out))
    return out


def _table_soa(chunks):
    return (_c(chunks["pool_offset"], np.int64), _c(chunks["len"], np.int64),
            _c(chunks["p_src"], np.int64), _c(chunks["p_tgt"], np.int64),
            _c(chunks["reused"], np.uint8))


def plan(chunks, indptr):
    """Per-row plan of a batch of chunk tables.

    Returns dict(ctx[B], row_start[B+1], src_row, delta, pos_src) with rows of request b at
    [row_start[b], row_start[b+1]).  Raises ValueError on a table the method does not allow.
    """
    indptr = _c(indptr, np.int64)
    B = indptr.shape[0] - 1
    po, ln, ps, pt, ru = _table_soa(chunks)
    total = int(ln.sum()) if ln.size else 0
    ctx = np.zeros(B, np.int64)
    src = np.empty(max(total, 1), np.int64)
    dl = np.empty(max(total, 1), np.int64)
    pss = np.empty(max(total, 1), np.int64)
    rc = _load().oracle_plan(B, _p(indptr), _p(po), _p(ln), _p(ps), _p(pt), _p(ru), _p(ctx),
                             _p(src), _p(dl), _p(pss))
    if rc != 0:
        raise ValueError({-1: "chunks do not tile [0, ctx) in order",
                          -2: "reused chunk inside the 32-token carve-out"}.get(rc, rc))
    row_start = np.zeros(B + 1, np.int64)
    row_start[1:] = np.cumsum(ctx)
    return dict(ctx=ctx, row_start=row_start, src_row=src[:total], delta=dl[:total],
                pos_src=pss[:total])


def assemble(kv_rows_bits, src_row, delta, rope=None) -> np.ndarray:
    """fp64 [n, 576] rows [cKV | R(delta) k_r] gathered from the bf16 row store."""
    kv = kv_rows_bits
    assert kv.dtype == np.uint16 and kv.ndim == 2 and kv.shape[1] == D_ROW
    kv = np.ascontiguousarray(kv)
    src_row = _c(src_row, np.int64)
    delta = _c(delta, np.int64)
    if src_row.size and (src_row.min() < 0 or src_row.max() >= kv.shape[0]):
        raise ValueError("source row outside the row store")
    out = np.empty((src_row.shape[0], D_ROW), np.float64)
    rp = _rope(rope)
    if rp is None:
        _load().oracle_assemble(_p(kv), src_row.shape[0], _p(src_row), _p(delta), _p(out))
    else:
        _load().oracle_assemble_ex(_p(kv), src_row.shape[0], _p(src_row), _p(delta), _p(rp[0]),
                                   rp[1], _p(out))
    return out


def attn(q, visible, K, scale):
    """Softmax attention of fp64 query rows q[R, 576] over keys K[:visible[r]] (fp64).

    Returns (O[R, 512], lse[R]) with lse in natural log units.
    """
    q = _c(np.atleast_2d(q), np.float64)
    K = _c(K, np.float64)
    visible = _c(np.broadcast_to(np.asarray(visible, np.int64), (q.shape[0],)), np.int64)
    if visible.size and (visible.min() < 1 or visible.max() > K.shape[0]):
        raise ValueError("visible key count out of range")
    O = np.empty((q.shape[0], D_LAT), np.float64)
    lse = np.empty(q.shape[0], np.float64)
    _load().oracle_attn(_p(q), _p(visible), q.shape[0], _p(K), K.shape[0], float(scale), _p(O),
                        _p(lse))
    return O, lse


def mla_attention(q_lat_bits, q_rope_bits, chunks, indptr, kv_rows_bits, scale, select=None,
                  rope=None):
    """fp64 MLA attention of a batch, following the reuse-time reconstruction.

    q_lat_bits [B, n_q, H, 512] and q_rope_bits [B, n_q, H, 64] are bf16 bit patterns;
    query i of request b sits at position ctx_b - n_q + i and sees keys 0..that position.
    select: None for every (b, i, h), else an int array [R, 3] of (b, i, h).
    Returns (O, lse): [B, n_q, H, 512] / [B, n_q, H] for select=None, else [R, 512] / [R].
    """
    B, n_q, H = q_lat_bits.shape[:3]
    pl = plan(chunks, indptr)
    if select is None:
        sel = np.stack(np.meshgrid(np.arange(B), np.arange(n_q), np.arange(H), indexing="ij"),
                       -1).reshape(-1, 3)
    else:
        sel = np.asarray(select, np.int64).reshape(-1, 3)
    O = np.empty((sel.shape[0], D_LAT))
    lse = np.empty(sel.shape[0])
    for b in np.unique(sel[:, 0]):
        rows = np.nonzero(sel[:, 0] == b)[0]
        r0, r1 = pl["row_start"][b], pl["row_start"][b + 1]
        ctx = int(r1 - r0)
        K = assemble(kv_rows_bits, pl["src_row"][r0:r1], pl["delta"][r0:r1], rope)
        ii, hh = sel[rows, 1], sel[rows, 2]
        q = np.concatenate([widen(q_lat_bits[b, ii, hh]), widen(q_rope_bits[b, ii, hh])], axis=1)
        visible = ctx - n_q + ii + 1
        O[rows], lse[rows] = attn(q, visible, K, scale)
    if select is None:
        return O.reshape(B, n_q, H, D_LAT), lse.reshape(B, n_q, H)
    return O, lse


def rotate_gather(kv_rows_bits, chunks, indptr, page_table, rows=None, rope=None):
    """Expected paged rows of the standalone rotate+gather path.

    Target row t of request b lands in slot page_table[b, t // 64] * 64 + t % 64 with value
    [cKV | R(delta) k_r] of its source row (fp64).  rows: None for all target rows, else an
    int array [R, 2] of (b, t).  Returns (slot[R], values[R, 576]).
    """
    pl = plan(chunks, indptr)
    page_table = np.asarray(page_table)
    if rows is None:
        b_of = np.repeat(np.arange(len(pl["ctx"])), pl["ctx"])
        t_of = np.arange(pl["src_row"].shape[0]) - pl["row_start"][b_of]
    else:
        rows = np.asarray(rows, np.int64).reshape(-1, 2)
        b_of, t_of = rows[:, 0], rows[:, 1]
    flat = pl["row_start"][b_of] + t_of
    slot = page_table[b_of, t_of // 64].astype(np.int64) * 64 + t_of % 64
    vals = assemble(kv_rows_bits, pl["src_row"][flat], pl["delta"][flat], rope)
    return slot, vals


# ------------------------------------------------------------------- content-defined chunking

def gear_hash(tokens, gear) -> np.ndarray:
    """h_i = sum_{k<64, k<=i} gear[tokens[i-k]] * 2^k mod 2^64 for every position (uint64)."""
    tokens = _c(tokens, np.int32)
    gear = _c(gear, np.uint64)
    if tokens.size and (tokens.min() < 0 or tokens.max() >= gear.shape[0]):
        raise ValueError("token id outside the Gear table")
    out = np.empty(tokens.shape[0], np.uint64)
    _load().oracle_gear_hash(_p(tokens), tokens.shape[0], _p(gear), _p(out))
    return out


def cdc(tokens, gear, min_len=32, max_len=512, bits=7, mode=0):
    """Content-defined chunks of one stream: (starts, lens) int64 arrays."""
    tokens = _c(tokens, np.int32)
    gear = _c(gear, np.uint64)
    if tokens.size and (tokens.min() < 0 or tokens.max() >= gear.shape[0]):
        raise ValueError("token id outside the Gear table")
    n = tokens.shape[0]
    starts = np.empty(max(n, 1), np.int64)
    lens = np.empty(max(n, 1), np.int64)
    c = _load().oracle_cdc(_p(tokens), n, _p(gear), int(min_len), int(max_len), int(bits),
                           int(mode), _p(starts), _p(lens))
    return starts[:c], lens[:c]


def xxh64(data: bytes, seed: int = 0) -> int:
    buf = np.frombuffer(bytes(data) + b"\0", np.uint8)
    return int(_load().oracle_xxh64(_p(buf), len(data), ctypes.c_uint64(seed)))


def chunk_fingerprint(tokens, start, length, seed: int = 0) -> int:
    tokens = _c(tokens, np.int32)
    return int(_load().oracle_chunk_fingerprint(_p(tokens), int(start), int(length),
                                                ctypes.c_uint64(seed)))


def splitmix_gear(vocab: int, seed: int = 0) -> np.ndarray:
    """Gear table whose word t is the (t+1)-th SplitMix64 output for `seed`."""
    out = np.empty(int(vocab), np.uint64)
    _load().oracle_splitmix_gear(int(vocab), ctypes.c_uint64(seed), _p(out))
    return out
