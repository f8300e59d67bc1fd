"""Thin ctypes binding over libirm.so (include/irm.h).

Argument marshalling only: every step of the path runs in the library's CUDA kernels.
PyTorch supplies device memory and the current stream.  If libirm.so is missing the first
call raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np
import torch

from .synth import CHUNK_DTYPE

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libirm.so")
_lib = None

WORKSPACE_HEADER = 256
DEFAULT_SCALE = 1.0 / math.sqrt(192.0)

EXPORTS = ["irm_status_string", "irm_last_error", "irm_version", "irm_validate_chunks",
           "irm_device_status", "irm_assemble_kv_workspace_size", "irm_assemble_kv",
           "irm_assemble_kv_rope", "irm_mla_attn_decode_workspace_size", "irm_mla_attn_decode",
           "irm_mla_attn_decode_rope", "irm_mla_attn_decode_noalloc", "irm_decode_noalloc_status",
           "irm_mla_attn_prefill_workspace_size", "irm_mla_attn_prefill", "irm_mla_attn_prefill_rope",
           "irm_cdc_sizes", "irm_cdc_chunk", "irm_registry_create", "irm_registry_stats",
           "irm_registry_assemble", "irm_selftest_wait_timeout"]

ROPE_NEOX, ROPE_INTERLEAVED = 0, 1


class Rope(ctypes.Structure):
    """irm_rope: the model's RoPE variant (32 frequencies theta_j in radians per position and
    the pairing, ROPE_NEOX = dims (j, j+32) or ROPE_INTERLEAVED = dims (2j, 2j+1))."""
    _fields_ = [("inv_freq", ctypes.c_double * 32), ("pairing", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]

    @classmethod
    def make(cls, inv_freq, pairing=ROPE_NEOX):
        f = np.asarray(inv_freq, np.float64).reshape(32)
        return cls((ctypes.c_double * 32)(*f.tolist()), int(pairing), 0)


CDC_THRESHOLD, CDC_LOW_BITS = 0, 1


class CdcParams(ctypes.Structure):
    """irm_cdc_params: chunk length clip, boundary test and fingerprint seed."""
    _fields_ = [("min_len", ctypes.c_int32), ("max_len", ctypes.c_int32), ("bits", ctypes.c_int32),
                ("mode", ctypes.c_int32), ("seed", ctypes.c_uint64), ("gear_seed", ctypes.c_uint64)]

    @classmethod
    def make(cls, min_len=32, max_len=512, bits=7, mode=CDC_THRESHOLD, seed=0, gear_seed=0):
        return cls(int(min_len), int(max_len), int(bits), int(mode), int(seed), int(gear_seed))


def _rope_ptr(rope):
    return None if rope is None else ctypes.cast(ctypes.pointer(rope), ctypes.c_void_p)


class IrmError(RuntimeError):
    def __init__(self, status: int, text: str, detail: str):
        super().__init__(f"irm status {status} ({text}): {detail}")
        self.status = status


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is not built: run __graft_entry__.build() "
                               "(the CUDA library is required; there is no fallback)")
        L = ctypes.CDLL(_LIB_PATH)
        P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        L.irm_status_string.restype = ctypes.c_char_p
        L.irm_status_string.argtypes = [I]
        L.irm_last_error.restype = ctypes.c_char_p
        L.irm_version.restype = ctypes.c_char_p
        L.irm_validate_chunks.argtypes = [P, P, I, I64, P]
        L.irm_device_status.argtypes = [P, P]
        L.irm_selftest_wait_timeout.argtypes = [P, SZ, P]
        L.irm_assemble_kv_workspace_size.argtypes = [P, P, I, P]
        L.irm_assemble_kv.argtypes = [P, P, I, P, I64, P, I64, P, I, P, P, P, P, SZ, P]
        L.irm_mla_attn_decode_workspace_size.argtypes = [P, P, I, I, P]
        L.irm_mla_attn_decode.argtypes = [P, P, I, I, P, P, P, I64, ctypes.c_float, P, P, P, SZ, P]
        L.irm_mla_attn_decode_noalloc.argtypes = [P, P, I, I, P, P, P, I64, ctypes.c_float, P, P, P]
        L.irm_decode_noalloc_status.argtypes = [P]
        L.irm_mla_attn_prefill_workspace_size.argtypes = [P, P, I, I, I, P]
        L.irm_mla_attn_prefill.argtypes = [P, P, I, I, I, P, P, P, I64, ctypes.c_float, P, P, P,
                                           SZ, P]
        L.irm_assemble_kv_rope.argtypes = [P, P, I, P, I64, P, I64, P, I, P, P, P, P, P, SZ, P]
        L.irm_mla_attn_decode_rope.argtypes = [P, P, I, I, P, P, P, I64, ctypes.c_float, P, P, P,
                                               P, SZ, P]
        L.irm_mla_attn_prefill_rope.argtypes = [P, P, I, I, I, P, P, P, I64, ctypes.c_float, P, P,
                                                P, P, SZ, P]
        L.irm_cdc_sizes.argtypes = [P, I, P, P, P]
        L.irm_cdc_chunk.argtypes = [P, P, I, P, ctypes.c_int32, P, P, P, P, P, P, SZ, P]
        L.irm_registry_create.argtypes = [I64, I64, I64, P]
        L.irm_registry_destroy.argtypes = [P]
        L.irm_registry_destroy.restype = None
        L.irm_registry_stats.argtypes = [P, P, P]
        L.irm_registry_assemble.argtypes = [P, P, I64, I64, I64, P, P, P, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_uint64, P, P, ctypes.c_int32, P]
        for name in EXPORTS:
            if name not in ("irm_status_string", "irm_last_error", "irm_version"):
                getattr(L, name).restype = I
        _lib = L
    return _lib


def _check(st: int):
    if st != 0:
        L = lib()
        raise IrmError(st, L.irm_status_string(st).decode(), L.irm_last_error().decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, name, ndim=None):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on the GPU")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")


class ChunkTable:
    """A batch of chunk tables in host memory, as the library takes them.  With CUDA present
    the table sits in one page-locked block laid out as the library's workspace table area
    (indptr [B+1] int32, padded to 8 bytes, then the chunk records), so a call stages it with
    one asynchronous host-to-device copy; keep it unchanged while calls that use it are in
    flight.  Without CUDA (host-only validation) it is plain pageable memory."""

    def __init__(self, chunks: np.ndarray, indptr: np.ndarray, pinned: bool | None = None):
        chunks = np.ascontiguousarray(chunks, dtype=CHUNK_DTYPE)
        indptr = np.ascontiguousarray(indptr, dtype=np.int32)
        self.B = int(indptr.shape[0] - 1)
        ia = (4 * (self.B + 1) + 7) // 8 * 8
        nbytes = ia + chunks.nbytes
        if pinned is None:
            pinned = torch.cuda.is_available()
        buf = torch.zeros(nbytes, dtype=torch.uint8)
        if pinned:
            buf = buf.pin_memory()
        self._buf = buf  # keeps the block alive
        raw = buf.numpy()
        self.indptr_host = raw[:4 * (self.B + 1)].view(np.int32)
        self.chunks_host = raw[ia:ia + chunks.nbytes].view(CHUNK_DTYPE)
        self.indptr_host[:] = indptr
        self.chunks_host[:] = chunks
        self.n_chunks = int(chunks.shape[0])

    def validate(self, n_rows: int) -> np.ndarray:
        ctx = np.zeros(self.B, np.int64)
        _check(lib().irm_validate_chunks(_ptr(self.chunks_host), _ptr(self.indptr_host), self.B,
                                         int(n_rows), _ptr(ctx)))
        return ctx


def validate_chunks(chunks: np.ndarray, indptr: np.ndarray, n_rows: int) -> np.ndarray:
    """Host-only validation (no GPU needed).  Returns each request's context length."""
    chunks = np.ascontiguousarray(chunks, dtype=CHUNK_DTYPE)
    indptr = np.ascontiguousarray(indptr, dtype=np.int32)
    B = int(indptr.shape[0] - 1)
    ctx = np.zeros(max(B, 1), np.int64)
    _check(lib().irm_validate_chunks(_ptr(chunks), _ptr(indptr), B, int(n_rows), _ptr(ctx)))
    return ctx[:B]


def new_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Zero-initialised workspace (the first 256 bytes hold the device status word)."""
    return torch.zeros(max(int(nbytes), WORKSPACE_HEADER), dtype=torch.uint8, device=device)


def device_status(workspace: torch.Tensor, stream=None):
    """Raises IrmError if a kernel recorded a timeout or an out-of-range row (and clears it)."""
    _check(lib().irm_device_status(_ptr(workspace), _stream(stream)))


def selftest_wait_timeout(workspace: torch.Tensor, stream=None):
    """Launches the bounded-wait self-test (a wait nothing ever completes); after it,
    device_status(workspace) raises the timeout it recorded."""
    _check(lib().irm_selftest_wait_timeout(_ptr(workspace), workspace.numel(), _stream(stream)))


def assemble_kv_workspace_size(table: ChunkTable) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().irm_assemble_kv_workspace_size(_ptr(table.chunks_host), _ptr(table.indptr_host),
                                                table.B, ctypes.byref(n)))
    return n.value


def irm_assemble_kv(table: ChunkTable, kv_rows: torch.Tensor, paged_out=None, page_table=None,
                    out_src_row=None, out_delta=None, out_pos_src=None, workspace=None,
                    stream=None, rope: Rope | None = None):
    """Rotate+gather and/or the assembly plan; rope selects the model's RoPE variant
    (irm_assemble_kv_rope), None the default."""
    _need(kv_rows, torch.bfloat16, "kv_rows", 2)
    n_pages, max_pages = 0, 0
    if paged_out is not None:
        _need(paged_out, torch.bfloat16, "paged_out", 3)
        _need(page_table, torch.int32, "page_table", 2)
        n_pages, max_pages = int(paged_out.shape[0]), int(page_table.shape[1])
    for t, n in ((out_src_row, "out_src_row"), (out_delta, "out_delta"), (out_pos_src, "out_pos_src")):
        if t is not None:
            _need(t, torch.int32, n, 1)
    if workspace is None:
        workspace = new_workspace(assemble_kv_workspace_size(table), kv_rows.device)
    _check(lib().irm_assemble_kv_rope(
        _ptr(table.chunks_host), _ptr(table.indptr_host), table.B,
        _ptr(kv_rows), int(kv_rows.shape[0]), _ptr(paged_out), n_pages,
        _ptr(page_table), max_pages, _ptr(out_src_row), _ptr(out_delta), _ptr(out_pos_src),
        _rope_ptr(rope), _ptr(workspace), workspace.numel(), _stream(stream)))
    return workspace


def decode_workspace_size(table: ChunkTable, H: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().irm_mla_attn_decode_workspace_size(_ptr(table.chunks_host),
                                                    _ptr(table.indptr_host), table.B, int(H),
                                                    ctypes.byref(n)))
    return n.value


def prefill_workspace_size(table: ChunkTable, n_q: int, H: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().irm_mla_attn_prefill_workspace_size(_ptr(table.chunks_host), _ptr(table.indptr_host),
                                                     table.B, int(n_q), int(H), ctypes.byref(n)))
    return n.value


def irm_mla_attn_decode(q_lat, q_rope, table: ChunkTable, kv_rows, softmax_scale=DEFAULT_SCALE,
                        out=None, lse=None, workspace=None, stream=None, rope: Rope | None = None):
    """q_lat [B, H, 512] / q_rope [B, H, 64] bf16 (a [B, 1, H, *] view is accepted); rope
    selects the model's RoPE variant (irm_mla_attn_decode_rope), None the default."""
    B, H = int(q_lat.shape[0]), int(q_lat.shape[-2])
    _need(q_lat, torch.bfloat16, "q_lat")
    _need(q_rope, torch.bfloat16, "q_rope")
    _need(kv_rows, torch.bfloat16, "kv_rows", 2)
    if out is None:
        out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=q_lat.device)
    _need(out, torch.bfloat16, "out")
    if lse is not None:
        _need(lse, torch.float32, "lse")
    if workspace is None:
        workspace = new_workspace(decode_workspace_size(table, H), q_lat.device)
    _check(lib().irm_mla_attn_decode_rope(
        _ptr(q_lat), _ptr(q_rope), B, H, _ptr(table.chunks_host), _ptr(table.indptr_host),
        _ptr(kv_rows), int(kv_rows.shape[0]),
        float(softmax_scale), _ptr(out), _ptr(lse), _rope_ptr(rope), _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return out, lse, workspace


def irm_mla_attn_decode_noalloc(q_lat, q_rope, table: ChunkTable, kv_rows,
                                softmax_scale=DEFAULT_SCALE, out=None, lse=None, stream=None):
    """Decode for callers that cannot allocate device memory: the library's own fixed
    scratch array replaces the workspace (see include/irm.h for the limit)."""
    B, H = int(q_lat.shape[0]), int(q_lat.shape[-2])
    _need(q_lat, torch.bfloat16, "q_lat")
    _need(q_rope, torch.bfloat16, "q_rope")
    _need(kv_rows, torch.bfloat16, "kv_rows", 2)
    if out is None:
        out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=q_lat.device)
    _need(out, torch.bfloat16, "out")
    if lse is not None:
        _need(lse, torch.float32, "lse")
    _check(lib().irm_mla_attn_decode_noalloc(
        _ptr(q_lat), _ptr(q_rope), B, H, _ptr(table.chunks_host), _ptr(table.indptr_host),
        _ptr(kv_rows), int(kv_rows.shape[0]),
        float(softmax_scale), _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def decode_noalloc_status(stream=None):
    """Raises IrmError if a no-allocation decode recorded a timeout or an out-of-range row in
    the library's scratch array (and clears it)."""
    _check(lib().irm_decode_noalloc_status(_stream(stream)))


def irm_mla_attn_prefill(q_lat, q_rope, table: ChunkTable, kv_rows, softmax_scale=DEFAULT_SCALE,
                         out=None, lse=None, workspace=None, stream=None, rope: Rope | None = None):
    """q_lat [B, n_q, H, 512] / q_rope [B, n_q, H, 64] bf16, causal over the last n_q rows;
    rope selects the model's RoPE variant (irm_mla_attn_prefill_rope), None the default."""
    B, n_q, H = (int(x) for x in q_lat.shape[:3])
    _need(q_lat, torch.bfloat16, "q_lat", 4)
    _need(q_rope, torch.bfloat16, "q_rope", 4)
    _need(kv_rows, torch.bfloat16, "kv_rows", 2)
    if out is None:
        out = torch.empty((B, n_q, H, 512), dtype=torch.bfloat16, device=q_lat.device)
    _need(out, torch.bfloat16, "out")
    if lse is not None:
        _need(lse, torch.float32, "lse")
    if workspace is None:
        workspace = new_workspace(prefill_workspace_size(table, n_q, H), q_lat.device)
    _check(lib().irm_mla_attn_prefill_rope(
        _ptr(q_lat), _ptr(q_rope), B, n_q, H, _ptr(table.chunks_host), _ptr(table.indptr_host),
        _ptr(kv_rows), int(kv_rows.shape[0]),
        float(softmax_scale), _ptr(out), _ptr(lse), _rope_ptr(rope), _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return out, lse, workspace


def cdc_sizes(offsets: np.ndarray, params: CdcParams | None = None):
    """(workspace bytes, output slots) of irm_cdc_chunk for these stream offsets."""
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    nb, sl = ctypes.c_size_t(0), ctypes.c_int64(0)
    pp = None if params is None else ctypes.cast(ctypes.pointer(params), ctypes.c_void_p)
    _check(lib().irm_cdc_sizes(_ptr(offsets), int(offsets.shape[0] - 1), pp, ctypes.byref(nb),
                               ctypes.byref(sl)))
    return nb.value, sl.value


def cdc_slot_base(offsets: np.ndarray, min_len: int = 32) -> np.ndarray:
    """First output slot of each stream (the layout irm_cdc_sizes documents)."""
    lens = np.diff(np.asarray(offsets, np.int64))
    return np.concatenate([[0], np.cumsum(lens // min_len + 1)])[:-1]


def irm_cdc_chunk(tokens: torch.Tensor, offsets: np.ndarray, gear: torch.Tensor | None,
                  params: CdcParams | None = None, fingerprints=True, out=None, workspace=None,
                  stream=None, vocab: int | None = None):
    """Content-defined chunks of token streams (tokens int32 on the GPU, streams at host
    offsets; gear: the 64-bit Gear table as an int64 tensor on the GPU, or None for Gear
    words generated from params.gear_seed, with token ids in [0, vocab)).  Returns
    (n_chunks [S], chunk_start [slots], chunk_len [slots], chunk_hash [slots] or None,
    workspace); stream s's chunks sit at slots cdc_slot_base(offsets)[s] onwards."""
    _need(tokens, torch.int32, "tokens", 1)
    if gear is not None:
        _need(gear, torch.int64, "gear", 1)
        vocab = int(gear.shape[0])
    elif vocab is None:
        raise ValueError("generated Gear words need the vocab size")
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    S = int(offsets.shape[0] - 1)
    nbytes, slots = cdc_sizes(offsets, params)
    dev = tokens.device
    if out is None:
        out = (torch.empty(S, dtype=torch.int32, device=dev),
               torch.empty(max(slots, 1), dtype=torch.int32, device=dev),
               torch.empty(max(slots, 1), dtype=torch.int32, device=dev),
               torch.empty(max(slots, 1), dtype=torch.int64, device=dev) if fingerprints else None)
    n_chunks, c_start, c_len, c_hash = out
    if workspace is None:
        workspace = new_workspace(nbytes, dev)
    pp = None if params is None else ctypes.cast(ctypes.pointer(params), ctypes.c_void_p)
    _check(lib().irm_cdc_chunk(_ptr(tokens), _ptr(offsets), S, _ptr(gear),
                               int(vocab), pp, _ptr(n_chunks), _ptr(c_start), _ptr(c_len),
                               _ptr(c_hash), _ptr(workspace), workspace.numel(), _stream(stream)))
    return n_chunks, c_start, c_len, c_hash, workspace


ASSEMBLE_S1 = 1


class Registry:
    """Content-addressed chunk registry (host side, libirm's irm_registry): keeps cached chunks'
    rows in a ring of pool rows and turns a request's CDC segments into a chunk table."""

    def __init__(self, pool_rows: int, pool_base: int = 0, capacity: int = 1 << 16):
        h = ctypes.c_void_p()
        _check(lib().irm_registry_create(int(pool_base), int(pool_rows), int(capacity), ctypes.byref(h)))
        self._h = h

    def close(self):
        if self._h:
            lib().irm_registry_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def stats(self):
        live, rows = ctypes.c_int64(0), ctypes.c_int64(0)
        _check(lib().irm_registry_stats(self._h, ctypes.byref(live), ctypes.byref(rows)))
        return live.value, rows.value

    def assemble(self, tokens, prefix_len, prefix_row, seg_start, seg_len, seg_hash, s1=False,
                 seed=0):
        """(chunk table as a CHUNK_DTYPE array, prefill flags uint8) of one request."""
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        st = np.ascontiguousarray(seg_start, dtype=np.int32)
        ln = np.ascontiguousarray(seg_len, dtype=np.int32)
        hs = np.ascontiguousarray(np.asarray(seg_hash, dtype=np.uint64))
        cap = 1 + (int(((ln.astype(np.int64) + 127) // 128).sum()) if s1 else len(ln))
        out = np.zeros(cap, CHUNK_DTYPE)
        pre = np.zeros(cap, np.uint8)
        n = ctypes.c_int32(0)
        _check(lib().irm_registry_assemble(self._h, _ptr(tokens), int(tokens.shape[0]), int(prefix_len),
                                           int(prefix_row), _ptr(st), _ptr(ln), _ptr(hs), int(len(st)),
                                           ASSEMBLE_S1 if s1 else 0, ctypes.c_uint64(seed), _ptr(out),
                                           _ptr(pre), cap, ctypes.byref(n)))
        return out[:n.value], pre[:n.value]
