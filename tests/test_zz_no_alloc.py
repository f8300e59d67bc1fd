"""The no-allocation decode entry point (irm_mla_attn_decode_noalloc), called through the C
ABI.  It serves callers that cannot call cudaMalloc themselves -- a plugin inside an
application that owns the device memory pool, or code that must not allocate while a CUDA
graph is being built -- so its split-KV scratch and copied chunk table live in a fixed array
inside the library instead of a caller workspace.  It runs the same kernel with the same
split as irm_mla_attn_decode whenever that split's scratch fits the array, so on two calls in
a row its output must equal the workspace decode's bit for bit (and both match the fp64
oracle within the parity tolerance); where it does not fit, it takes the split that does.

This file is collected last on purpose, so that a run stopping at the first failure has
already run every other test.  It must pass in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from mla_position_independent_gb300 import synth
from helpers import SCALE, TOL_MAX_ABS, TOL_REL_L2, max_abs, rel_l2

pytestmark = pytest.mark.gpu


def _call_noalloc(L, case, table, ql, qr, out, lse):
    st = L.irm_mla_attn_decode_noalloc(
        ql.data_ptr(), qr.data_ptr(), ql.shape[0], ql.shape[1], table.chunks_host.ctypes.data,
        table.indptr_host.ctypes.data, case.kv_rows.data_ptr(), case.kv_rows.shape[0],
        ctypes.c_float(SCALE), out.data_ptr(), lse.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_noalloc_decode_matches_workspace_decode():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import mla_position_independent_gb300 as irm
    import oracle
    oracle.build()
    L = irm.lib()
    case = synth.v2lite_decode(0, device="cuda")
    table = irm.ChunkTable(case.chunks, case.indptr)
    ql, qr = case.q_lat[:, 0].contiguous(), case.q_rope[:, 0].contiguous()
    ref, ref_lse, ws = irm.irm_mla_attn_decode(
        ql, qr, table, case.kv_rows, SCALE,
        lse=torch.empty(ql.shape[:2], dtype=torch.float32, device="cuda"))
    irm.device_status(ws)
    for _ in range(2):  # the scratch keeps the previous call's contents
        out = torch.full_like(case.q_lat[:, 0], float("nan"))
        lse = torch.full(ql.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        assert _call_noalloc(L, case, table, ql, qr, out, lse) == 0, L.irm_last_error().decode()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        assert torch.equal(lse, ref_lse)
    irm.decode_noalloc_status()  # no device error recorded in the array's status word
    # and against the fp64 oracle on a few (request, head) rows
    sel = np.array([[b, 0, h] for b in (0, 3, 7) for h in (0, 9, 15)])
    O, _ = oracle.mla_attention(synth.bits(case.q_lat), synth.bits(case.q_rope), case.chunks,
                                case.indptr, synth.bits(case.kv_rows), SCALE, select=sel)
    got = out.float().cpu().numpy().astype(np.float64)[sel[:, 0], sel[:, 2]]
    assert rel_l2(got, O) <= TOL_REL_L2 and max_abs(got, O) <= TOL_MAX_ABS


def test_noalloc_decode_within_its_scratch():
    """The V3-shaped decode: the workspace decode's long-first split needs more scratch than the
    array holds (two fp32 partials per request), so the no-allocation call takes the split
    that fits, and still matches the fp64 oracle."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import mla_position_independent_gb300 as irm
    import oracle
    oracle.build()
    L = irm.lib()
    case = synth.v3_decode(0, device="cuda")
    table = irm.ChunkTable(case.chunks, case.indptr)
    ql, qr = case.q_lat[:, 0].contiguous(), case.q_rope[:, 0].contiguous()
    out = torch.full_like(case.q_lat[:, 0], float("nan"))
    lse = torch.full(ql.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    assert _call_noalloc(L, case, table, ql, qr, out, lse) == 0, L.irm_last_error().decode()
    torch.cuda.synchronize()
    irm.decode_noalloc_status()
    sel = np.array([[b, 0, h] for b in (0, 21, 63) for h in (0, 64, 127)])
    O, Lo = oracle.mla_attention(synth.bits(case.q_lat), synth.bits(case.q_rope), case.chunks,
                                 case.indptr, synth.bits(case.kv_rows), SCALE, select=sel)
    got = out.float().cpu().numpy().astype(np.float64)[sel[:, 0], sel[:, 2]]
    assert rel_l2(got, O) <= TOL_REL_L2 and max_abs(got, O) <= TOL_MAX_ABS
    gl = lse.cpu().numpy().astype(np.float64)[sel[:, 0], sel[:, 2]]
    assert np.max(np.abs(gl - Lo)) < 2e-2


def test_noalloc_rejects_decode_larger_than_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import mla_position_independent_gb300 as irm
    L = irm.lib()
    # one request whose chunk table alone (1.5M records of 24 bytes) is more than the array
    # holds, whatever the split
    n = 1_500_000
    chunks = np.zeros(n, dtype=synth.CHUNK_DTYPE)
    chunks["pool_offset"] = np.arange(n) % 1000
    chunks["len"] = 1
    chunks["p_tgt"] = np.arange(n)
    indptr = np.array([0, n], dtype=np.int32)
    B = 1
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")  # never read: rejected first
    st = L.irm_mla_attn_decode_noalloc(
        dummy.data_ptr(), dummy.data_ptr(), B, 128, chunks.ctypes.data, indptr.ctypes.data,
        dummy.data_ptr(), 40000, ctypes.c_float(SCALE), dummy.data_ptr(), None, None)
    assert st == -8 and b"no-allocation" in L.irm_last_error()
