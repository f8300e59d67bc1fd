"""Host-side checks of the C ABI (no GPU): the library loads, exports every entry point the
header declares, and rejects bad chunk tables with status codes before any launch."""
import ctypes
import os
import re

import numpy as np
import pytest

from mla_position_independent_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def irm():
    from mla_position_independent_gb300 import build
    build.build()
    import mla_position_independent_gb300 as m
    m.lib()
    return m


def test_exports_every_declared_symbol(irm):
    hdr = open(os.path.join(ROOT, "include", "irm.h")).read()
    declared = set(re.findall(r"^(?:irm_status|const char\*)\s+(irm_\w+)\(", hdr, re.M))
    assert {"irm_assemble_kv", "irm_mla_attn_decode", "irm_mla_attn_prefill"} <= declared
    L = irm.lib()
    for name in sorted(declared):
        assert hasattr(L, name), name
    assert L.irm_version().decode().endswith("sm_103a")


def _codes(irm):
    return {"ok": 0, "arg": -1, "table": -2, "carve": -3, "unsup": -4, "ws": -8}


def _validate(irm, reqs, n_rows=1000):
    chunks, indptr = synth.make_table(reqs)
    try:
        return 0, irm.validate_chunks(chunks, indptr, n_rows)
    except irm.IrmError as e:
        return e.status, None


def test_validate_good_table(irm):
    st, ctx = _validate(irm, [[(0, 32, 0, 0), (100, 50, 7, 1)], [(500, 3, 0, 0)]])
    assert st == 0 and list(ctx) == [82, 3]


@pytest.mark.parametrize("reqs,code", [
    ([[(0, 16, 0, 0), (100, 50, 7, 1)]], -3),          # reused chunk at p_tgt 16 < 32
    ([[(0, 32, 0, 0), (100, 0, 7, 1)]], -2),           # len 0
    ([[(0, 32, 0, 0), (990, 50, 7, 1)]], -2),          # rows past the row store
    ([[(-5, 32, 0, 0)]], -2),                          # negative pool offset
    ([[(0, 40, 0, 1)]], -3),                           # reused chunk covering position 0
])
def test_validate_rejects(irm, reqs, code):
    assert _validate(irm, reqs)[0] == code


def test_validate_rejects_gap_and_order(irm):
    chunks, indptr = synth.make_table([[(0, 32, 0, 0), (100, 50, 7, 1)]])
    chunks["p_tgt"][1] = 40   # gap
    with pytest.raises(irm.IrmError) as e:
        irm.validate_chunks(chunks, indptr, 1000)
    assert e.value.status == -2
    chunks, indptr = synth.make_table([[(0, 32, 0, 0)], []])
    with pytest.raises(irm.IrmError) as e:     # request without chunks
        irm.validate_chunks(chunks, indptr, 1000)
    assert e.value.status == -2
    chunks, indptr = synth.make_table([[(0, 32, 0, 0)]])
    indptr = indptr.copy()
    indptr[0] = 1
    with pytest.raises(irm.IrmError):
        irm.validate_chunks(chunks, indptr, 1000)


def test_validate_rejects_delta_overflow(irm):
    chunks, indptr = synth.make_table([[(0, 32, 0, 0), (100, 50, 0, 1)]])
    chunks["p_src"][1] = -(2 ** 31) + 1        # delta = 32 - p_src overflows int32
    with pytest.raises(irm.IrmError) as e:
        irm.validate_chunks(chunks, indptr, 1000)
    assert e.value.status == -2


def test_null_and_error_paths_return_codes(irm):
    L = irm.lib()
    assert L.irm_validate_chunks(None, None, 1, 10, None) == -1
    assert L.irm_device_status(None, None) == -1
    n = ctypes.c_size_t(0)
    chunks, indptr = synth.make_table([[(0, 32, 0, 0)], [(40, 5, 0, 0)], [(60, 7, 0, 0)]])
    assert L.irm_assemble_kv_workspace_size(chunks.ctypes.data, indptr.ctypes.data, 0, ctypes.byref(n)) == -1
    assert L.irm_assemble_kv_workspace_size(None, None, 3, ctypes.byref(n)) == -1
    assert L.irm_assemble_kv_workspace_size(chunks.ctypes.data, indptr.ctypes.data, 3, ctypes.byref(n)) == 0
    assert n.value >= 256 + 16 + 3 * 24 + 32
    assert L.irm_mla_attn_prefill_workspace_size(chunks.ctypes.data, indptr.ctypes.data, 1, 1, 129,
                                                 ctypes.byref(n)) == -4
    assert L.irm_status_string(-3).decode().startswith("reused chunk")


def test_workspace_holds_the_copied_table(irm):
    """Every workspace size counts the table area the library copies the validated table
    into (status header, indptr padded to 8 bytes, 24-byte records, rounded to 256 bytes), so
    it grows with the number of chunks."""
    L = irm.lib()
    n = ctypes.c_size_t(0)
    sizes = {}
    for k in (1, 9, 10, 100):
        reqs = [[(0, 32, 0, 0)] + [(100 + 10 * i, 10, 7, 1) for i in range(k)]]
        chunks, indptr = synth.make_table(reqs)
        assert L.irm_assemble_kv_workspace_size(chunks.ctypes.data, indptr.ctypes.data, 1, ctypes.byref(n)) == 0
        asm = n.value
        assert L.irm_mla_attn_prefill_workspace_size(chunks.ctypes.data, indptr.ctypes.data, 1, 4, 16,
                                                     ctypes.byref(n)) == 0
        sizes[k] = (asm, n.value)
        tab = -(-(8 + 24 * (k + 1)) // 256) * 256
        assert n.value == 256 + tab                       # prefill: header + table
        assert asm == 256 + tab + 256                     # rotate+gather: + row starts [B+1] int64
    assert sizes[1] == sizes[9] and sizes[10][0] > sizes[9][0] and sizes[100][1] > sizes[10][1]


def test_chunk_table_block_layout(irm):
    """The binding's ChunkTable keeps indptr and the records in one block laid out as the
    workspace's table area (records at the next 8-byte boundary after indptr), which lets the
    library copy a page-locked table with one transfer."""
    chunks, indptr = synth.make_table([[(0, 32, 0, 0), (100, 50, 7, 1)], [(500, 3, 0, 0)]])
    t = irm.ChunkTable(chunks, indptr, pinned=False)
    base = t.indptr_host.ctypes.data
    assert t.chunks_host.ctypes.data - base == 16 and t.chunks_host.ctypes.data % 8 == 0
    assert list(t.indptr_host) == [0, 2, 3] and t.chunks_host.tobytes() == chunks.tobytes()
    assert list(t.validate(1000)) == [82, 3]


def test_attention_rejects_before_launch(irm):
    """Shape and workspace errors are reported before anything touches the GPU (the device
    pointers below are never dereferenced)."""
    L = irm.lib()
    chunks, indptr = synth.make_table([[(0, 32, 0, 0), (100, 50, 7, 1)]])
    fake = ctypes.c_void_p(1 << 20)
    ws = ctypes.c_void_p(1 << 21)
    args = lambda H, ws_bytes: (fake, fake, 1, H, chunks.ctypes.data, indptr.ctypes.data,
                                fake, 1000, ctypes.c_float(0.07), fake, None, ws, ws_bytes, None)
    assert L.irm_mla_attn_decode(*args(0, 1 << 20)) == -4
    assert L.irm_mla_attn_decode(*args(200, 1 << 20)) == -4
    n = ctypes.c_size_t(0)
    assert L.irm_mla_attn_decode_workspace_size(chunks.ctypes.data, indptr.ctypes.data, 1, 16,
                                                ctypes.byref(n)) == 0
    assert L.irm_mla_attn_decode(*args(16, n.value - 1)) == -8
    # n_q larger than the context
    assert L.irm_mla_attn_prefill(fake, fake, 1, 83, 16, chunks.ctypes.data, indptr.ctypes.data,
                                  fake, 1000, ctypes.c_float(0.07), fake, None, ws,
                                  1 << 20, None) == -1
    # misaligned q pointer
    bad = ctypes.c_void_p((1 << 20) + 2)
    assert L.irm_mla_attn_prefill(bad, fake, 1, 1, 16, chunks.ctypes.data, indptr.ctypes.data,
                                  fake, 1000, ctypes.c_float(0.07), fake, None, ws,
                                  1 << 20, None) == -1
    # a workspace too small for the copied table is refused before the copy
    assert L.irm_mla_attn_prefill(fake, fake, 1, 1, 16, chunks.ctypes.data, indptr.ctypes.data,
                                  fake, 1000, ctypes.c_float(0.07), fake, None, ws,
                                  256, None) == -8


def test_chunk_struct_layout_matches_header(irm):
    hdr = open(os.path.join(ROOT, "include", "irm.h")).read()
    assert "int64_t pool_offset;" in hdr and "uint8_t pad[3];" in hdr
    assert synth.CHUNK_DTYPE.itemsize == 24
    assert [synth.CHUNK_DTYPE.fields[k][1] for k in ("pool_offset", "len", "p_src", "p_tgt", "reused")] == \
        [0, 8, 12, 16, 20]


def test_rope_struct_layout_matches_header(irm):
    """irm_rope is 32 doubles + two int32 (264 bytes), as the header declares."""
    assert ctypes.sizeof(irm.Rope) == 32 * 8 + 8
    r = irm.Rope.make(np.arange(32) * 0.5, irm.ROPE_INTERLEAVED)
    assert r.inv_freq[3] == 1.5 and r.pairing == 1 and r.reserved == 0


@pytest.mark.parametrize("bad", ["pairing", "nan", "inf", "reserved"])
def test_rope_entry_points_reject_bad_specs(irm, bad):
    """The *_rope entry points check the spec on the host, before any pointer or launch."""
    r = irm.Rope.make(10000.0 ** (-2.0 * np.arange(32) / 64.0))
    if bad == "pairing":
        r.pairing = 2
    elif bad == "nan":
        r.inv_freq[7] = float("nan")
    elif bad == "inf":
        r.inv_freq[0] = float("inf")
    else:
        r.reserved = 1
    chunks, indptr = synth.make_table([[(0, 32, 0, 0), (100, 50, 7, 1)]])
    L = irm.lib()
    rp = ctypes.cast(ctypes.pointer(r), ctypes.c_void_p)
    st = L.irm_assemble_kv_rope(chunks.ctypes.data, indptr.ctypes.data, 1, None, 1000,
                                None, 0, None, 0, None, None, None, rp, None, 0, None)
    assert st == -1, L.irm_last_error()
    st = L.irm_mla_attn_decode_rope(None, None, 1, 16, chunks.ctypes.data, indptr.ctypes.data,
                                    None, 1000, 0.1, None, None, rp, None, 0, None)
    assert st == -1
    st = L.irm_mla_attn_prefill_rope(None, None, 1, 4, 16, chunks.ctypes.data, indptr.ctypes.data,
                                     None, 1000, 0.1, None, None, rp, None, 0, None)
    assert st == -1
    assert "rope" in L.irm_last_error().decode()


def test_cdc_sizes_and_slot_layout(irm):
    nb, slots = irm.cdc_sizes(np.array([0, 100, 100, 1100]))
    assert slots == (100 // 32 + 1) + 1 + (1000 // 32 + 1)
    assert list(irm.cdc_slot_base(np.array([0, 100, 100, 1100]))) == [0, 4, 5]
    assert nb >= 256


@pytest.mark.parametrize("bad", [dict(min_len=0), dict(min_len=64, max_len=32), dict(bits=64),
                                 dict(mode=2), dict(max_len=70000)])
def test_cdc_rejects_bad_params(irm, bad):
    with pytest.raises(irm.IrmError) as e:
        irm.cdc_sizes(np.array([0, 100]), irm.CdcParams.make(**bad))
    assert e.value.status == -1


def test_cdc_rejects_bad_offsets(irm):
    for offs in ([1, 100], [0, 100, 50]):
        with pytest.raises(irm.IrmError) as e:
            irm.cdc_sizes(np.array(offs))
        assert e.value.status == -1
