"""Pins of the reference assembler (CPU only) against what the assembly loop of
"Irminsul论文详解" §5 fixes: exact prefix first, carve-out prefill below position 32, a registry
hit reuses the cached rows with delta = p - p_src, a miss is prefilled and registered; and the
S1 fallback of §6 (128-token sub-windows of a missed chunk)."""
import numpy as np
import pytest

from mla_position_independent_gb300 import synth


def _cdc(oracle_mod, tokens, gear):
    st, ln = oracle_mod.cdc(tokens, gear)
    hs = [oracle_mod.chunk_fingerprint(tokens, s, l) for s, l in zip(st, ln)]
    return st, ln, hs


def _check_table(out, ctx):
    """Chunks tile [0, ctx) in order, positions below 32 are never reused."""
    p = 0
    for off, ln, ps, pt, reused, prefill in out:
        assert pt == p and ln > 0
        assert not (reused and pt < 32)
        assert not (reused and prefill)
        p += ln
    assert p == ctx


def test_first_request_prefills_everything(oracle_mod):
    from oracle.assembler import Registry
    rng = np.random.default_rng(70)
    gear = synth.gear_table(5000, seed=1)
    tok = rng.integers(0, 5000, 3000).astype(np.int32)
    reg = Registry(pool_rows=100000)
    out = reg.assemble(tok, 0, 0, *_cdc(oracle_mod, tok, gear))
    _check_table(out, 3000)
    assert all(prefill == 1 and reused == 0 for *_, reused, prefill in out)
    # rows of consecutive fresh chunks are consecutive in the ring
    offs = [o for o, *_ in out]
    assert offs == sorted(offs) and offs[0] == 0


def test_moved_document_is_reused_with_delta(oracle_mod):
    """Walkthrough §5: the same document at another position hits the registry; its chunks
    are reused with p_src = the position they were prefilled at (delta = p_tgt - p_src)."""
    from oracle.assembler import Registry
    rng = np.random.default_rng(71)
    gear = synth.gear_table(50000, seed=2)
    doc = rng.integers(0, 50000, 4000).astype(np.int32)
    a = np.concatenate([rng.integers(0, 50000, 700).astype(np.int32), doc])
    b = np.concatenate([rng.integers(0, 50000, 1913).astype(np.int32), doc])
    reg = Registry(pool_rows=1 << 20)
    out_a = reg.assemble(a, 0, 0, *_cdc(oracle_mod, a, gear))
    out_b = reg.assemble(b, 0, 0, *_cdc(oracle_mod, b, gear))
    _check_table(out_b, len(b))
    reused = [c for c in out_b if c[4] == 1]
    assert sum(c[1] for c in reused) > 0.8 * len(doc)
    fresh_a = {c[3]: c for c in out_a if c[5] == 1}
    for off, ln, ps, pt, _, _ in reused:
        src = fresh_a[ps]                       # prefilled in request a at position p_src
        assert src[0] == off and src[1] == ln
        assert pt - ps == 1913 - 700            # the document moved by 1213 positions
        np.testing.assert_array_equal(b[pt:pt + ln], a[ps:ps + ln])


def test_exact_prefix_and_carve_out(oracle_mod):
    from oracle.assembler import Registry
    rng = np.random.default_rng(72)
    gear = synth.gear_table(1000, seed=3)
    tok = rng.integers(0, 1000, 2000).astype(np.int32)
    reg = Registry(pool_rows=1 << 16, pool_base=5000)
    # a prefix of 20 tokens (shorter than the carve-out): the first tail chunk starts below 32
    st, ln, hs = _cdc(oracle_mod, tok[20:], gear)
    out = reg.assemble(tok, 20, 777, st, ln, hs)
    _check_table(out, 2000)
    assert out[0] == (777, 20, 0, 0, 0, 0)
    assert out[1][3] == 20 and out[1][5] == 1 and out[1][0] == 5000
    # the same request again: the prefix is reused in place, the chunk that started at 20 is
    # a carve-out prefill again (never registered), the others hit
    out2 = reg.assemble(tok, 20, 777, st, ln, hs)
    assert out2[1][5] == 1 and out2[1][4] == 0
    assert all(c[4] == 1 and c[3] - c[2] == 0 for c in out2[2:])


def test_duplicates_within_one_request_are_not_hits(oracle_mod):
    from oracle.assembler import Registry
    rng = np.random.default_rng(73)
    gear = synth.gear_table(3000, seed=4)
    doc = rng.integers(0, 3000, 2000).astype(np.int32)
    tok = np.concatenate([rng.integers(0, 3000, 100).astype(np.int32), doc, doc])
    reg = Registry(pool_rows=1 << 16)
    out = reg.assemble(tok, 0, 0, *_cdc(oracle_mod, tok, gear))
    assert all(c[4] == 0 for c in out)
    out2 = reg.assemble(tok, 0, 0, *_cdc(oracle_mod, tok, gear))
    assert sum(c[1] for c in out2 if c[4]) > 3000


def test_ring_eviction_makes_entries_stale(oracle_mod):
    from oracle.assembler import Registry
    rng = np.random.default_rng(74)
    gear = synth.gear_table(3000, seed=5)
    a = rng.integers(0, 3000, 3000).astype(np.int32)
    reg = Registry(pool_rows=4096)
    seg_a = _cdc(oracle_mod, a, gear)
    reg.assemble(a, 0, 0, *seg_a)
    filler = rng.integers(0, 3000, 3000).astype(np.int32)
    reg.assemble(filler, 0, 0, *_cdc(oracle_mod, filler, gear))  # the ring turns past a's rows
    out = reg.assemble(a, 0, 0, *seg_a)
    hits = sum(c[1] for c in out if c[4])
    assert hits < 2000  # most of a's rows were overwritten
    for off, ln, *_ in out:
        assert 0 <= off and off + ln <= 4096


def test_s1_recovers_windows_of_a_missed_chunk(oracle_mod):
    """Walkthrough §6: a CDC chunk that misses is split into 128-token windows that are
    looked up again; windows prefilled before (as windows of an earlier chunk) are reused."""
    from oracle.assembler import Registry
    rng = np.random.default_rng(75)
    body = rng.integers(0, 9000, 512).astype(np.int32)
    a = np.concatenate([rng.integers(0, 9000, 64).astype(np.int32), body])
    b = np.concatenate([rng.integers(0, 9000, 64).astype(np.int32), body[:384], rng.integers(0, 9000, 128).astype(np.int32)])
    reg = Registry(pool_rows=1 << 16)
    # hand-made segments: one 64-token head, then one 512-token chunk
    seg = lambda t: ([0, 64], [64, 512], [12345, oracle_mod.chunk_fingerprint(t, 64, 512)])
    reg.assemble(a, 0, 0, *seg(a), s1=True)
    out = reg.assemble(b, 0, 0, *seg(b), s1=True)
    _check_table(out, len(b))
    reused = [c for c in out if c[4]]
    assert [c[1] for c in reused] == [128, 128, 128]
    assert [c[3] for c in reused] == [64, 192, 320]
    assert out[-1][5] == 1 and out[-1][1] == 128
    # without S1 the changed chunk misses as a whole
    reg2 = Registry(pool_rows=1 << 16)
    reg2.assemble(a, 0, 0, *seg(a))
    assert not any(c[4] for c in reg2.assemble(b, 0, 0, *seg(b)))
