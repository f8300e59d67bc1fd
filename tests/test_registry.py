"""The library's host-side registry and assembler (irm_registry_*) against the reference
assembler, on sequences of requests: the chunk tables and prefill flags must agree exactly
(integer work) ["Irminsul论文详解" §5 assembly loop, §6 S1 fallback].  CPU only."""
import numpy as np
import pytest

from mla_position_independent_gb300 import synth


@pytest.fixture(scope="module")
def irm():
    from mla_position_independent_gb300 import build
    build.build()
    import mla_position_independent_gb300 as m
    m.lib()
    return m


def _segments(oracle_mod, tokens, gear, prefix_len, seed=0):
    tail = tokens[prefix_len:]
    st, ln = oracle_mod.cdc(tail, gear)
    hs = [oracle_mod.chunk_fingerprint(tail, s, l, seed) for s, l in zip(st, ln)]
    return st, ln, np.array(hs, np.uint64)


def _as_tuples(table, pre):
    return [(int(c["pool_offset"]), int(c["len"]), int(c["p_src"]), int(c["p_tgt"]), int(c["reused"]),
             int(p)) for c, p in zip(table, pre)]


def _requests(seed, n_req, vocab=20000):
    """Agentic-like requests: shared documents in shuffled order between random filler."""
    rng = np.random.default_rng(seed)
    docs = [rng.integers(0, vocab, int(rng.integers(300, 3000))).astype(np.int32) for _ in range(8)]
    reqs = []
    for _ in range(n_req):
        parts = [rng.integers(0, vocab, int(rng.integers(1, 400))).astype(np.int32)]
        for d in rng.permutation(8)[:int(rng.integers(2, 6))]:
            parts.append(docs[d])
            parts.append(rng.integers(0, vocab, int(rng.integers(0, 200))).astype(np.int32))
        reqs.append(np.concatenate(parts))
    return reqs


@pytest.mark.parametrize("s1", [False, True])
@pytest.mark.parametrize("pool_rows", [1 << 20, 6000])
def test_registry_matches_reference(irm, oracle_mod, s1, pool_rows):
    from oracle.assembler import Registry as RefRegistry
    gear = synth.gear_table(20000, seed=9)
    reg = irm.Registry(pool_rows=pool_rows, pool_base=1000, capacity=64)
    ref = RefRegistry(pool_rows=pool_rows, pool_base=1000)
    reused_total = 0
    for i, tok in enumerate(_requests(80, 12)):
        prefix = [0, 0, 17, 300][i % 4] if len(tok) > 400 else 0
        segs = _segments(oracle_mod, tok, gear, prefix)
        got, pre = reg.assemble(tok, prefix, 77, *segs, s1=s1)
        want = ref.assemble(tok, prefix, 77, *segs, s1=s1)
        assert _as_tuples(got, pre) == want, f"request {i}"
        irm.validate_chunks(got, np.array([0, len(got)], np.int32), 1000 + pool_rows)
        reused_total += sum(c[1] for c in want if c[4])
    assert reused_total > 0
    live, rows = reg.stats()
    assert rows == ref.cursor and live > 0


def test_registry_rejects_bad_segments(irm):
    reg = irm.Registry(pool_rows=1000)
    with pytest.raises(irm.IrmError):
        reg.assemble(np.zeros(100, np.int32), 0, 0, [0, 60], [50, 50], [1, 2])   # gap
    with pytest.raises(irm.IrmError):
        reg.assemble(np.zeros(100, np.int32), 0, 0, [0], [90], [1])             # does not cover
    with pytest.raises(irm.IrmError):
        reg.assemble(np.zeros(2000, np.int32), 0, 0, [0], [2000], [1])         # longer than the pool


def test_registry_heavy_eviction_with_s1(irm, oracle_mod):
    """A pool of 2500 rows (a fraction of one request) with S1: entries go stale all the time;
    the library and the reference still agree request by request."""
    from oracle.assembler import Registry as RefRegistry
    gear = synth.gear_table(20000, seed=10)
    reg = irm.Registry(pool_rows=2500, capacity=16)
    ref = RefRegistry(pool_rows=2500)
    for i, tok in enumerate(_requests(81, 20)):
        segs = _segments(oracle_mod, tok, gear, 0)
        got, pre = reg.assemble(tok, 0, 0, *segs, s1=True)
        assert _as_tuples(got, pre) == ref.assemble(tok, 0, 0, *segs, s1=True), f"request {i}"
