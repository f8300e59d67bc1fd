"""Pins of the oracle's content-defined chunking (CPU only): the 64-token-window Gear hash
[summary §2.2: rolling Gear hash over 64-token windows], the 7-bit boundary test and the
[32, 512] chunk clip [walkthrough §6], and the xxHash64 chunk fingerprint [summary §2.2]."""
import json
import os

import numpy as np
import pytest

from mla_position_independent_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
M64 = (1 << 64) - 1


def _recurrence(tokens, gear):
    """h_i = 2 h_{i-1} + G[x_i] mod 2^64 (Python ints): the window sum written as a recurrence."""
    out, h = [], 0
    for t in tokens:
        h = ((h << 1) + int(gear[t])) & M64
        out.append(h)
    return np.array(out, dtype=np.uint64)


def _candidates(h, bits=7, mode=0):
    h = h.astype(np.uint64)
    if mode == 1:
        return (h & np.uint64((1 << bits) - 1)) == 0
    return (h >> np.uint64(64 - bits)) == 0


def test_xxh64_reference_values(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "xxh64_reference.json")))
    for c in g["cases"]:
        assert oracle_mod.xxh64(c["input_utf8"].encode(), c["seed"]) == int(c["xxh64"], 16)


def test_xxh64_lengths_and_seed(oracle_mod):
    """Every input length from 0 to 100 (all tail paths) gives a distinct hash, a one-byte
    change or another seed changes it."""
    rng = np.random.default_rng(40)
    data = rng.integers(0, 256, 100, dtype=np.uint8).tobytes()
    hs = {oracle_mod.xxh64(data[:n]) for n in range(101)}
    assert len(hs) == 101
    for n in (1, 7, 8, 31, 32, 33, 64, 100):
        b = bytearray(data[:n])
        b[n // 2] ^= 1
        assert oracle_mod.xxh64(bytes(b)) != oracle_mod.xxh64(data[:n])
        assert oracle_mod.xxh64(data[:n], 1) != oracle_mod.xxh64(data[:n], 0)


def test_chunk_fingerprint_is_xxh64_of_le_int32(oracle_mod):
    tok = np.array([1, 258, 70000, 102399, 0, 5], np.int32)
    assert oracle_mod.chunk_fingerprint(tok, 1, 4, 9) == oracle_mod.xxh64(tok[1:5].astype("<i4").tobytes(), 9)


def test_gear_window_sum_is_the_recurrence(oracle_mod):
    rng = np.random.default_rng(41)
    gear = synth.gear_table(5000, seed=3)
    tokens = rng.integers(0, 5000, 700).astype(np.int32)
    np.testing.assert_array_equal(oracle_mod.gear_hash(tokens, gear), _recurrence(tokens, gear))


def test_gear_hash_sees_exactly_64_tokens(oracle_mod):
    """h_i does not depend on tokens 64 or more positions back, and does on the token 63 back
    (through the top bit, which the threshold test reads)."""
    rng = np.random.default_rng(42)
    gear = synth.gear_table(1000, seed=4)
    tokens = rng.integers(0, 1000, 400).astype(np.int32)
    h0 = oracle_mod.gear_hash(tokens, gear)
    t2 = tokens.copy()
    t2[:200] = rng.integers(0, 1000, 200)
    h2 = oracle_mod.gear_hash(t2, gear)
    np.testing.assert_array_equal(h0[263:], h2[263:])
    a, b = next((a, b) for a in range(1000) for b in range(1000) if (int(gear[a]) - int(gear[b])) & 1)
    t3 = tokens.copy()
    t3[300 - 63] = a
    t4 = tokens.copy()
    t4[300 - 63] = b
    assert oracle_mod.gear_hash(t3, gear)[300] != oracle_mod.gear_hash(t4, gear)[300]


@pytest.mark.parametrize("mode", [0, 1])
def test_cdc_rules_by_brute_force(oracle_mod, mode):
    """Chunks tile the stream; every chunk but the last ends at a candidate with length >= 32
    or at length 512; no candidate lies in [start + 31, end - 1]."""
    rng = np.random.default_rng(43 + mode)
    gear = synth.gear_table(3000, seed=5)
    for n in (1, 31, 32, 33, 600, 5000):
        tokens = rng.integers(0, 3000, n).astype(np.int32)
        starts, lens = oracle_mod.cdc(tokens, gear, mode=mode)
        cand = _candidates(_recurrence(tokens, gear), mode=mode)
        assert starts[0] == 0 and lens.sum() == n
        np.testing.assert_array_equal(starts[1:], (starts + lens)[:-1])
        for s, L in zip(starts, lens):
            e = s + L - 1
            assert 1 <= L <= 512
            if e != n - 1:
                assert (L >= 32 and cand[e]) or L == 512
            assert not cand[s + 31:e].any()


def test_cdc_forced_boundaries_every_512_without_candidates(oracle_mod):
    """A table whose hashes never pass the test gives chunks of exactly 512 (and a tail)."""
    gear = np.full(10, np.uint64(1) << np.uint64(63), np.uint64) | np.uint64(0x8000)
    tokens = np.arange(2000, dtype=np.int32) % 10
    starts, lens = oracle_mod.cdc(tokens, gear)
    assert list(lens) == [512, 512, 512, 464]


def test_cdc_mean_length_follows_the_7bit_test(oracle_mod):
    """On random tokens a position passes the test with probability 2^-7, so after the 31
    positions a chunk skips, its length is 31 + geometric(1/128) clipped at 512: mean
    31 + 128 (1 - (127/128)^481) = 155.9 (the pages quote about 128)."""
    rng = np.random.default_rng(44)
    gear = synth.gear_table(102400, seed=6)
    tokens = rng.integers(0, 102400, 400000).astype(np.int32)
    for mode in (0, 1):
        starts, lens = oracle_mod.cdc(tokens, gear, mode=mode)
        expect = 31 + 128 * (1 - (127 / 128) ** 481)
        assert abs(lens[:-1].mean() - expect) / expect < 0.05


def test_cdc_boundaries_follow_content_after_a_shift(oracle_mod):
    """Walkthrough §6: the same document behind prefixes of different lengths (a 13-token
    shift) gets the same chunk boundaries relative to the document once the chunkers have
    met a common boundary; fixed-offset blocks would not line up."""
    rng = np.random.default_rng(45)
    gear = synth.gear_table(50000, seed=7)
    doc = rng.integers(0, 50000, 6000).astype(np.int32)
    pa = rng.integers(0, 50000, 1024).astype(np.int32)
    pb = rng.integers(0, 50000, 1037).astype(np.int32)
    sa, _ = oracle_mod.cdc(np.concatenate([pa, doc]), gear)
    sb, _ = oracle_mod.cdc(np.concatenate([pb, doc]), gear)
    ra = set((sa[sa >= 1024] - 1024).tolist())
    rb = set((sb[sb >= 1037] - 1037).tolist())
    tail_a = {x for x in ra if x >= 2048}
    tail_b = {x for x in rb if x >= 2048}
    assert tail_a and tail_a == tail_b


def test_splitmix_gear_reference_values(oracle_mod):
    """Gear words from SplitMix64: word t is the generator's (t+1)-th output."""
    g = json.load(open(os.path.join(GOLDEN, "splitmix64_reference.json")))
    for c in g["cases"]:
        got = oracle_mod.splitmix_gear(len(c["outputs"]), c["seed"])
        assert [int(x) for x in got] == [int(h, 16) for h in c["outputs"]]
