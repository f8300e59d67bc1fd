"""GPU parity of content-defined chunking (irm_cdc_chunk) against the oracle: chunk starts,
lengths and xxHash64 fingerprints are integer results and must match bit for bit
[summary §2.2: Gear hash over 64-token windows, xxHash64 fingerprints; walkthrough §6:
7-bit boundary test, [32, 512] clip]."""
import numpy as np
import pytest
import torch

from mla_position_independent_gb300 import synth
import mla_position_independent_gb300 as irm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    irm.lib()


def _gear_dev(gear):
    return torch.from_numpy(gear.view(np.int64).copy()).cuda()


def _run_and_check(oracle_mod, tokens, offsets, gear, params=None, check_hash=True, generated=False):
    """gear: the table both sides use; generated=True passes no table to the library, which
    then derives the same words from params.gear_seed (gear must be oracle.splitmix_gear)."""
    p = params or irm.CdcParams.make()
    n_chunks, c_start, c_len, c_hash, ws = irm.irm_cdc_chunk(
        torch.from_numpy(tokens).cuda(), offsets, None if generated else _gear_dev(gear), params,
        vocab=len(gear))
    irm.device_status(ws)
    n_chunks = n_chunks.cpu().numpy()
    c_start, c_len = c_start.cpu().numpy(), c_len.cpu().numpy()
    c_hash = c_hash.cpu().numpy().view(np.uint64) if c_hash is not None else None
    base = irm.cdc_slot_base(offsets, p.min_len)
    total = 0
    for s in range(len(offsets) - 1):
        tok = tokens[offsets[s]:offsets[s + 1]]
        st, ln = oracle_mod.cdc(tok, gear, p.min_len, p.max_len, p.bits, p.mode)
        k = int(n_chunks[s])
        assert k == len(st), f"stream {s}: {k} chunks, oracle {len(st)}"
        np.testing.assert_array_equal(c_start[base[s]:base[s] + k], st)
        np.testing.assert_array_equal(c_len[base[s]:base[s] + k], ln)
        if check_hash:
            idx = np.arange(k) if k <= 400 else np.unique(np.r_[0:50, k - 50:k,
                                                                np.random.default_rng(s).integers(0, k, 300)])
            for i in idx:
                want = oracle_mod.chunk_fingerprint(tok, st[i], ln[i], p.seed)
                assert int(c_hash[base[s] + i]) == want, f"stream {s} chunk {i} fingerprint"
        total += k
    return total


@pytest.mark.parametrize("mode", [irm.CDC_THRESHOLD, irm.CDC_LOW_BITS])
def test_cdc_edge_lengths(oracle_mod, mode):
    rng = np.random.default_rng(60 + mode)
    gear = synth.gear_table(4000, seed=1)
    lens = [0, 1, 31, 32, 33, 63, 64, 65, 511, 512, 513, 1023, 1024, 1025, 3000, 20000]
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    tokens = rng.integers(0, 4000, offsets[-1]).astype(np.int32)
    _run_and_check(oracle_mod, tokens, offsets, gear, irm.CdcParams.make(mode=mode, seed=123))


@pytest.mark.parametrize("params", [dict(min_len=1, max_len=8, bits=2), dict(min_len=16, max_len=64, bits=4),
                                    dict(min_len=100, max_len=100), dict(min_len=7, max_len=3000, bits=12)])
def test_cdc_other_parameters(oracle_mod, params):
    rng = np.random.default_rng(61)
    gear = synth.gear_table(1000, seed=2)
    offsets = np.array([0, 777, 5000, 5001, 12000], np.int64)
    tokens = rng.integers(0, 1000, offsets[-1]).astype(np.int32)
    _run_and_check(oracle_mod, tokens, offsets, gear, irm.CdcParams.make(**params))


def test_cdc_forced_boundaries(oracle_mod):
    gear = np.full(10, np.uint64(1) << np.uint64(63), np.uint64) | np.uint64(0x8000)
    tokens = (np.arange(5000) % 10).astype(np.int32)
    n = _run_and_check(oracle_mod, tokens, np.array([0, 2000, 5000], np.int64), gear)
    assert n == 4 + 6


def test_cdc_agentic_streams_full(oracle_mod):
    """The benchmark's stream shape at a smaller size: 8 streams x 64K tokens of shared
    documents at shifting offsets, every boundary and sampled fingerprints."""
    tokens, offsets = synth.cdc_streams(8, 1 << 16, seed=0)
    gear = synth.gear_table(102400, seed=0)
    n = _run_and_check(oracle_mod, tokens, offsets, gear)
    assert 2500 < n < 4500


def test_cdc_token_out_of_range_is_recorded(oracle_mod):
    gear = synth.gear_table(100, seed=3)
    tokens = np.arange(300, dtype=np.int32) % 100
    tokens[150] = 5000
    n_chunks, _, _, _, ws = irm.irm_cdc_chunk(torch.from_numpy(tokens).cuda(),
                                              np.array([0, 300], np.int64), _gear_dev(gear))
    with pytest.raises(irm.IrmError) as e:
        irm.device_status(ws)
    assert e.value.status == -7


@pytest.mark.parametrize("gear_seed", [0, 1234567])
def test_cdc_generated_gear_words(oracle_mod, gear_seed):
    """gear == NULL: the kernels derive Gear word t as the (t+1)-th SplitMix64 output; the
    oracle runs on the table of the same words."""
    tokens, offsets = synth.cdc_streams(4, 40000, seed=1)
    gear = oracle_mod.splitmix_gear(102400, gear_seed)
    _run_and_check(oracle_mod, tokens, offsets, gear, irm.CdcParams.make(gear_seed=gear_seed, seed=5),
                   generated=True)


def test_cdc_one_long_stream(oracle_mod):
    """One stream of 1M tokens: 256 speculative segments whose true starts the fix-up resolves
    in order; every boundary and sampled fingerprints."""
    tokens, offsets = synth.cdc_streams(1, 1 << 20, seed=3)
    gear = oracle_mod.splitmix_gear(102400, 11)
    n = _run_and_check(oracle_mod, tokens, offsets, gear, irm.CdcParams.make(gear_seed=11), generated=True)
    assert n > 5000


def test_cdc_long_chunks_cross_segments(oracle_mod):
    """max_len larger than a walk segment (chunks spanning several segments) and a sparse test."""
    tokens, offsets = synth.cdc_streams(3, 100000, seed=4)
    gear = oracle_mod.splitmix_gear(102400, 5)
    _run_and_check(oracle_mod, tokens, offsets, gear,
                   irm.CdcParams.make(min_len=3000, max_len=20000, bits=12, gear_seed=5), generated=True)


def test_cdc_many_streams(oracle_mod):
    """More streams than the launch parameters carry (1500, lengths 0 to 700): the offsets go
    through the workspace and the per-stream bases are computed on the device."""
    rng = np.random.default_rng(62)
    gear = synth.gear_table(5000, seed=6)
    lens = rng.integers(0, 700, 1500)
    lens[::97] = 0
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    tokens = rng.integers(0, 5000, offsets[-1]).astype(np.int32)
    _run_and_check(oracle_mod, tokens, offsets, gear, irm.CdcParams.make(seed=9))


def test_cdc_segment_boundaries(oracle_mod):
    """Streams whose lengths sit at and around multiples of the 4096-token walk segment, with
    chunk limits that make chunks end exactly at, before and after segment ends."""
    rng = np.random.default_rng(63)
    gear = synth.gear_table(3000, seed=7)
    lens = [4095, 4096, 4097, 8191, 8192, 8193, 12288 + 511, 12288 + 512]
    offsets = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    tokens = rng.integers(0, 3000, offsets[-1]).astype(np.int32)
    for params in (irm.CdcParams.make(), irm.CdcParams.make(min_len=64, max_len=64),
                   irm.CdcParams.make(min_len=512, max_len=4096, bits=9)):
        _run_and_check(oracle_mod, tokens, offsets, gear, params)
