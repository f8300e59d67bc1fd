"""End to end through the library: token streams -> GPU content-defined chunking -> host registry
assembly -> (the test writes the rows a prefill would produce) -> fused delta-rotate decode
attention.  A second request that reorders the first one's documents reuses their cached rows
at new positions; its attention must equal the oracle's attention over a fresh encoding of
every row at its true position ("Irminsul论文详解" §5: reused chunks keep cKV and rotate k_r by
delta = p_tgt - p_src, so R(delta) R(p_src) = R(p_tgt))."""
import numpy as np
import pytest
import torch

from mla_position_independent_gb300 import synth
import mla_position_independent_gb300 as irm
from helpers import SCALE, assert_close, widen_bf16

pytestmark = pytest.mark.gpu
VOCAB = 30000


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    irm.lib()


def _token_content(seed=0):
    """A stand-in model: cKV and the RoPE content vector depend on the token id only."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((VOCAB, 512)).astype(np.float32),
            rng.standard_normal((VOCAB, 64)))


def _rows(oracle_mod, tokens, positions, ckv, kv_content):
    """bf16 KV rows [cKV(token) | RoPE(position) v(token)] (a prefill at those positions)."""
    kr = oracle_mod.rotate(kv_content[tokens], positions)
    return torch.from_numpy(np.concatenate([ckv[tokens], kr.astype(np.float32)], 1)).to(torch.bfloat16)


def test_cdc_registry_decode_pipeline(oracle_mod):
    rng = np.random.default_rng(90)
    ckv, kvc = _token_content(1)
    docs = [rng.integers(0, VOCAB, n).astype(np.int32) for n in (1500, 2200, 900)]
    filler = lambda n: rng.integers(0, VOCAB, n).astype(np.int32)
    req_a = np.concatenate([filler(100), docs[0], filler(37), docs[1], docs[2]])
    req_b = np.concatenate([filler(250), docs[2], filler(11), docs[0], docs[1], filler(60)])
    pool_rows = 16384
    kv = torch.zeros((pool_rows, 576), dtype=torch.bfloat16, device="cuda")
    reg = irm.Registry(pool_rows=pool_rows)
    H = 16
    for name, tok in (("a", req_a), ("b", req_b)):
        # 1. content-defined chunks and fingerprints on the GPU (generated Gear words)
        offs = np.array([0, len(tok)], np.int64)
        n_chunks, c_start, c_len, c_hash, ws = irm.irm_cdc_chunk(
            torch.from_numpy(tok).cuda(), offs, None, irm.CdcParams.make(gear_seed=3), vocab=VOCAB)
        irm.device_status(ws)
        k = int(n_chunks[0])
        seg = (c_start[:k].cpu().numpy(), c_len[:k].cpu().numpy(), c_hash[:k].cpu().numpy().view(np.uint64))
        # 2. chunk table from the registry
        table, prefill = reg.assemble(tok, 0, 0, *seg)
        # 3. the rows a prefill writes for the chunks it computes
        for c, pre in zip(table, prefill):
            if pre:
                p0, n, off = int(c["p_tgt"]), int(c["len"]), int(c["pool_offset"])
                kv[off:off + n] = _rows(oracle_mod, tok[p0:p0 + n], np.arange(p0, p0 + n), ckv, kvc).cuda()
        reused = int(sum(int(c["len"]) for c in table if c["reused"]))
        if name == "a":
            assert reused == 0
            continue
        # chunks straddling a document edge differ between the requests; the rest is reused
        assert reused > 0.6 * sum(len(d) for d in docs)
        # 4. decode attention for the request's next token, over the assembled table
        ql = torch.from_numpy((rng.standard_normal((1, H, 512))).astype(np.float32)).to(torch.bfloat16).cuda()
        qr = torch.from_numpy((rng.standard_normal((1, H, 64))).astype(np.float32)).to(torch.bfloat16).cuda()
        out, _, ws = irm.irm_mla_attn_decode(ql, qr, irm.ChunkTable(table, np.array([0, len(table)], np.int32)),
                                             kv, SCALE)
        irm.device_status(ws)
        # the oracle: every row freshly encoded at its true position (a full recompute)
        fresh = _rows(oracle_mod, tok, np.arange(len(tok)), ckv, kvc)
        fresh_table = synth.make_table([[(0, len(tok), 0, 0)]])
        O, _ = oracle_mod.mla_attention(synth.bits(ql[:, None]), synth.bits(qr[:, None]), *fresh_table,
                                        synth.bits(fresh), SCALE)
        assert_close(widen_bf16(out), O[:, 0], "pipeline decode vs full recompute")
