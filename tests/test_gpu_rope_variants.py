"""GPU parity of the RoPE-variant entry points ("Irminsul论文详解" §11: the delta-rotation must
use the model's own rotary class and inv_freq).  Cached k_r rows are encoded by the oracle at
their source positions with a variant (a frequency table and NeoX or interleaved pairing);
the CUDA path, given the same variant through the *_rope entry points, must match the fp64
oracle with the same variant: rotated k_r within the pages' bf16 error, attention outputs
within the bf16 output tolerances."""
import numpy as np
import pytest
import torch

from mla_position_independent_gb300 import synth
import mla_position_independent_gb300 as irm
from helpers import (SCALE, TOL_KR_REL_L2, assert_close, rel_l2, rope_tables, to_device,
                     widen_bf16)

pytestmark = pytest.mark.gpu

VARIANTS = [("base10k", irm.ROPE_INTERLEAVED), ("base500k", irm.ROPE_NEOX),
            ("yarn", irm.ROPE_NEOX), ("yarn", irm.ROPE_INTERLEAVED)]
IDS = [f"{n}-{'il' if p else 'neox'}" for n, p in VARIANTS]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    irm.lib()


def _spec(name, pairing):
    th = rope_tables()[name]
    return irm.Rope.make(th, pairing), (th, pairing)


def _encode(case, oracle_mod, rope_o):
    """Cached rows carry RoPE(position) of their content under the variant (bf16; rope_o None:
    the default convention)."""
    if case.rope_rows is None:
        return case
    enc = oracle_mod.rotate(case.rope_content, case.rope_pos, rope=rope_o)
    kr = torch.from_numpy(enc).to(torch.bfloat16).to(case.kv_rows.device)
    case.kv_rows[torch.as_tensor(case.rope_rows, device=case.kv_rows.device), 512:] = kr
    return case


@pytest.mark.parametrize("variant", VARIANTS, ids=IDS)
def test_rotate_gather_variant(oracle_mod, variant):
    rope_c, rope_o = _spec(*variant)
    rng = np.random.default_rng(7)
    reqs, p = [[]], 0
    for k, n in enumerate([32, 1, 31, 64, 65, 200, 512, 7]):
        reused = p >= 32
        d = [1, -1, 65536, -65536, 12345, 3][k % 6] if reused else 0
        reqs[0].append((int(rng.integers(0, 3000 - n)), n, p - d, reused))
        p += n
    case = to_device(synth.custom_case(reqs, n_rows=3000, n_q=0, pages=True))
    table = irm.ChunkTable(case.chunks, case.indptr)
    paged = torch.zeros((case.n_pages, 64, 576), dtype=torch.bfloat16, device="cuda")
    ws = irm.irm_assemble_kv(table, case.kv_rows, paged, torch.from_numpy(case.page_table).cuda(),
                             rope=rope_c)
    irm.device_status(ws)
    kv = synth.bits(case.kv_rows)
    slot, ref = oracle_mod.rotate_gather(kv, case.chunks, case.indptr, case.page_table, rope=rope_o)
    got = synth.bits(paged.view(-1, 576))[slot]
    pl = oracle_mod.plan(case.chunks, case.indptr)
    src = kv[pl["src_row"]]
    assert np.array_equal(got[:, :512], src[:, :512])
    z = pl["delta"] == 0
    assert np.array_equal(got[z, 512:], src[z, 512:])
    assert rel_l2(oracle_mod.widen(got[~z, 512:]), ref[~z, 512:]) <= TOL_KR_REL_L2


def _attn(case, rope_c, prefill):
    table = irm.ChunkTable(case.chunks, case.indptr)
    if prefill:
        out, _, ws = irm.irm_mla_attn_prefill(case.q_lat, case.q_rope, table, case.kv_rows, SCALE,
                                              rope=rope_c)
    else:
        out, _, ws = irm.irm_mla_attn_decode(case.q_lat[:, 0], case.q_rope[:, 0], table,
                                             case.kv_rows, SCALE, rope=rope_c)
        out = out[:, None]
    irm.device_status(ws)
    return widen_bf16(out)


@pytest.mark.parametrize("variant", VARIANTS, ids=IDS)
@pytest.mark.parametrize("H", [16, 128])
def test_attention_variant_tiny(oracle_mod, variant, H):
    """The tiny reuse workload with its cached rows encoded under the variant, queries sharp
    (std 1) so that rotation errors show in O; prefill and decode."""
    rope_c, rope_o = _spec(*variant)
    case = to_device(_encode(synth.tiny_case(0, q_std=1.0, H=H), oracle_mod, rope_o))
    kv = synth.bits(case.kv_rows)
    ql, qr = synth.bits(case.q_lat), synth.bits(case.q_rope)
    O, _ = oracle_mod.mla_attention(ql, qr, case.chunks, case.indptr, kv, SCALE, rope=rope_o)
    assert_close(_attn(case, rope_c, prefill=True), O, f"prefill H={H} {variant}")
    Od, _ = oracle_mod.mla_attention(ql[:, -1:], qr[:, -1:], case.chunks, case.indptr, kv, SCALE,
                                     rope=rope_o)
    case.q_lat, case.q_rope = case.q_lat[:, -1:].contiguous(), case.q_rope[:, -1:].contiguous()
    assert_close(_attn(case, rope_c, prefill=False), Od, f"decode H={H} {variant}")


@pytest.mark.parametrize("variant", [("yarn", irm.ROPE_INTERLEAVED), ("base500k", irm.ROPE_NEOX)],
                         ids=["yarn-il", "base500k-neox"])
def test_decode_v2lite_variant(oracle_mod, variant):
    """The V2-Lite-shaped decode (decode kernel) with a variant, sharp queries, all outputs."""
    rope_c, rope_o = _spec(*variant)
    case = to_device(synth.v2lite_decode(0, q_std=1.0))
    kv = synth.bits(case.kv_rows)
    ql, qr = synth.bits(case.q_lat), synth.bits(case.q_rope)
    O, _ = oracle_mod.mla_attention(ql, qr, case.chunks, case.indptr, kv, SCALE, rope=rope_o)
    assert_close(_attn(case, rope_c, prefill=False), O, f"v2lite decode {variant}")


def test_wrong_rotary_class_changes_the_result(oracle_mod):
    """Rows cached under an interleaved YaRN-like class: the matching spec reproduces the
    oracle, while the default class (what a plain base-10000 fallback would do) does not."""
    rope_c, rope_o = _spec("yarn", irm.ROPE_INTERLEAVED)
    case = to_device(_encode(synth.tiny_case(0, q_std=1.0), oracle_mod, rope_o))
    kv = synth.bits(case.kv_rows)
    O, _ = oracle_mod.mla_attention(synth.bits(case.q_lat), synth.bits(case.q_rope), case.chunks,
                                    case.indptr, kv, SCALE, rope=rope_o)
    assert_close(_attn(case, rope_c, prefill=True), O, "matching class")
    assert rel_l2(_attn(case, None, prefill=True), O) > 2e-2


def test_v3_decode_variant_sampled(oracle_mod):
    """The V3-shaped decode (tile kernel, split-KV) with an interleaved YaRN-like variant on
    request-private rows encoded by the oracle; sampled (request, head) outputs."""
    rope_c, rope_o = _spec("yarn", irm.ROPE_INTERLEAVED)
    case = synth.v3_decode(0, q_std=1.0, device="cuda")
    rng = np.random.default_rng(8)
    sel = np.array([[b, 0, h] for b in (0, 31, 63) for h in rng.choice(128, 6, replace=False)])
    kv = synth.bits(case.kv_rows)
    O, _ = oracle_mod.mla_attention(synth.bits(case.q_lat), synth.bits(case.q_rope), case.chunks,
                                    case.indptr, kv, SCALE, select=sel, rope=rope_o)
    got = _attn(case, rope_c, prefill=False)[sel[:, 0], sel[:, 1], sel[:, 2]]
    assert_close(got, O, "v3 decode yarn-il")


def test_chunked_prefill_variant_sampled(oracle_mod):
    rope_c, rope_o = _spec("base500k", irm.ROPE_INTERLEAVED)
    case = synth.chunked_prefill(0, device="cuda", n_q=256)
    sel = np.array([[b, i, h] for b in (0, 3) for i in (0, 128, 255) for h in (0, 77, 127)])
    kv = synth.bits(case.kv_rows)
    O, _ = oracle_mod.mla_attention(synth.bits(case.q_lat), synth.bits(case.q_rope), case.chunks,
                                    case.indptr, kv, SCALE, select=sel, rope=rope_o)
    got = _attn(case, rope_c, prefill=True)[sel[:, 0], sel[:, 1], sel[:, 2]]
    assert_close(got, O, "chunked prefill base500k-il")


def test_plain_entry_points_equal_the_default_variant(oracle_mod):
    """The entry points without a RoPE argument give bit-identical results to the *_rope ones
    called with NULL (they are the default convention)."""
    import ctypes
    case = to_device(_encode(synth.tiny_case(0, q_std=1.0), oracle_mod, None))
    table = irm.ChunkTable(case.chunks, case.indptr)
    L = irm.lib()
    ql, qr = case.q_lat[:, -1].contiguous(), case.q_rope[:, -1].contiguous()
    ref, _, _ = irm.irm_mla_attn_decode(ql, qr, table, case.kv_rows, SCALE)
    out = torch.empty_like(ref)
    ws = irm.new_workspace(irm.decode_workspace_size(table, 16))
    st = L.irm_mla_attn_decode(ql.data_ptr(), qr.data_ptr(), 1, 16, table.chunks_host.ctypes.data,
                               table.indptr_host.ctypes.data, case.kv_rows.data_ptr(), case.kv_rows.shape[0],
                               ctypes.c_float(SCALE), out.data_ptr(), None, ws.data_ptr(), ws.numel(),
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    pref, _, _ = irm.irm_mla_attn_prefill(case.q_lat, case.q_rope, table, case.kv_rows, SCALE)
    out2 = torch.empty_like(pref)
    ws2 = irm.new_workspace(irm.prefill_workspace_size(table, 16, 16))
    st = L.irm_mla_attn_prefill(case.q_lat.data_ptr(), case.q_rope.data_ptr(), 1, 16, 16,
                                table.chunks_host.ctypes.data, table.indptr_host.ctypes.data,
                                case.kv_rows.data_ptr(), case.kv_rows.shape[0], ctypes.c_float(SCALE),
                                out2.data_ptr(), None, ws2.data_ptr(), ws2.numel(),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(out2, pref)
