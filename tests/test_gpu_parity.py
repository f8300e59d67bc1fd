"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, on the same seeded
inputs.  Indices and positions are compared bit for bit; bf16 outputs within relative L2
5e-3 and max-abs 2e-2; rotated k_r within relative L2 4.7e-3 (the pages' bf16 figure)."""
import numpy as np
import pytest
import torch

from mla_position_independent_gb300 import synth
import mla_position_independent_gb300 as irm
from helpers import (SCALE, TOL_KR_REL_L2, assert_close, encode_rope_rows, rel_l2, to_device,
                     widen_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    irm.lib()


# ----------------------------------------------------------------------------- assembly

def _assemble_and_check(case, oracle_mod, check_plan=True):
    case = to_device(case)
    table = irm.ChunkTable(case.chunks, case.indptr)
    n_rows = case.kv_rows.shape[0]
    total = int(case.chunks["len"].astype(np.int64).sum())
    paged = torch.zeros((case.n_pages, 64, 576), dtype=torch.bfloat16, device="cuda")
    pt = torch.from_numpy(case.page_table).cuda()
    outs = [torch.full((total,), -7, dtype=torch.int32, device="cuda") for _ in range(3)]
    ws = irm.irm_assemble_kv(table, case.kv_rows, paged, pt, *outs)
    irm.device_status(ws)
    kv_bits = synth.bits(case.kv_rows)
    if check_plan:
        pl = oracle_mod.plan(case.chunks, case.indptr)
        assert np.array_equal(outs[0].cpu().numpy(), pl["src_row"])
        assert np.array_equal(outs[1].cpu().numpy(), pl["delta"])
        assert np.array_equal(outs[2].cpu().numpy(), pl["pos_src"])
    slot, ref = oracle_mod.rotate_gather(kv_bits, case.chunks, case.indptr, case.page_table)
    got_bits = synth.bits(paged.view(-1, 576))[slot]
    # cKV: byte-identical; rows with delta == 0: byte-identical k_r
    src_bits = kv_bits[oracle_mod.plan(case.chunks, case.indptr)["src_row"]]
    assert np.array_equal(got_bits[:, :512], src_bits[:, :512])
    pl = oracle_mod.plan(case.chunks, case.indptr)
    zero = pl["delta"] == 0
    assert np.array_equal(got_bits[zero, 512:], src_bits[zero, 512:])
    if (~zero).any():
        got = oracle_mod.widen(got_bits[~zero, 512:])
        r = rel_l2(got, ref[~zero, 512:])
        assert r <= TOL_KR_REL_L2, f"rotated k_r rel L2 {r:.3e}"
        return r
    return 0.0


def test_assemble_tiny(oracle_mod):
    case = encode_rope_rows(synth.tiny_case(0), oracle_mod)
    case.page_table = np.random.default_rng(3).permutation(8).astype(np.int32)[None]
    case.n_pages = 8
    _assemble_and_check(case, oracle_mod)


@pytest.mark.parametrize("lens", [[32, 1, 31, 32, 33, 63, 64, 65, 512], [40], [32, 7], [32, 100, 3]])
@pytest.mark.parametrize("deltas", [(0, 1, -1), (65536, -65536, 12345)])
def test_assemble_edge_cases(oracle_mod, lens, deltas):
    rng = np.random.default_rng(sum(lens))
    n_rows = 2048
    reqs, p = [[]], 0
    for k, n in enumerate(lens):
        reused = p >= 32
        d = deltas[k % len(deltas)] if reused else 0
        off = int(rng.integers(0, n_rows - n))
        reqs[0].append((off, n, p - d, reused))
        p += n
    case = synth.custom_case(reqs, n_rows=n_rows, n_q=0, pages=True)
    _assemble_and_check(case, oracle_mod)


def test_assemble_multi_request(oracle_mod):
    case = synth.custom_case([[(0, 32, 0, 0), (500, 70, 9, 1), (100, 1, 50, 1)],
                              [(900, 5, 0, 0)], [(1000, 32, 0, 0), (32, 129, -4000, 1)]],
                             n_rows=1200, n_q=0, pages=True)
    _assemble_and_check(case, oracle_mod)


def test_assemble_long_chunks_split_across_ctas(oracle_mod):
    """Chunks far longer than a CTA's share of the rows: the CTAs split the batch's rows in
    equal ranges, so many of them copy parts of one chunk (and a range can end inside one)."""
    case = synth.custom_case([[(0, 32, 0, 0), (40, 30000, 100, 1), (30100, 7, 9000, 1)],
                              [(31000, 5000, 0, 0), (36100, 3333, -777, 1)]],
                             n_rows=40000, n_q=0, pages=True)
    _assemble_and_check(case, oracle_mod)


def test_assemble_many_requests(oracle_mod):
    """300 requests (more than the launch parameters carry row offsets for, so the kernel
    reads them from the device): ragged lengths, reused and fresh chunks, paged output and
    the per-row plan."""
    rng = np.random.default_rng(61)
    n_rows = 9000
    reqs = []
    for b in range(300):
        p, req = 0, [(int(rng.integers(0, n_rows - 32)), 32, 0, 0)]
        p = 32
        for _ in range(int(rng.integers(0, 4))):
            n = int(rng.integers(1, 300))
            reused = rng.random() < 0.7
            d = int(rng.integers(-5000, 5001)) if reused else 0
            req.append((int(rng.integers(0, n_rows - n)), n, p - d, int(reused)))
            p += n
        reqs.append(req)
    case = synth.custom_case(reqs, n_rows=n_rows, n_q=0, pages=True)
    _assemble_and_check(case, oracle_mod)


def test_rotate_gather_64k_rows_full(oracle_mod):
    case = synth.rotate_gather_case(1 << 16, seed=0, device="cuda")
    r = _assemble_and_check(case, oracle_mod)
    assert r < 2.5e-3


def _check_gather_sampled(case, oracle_mod, n_rows):
    """Rotate+gather of a workload, checked on sampled target rows plus every chunk's
    endpoints (the first 20000 of each kind): cKV and unrotated k_r bit-exact, rotated k_r
    within the pages' bf16 error."""
    table = irm.ChunkTable(case.chunks, case.indptr)
    paged = torch.empty((case.n_pages, 64, 576), dtype=torch.bfloat16, device="cuda")
    pt = torch.from_numpy(case.page_table).cuda()
    ws = irm.irm_assemble_kv(table, case.kv_rows, paged, pt)
    irm.device_status(ws)
    rng = np.random.default_rng(1)
    ends = np.concatenate([case.chunks["p_tgt"], case.chunks["p_tgt"] + case.chunks["len"] - 1])
    t = np.unique(np.concatenate([rng.integers(0, n_rows, 20000), ends[:20000], ends[-2000:]]))
    # only the rows the oracle needs are copied to the host
    pl = oracle_mod.plan(case.chunks, case.indptr)
    src = pl["src_row"][t]
    kv_sub = synth.bits(case.kv_rows[torch.from_numpy(src).cuda()])
    ref = oracle_mod.assemble(kv_sub, np.arange(len(t)), pl["delta"][t])
    slot = case.page_table[0, t // 64].astype(np.int64) * 64 + t % 64
    got = synth.bits(paged.view(-1, 576)[torch.from_numpy(slot).cuda()])
    assert np.array_equal(got[:, :512], kv_sub[:, :512])
    nz = pl["delta"][t] != 0
    assert np.array_equal(got[~nz, 512:], kv_sub[~nz, 512:])
    assert rel_l2(oracle_mod.widen(got[nz, 512:]), ref[nz, 512:]) <= TOL_KR_REL_L2


@pytest.mark.parametrize("n_rows", [1 << 20, 1 << 22])
def test_rotate_gather_full_size_sampled(oracle_mod, n_rows):
    """The configured sizes, checked on sampled target rows plus every chunk's endpoints."""
    case = synth.rotate_gather_case(n_rows, seed=0, device="cuda")
    _check_gather_sampled(case, oracle_mod, n_rows)


@pytest.mark.parametrize("n_rows", [1 << 24, 1 << 26])
def test_rotate_gather_largest_sizes_sampled(oracle_mod, n_rows):
    """The sweep's 16M- and 64M-row sizes (38.6 and 154.6 GB of row store plus pages), when
    the device has the memory free; the row store is filled 1M rows at a time."""
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    if free < 2 * n_rows * 1152 + (2 << 30):
        pytest.skip(f"needs {2 * n_rows * 1152 / 1e9:.1f} GB of free device memory")
    case = synth.rotate_gather_case(n_rows, seed=0, device="cuda", fill_kv=False)
    g = torch.Generator(device="cuda")
    g.manual_seed(123)
    step = 1 << 20
    for i in range(0, n_rows, step):
        case.kv_rows[i:i + step] = torch.randn((min(step, n_rows - i), 576), generator=g,
                                               device="cuda").to(torch.bfloat16)
    try:
        _check_gather_sampled(case, oracle_mod, n_rows)
    finally:
        del case
        torch.cuda.empty_cache()


# ----------------------------------------------------------------------------- attention

def _attn_gpu(case, prefill):
    table = irm.ChunkTable(case.chunks, case.indptr)
    B, n_q, H = case.q_lat.shape[:3]
    if prefill:
        lse = torch.empty((B, n_q, H), dtype=torch.float32, device="cuda")
        out, lse, ws = irm.irm_mla_attn_prefill(case.q_lat, case.q_rope, table, case.kv_rows,
                                                SCALE, lse=lse)
    else:
        lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
        out, lse, ws = irm.irm_mla_attn_decode(case.q_lat[:, 0], case.q_rope[:, 0], table,
                                               case.kv_rows, SCALE, lse=lse)
        out, lse = out[:, None], lse[:, None]
    irm.device_status(ws)
    return out, lse


def _check_attn(case, oracle_mod, prefill, select=None, what=""):
    out, lse = _attn_gpu(case, prefill)
    kv = synth.bits(case.kv_rows)
    ql, qr = synth.bits(case.q_lat), synth.bits(case.q_rope)
    O, L = oracle_mod.mla_attention(ql, qr, case.chunks, case.indptr, kv, SCALE, select=select)
    got = widen_bf16(out)
    gl = lse.cpu().numpy().astype(np.float64)
    if select is not None:
        s = np.asarray(select)
        got, gl = got[s[:, 0], s[:, 1], s[:, 2]], gl[s[:, 0], s[:, 1], s[:, 2]]
    r, m = assert_close(got, O, what or case.name)
    assert np.max(np.abs(gl - L)) < 2e-2, f"lse max abs {np.max(np.abs(gl - L)):.3e}"
    return r, m


@pytest.mark.parametrize("q_std", [synth.Q_STD, 1.0])
def test_prefill_tiny(oracle_mod, q_std):
    case = to_device(encode_rope_rows(synth.tiny_case(0, q_std=q_std), oracle_mod))
    _check_attn(case, oracle_mod, prefill=True)


@pytest.mark.parametrize("q_std", [synth.Q_STD, 1.0])
def test_decode_v2lite_full(oracle_mod, q_std):
    case = to_device(synth.v2lite_decode(0, q_std=q_std))
    _check_attn(case, oracle_mod, prefill=False)


def test_decode_v3_sampled(oracle_mod):
    """The full V3-shaped decode, checked on 4 heads of every one of the 64 requests (head 0,
    head 127 and two seeded ones), so every request's KV split and merge is covered."""
    case = synth.v3_decode(0, device="cuda")
    rng = np.random.default_rng(5)
    sel = np.array([[b, 0, h] for b in range(64)
                    for h in np.unique(np.concatenate([[0, 127], rng.choice(126, 2, replace=False) + 1]))])
    _check_attn(case, oracle_mod, prefill=False, select=sel)


def test_decode_v3_sharp_sampled(oracle_mod):
    case = synth.v3_decode(0, q_std=1.0, device="cuda")
    sel = np.array([[b, 0, h] for b in (0, 63) for h in (0, 77, 127)])
    _check_attn(case, oracle_mod, prefill=False, select=sel)


def test_prefill_chunked_sampled(oracle_mod):
    """The full chunked prefill (128 heads: a 128-row query tile is one query), checked in
    every request on one query of every block of 64 consecutive query tiles (two heads each)
    and on the first, second and last query (three heads each).  Every query sees the whole
    prefix, so every KV tile, including each one that straddles a chunk boundary, enters
    every sampled row."""
    case = synth.chunked_prefill(0, device="cuda")
    rng = np.random.default_rng(6)
    sel = []
    for b in range(4):
        for blk in range(0, 2048, 64):
            i = blk + int(rng.integers(0, 64))
            sel += [[b, i, int(h)] for h in rng.choice(128, 2, replace=False)]
        sel += [[b, i, h] for i in (0, 1, 2047) for h in (0, 64, 127)]
    _check_attn(case, oracle_mod, prefill=True, select=np.array(sel))


@pytest.mark.parametrize("H", [8, 16, 32, 64, 128])
@pytest.mark.parametrize("lens", [[40], [32, 1, 31, 33, 63, 64, 65], [32, 17], [32, 200, 128, 3]])
def test_attention_edge_cases(oracle_mod, H, lens):
    rng = np.random.default_rng(H + len(lens))
    n_rows = 2048
    reqs = []
    for b in range(2):
        p, req = 0, []
        for k, n in enumerate(lens):
            reused = p >= 32 and k % 2 == 1
            d = [1, -1, 65536, -65536, 0, 777][k % 6] if reused else 0
            req.append((int(rng.integers(0, n_rows - n)), n, p - d, reused))
            p += n
        reqs.append(req)
    ctx = sum(lens)
    for n_q in sorted({1, min(5, ctx), min(ctx, 70)}):
        case = to_device(synth.custom_case(reqs, n_rows=n_rows, n_q=n_q, H=H, q_std=1.0,
                                           seed=n_q))
        _check_attn(case, oracle_mod, prefill=True, what=f"H={H} lens={lens} n_q={n_q}")
        if n_q == 1:
            _check_attn(case, oracle_mod, prefill=False, what=f"decode H={H} lens={lens}")


@pytest.mark.parametrize("H", [3, 40, 100])
def test_attention_head_counts_not_dividing_the_tile(oracle_mod, H):
    """A query tile holds floor(128 / H) queries of H heads (rows past them unused); prefill
    over several query tiles and decode, with ragged chunks and large deltas."""
    rng = np.random.default_rng(H)
    n_rows = 4096
    reqs = []
    for b in range(2):
        p, req = 0, []
        for k, n in enumerate([32, 200, 128, 3, 77]):
            reused = p >= 32 and k % 2 == 1
            d = [1, -1, 65536, -65536, 0, 777][k % 6] if reused else 0
            req.append((int(rng.integers(0, n_rows - n)), n, p - d, reused))
            p += n
        reqs.append(req)
    for n_q in (1, 70):
        case = to_device(synth.custom_case(reqs, n_rows=n_rows, n_q=n_q, H=H, q_std=1.0, seed=n_q + H))
        _check_attn(case, oracle_mod, prefill=True, what=f"H={H} n_q={n_q}")
        if n_q == 1:
            _check_attn(case, oracle_mod, prefill=False, what=f"decode H={H}")


def _ragged_decode_case(ctxs, H, seed):
    """Requests of very different context lengths in one decode batch: with the splits of a
    request sized for the longest one, short requests leave whole splits without tiles."""
    rng = np.random.default_rng(seed)
    n_rows = 12000
    reqs = []
    for ctx in ctxs:
        p, req = 0, []
        while p < ctx:
            n = 32 if p == 0 else int(min(ctx - p, rng.integers(1, 300)))
            n = min(n, ctx - p)
            reused = p >= 32 and rng.random() < 0.75
            d = int(rng.integers(-4096, 4097)) if reused else 0
            req.append((int(rng.integers(0, n_rows - n)), n, p - d, reused))
            p += n
        reqs.append(req)
    return to_device(synth.custom_case(reqs, n_rows=n_rows, n_q=1, H=H, q_std=1.0, seed=seed))


@pytest.mark.parametrize("H", [16, 32])
@pytest.mark.parametrize("ctxs", [[9000], [33, 100, 4000, 64, 9000], [64] * 3 + [4097]])
def test_decode_ragged_batch(oracle_mod, H, ctxs):
    case = _ragged_decode_case(ctxs, H, seed=len(ctxs) + H)
    _check_attn(case, oracle_mod, prefill=False, what=f"decode H={H} ctxs={ctxs}")


def test_decode_many_requests(oracle_mod):
    """More clusters than fit at once (several waves), sampled outputs."""
    case = _ragged_decode_case([700 + 37 * b for b in range(40)], 16, seed=3)
    sel = np.array([[b, 0, h] for b in (0, 17, 39) for h in (0, 5, 15)])
    _check_attn(case, oracle_mod, prefill=False, select=sel, what="decode 40 requests")


@pytest.mark.parametrize("H", [64, 128])
@pytest.mark.parametrize("ctxs", [[8192], [8192, 3000]])
def test_decode_split_kv(oracle_mod, H, ctxs):
    """One or two long requests with many heads: the tile kernel splits each request's KV
    over several clusters and merges their partials (the last cluster of a query tile)."""
    case = _ragged_decode_case(ctxs, H, seed=7 + H)
    sel = np.array([[b, 0, h] for b in range(len(ctxs)) for h in (0, 1, H // 2, H - 1)])
    _check_attn(case, oracle_mod, prefill=False, select=sel, what=f"split-KV decode H={H} ctxs={ctxs}")


@pytest.mark.parametrize("H", [64, 128])
def test_decode_many_heads_ragged_batch(oracle_mod, H):
    """96 requests of ragged contexts (24 to 250 KV tiles) with many heads: more query tiles
    than fit on the GPU at once, so the tile kernel runs in waves; sampled on every request."""
    rng = np.random.default_rng(40 + H)
    ctxs = [int(c) for c in rng.integers(1500, 16000, 96)]
    case = _ragged_decode_case(ctxs, H, seed=41 + H)
    sel = np.array([[b, 0, h] for b in range(96) for h in (0, int(rng.integers(1, H - 1)), H - 1)])
    _check_attn(case, oracle_mod, prefill=False, what=f"ragged decode H={H}", select=sel)


@pytest.mark.parametrize("H", [64, 128])
def test_decode_long_first_split(oracle_mod, H):
    """40 requests (fewer query tiles than cluster slots) of ragged contexts, some of a single KV
    tile: each query tile's KV is cut into a long leading split, all scheduled first, and a short
    trailing one run on the cluster slots left (empty for the one-tile requests); the two
    partials are merged by whichever finishes last.  Sampled on every request."""
    rng = np.random.default_rng(50 + H)
    ctxs = [int(c) for c in rng.integers(4000, 9000, 40)]
    ctxs[3], ctxs[17], ctxs[30] = 33, 64, 65
    case = _ragged_decode_case(ctxs, H, seed=51 + H)
    sel = np.array([[b, 0, h] for b in range(40) for h in (0, int(rng.integers(1, H - 1)), H - 1)])
    _check_attn(case, oracle_mod, prefill=False, what=f"long-first decode H={H}", select=sel)


def test_decode_single_tile_requests(oracle_mod):
    """100 requests of at most one KV tile each, 128 heads; every output row is checked."""
    ctxs = [33 + (13 * b) % 32 for b in range(100)]
    case = _ragged_decode_case(ctxs, 128, seed=43)
    _check_attn(case, oracle_mod, prefill=False, what="decode, one tile per request")


@pytest.mark.parametrize("H", [16, 32])
def test_decode_beyond_launch_hints(oracle_mod, H):
    """300 short requests: more decode splits than the launch arguments carry start hints for,
    so every CTA finds its request's chunk range and first chunk from the device table."""
    ctxs = [40 + (7 * b) % 170 for b in range(300)]
    case = _ragged_decode_case(ctxs, H, seed=11 + H)
    sel = np.array([[b, 0, h] for b in (0, 1, 150, 257, 299) for h in (0, H // 2, H - 1)])
    _check_attn(case, oracle_mod, prefill=False, select=sel, what=f"decode 300 requests H={H}")


def _long_table_case(n_chunks=1500, n_q=1):
    """One request whose table is too long to travel in the launch parameters (more than 1024
    records), so the library copies it into the workspace."""
    rng = np.random.default_rng(9)
    reqs, p = [[(0, 32, 0, 0)]], 32
    for k in range(n_chunks):
        n = 1 + k % 5
        reqs[0].append((int(rng.integers(0, 8000 - n)), n, p - int(rng.integers(-3000, 3000)), 1))
        p += n
    return to_device(synth.custom_case(reqs, n_rows=8000, n_q=n_q, H=16, q_std=1.0))


@pytest.mark.parametrize("long_table", [False, True])
def test_pageable_table_is_read_before_the_call_returns(oracle_mod, long_table):
    """The library hands the validated host table to the kernels itself (in the launch
    parameters when short, by a copy into the workspace when long).  A pageable table has
    been read when the call returns, so overwriting it right after the call (before the GPU
    has run anything) changes nothing: the kernels run on the table that was validated."""
    if long_table:
        case = _long_table_case()
        ql, qr = case.q_lat[:, 0].contiguous(), case.q_rope[:, 0].contiguous()
    else:
        case = to_device(encode_rope_rows(synth.tiny_case(0, q_std=1.0), oracle_mod))
        ql, qr = case.q_lat[:, -1].contiguous(), case.q_rope[:, -1].contiguous()
    table = irm.ChunkTable(case.chunks, case.indptr, pinned=False)
    ref, _, _ = irm.irm_mla_attn_decode(ql, qr, irm.ChunkTable(case.chunks, case.indptr), case.kv_rows, SCALE)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    block = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(side):
        block.fill_(1)  # keeps the stream busy while the host table is overwritten
        out, _, ws = irm.irm_mla_attn_decode(ql, qr, table, case.kv_rows, SCALE, stream=side)
        table.chunks_host["pool_offset"][:] = 10_000_000
        table.chunks_host["p_src"][:] = 7
        table.indptr_host[:] = 0
    torch.cuda.synchronize()
    irm.device_status(ws)
    assert torch.equal(out, ref)


@pytest.mark.parametrize("long_table", [False, True])
@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")  # the refused capture leaves it empty
def test_graph_capture_of_the_table(oracle_mod, long_table):
    """A call captured into a CUDA graph replays the table it validated at capture time.  A
    short table travels in the launch parameters, so any host memory works; a long one is
    copied into the workspace by a captured copy, which needs page-locked host memory (a
    pageable one is refused during capture)."""
    if long_table:
        case = _long_table_case()
        ql, qr = case.q_lat[:, 0].contiguous(), case.q_rope[:, 0].contiguous()
    else:
        case = to_device(encode_rope_rows(synth.tiny_case(0, q_std=1.0), oracle_mod))
        ql, qr = case.q_lat[:, -1].contiguous(), case.q_rope[:, -1].contiguous()
    pinned = irm.ChunkTable(case.chunks, case.indptr)
    pageable = irm.ChunkTable(case.chunks, case.indptr, pinned=False)
    ref, _, ws = irm.irm_mla_attn_decode(ql, qr, pinned, case.kv_rows, SCALE)
    out = torch.empty_like(ref)
    side = torch.cuda.Stream()
    for table, ok in ((pinned, True), (pageable, not long_table)):
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        if not ok:
            with pytest.raises(irm.IrmError) as e:
                with torch.cuda.stream(side):
                    with torch.cuda.graph(g, stream=side):
                        irm.irm_mla_attn_decode(ql, qr, table, case.kv_rows, SCALE, out=out,
                                                workspace=ws, stream=side)
            assert e.value.status == -1 and "page-locked" in str(e.value)
            torch.cuda.synchronize()
            continue
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                irm.irm_mla_attn_decode(ql, qr, table, case.kv_rows, SCALE, out=out, workspace=ws,
                                        stream=side)
        for _ in range(2):
            out.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(out, ref)
        irm.device_status(ws)


def test_long_table_decode_and_prefill(oracle_mod):
    """Tables copied into the workspace (more records than the launch parameters carry) give
    the same results as the oracle, for decode and for prefill."""
    case = _long_table_case()
    sel = np.array([[0, 0, h] for h in range(16)])
    _check_attn(case, oracle_mod, prefill=False, select=sel, what="decode, 1501-chunk table")
    pcase = _long_table_case(n_q=9)
    sel = np.array([[0, i, h] for i in (0, 4, 8) for h in (0, 7, 15)])
    _check_attn(pcase, oracle_mod, prefill=True, select=sel, what="prefill, 1501-chunk table")


def test_bad_page_index_is_recorded_not_faulted(oracle_mod):
    """Page indices live in device memory and are not seen by the host: one outside the paged
    output is caught by the gather kernel (the rows of that page are skipped, the status word
    records IRM_ERR_DEVICE_BOUNDS) while every other page is still written."""
    case = encode_rope_rows(synth.tiny_case(0), oracle_mod)
    case = to_device(case)
    table = irm.ChunkTable(case.chunks, case.indptr)
    pt_np = np.arange(8, dtype=np.int32)[None].copy()
    pt_np[0, 3] = 8  # rows 192..255 would land past the 8 pages
    paged = torch.zeros((8, 64, 576), dtype=torch.bfloat16, device="cuda")
    ws = irm.irm_assemble_kv(table, case.kv_rows, paged, torch.from_numpy(pt_np).cuda())
    with pytest.raises(irm.IrmError) as e:
        irm.device_status(ws)
    assert e.value.status == -7
    irm.device_status(ws)  # cleared
    got = synth.bits(paged.view(-1, 576))
    pl = oracle_mod.plan(case.chunks, case.indptr)
    src = synth.bits(case.kv_rows)[pl["src_row"]]
    keep = np.ones(512, bool)
    keep[192:256] = False
    assert np.array_equal(got[np.arange(512)[keep], :512], src[keep, :512])
    assert not got[192:256].any()
