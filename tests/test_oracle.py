"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than itself: the worked example of the
walkthrough page (§15), the composition law R(delta) R(p_src) = R(p_tgt) (§4), closed
forms, invariants, special cases and brute-force enumeration.  The last group plants
mistakes in a copy of the oracle's steps (on the CPU) and shows the pins catch them.
"""
import json
import math
import os

import numpy as np
import pytest

from mla_position_independent_gb300 import synth
from helpers import rope_tables

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SCALE = 1.0 / math.sqrt(192.0)


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------- rotation

def test_worked_example_delta_and_composition(oracle_mod):
    """Walkthrough §15: 100 -> 350 gives delta 250; 360 -> 110 gives delta -250, and the
    rotated k_r equals the key encoded at the target position."""
    g = _golden("worked_example.json")
    rng = np.random.default_rng(1)
    for case in g["cases"]:
        ps, pt = case["p_src"], case["p_tgt"]
        # the plan's delta for a one-chunk reuse at pt of a chunk cached at ps
        chunks, indptr = synth.make_table([[(0, 32, 0, 0), (32, pt - 32, 0, 0), (100, 8, ps, 1)]])
        pl = oracle_mod.plan(chunks, indptr)
        assert int(pl["delta"][pt]) == case["delta"]
        assert int(pl["pos_src"][pt]) == ps
        k = rng.standard_normal((4, 64))
        kb = oracle_mod.rotate(k, ps)
        np.testing.assert_allclose(oracle_mod.rotate(kb, case["delta"]), oracle_mod.rotate(k, pt),
                                   rtol=0, atol=1e-12)


def test_composition_small_positions(oracle_mod):
    """R(delta) R(p_src) k = R(p_tgt) k to 1e-12 for positions where fp64 angles are exact
    to ~1e-13 (|p| <= 4096)."""
    rng = np.random.default_rng(2)
    k = rng.standard_normal((256, 64))
    ps = rng.integers(0, 4096, 256)
    d = rng.integers(-4096, 4096, 256)
    lhs = oracle_mod.rotate(oracle_mod.rotate(k, ps), d)
    rhs = oracle_mod.rotate(k, ps + d)
    assert np.max(np.abs(lhs - rhs)) < 1e-12


def test_composition_large_positions(oracle_mod):
    """Same law for p_src in [0, 2^17] and delta in [-65536, 65536].  fp64 angle rounding is
    |angle| * 2^-53 per product, so the bound is 4 * 2^18 * 2^-53 * |k|_inf-ish."""
    rng = np.random.default_rng(3)
    k = rng.standard_normal((256, 64))
    ps = rng.integers(0, 1 << 17, 256)
    d = rng.integers(-65536, 65536, 256)
    lhs = oracle_mod.rotate(oracle_mod.rotate(k, ps), d)
    rhs = oracle_mod.rotate(k, ps + d)
    bound = 4 * (1 << 18) * 2.0 ** -53 * np.abs(k).max() * 8
    assert np.max(np.abs(lhs - rhs)) < bound


def test_delta_zero_is_identity(oracle_mod):
    rng = np.random.default_rng(4)
    k = rng.standard_normal((32, 64))
    assert np.array_equal(oracle_mod.rotate(k, 0), k)


def test_norm_preserved_and_inverse(oracle_mod):
    rng = np.random.default_rng(5)
    k = rng.standard_normal((128, 64))
    d = rng.integers(-65536, 65536, 128)
    r = oracle_mod.rotate(k, d)
    np.testing.assert_allclose(np.linalg.norm(r, axis=1), np.linalg.norm(k, axis=1), rtol=1e-13)
    np.testing.assert_allclose(oracle_mod.rotate(r, -d), k, rtol=0, atol=1e-12)


def test_neox_pairing_and_frequencies(oracle_mod):
    """Pair j couples dims (j, j+32) (NeoX half split) and turns by delta * theta_j with
    theta_0 = 1, theta_16 = 10000^-1/2 = 0.01, and a constant ratio 10000^(-1/32) between
    neighbouring pairs."""
    theta = oracle_mod.rope_theta()
    assert theta[0] == 1.0
    assert abs(theta[16] - 0.01) < 1e-15
    np.testing.assert_allclose(theta[1:] / theta[:-1], 10000.0 ** (-1.0 / 32), rtol=1e-13)
    for j in (0, 1, 7, 16, 31):
        k = np.zeros(64)
        k[j] = 0.6
        k[j + 32] = -0.8
        for delta in (1, 3, -2, 250):
            r = oracle_mod.rotate(k, delta)[0]
            others = np.delete(r, [j, j + 32])
            assert np.all(others == 0.0)
            ang_in = math.atan2(k[j + 32], k[j])
            ang_out = math.atan2(r[j + 32], r[j])
            turned = (ang_out - ang_in) % (2 * math.pi)
            expect = (delta * theta[j]) % (2 * math.pi)
            assert min(abs(turned - expect), 2 * math.pi - abs(turned - expect)) < 1e-12


def test_first_pair_closed_form(oracle_mod):
    """theta_0 = 1: pair 0 is the plain 2-D rotation by delta radians."""
    k = np.zeros(64)
    k[0], k[32] = 1.0, 0.0
    for delta in (1, 2, 100, -7):
        r = oracle_mod.rotate(k, delta)[0]
        assert abs(r[0] - math.cos(delta)) < 1e-15 and abs(r[32] - math.sin(delta)) < 1e-15


def test_bf16_rotation_within_pages_error(oracle_mod):
    """Summary §3: bf16 delta-rotation has relative L2 error 4.7e-3.  The exact rotation
    rounded once to bf16 must stay below it (it sits at the bf16 floor, ~1.1e-3)."""
    import torch
    g = _golden("structural_constants.json")
    rng = np.random.default_rng(6)
    k = rng.standard_normal((4096, 64))
    d = rng.integers(-65536, 65536, 4096)
    r = oracle_mod.rotate(k, d)
    r16 = torch.from_numpy(r).to(torch.bfloat16).double().numpy()
    rel = np.linalg.norm(r16 - r) / np.linalg.norm(r)
    assert 5e-4 < rel < g["bf16_rotation_rel_l2"]


# --------------------------------------------------------------------------- assembly

def _brute_plan(chunks, indptr):
    """Row-by-row enumeration: for each target position scan the table for its chunk."""
    src, dl, ps = [], [], []
    for b in range(len(indptr) - 1):
        c = chunks[indptr[b]:indptr[b + 1]]
        ctx = int(c["len"].sum())
        for t in range(ctx):
            hit = [x for x in c if x["p_tgt"] <= t < x["p_tgt"] + x["len"]]
            assert len(hit) == 1
            x = hit[0]
            d = int(x["p_tgt"]) - int(x["p_src"]) if x["reused"] else 0
            src.append(int(x["pool_offset"]) + t - int(x["p_tgt"]))
            dl.append(d)
            ps.append(t - d)
    return np.array(src), np.array(dl), np.array(ps)


def _random_table(rng, B, n_rows):
    reqs = []
    for _ in range(B):
        ctx = int(rng.integers(1, 300))
        lens = []
        while sum(lens) < ctx:
            lens.append(int(min(rng.integers(1, 70), ctx - sum(lens))))
        p, req = 0, []
        for n in lens:
            reused = p >= 32 and rng.random() < 0.7
            off = int(rng.integers(0, n_rows - n + 1))
            req.append((off, n, int(rng.integers(-5000, 5000)), reused))
            p += n
        reqs.append(req)
    return synth.make_table(reqs)


def test_plan_matches_bruteforce(oracle_mod):
    rng = np.random.default_rng(7)
    for _ in range(20):
        chunks, indptr = _random_table(rng, int(rng.integers(1, 5)), 1000)
        pl = oracle_mod.plan(chunks, indptr)
        s, d, p = _brute_plan(chunks, indptr)
        assert np.array_equal(pl["src_row"], s)
        assert np.array_equal(pl["delta"], d)
        assert np.array_equal(pl["pos_src"], p)
        # invariants: sum of lengths, pos_src + delta = t, carve-out rows unrotated
        t = np.concatenate([np.arange(c) for c in pl["ctx"]])
        assert pl["src_row"].shape[0] == int(chunks["len"].sum())
        assert np.array_equal(pl["pos_src"] + pl["delta"], t)
        assert np.all(pl["delta"][t < 32] == 0)


def test_plan_rejects_bad_tables(oracle_mod):
    chunks, indptr = synth.make_table([[(0, 16, 0, 0), (16, 40, 500, 1)]])   # reused at p=16
    with pytest.raises(ValueError):
        oracle_mod.plan(chunks, indptr)
    chunks, indptr = synth.make_table([[(0, 40, 0, 0)]])
    chunks["p_tgt"][0] = 3                                                     # gap at 0
    with pytest.raises(ValueError):
        oracle_mod.plan(chunks, indptr)


def test_assemble_keeps_ckv_and_rotates_kr(oracle_mod):
    rng = np.random.default_rng(8)
    kv = synth.bits(synth.normal_bf16((64, 576), 11))
    src = rng.integers(0, 64, 200)
    d = rng.integers(-9000, 9000, 200)
    d[:50] = 0
    out = oracle_mod.assemble(kv, src, d)
    w = oracle_mod.widen(kv[src])
    assert np.array_equal(out[:, :512], w[:, :512])          # cKV passes through untouched
    assert np.array_equal(out[:50, 512:], w[:50, 512:])      # delta = 0 rows unchanged
    np.testing.assert_allclose(out[50:, 512:], oracle_mod.rotate(w[50:, 512:], d[50:]),
                               rtol=0, atol=1e-13)


# --------------------------------------------------------------------------- attention

def _rand_keys(rng, n):
    return rng.standard_normal((n, 576))


def test_attn_single_key(oracle_mod):
    rng = np.random.default_rng(9)
    K = _rand_keys(rng, 5)
    q = rng.standard_normal((3, 576))
    O, lse = oracle_mod.attn(q, 1, K, SCALE)
    np.testing.assert_array_equal(O, np.repeat(K[:1, :512], 3, 0))
    np.testing.assert_allclose(lse, SCALE * (q @ K[0]), rtol=1e-13)


def test_attn_zero_query_is_mean(oracle_mod):
    rng = np.random.default_rng(10)
    K = _rand_keys(rng, 37)
    O, lse = oracle_mod.attn(np.zeros((1, 576)), 37, K, SCALE)
    np.testing.assert_allclose(O[0], K[:, :512].mean(0), rtol=0, atol=1e-13)
    assert abs(lse[0] - math.log(37)) < 1e-13


def test_attn_two_keys_logistic(oracle_mod):
    """Two keys whose scaled scores differ by ln 3: weights are exactly 3/4 and 1/4."""
    K = np.zeros((2, 576))
    K[0, 0] = 1.0
    K[1, 1] = 1.0
    K[0, 512] = 2.0        # k_r participates in the score
    q = np.zeros((1, 576))
    q[0, 512] = math.log(3.0) / (2.0 * SCALE)
    O, lse = oracle_mod.attn(q, 2, K, SCALE)
    assert abs(O[0, 0] - 0.75) < 1e-15 and abs(O[0, 1] - 0.25) < 1e-15
    assert abs(lse[0] - math.log(4.0)) < 1e-14


def test_attn_sharp_query_selects_key(oracle_mod):
    rng = np.random.default_rng(11)
    K = _rand_keys(rng, 20)
    q = 200.0 * K[7:8] / np.linalg.norm(K[7]) / SCALE
    O, _ = oracle_mod.attn(q, 20, K, SCALE)
    np.testing.assert_allclose(O[0], K[7, :512], atol=1e-9)


def test_attn_causal_prefix_only(oracle_mod):
    rng = np.random.default_rng(12)
    K = _rand_keys(rng, 30)
    q = rng.standard_normal((1, 576))
    O1, l1 = oracle_mod.attn(q, 17, K, SCALE)
    K2 = K.copy()
    K2[17:] = 1e3 * rng.standard_normal((13, 576))       # invisible keys do not matter
    O2, l2 = oracle_mod.attn(q, 17, K2, SCALE)
    assert np.array_equal(O1, O2) and np.array_equal(l1, l2)


def test_attn_shift_invariance(oracle_mod):
    """A shared component c along dim 0 of every cKV row shifts all scores by the same
    amount when q_lat[0] changes: O is unchanged and lse moves by that amount."""
    rng = np.random.default_rng(13)
    K = _rand_keys(rng, 25)
    K[:, 0] = 0.5
    q = rng.standard_normal((1, 576))
    q2 = q.copy()
    q2[0, 0] += 3.0
    O1, l1 = oracle_mod.attn(q, 25, K, SCALE)
    O2, l2 = oracle_mod.attn(q2, 25, K, SCALE)
    np.testing.assert_allclose(O2, O1, rtol=0, atol=1e-13)
    assert abs((l2 - l1)[0] - SCALE * 1.5) < 1e-13


def test_query_rotation_identity(oracle_mod):
    """q_rope . R(delta) k = (R(-delta) q_rope) . k: attention over rotated keys equals
    attention of the counter-rotated query over the unrotated keys."""
    rng = np.random.default_rng(14)
    K = _rand_keys(rng, 40)
    q = rng.standard_normal((1, 576))
    d = 1234
    Kr = K.copy()
    Kr[:, 512:] = oracle_mod.rotate(K[:, 512:], d)
    qr = q.copy()
    qr[:, 512:] = oracle_mod.rotate(q[:, 512:], -d)
    O1, l1 = oracle_mod.attn(q, 40, Kr, SCALE)
    O2, l2 = oracle_mod.attn(qr, 40, K, SCALE)
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def test_full_recompute_equivalence(oracle_mod):
    """Brute force on the tiny workload: attention over the reused rows (cached at p_src,
    rotated by delta) equals attention over the same content freshly encoded at p_tgt."""
    case = synth.tiny_case(seed=0)
    kv = synth.bits(case.kv_rows).copy()
    enc = oracle_mod.rotate(case.rope_content, case.rope_pos)
    # keep fp64 keys for the equivalence (no bf16 rounding on either side)
    pl = oracle_mod.plan(case.chunks, case.indptr)
    K_reuse = oracle_mod.assemble(kv, pl["src_row"], pl["delta"])
    K_reuse[:, 512:] = oracle_mod.rotate(enc[pl["src_row"]], pl["delta"])
    t = np.arange(512)
    K_fresh = K_reuse.copy()
    K_fresh[:, 512:] = oracle_mod.rotate(case.rope_content[pl["src_row"]], t)
    np.testing.assert_allclose(K_reuse[:, 512:], K_fresh[:, 512:], rtol=0, atol=1e-11)
    ql = oracle_mod.widen(synth.bits(case.q_lat))[0]
    qr = oracle_mod.widen(synth.bits(case.q_rope))[0]
    q = np.concatenate([ql, qr], -1).reshape(-1, 576)
    vis = np.repeat(512 - 16 + np.arange(16) + 1, 16)
    O1, l1 = oracle_mod.attn(q, vis, K_reuse, SCALE)
    O2, l2 = oracle_mod.attn(q, vis, K_fresh, SCALE)
    np.testing.assert_allclose(O1, O2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def test_mla_attention_composes_steps(oracle_mod):
    """mla_attention (plan -> assemble -> attn per request) agrees with the steps called one
    by one, for all rows and for a sampled subset, with causal positions ctx - n_q + i."""
    case = synth.custom_case([[(0, 32, 0, 0), (100, 50, 7, 1), (40, 20, 0, 0)],
                              [(200, 40, 0, 0), (300, 33, -90, 1)]], n_rows=400, n_q=3, H=2)
    kv = synth.bits(case.kv_rows)
    ql, qr = synth.bits(case.q_lat), synth.bits(case.q_rope)
    O, lse = oracle_mod.mla_attention(ql, qr, case.chunks, case.indptr, kv, SCALE)
    pl = oracle_mod.plan(case.chunks, case.indptr)
    for b in range(2):
        r0, r1 = pl["row_start"][b], pl["row_start"][b + 1]
        K = oracle_mod.assemble(kv, pl["src_row"][r0:r1], pl["delta"][r0:r1])
        for i in range(3):
            for h in range(2):
                q = np.concatenate([oracle_mod.widen(ql[b, i, h]), oracle_mod.widen(qr[b, i, h])])
                o, l = oracle_mod.attn(q, (r1 - r0) - 3 + i + 1, K, SCALE)
                np.testing.assert_array_equal(O[b, i, h], o[0])
                assert lse[b, i, h] == l[0]
    sel = np.array([[1, 2, 1], [0, 0, 0]])
    Os, ls = oracle_mod.mla_attention(ql, qr, case.chunks, case.indptr, kv, SCALE, select=sel)
    np.testing.assert_array_equal(Os[0], O[1, 2, 1])
    np.testing.assert_array_equal(Os[1], O[0, 0, 0])


def test_rotate_gather_slots(oracle_mod):
    case = synth.custom_case([[(0, 32, 0, 0), (64, 70, 9, 1)], [(500, 65, 0, 0)]], n_rows=600,
                             n_q=0, pages=True)
    kv = synth.bits(case.kv_rows)
    slot, vals = oracle_mod.rotate_gather(kv, case.chunks, case.indptr, case.page_table)
    assert slot.shape[0] == 167 and np.unique(slot).shape[0] == 167
    assert np.all(slot // 64 < case.n_pages)
    pl = oracle_mod.plan(case.chunks, case.indptr)
    np.testing.assert_array_equal(vals, oracle_mod.assemble(kv, pl["src_row"], pl["delta"]))


# --------------------------------------------------------------------------- RoPE variants
# Walkthrough §11: the delta-rotation must use the model's own rotary class and inv_freq
# (a plain base-10000 fallback made reuse collapse in the pages' TransMLA case study).  The
# oracle takes the spec as (theta[32] radians per position, pairing: 0 NeoX, 1 interleaved).

def test_rope_table_of_default_is_the_default(oracle_mod):
    """The spec path with the default table and NeoX pairing is the default rotation, bit
    for bit; the test's base-10000 table is that table to the last ulp."""
    rng = np.random.default_rng(31)
    k = rng.standard_normal((16, 64))
    d = rng.integers(-70000, 70000, 16)
    np.testing.assert_array_equal(oracle_mod.rotate(k, d, rope=(oracle_mod.rope_theta(), 0)),
                                  oracle_mod.rotate(k, d))
    np.testing.assert_allclose(rope_tables()["base10k"], oracle_mod.rope_theta(), rtol=2.3e-16)


@pytest.mark.parametrize("name", ["base10k", "base500k", "yarn"])
def test_interleaved_is_neox_on_even_odd_split(oracle_mod, name):
    """Interleaved pairs (2j, 2j+1) are the NeoX pairs (j, j+32) of the vector whose first
    half holds the even dims and second half the odd dims: R_int = P^T R_neox P."""
    th = rope_tables()[name]
    rng = np.random.default_rng(32)
    k = rng.standard_normal((12, 64))
    d = rng.integers(-5000, 5000, 12)
    perm = np.concatenate([np.arange(0, 64, 2), np.arange(1, 64, 2)])
    via_neox = np.empty_like(k)
    via_neox[:, perm] = oracle_mod.rotate(k[:, perm], d, rope=(th, 0))
    np.testing.assert_array_equal(oracle_mod.rotate(k, d, rope=(th, 1)), via_neox)


def test_interleaved_pairs_and_angles(oracle_mod):
    """Pairing 1: pair j moves only dims 2j, 2j+1, turned by delta * theta_j."""
    th = rope_tables()["yarn"]
    for j in (0, 5, 16, 20, 31):
        k = np.zeros(64)
        k[2 * j], k[2 * j + 1] = 0.6, -0.8
        for delta in (1, -3, 250, 40000):
            r = oracle_mod.rotate(k, delta, rope=(th, 1))[0]
            assert np.all(np.delete(r, [2 * j, 2 * j + 1]) == 0.0)
            turned = (math.atan2(r[2 * j + 1], r[2 * j]) - math.atan2(k[2 * j + 1], k[2 * j])) % (2 * math.pi)
            expect = (delta * th[j]) % (2 * math.pi)
            assert min(abs(turned - expect), 2 * math.pi - abs(turned - expect)) < 1e-10


@pytest.mark.parametrize("pairing", [0, 1])
@pytest.mark.parametrize("name", ["base500k", "yarn"])
def test_variant_composition_identity_and_norm(oracle_mod, name, pairing):
    """R(delta) R(p_src) = R(p_tgt) for any frequency table and pairing; delta = 0 is the
    identity and R preserves the norm."""
    rope = (rope_tables()[name], pairing)
    rng = np.random.default_rng(33)
    k = rng.standard_normal((128, 64))
    ps = rng.integers(0, 4096, 128)
    d = rng.integers(-4096, 4096, 128)
    lhs = oracle_mod.rotate(oracle_mod.rotate(k, ps, rope=rope), d, rope=rope)
    # each angle p * theta_j (|angle| <= 8192 rad) carries fp64 rounding of up to 2^-53
    # relative, i.e. <= 9.1e-13 rad, and three such angles enter the comparison
    assert np.max(np.abs(lhs - oracle_mod.rotate(k, ps + d, rope=rope))) < 4e-12
    np.testing.assert_array_equal(oracle_mod.rotate(k, 0, rope=rope), k)
    r = oracle_mod.rotate(k, d, rope=rope)
    np.testing.assert_allclose(np.linalg.norm(r, axis=1), np.linalg.norm(k, axis=1), rtol=1e-14)


def test_wrong_rotary_class_breaks_reuse(oracle_mod):
    """Walkthrough §11: keys cached under the model's rotary class (here interleaved pairs
    with a YaRN-like table) are moved correctly only by the same class; the default class
    (NeoX, base 10000) moves them somewhere else and changes the attention output."""
    rng = np.random.default_rng(34)
    content = rng.standard_normal((96, 64))
    p_src = 700 + np.arange(96)
    p_tgt = 3100 + np.arange(96)
    model = (rope_tables()["yarn"], 1)
    cached = oracle_mod.rotate(content, p_src, rope=model)
    fresh = oracle_mod.rotate(content, p_tgt, rope=model)
    right = oracle_mod.rotate(cached, p_tgt - p_src, rope=model)
    wrong = oracle_mod.rotate(cached, p_tgt - p_src)
    assert np.max(np.abs(right - fresh)) < 1e-11
    assert np.linalg.norm(wrong - fresh) / np.linalg.norm(fresh) > 0.5
    K = np.concatenate([rng.standard_normal((96, 512)), fresh], 1)
    q = rng.standard_normal((4, 576))
    O_ref, _ = oracle_mod.attn(q, 96, K, 1.0 / 8)
    K_right, K_wrong = K.copy(), K.copy()
    K_right[:, 512:], K_wrong[:, 512:] = right, wrong
    assert np.max(np.abs(oracle_mod.attn(q, 96, K_right, 1.0 / 8)[0] - O_ref)) < 1e-10
    assert np.max(np.abs(oracle_mod.attn(q, 96, K_wrong, 1.0 / 8)[0] - O_ref)) > 1e-2


def test_assemble_and_gather_follow_the_rope_spec(oracle_mod):
    """assemble / rotate_gather apply the spec they are given to exactly the rows rotate
    would, and leave cKV untouched."""
    case = synth.custom_case([[(0, 32, 0, 0), (64, 70, 9, 1), (300, 40, 5000, 1)]], n_rows=600,
                             n_q=0, pages=True)
    kv = synth.bits(case.kv_rows)
    rope = (rope_tables()["yarn"], 1)
    pl = oracle_mod.plan(case.chunks, case.indptr)
    K = oracle_mod.assemble(kv, pl["src_row"], pl["delta"], rope)
    np.testing.assert_array_equal(K[:, :512], oracle_mod.widen(kv[pl["src_row"], :512]))
    kr = oracle_mod.widen(kv[pl["src_row"], 512:])
    np.testing.assert_array_equal(K[:, 512:], oracle_mod.rotate(kr, pl["delta"], rope=rope))
    slot, vals = oracle_mod.rotate_gather(kv, case.chunks, case.indptr, case.page_table, rope=rope)
    np.testing.assert_array_equal(vals, K)


# --------------------------------------------------------------------------- planted mistakes

def _theta():
    return 10000.0 ** (-2.0 * np.arange(32) / 64.0)


def _rotate_variant(k, steps, mode):
    """A CPU copy of the rotation with one planted mistake, to show the pins catch it."""
    k = np.atleast_2d(k).astype(np.float64)
    steps = np.broadcast_to(np.asarray(steps), (k.shape[0],))
    th = _theta()
    if mode == "freq":
        th = 10000.0 ** (-np.arange(32) / 64.0)
    ang = steps[:, None] * th[None, :]
    c, s = np.cos(ang), np.sin(ang)
    if mode == "sign":
        s = -s
    if mode == "interleaved":
        x, y = k[:, 0::2], k[:, 1::2]
        out = np.empty_like(k)
        out[:, 0::2], out[:, 1::2] = x * c - y * s, x * s + y * c
        return out
    x, y = k[:, :32], k[:, 32:]
    return np.concatenate([x * c - y * s, x * s + y * c], 1)


@pytest.mark.parametrize("mode", ["sign", "freq", "interleaved"])
def test_pins_catch_planted_rotation_mistakes(oracle_mod, mode):
    """Each planted mistake disagrees with the oracle on the pinned special cases, while the
    unplanted copy agrees: the pins are sensitive to sign, frequency and pairing."""
    rng = np.random.default_rng(15)
    k = rng.standard_normal((8, 64))
    good = _rotate_variant(k, 250, "none")
    np.testing.assert_allclose(good, oracle_mod.rotate(k, 250), atol=1e-12)
    bad = _rotate_variant(k, 250, mode)
    assert np.max(np.abs(bad - oracle_mod.rotate(k, 250))) > 1e-3


def _rotate_interleaved_variant(k, steps, theta, mode):
    """A CPU copy of the interleaved rotation with one planted mistake."""
    k = np.atleast_2d(k).astype(np.float64)
    steps = np.broadcast_to(np.asarray(steps), (k.shape[0],))
    th = theta[::-1] if mode == "freq_order" else theta
    ang = steps[:, None] * th[None, :]
    c, s = np.cos(ang), np.sin(ang)
    if mode == "sign":
        s = -s
    if mode == "neox":
        x, y = k[:, :32], k[:, 32:]
        return np.concatenate([x * c - y * s, x * s + y * c], 1)
    x, y = k[:, 0::2], k[:, 1::2]
    out = np.empty_like(k)
    out[:, 0::2], out[:, 1::2] = x * c - y * s, x * s + y * c
    return out


@pytest.mark.parametrize("mode", ["sign", "freq_order", "neox"])
def test_variant_pins_catch_planted_mistakes(oracle_mod, mode):
    """The unplanted copy matches the oracle's interleaved YaRN-like rotation; each planted
    mistake (sign, frequency order, pairing) does not."""
    th = rope_tables()["yarn"]
    rng = np.random.default_rng(35)
    k = rng.standard_normal((8, 64))
    ref = oracle_mod.rotate(k, 777, rope=(th, 1))
    np.testing.assert_allclose(_rotate_interleaved_variant(k, 777, th, "none"), ref, atol=1e-12)
    assert np.max(np.abs(_rotate_interleaved_variant(k, 777, th, mode) - ref)) > 1e-3
