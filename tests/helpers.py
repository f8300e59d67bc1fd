"""Shared helpers for the parity tests (test-side only)."""
import math

import numpy as np
import torch

from mla_position_independent_gb300 import synth

SCALE = 1.0 / math.sqrt(192.0)
# bf16 outputs vs the fp64 oracle, and the rotated k_r bound (the pages' bf16 error).
TOL_REL_L2 = 5e-3
TOL_MAX_ABS = 2e-2
TOL_KR_REL_L2 = 4.7e-3


def rel_l2(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


def max_abs(x, ref):
    return float(np.max(np.abs(np.asarray(x, np.float64) - np.asarray(ref, np.float64))))


def encode_rope_rows(case, oracle_mod):
    """Fill k_r of the rows a workload asks for with RoPE(position) of their content vector,
    rounded to bf16 (the cached rows a prefill at that position would have produced)."""
    if case.rope_rows is None:
        return case
    enc = oracle_mod.rotate(case.rope_content, case.rope_pos)
    kv = case.kv_rows
    kr = torch.from_numpy(enc).to(torch.bfloat16).to(kv.device)
    kv[torch.as_tensor(case.rope_rows, device=kv.device), 512:] = kr
    return case


def to_device(case, device="cuda"):
    case.kv_rows = case.kv_rows.to(device)
    if case.q_lat is not None:
        case.q_lat = case.q_lat.to(device)
        case.q_rope = case.q_rope.to(device)
    return case


def widen_bf16(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(out, ref, what, rel=TOL_REL_L2, mx=TOL_MAX_ABS):
    r, m = rel_l2(out, ref), max_abs(out, ref)
    assert np.all(np.isfinite(np.asarray(out, np.float64))), f"{what}: non-finite output"
    assert r <= rel and m <= mx, f"{what}: rel L2 {r:.3e} (<= {rel}), max abs {m:.3e} (<= {mx})"
    return r, m


def rope_tables():
    """Frequency tables used as inputs by the RoPE-variant tests (model configurations, not
    method arithmetic): the default base 10000, a plain base 500000, and a YaRN-like table
    whose low-frequency pairs are slowed down by up to 40x with a linear ramp."""
    j = np.arange(32)
    base10k = 10000.0 ** (-2.0 * j / 64.0)
    base500k = 500000.0 ** (-2.0 * j / 64.0)
    ramp = np.clip((j - 16) / 8.0, 0.0, 1.0)
    yarn = base10k / (1.0 + 39.0 * ramp)
    return {"base10k": base10k, "base500k": base500k, "yarn": yarn}
