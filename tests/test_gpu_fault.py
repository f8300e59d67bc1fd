"""Failure detection on the GPU without a fault: a pipeline wait that can never complete gives
up after its time limit, the kernel records IRM_ERR_DEVICE_TIMEOUT in the workspace status word
and returns, and the context stays usable for the next call."""
import time

import numpy as np
import pytest
import torch

import mla_position_independent_gb300 as irm
from mla_position_independent_gb300 import synth
from helpers import SCALE, assert_close, to_device, widen_bf16

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    ws = irm.new_workspace(256)
    t0 = time.perf_counter()
    irm.selftest_wait_timeout(ws)
    with pytest.raises(irm.IrmError) as e:
        irm.device_status(ws)  # synchronizes: the wait gave up by itself
    waited = time.perf_counter() - t0
    assert e.value.status == -6, e.value  # IRM_ERR_DEVICE_TIMEOUT
    assert 1.0 < waited < 30.0, waited
    irm.device_status(ws)  # the status word was cleared
    # the context is still usable: a small decode matches the oracle
    case = to_device(synth.custom_case([[(0, 32, 0, 0), (40, 100, 7, 1), (300, 61, 500, 1)]],
                                       n_rows=512, n_q=1, H=16, q_std=1.0))
    table = irm.ChunkTable(case.chunks, case.indptr)
    out, _, ws2 = irm.irm_mla_attn_decode(case.q_lat[:, 0], case.q_rope[:, 0], table, case.kv_rows, SCALE)
    irm.device_status(ws2)
    O, _ = oracle_mod.mla_attention(synth.bits(case.q_lat), synth.bits(case.q_rope), case.chunks,
                                    case.indptr, synth.bits(case.kv_rows), SCALE)
    assert_close(widen_bf16(out[:, None]), O, "decode after the timeout")
