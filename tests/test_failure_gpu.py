"""Failure path on the GPU without a fault: the GEMM core's bounded waits.

rf_selftest_wait_timeout runs the real single-CTA and CTA-pair GEMM kernels, in
round-robin and in dynamic unit order, on a problem whose operand copies are never
issued, so the MMA thread waits for data that nothing sends. With a 200 ms wait limit each role must give up, drain, free
TMEM, report RF_ERR_TIMEOUT in the status word and exit; afterwards the context
must still run a fill correctly.
"""
import time

import pytest
import torch

import oracle as O
import ridge_map_kv_gb300 as rf
import synth
from fillcheck import assert_bookkeeping, assert_values, run_fill

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", [0, 1, 2, 3],
                         ids=["single-cta", "cta-pair", "single-cta-dynamic-order", "cta-pair-dynamic-order"])
def test_gemm_wait_runs_out_reports_timeout_and_context_survives(mode):
    pair = mode & 1
    rf.rf_set_wait_timeout_ms(200)
    try:
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        t0 = time.monotonic()
        rf.rf_selftest_wait_timeout(mode, status)
        torch.cuda.synchronize()
        elapsed = time.monotonic() - t0
    finally:
        rf.rf_set_wait_timeout_ms(0)        # back to the default limit
    assert int(status.item()) == rf.RF_ERR_TIMEOUT
    assert 0.15 < elapsed < 10.0, elapsed
    cfg = synth.TOY
    inp = synth.fill_inputs(cfg)
    res = run_fill(cfg, inp, flags=rf.RF_FLAG_CTA_PAIR if pair else rf.RF_FLAG_SINGLE_CTA)
    assert res["status"] == 0
    mnp = inp["mask"].cpu().numpy()
    assert_bookkeeping(cfg, res, mnp)
    assert_values(cfg, inp, res, O.prefix_partition(cfg.N, cfg.T, mnp))
