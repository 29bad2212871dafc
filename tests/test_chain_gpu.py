"""The toy workload end to end on the GPU against the same chain in the oracle.

[RF] "Ridge map": the maps are fitted once, in closed form, from one pass of
calibration statistics, and the fill then runs them with the layer's own norm,
projections and RoPE. Here the whole chain runs through the C ABI:

  rf_calib_accumulate (2,048 planted rows, two batches) -> rf_solve (λ = 0.03,
  one refinement sweep, bf16 copy of the maps) -> rf_fill_kv (the toy fill),

and the oracle runs calib_stats -> ridge_solve -> the fill on the same rows. The
maps enter the fill as bf16 on both sides (the pages store them in bf16, 32 MiB
per layer at d = 4096); the oracle rounds its fp64 maps to bf16 (round to nearest
even) and its offsets to fp32, the widths the boundary takes. The solved maps must
match within 1e-5, the filled K/V within the per-head tolerance, and the cache
bookkeeping bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle as O
import ridge_map_kv_gb300 as rf
import synth
from fillcheck import assert_bookkeeping, assert_values, run_fill

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _round_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bf16 value (8 significant bits, ties to even), as fp64."""
    m, e = np.frexp(x)                 # x = m 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.round(m * 256.0) / 256.0, e)


def test_toy_calibrate_solve_fill_chain_matches_oracle_chain():
    cfg = synth.TOY
    P, d = cfg.P, cfg.d
    cal = synth.calib_inputs(d, d, P, cfg.calib_n, index=cfg.index)

    # GPU chain: sums -> solve -> fill
    X, Y = cal["X"].to(DEV), cal["Y"].to(DEV)
    st = {"G": torch.zeros((d, d), dtype=torch.float64, device=DEV),
          "C": torch.zeros((P, d, d), dtype=torch.float64, device=DEV),
          "sx": torch.zeros(d, dtype=torch.float64, device=DEV),
          "sy": torch.zeros((P, d), dtype=torch.float64, device=DEV),
          "n": torch.zeros(1, dtype=torch.int64, device=DEV)}
    cs = rf.calib_stats_struct(st["G"], st["C"], st["sx"], st["sy"], st["n"])
    cd = rf.rf_calib_desc(d_in=d, d_out=d, n_maps=P)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    n = cfg.calib_n
    for a, b in ((0, 1000), (1000, n)):
        rf.rf_calib_accumulate(cd, X[a:], d, Y[:, a:], d, n * d, b - a, cs, status)
    A = torch.empty((P, d, d), dtype=torch.float32, device=DEV)
    bvec = torch.empty((P, d), dtype=torch.float32, device=DEV)
    Ab = torch.empty((P, d, d), dtype=torch.bfloat16, device=DEV)
    wsb = rf.rf_solve_workspace_bytes(cd)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    rf.rf_solve(cd, cs, cfg.lam, rf.RF_ALPHA_TRACE, 1, A, bvec, Ab, None, status, ws, wsb)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    inp = synth.fill_inputs(cfg)
    gpu_inp = dict(inp, A=Ab.cpu(), b=bvec.cpu())
    res = run_fill(cfg, gpu_inp)
    assert res["status"] == 0

    # oracle chain: sums -> solve -> fill (maps rounded to bf16, offsets to fp32)
    f64 = O.bf16_bits_to_f64
    Ar, br, _ = O.ridge_solve(O.calib_stats(f64(synth.bits(cal["X"])), f64(synth.bits(cal["Y"]))), cfg.lam)
    A_gpu = A.cpu().numpy().astype(np.float64)
    for p in range(P):
        assert np.linalg.norm(A_gpu[p] - Ar[p]) <= 1e-5 * np.linalg.norm(Ar[p])
    ora_inp = dict(inp, A=torch.as_tensor(_round_bf16(Ar)), b=torch.as_tensor(br, dtype=torch.float32))

    mask = None if inp["mask"] is None else inp["mask"].numpy()
    idx = O.prefix_partition(cfg.N, cfg.T, mask)
    assert res["n_fill"] == len(idx) == 5
    assert_bookkeeping(cfg, res, mask)
    assert_values(cfg, ora_inp, res, idx)
