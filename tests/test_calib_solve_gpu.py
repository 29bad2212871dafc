"""GPU parity of rf_calib_accumulate and rf_solve against the fp64 oracle.

Calibration sums: every entry on small cases (ragged batches and row chunks),
sampled entries at full width (27B-shaped d=5120, and the cross-model Gram 8192^2
over 131,072 rows). Tolerance: |ΔG_ij| <= 1e-5 sqrt(G_ii G_jj), the same scale for C
with the y column's sum of squares.
Solve: on the toy, the fp32 solve (with fp64 refinement) equals the oracle's A
and b within 1e-5 relative (Frobenius per map); widths that split unevenly in
the recursive factorisation (768, 1280, 2560) match every entry; at the configs'
own sizes (d=4096 sampled rows; d=5120 for the 27B shape and 8192 -> 1024 for
the cross-model mapper, every entry) A matches and satisfies the normal equations.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import ridge_map_kv_gb300 as rf
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _zeros_stats(d_in, d_out, P):
    return {"G": torch.zeros((d_in, d_in), dtype=torch.float64, device=DEV),
            "C": torch.zeros((max(P, 1), d_in, d_out), dtype=torch.float64, device=DEV),
            "sx": torch.zeros(d_in, dtype=torch.float64, device=DEV),
            "sy": torch.zeros((max(P, 1), d_out), dtype=torch.float64, device=DEV),
            "n": torch.zeros(1, dtype=torch.int64, device=DEV)}


def _struct(st):
    return rf.calib_stats_struct(st["G"], st["C"], st["sx"], st["sy"], st["n"])


def _accumulate(X, Y, st, row_splits, flags=0, workspace=True):
    """Adds the rows of X, Y to ``st`` in the batches ``row_splits`` cuts; with
    ``workspace`` the GEMM takes its tiles in dynamic order (a device counter)."""
    n, d_in = X.shape
    P, _, d_out = Y.shape
    desc = rf.rf_calib_desc(d_in=d_in, d_out=d_out, n_maps=P, flags=flags)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(rf.rf_calib_workspace_bytes(desc, n), dtype=torch.uint8, device=DEV) if workspace else None
    bounds = [0] + list(row_splits) + [n]
    for a, b in zip(bounds[:-1], bounds[1:]):
        rf.rf_calib_accumulate(desc, X[a:], d_in, Y[:, a:], d_out, n * d_out, b - a, _struct(st), status,
                               ws, 0 if ws is None else ws.numel())
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def _f64(t):
    return O.bf16_bits_to_f64(synth.bits(t))


def _check_stats(st, ref, Yref_sq=None, rows=None, cols_x=None, cols_y=None):
    G = st["G"].cpu().numpy()
    C = st["C"].cpu().numpy()
    if cols_x is not None:
        G = G[np.ix_(cols_x, cols_x)]
        C = C[:, cols_x][:, :, cols_y]
    dg = np.sqrt(np.diag(ref["G"]))
    tolG = 1e-5 * np.outer(dg, dg)
    assert np.all(np.abs(G - ref["G"]) <= tolG), np.max(np.abs(G - ref["G"]) / tolG)
    if ref["C"].shape[0] and C.size:
        ysq = np.sqrt(Yref_sq)                                       # [P, d_out]
        tolC = 1e-5 * dg[None, :, None] * ysq[:, None, :]
        assert np.all(np.abs(C - ref["C"]) <= tolC), np.max(np.abs(C - ref["C"]) / tolC)


@pytest.mark.parametrize("shape", [(256, 256, 4, 2048, [1000]), (512, 768, 3, 3000, []), (256, 512, 1, 100, [40]),
                                   (256, 512, 2, 40000, [])],
                         ids=["toy two batches", "3 chunks ragged", "tiny ragged batches", "three slabs, ragged last"])
@pytest.mark.parametrize("flags", [rf.RF_FLAG_SINGLE_CTA, rf.RF_FLAG_CTA_PAIR], ids=["single-cta", "cta-pair"])
def test_calib_sums_match_oracle(shape, flags):
    d_in, d_out, P, n, splits = shape
    cal = synth.calib_inputs(d_in, d_out, P, n, index=0 if d_in == 256 and P == 4 else 93)
    X, Y = cal["X"].to(DEV), cal["Y"].to(DEV)
    st = _zeros_stats(d_in, d_out, P)
    _accumulate(X, Y, st, splits, flags)
    Xf, Yf = _f64(cal["X"]), _f64(cal["Y"])
    ref = O.calib_stats(Xf, Yf)
    _check_stats(st, ref, (Yf ** 2).sum(axis=1))
    assert int(st["n"].item()) == n
    np.testing.assert_allclose(st["sx"].cpu().numpy(), ref["sx"], rtol=0, atol=1e-6 * np.abs(Xf).sum(0).max())
    np.testing.assert_allclose(st["sy"].cpu().numpy(), ref["sy"], rtol=0, atol=1e-6 * np.abs(Yf).sum(1).max())


@pytest.mark.slow
@pytest.mark.parametrize("d_in,d_out,P,n", [(5120, 5120, 2, 16384), (8192, 256, 0, 131072)],
                         ids=["27b-shaped XtX and XtY", "cross-model Gram 8192^2 x 131072 rows"])
@pytest.mark.parametrize("flags", [rf.RF_FLAG_SINGLE_CTA, rf.RF_FLAG_CTA_PAIR], ids=["single-cta", "cta-pair"])
def test_calib_full_width_sampled(d_in, d_out, P, n, flags):
    cal = synth.calib_inputs(d_in, d_out, max(P, 1), n, index=3 if P else 4, device=DEV, noise=0.05)
    X, Y = cal["X"], cal["Y"][:P] if P else cal["Y"][:0]
    st = _zeros_stats(d_in, d_out, P)
    desc = rf.rf_calib_desc(d_in=d_in, d_out=d_out, n_maps=P, flags=flags)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(rf.rf_calib_workspace_bytes(desc, n), dtype=torch.uint8, device=DEV)
    rf.rf_calib_accumulate(desc, X, d_in, Y if P else None, d_out, n * d_out, n, _struct(st), status, ws, ws.numel())
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rng = np.random.default_rng(5)
    cx = np.sort(rng.choice(d_in, 96, replace=False))
    cy = np.sort(rng.choice(d_out, 64, replace=False))
    Xs = _f64(X[:, torch.as_tensor(cx, device=DEV)])
    if P:
        Ys = _f64(Y[:, :, torch.as_tensor(cy, device=DEV)])
        ref = O.calib_stats(Xs, Ys)
    else:  # Gram only: the oracle's sums of X, with its C (of a dummy Y) left unused
        ref = O.calib_stats(Xs, np.zeros((1, n, 1)))
        ref["C"] = np.zeros((0, len(cx), len(cy)))
    _check_stats(st, ref, (Ys ** 2).sum(axis=1) if P else None, cols_x=cx, cols_y=cy)


@pytest.mark.parametrize("flags", [rf.RF_FLAG_SINGLE_CTA, rf.RF_FLAG_CTA_PAIR], ids=["single-cta", "cta-pair"])
def test_calib_dynamic_and_round_robin_tile_orders_give_the_same_sums(flags):
    """With a workspace the calibration GEMM takes its tiles from a device counter,
    without one in a fixed round-robin order. Each tile is added to the fp64 totals
    once per 16 chunks of rows, in stream order, so the two orders give the same sums
    bit for bit: here over three row slabs with a ragged last one, in two batches."""
    cal = synth.calib_inputs(512, 256, 3, 16384 * 2 + 1288, index=96)
    X, Y = cal["X"].to(DEV), cal["Y"].to(DEV)
    a, b = _zeros_stats(512, 256, 3), _zeros_stats(512, 256, 3)
    _accumulate(X, Y, a, [20000], flags, workspace=True)
    _accumulate(X, Y, b, [20000], flags, workspace=False)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_calib_zero_rows_leaves_the_sums_unchanged():
    """n_rows = 0 is a valid call that adds nothing: every sum stays bit for bit."""
    cal = synth.calib_inputs(256, 256, 2, 512, index=93)
    X, Y = cal["X"].to(DEV), cal["Y"].to(DEV)
    st = _zeros_stats(256, 256, 2)
    _accumulate(X, Y, st, [])
    before = {k: v.clone() for k, v in st.items()}
    desc = rf.rf_calib_desc(d_in=256, d_out=256, n_maps=2)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rf.rf_calib_accumulate(desc, X, 256, Y, 256, 512 * 256, 0, _struct(st), status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for k in st:
        assert torch.equal(st[k], before[k]), k


# --------------------------------------------------------------------------- #
# Solve
# --------------------------------------------------------------------------- #
def test_solve_reports_a_non_positive_pivot():
    """Sums whose centred Gram has a negative eigenvalue (no rows give that, but a
    caller can pass any sums) make the fp32 Cholesky meet a pivot <= 0: the call
    returns RF_OK, RF_ERR_NOT_SPD lands in the status word, and the context
    stays usable (a well-posed solve follows in the same process)."""
    d, P = 256, 1
    G = np.eye(d)
    G[100, 100] = -1.0
    rng = np.random.default_rng(4)
    st = {"G": torch.as_tensor(G, device=DEV), "C": torch.as_tensor(rng.standard_normal((P, d, d)), device=DEV),
          "sx": torch.zeros(d, dtype=torch.float64, device=DEV),
          "sy": torch.zeros((P, d), dtype=torch.float64, device=DEV),
          "n": torch.tensor([10], dtype=torch.int64, device=DEV)}
    desc = rf.rf_calib_desc(d_in=d, d_out=d, n_maps=P)
    A = torch.empty((P, d, d), dtype=torch.float32, device=DEV)
    b = torch.empty((P, d), dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    wsb = rf.rf_solve_workspace_bytes(desc)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    rf.rf_solve(desc, _struct(st), 0.0, rf.RF_ALPHA_TRACE, 0, A, b, None, None, status, ws, wsb)
    torch.cuda.synchronize()
    assert int(status.item()) == rf.RF_ERR_NOT_SPD
    # the same process solves a well-posed system afterwards
    cal = synth.calib_inputs(256, 256, 2, 2048, index=0)
    ref = O.calib_stats(_f64(cal["X"]), _f64(cal["Y"]))
    A2, _, _, _ = _solve(_upload_stats(ref), 256, 256, 2, 0.03)
    Ar, _, _ = O.ridge_solve(ref, 0.03)
    assert max(_rel(A2[p], Ar[p]) for p in range(2)) <= 1e-5



def _upload_stats(ref):
    P = ref["C"].shape[0]
    return {"G": torch.as_tensor(ref["G"], device=DEV), "C": torch.as_tensor(ref["C"], device=DEV),
            "sx": torch.as_tensor(ref["sx"], device=DEV), "sy": torch.as_tensor(ref["sy"], device=DEV),
            "n": torch.tensor([ref["n"]], dtype=torch.int64, device=DEV)}


def _solve(st, d_in, d_out, P, lam, mode=rf.RF_ALPHA_TRACE, refine=1, flags=0):
    desc = rf.rf_calib_desc(d_in=d_in, d_out=d_out, n_maps=P, flags=flags)
    A = torch.empty((P, d_out, d_in), dtype=torch.float32, device=DEV)
    b = torch.empty((P, d_out), dtype=torch.float32, device=DEV)
    Ab = torch.empty((P, d_out, d_in), dtype=torch.bfloat16, device=DEV)
    alpha = torch.zeros(1, dtype=torch.float64, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    wsb = rf.rf_solve_workspace_bytes(desc)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    rf.rf_solve(desc, _struct(st), lam, mode, refine, A, b, Ab, alpha, status, ws, wsb)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return A.cpu().numpy().astype(np.float64), b.cpu().numpy().astype(np.float64), Ab, float(alpha.item())


def _rel(a, r, axis=None):
    return np.linalg.norm(a - r, axis=axis) / np.linalg.norm(r, axis=axis)


@pytest.mark.parametrize("mode,lam,refine", [(rf.RF_ALPHA_TRACE, 0.03, 1), (rf.RF_ALPHA_TRACE, 0.03, 0),
                                             (rf.RF_ALPHA_ABSOLUTE, 5.0, 1), (rf.RF_ALPHA_TRACE, 1.0, 2)])
def test_solve_toy_matches_oracle(mode, lam, refine):
    cal = synth.calib_inputs(256, 256, 4, 2048, index=0)
    ref = O.calib_stats(_f64(cal["X"]), _f64(cal["Y"]))
    A, b, Ab, alpha = _solve(_upload_stats(ref), 256, 256, 4, lam, mode, refine)
    Ar, br, alr = O.ridge_solve(ref, lam, "trace" if mode == rf.RF_ALPHA_TRACE else "absolute")
    assert abs(alpha - alr) <= 1e-12 * alr
    for p in range(4):
        assert _rel(A[p], Ar[p]) <= 1e-5, _rel(A[p], Ar[p])
        assert _rel(b[p], br[p]) <= 1e-5
    # the bf16 copy is the rounding of the fp32 maps
    np.testing.assert_array_equal(synth.bits(Ab), synth.bits(torch.as_tensor(A, dtype=torch.float32).to(torch.bfloat16)))


def test_solve_resolve_at_new_lambda_equals_fresh_solve():
    cal = synth.calib_inputs(256, 256, 2, 2048, index=0, salt=1)
    ref = O.calib_stats(_f64(cal["X"]), _f64(cal["Y"]))
    st = _upload_stats(ref)
    _solve(st, 256, 256, 2, 1.0)
    A1, b1, _, _ = _solve(st, 256, 256, 2, 0.01)
    A2, b2, _, _ = _solve(_upload_stats(ref), 256, 256, 2, 0.01)
    np.testing.assert_array_equal(A1, A2)
    np.testing.assert_array_equal(b1, b2)


def test_gpu_calibration_then_solve_recovers_planted_maps():
    """Planted toy: GPU accumulate + GPU solve gives the oracle's maps (from exact
    fp64 sums) within 1e-4, and both are near A_true at the noise level."""
    cal = synth.calib_inputs(256, 256, 4, 2048, index=0)
    st = _zeros_stats(256, 256, 4)
    _accumulate(cal["X"].to(DEV), cal["Y"].to(DEV), st, [777])
    A, b, _, _ = _solve(st, 256, 256, 4, 0.03)
    Ar, br, _ = O.ridge_solve(O.calib_stats(_f64(cal["X"]), _f64(cal["Y"])), 0.03)
    At = cal["A_true"].numpy().astype(np.float64)
    for p in range(4):
        assert _rel(A[p], Ar[p]) <= 1e-4
        assert _rel(A[p], At[p]) <= 0.05


def _conditioned_case(seed, n, decades):
    """Planted maps on rows whose spectrum falls geometrically over ``decades``
    (κ(Gc) about 10^(2·decades), times the sampling spread), λ = 1e-9: the oracle's
    A and the sums, with κ(H) from the oracle's H."""
    d, P = 512, 2
    rng = np.random.default_rng(seed)
    Q, _ = np.linalg.qr(rng.standard_normal((d, d)))
    X = (rng.standard_normal((n, d)) * np.geomspace(1.0, 10 ** -decades, d)) @ Q.T
    At = rng.standard_normal((P, d, d)) / math.sqrt(d)
    Y = np.einsum("pij,nj->pni", At, X) + 0.01 * rng.standard_normal((P, n, d))
    Xb = torch.as_tensor(X, dtype=torch.float32).to(torch.bfloat16)
    Yb = torch.as_tensor(Y, dtype=torch.float32).to(torch.bfloat16)
    ref = O.calib_stats(_f64(Xb), _f64(Yb))
    lam = 1e-9
    Ar, _, alpha = O.ridge_solve(ref, lam)
    Gc, _, _, _ = O.centre_stats(ref)
    ev = np.linalg.eigvalsh(Gc + alpha * np.eye(d))
    return ref, Ar, lam, ev[-1] / ev[0], d, P


DIGITS = pytest.mark.parametrize("flags", [0, rf.RF_SOLVE_DIGITS7], ids=["8-bit digits", "7-bit digits"])


@DIGITS
def test_solve_refinement_restores_accuracy_when_ill_conditioned(flags):
    """κ(Gc) ≈ 1e4: the fp32 factorisation alone loses about κ·2^-24; one sweep with the
    fp64-accurate residual (tensor-core digit products, exact integer chunk sums)
    brings A back to fp32 accuracy. A residual accurate only to fp32 would not."""
    ref, Ar, lam, kappa, d, P = _conditioned_case(21, 4096, 2.0)
    A0, _, _, _ = _solve(_upload_stats(ref), d, d, P, lam, refine=0, flags=flags)
    A1, _, _, _ = _solve(_upload_stats(ref), d, d, P, lam, refine=1, flags=flags)
    e0 = max(_rel(A0[p], Ar[p]) for p in range(P))
    e1 = max(_rel(A1[p], Ar[p]) for p in range(P))
    assert e0 > 1e-5, e0              # the case is hard enough to need refinement
    assert e1 <= 1e-5 and e1 < e0 / 20, (e0, e1)


def test_solve_refinement_in_the_four_digit_band():
    """κ(H) below 51: every estimate of it is too (the Rayleigh quotients approach from
    below), so the plan certainly keeps four 8-bit digits (10 digit pairs, a residual
    within 2^-31.7 of Σ|A||H|) and three correction terms. One sweep must still reach
    fp32-level accuracy (the residual's truncation times κ is about 1.4e-8 here)."""
    ref, Ar, lam, kappa, d, P = _conditioned_case(24, 4096, 0.7)
    assert 20 < kappa < 51, kappa
    A0, _, _, _ = _solve(_upload_stats(ref), d, d, P, lam, refine=0)
    A1, _, _, _ = _solve(_upload_stats(ref), d, d, P, lam, refine=1)
    e0 = max(_rel(A0[p], Ar[p]) for p in range(P))
    e1 = max(_rel(A1[p], Ar[p]) for p in range(P))
    assert e1 <= 1e-6 and e1 <= e0, (e0, e1)


@DIGITS
def test_solve_refinement_at_moderate_conditioning(flags):
    """κ(Gc) ≈ 90: with 8-bit digits the band where the plan keeps five digits (15
    pairs, 2^-39.4) and three correction terms; with 7-bit digits it keeps five as
    well (2^-34.4). One sweep must still reach fp32-level accuracy (the residual's
    truncation times κ, and the correction's error, about κ²·2^-40, are near 1e-8
    or below here)."""
    ref, Ar, lam, kappa, d, P = _conditioned_case(23, 4096, 0.9)
    A0, _, _, _ = _solve(_upload_stats(ref), d, d, P, lam, refine=0, flags=flags)
    A1, _, _, _ = _solve(_upload_stats(ref), d, d, P, lam, refine=1, flags=flags)
    e0 = max(_rel(A0[p], Ar[p]) for p in range(P))
    e1 = max(_rel(A1[p], Ar[p]) for p in range(P))
    assert e1 <= 1e-6 and e1 <= e0, (e0, e1)


@DIGITS
def test_solve_repeated_refinement_converges_when_badly_conditioned(flags):
    """κ(Gc) ≈ 1e5: the fp32 solve alone is off by about κ·2^-24 and each sweep shrinks
    the error by about that factor again, down to the residual's own accuracy or the
    fp32 rounding of A (about 6e-8). Reaching 1e-6 needs the residual good to about
    1e-6/κ ≈ 2^-36 of its terms; an fp32-accurate residual would stall near the
    unrefined error. (Measured on a GB300 with 7-bit digits: 1.7e-3 unrefined, 5.4e-8
    after four sweeps.)"""
    ref, Ar, lam, kappa, d, P = _conditioned_case(22, 8192, 2.5)
    errs = {}
    for refine in (0, 4):
        A, _, _, _ = _solve(_upload_stats(ref), d, d, P, lam, refine=refine, flags=flags)
        errs[refine] = max(_rel(A[p], Ar[p]) for p in range(P))
    assert errs[0] > 1e-4, errs   # hard enough that fp32 alone is far off
    assert errs[4] <= 1e-6 and errs[4] < errs[0] / 1000, errs


@DIGITS
def test_solve_degenerate_maps_with_refinement(flags):
    """Maps that exercise the refinement's corner cases, two sweeps: Y = 0 (Cc = 0, so A
    and b stay exactly 0: zero digit rows, T = 0), Y = X (the self map, A = Gc(Gc +
    αI)^-1, [RF] "Ridge map" at l = S), and Y = 1000 X + 7 (the same map scaled by 10^3,
    digits scaled by their row's power of two, b = μ_y − A μ_x). Each against the oracle."""
    d, P, n = 512, 3, 4096
    rng = np.random.default_rng(31)
    X = rng.standard_normal((n, d)) * np.geomspace(1.0, 0.3, d)
    Y = np.stack([np.zeros((n, d)), X, 1000.0 * X + 7.0])
    Xb = torch.as_tensor(X, dtype=torch.float32).to(torch.bfloat16)
    Yb = torch.as_tensor(Y, dtype=torch.float32).to(torch.bfloat16)
    ref = O.calib_stats(_f64(Xb), _f64(Yb))
    Ar, br, _ = O.ridge_solve(ref, 0.03)
    A, b, _, _ = _solve(_upload_stats(ref), d, d, P, 0.03, refine=2, flags=flags)
    assert not np.any(A[0]) and not np.any(b[0])
    for p in (1, 2):
        assert _rel(A[p], Ar[p]) <= 1e-6, (p, _rel(A[p], Ar[p]))
        assert _rel(b[p], br[p]) <= 1e-5, (p, _rel(b[p], br[p]))


@pytest.mark.slow
def test_solve_full_width_sampled_rows():
    d, P, n = 4096, 2, 8192
    cal = synth.calib_inputs(d, d, P, n, index=1, device=DEV)
    Xf, Yf = _f64(cal["X"]), _f64(cal["Y"])
    ref = O.calib_stats(Xf, Yf)
    A, b, _, alpha = _solve(_upload_stats(ref), d, d, P, 0.03)
    Gc, Cc, mx, my = O.centre_stats(ref)
    H = Gc + O.ridge_alpha(Gc, 0.03) * np.eye(d)
    rows = np.sort(np.random.default_rng(2).choice(d, 64, replace=False))
    for p in range(P):
        Ar = np.linalg.solve(H, Cc[p][:, rows]).T        # oracle rows of A_p
        assert _rel(A[p][rows], Ar) <= 1e-5, _rel(A[p][rows], Ar)
        ne = _rel(A[p][rows] @ H, Cc[p][:, rows].T)      # normal equations
        assert ne <= 1e-5, ne
        assert _rel(b[p][rows], my[p][rows] - Ar @ mx) <= 1e-5


# --------------------------------------------------------------------------- #
# Widths that are not powers of two, and the configs' own solve sizes
# --------------------------------------------------------------------------- #
def _solve_vs_oracle(d_in, d_out, P, n, lam, index, refines, device="cpu"):
    """Oracle sums of seeded planted rows -> GPU solve at each refinement count.
    Returns the oracle's (A, b, alpha, H, Cc) and the GPU results by refinement."""
    cal = synth.calib_inputs(d_in, d_out, P, n, index=index, device=device)
    ref = O.calib_stats(_f64(cal["X"]), _f64(cal["Y"]))
    del cal
    Ar, br, alr = O.ridge_solve(ref, lam)
    Gc, Cc, _, _ = O.centre_stats(ref)
    H = Gc + alr * np.eye(d_in)
    st = _upload_stats(ref)
    got = {r: _solve(st, d_in, d_out, P, lam, refine=r) for r in refines}
    return (Ar, br, alr, H, Cc), got


@pytest.mark.parametrize("d_in,d_out,P,n", [(1280, 768, 2, 4096), (768, 512, 3, 3072), (2560, 512, 2, 8192)],
                         ids=["1280: 640+640, then 256+384", "768: 384+384, then 128+256",
                              "2560: tensor-core halves of 1280"])
def test_solve_widths_that_split_unevenly_match_oracle(d_in, d_out, P, n):
    """The factorisation halves its width at multiples of 128 near the middle, so
    widths that are not powers of two split unevenly (640 -> 256 + 384, 384 -> 128 +
    256), and 2560 takes one tensor-core level before the SIMT recursion at 1280:
    the branches the 27B-shaped solve (d = 5120) takes. Every entry of A and b is
    checked against the oracle, unrefined and after one refinement sweep."""
    (Ar, br, alr, H, Cc), got = _solve_vs_oracle(d_in, d_out, P, n, 0.03, index=95, refines=(0, 1))
    for refine, (A, b, Ab, alpha) in got.items():
        assert abs(alpha - alr) <= 1e-12 * alr
        for p in range(P):
            assert _rel(A[p], Ar[p]) <= 1e-5, (refine, p, _rel(A[p], Ar[p]))
            assert _rel(b[p], br[p]) <= 1e-5, (refine, p, _rel(b[p], br[p]))
            assert _rel(A[p] @ H, Cc[p].T) <= 1e-5          # the normal equations


@pytest.mark.parametrize("flags", [rf.RF_FLAG_SINGLE_CTA, rf.RF_FLAG_CTA_PAIR], ids=["single-cta", "cta-pair"])
def test_solve_on_either_gemm_kernel_matches_oracle(flags):
    """d_in = 2560: the factorisation's top node runs its four products on the tensor
    cores (on CTA pairs skipping the factors' zero triangles and unread tiles, on single
    CTAs as full split products), and H^-1 = L^-T L^-1 likewise; both kernels' maps,
    unrefined and after one sweep, against the oracle and the normal equations."""
    d_in, d_out, P, n = 2560, 256, 2, 8192
    cal = synth.calib_inputs(d_in, d_out, P, n, index=96)
    ref = O.calib_stats(_f64(cal["X"]), _f64(cal["Y"]))
    Ar, br, alr = O.ridge_solve(ref, 0.03)
    Gc, Cc, _, _ = O.centre_stats(ref)
    H = Gc + alr * np.eye(d_in)
    st = _upload_stats(ref)
    for refine, tol in ((0, 1e-4), (1, 1e-5)):
        A, b, _, _ = _solve(st, d_in, d_out, P, 0.03, refine=refine, flags=flags)
        for p in range(P):
            assert _rel(A[p], Ar[p]) <= tol, (refine, p, _rel(A[p], Ar[p]))
            assert _rel(b[p], br[p]) <= tol, (refine, p, _rel(b[p], br[p]))
            assert _rel(A[p] @ H, Cc[p].T) <= tol, (refine, p, _rel(A[p] @ H, Cc[p].T))


def _full_width_solve(d_in, d_out, P, n, lam, index):
    (Ar, br, alr, H, Cc), got = _solve_vs_oracle(d_in, d_out, P, n, lam, index, refines=(0, 1), device=DEV)
    errs = {}
    for refine, (A, b, _, alpha) in got.items():
        assert abs(alpha - alr) <= 1e-12 * alr
        errs[refine] = max(_rel(A[p], Ar[p]) for p in range(P))
        for p in range(P):
            assert _rel(b[p], br[p]) <= (1e-5 if refine else 1e-4)
            rows = np.sort(np.random.default_rng(3 + p).choice(d_out, 64, replace=False))
            assert _rel(A[p][rows] @ H, Cc[p][:, rows].T) <= (1e-5 if refine else 1e-4)   # normal equations
    # fp32 factorisation and products alone: about κ·sqrt(d)·2^-24 (κ ≈ 13-30 here);
    # one sweep with the fp64-accurate residual brings A to fp32 accuracy
    assert errs[0] <= 1e-4, errs
    assert errs[1] <= 1e-5 and errs[1] <= errs[0], errs
    return errs


@pytest.mark.slow
def test_solve_27b_shape_matches_oracle():
    """The 27B-shaped solve, d = 5120 (5120 -> 2560 -> 1280 on the tensor cores,
    then 640 -> 256 + 384 in fp32 SIMT), from 16,384 planted calibration rows,
    λ = 0.03: every entry of two maps against the oracle, and the normal equations
    on sampled rows."""
    c = synth.DENSE27B
    _full_width_solve(c.d, c.d, 2, c.calib_n, c.lam, index=c.index)


@pytest.mark.slow
def test_solve_cross_model_gram_shape_matches_oracle():
    """The cross-model mapper's solve: d_in = 8192 concatenated features (k = 8 source
    layers x 8 heads x 128) onto d_out = 1024 target columns, λ = 0.01 with α
    trace-scaled. The fp64 sums come from 16,384 rows (fewer than the 131,072 of the
    calibration, to keep the oracle's Gram quick; the solve's sizes are the same)."""
    x = synth.XMODEL
    _full_width_solve(x.d_in, x.KV, 2, 16384, x.lam, index=x.index)


@pytest.mark.parametrize("world", [2, 3])
def test_calibration_and_solve_by_layer_block_equal_the_whole(world):
    """Calibration and solve shard by upper layer like the fill, with no collective:
    rank r accumulates C and sy for its block of maps from the same X (its G and sx
    are those of every rank) and solves just those maps. Run block by block on one
    GPU, the blocks' sums and maps (with a refinement sweep) equal the whole call's
    bit for bit: every map's sums, factorisation, products and residual are computed
    from its own columns and the shared G alone."""
    from ridge_map_kv_gb300 import shard as sh
    d, P, n = 512, 7, 4096
    cal = synth.calib_inputs(d, d, P, n, index=97)
    X, Y = cal["X"].to(DEV), cal["Y"].to(DEV)
    whole = _zeros_stats(d, d, P)
    _accumulate(X, Y, whole, [2048])
    Aw, bw, _, _ = _solve(whole, d, d, P, 0.03, refine=1)
    for r in range(world):
        blk = sh.layer_shard(P, 0, world, r)
        part = _zeros_stats(d, d, blk.layers)
        _accumulate(X, Y[blk.p0:blk.p1].contiguous(), part, [2048])
        for k in ("G", "sx", "n"):
            assert torch.equal(part[k], whole[k]), k
        assert torch.equal(part["C"], whole["C"][blk.p0:blk.p1]) and torch.equal(part["sy"], whole["sy"][blk.p0:blk.p1])
        A, b, _, _ = _solve(part, d, d, blk.layers, 0.03, refine=1)
        assert np.array_equal(A, Aw[blk.p0:blk.p1]) and np.array_equal(b, bw[blk.p0:blk.p1])
