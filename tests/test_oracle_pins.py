"""Pins for the fp64 oracle: closed forms, invariants, textbook routines, brute
force on tiny inputs and the pages' worked example. These run on CPU only.

Each pin is chosen so that a plausible mistake in the oracle (a dropped term, a
wrong sign or index, a transposed operand, the wrong RoPE pairing) fails at least
one of them. Sources: RidgeFill review (jaehun.me, English edition), sections
"Two numbers set the skip range" and "Ridge map: ..."; the cross-model KV cache
transfer digest, sections on per-head ridge regression and content-space mapping.
"""
import math
import os

import numpy as np
import pytest

import oracle as O

RNG = np.random.default_rng(12345)


def _bf16_round(x):
    """Round float64 -> bf16 bit patterns (round to nearest even) for test inputs."""
    f = np.asarray(x, np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


# --------------------------------------------------------------------------- #
# bf16 decoding
# --------------------------------------------------------------------------- #
def test_bf16_decode_known_values():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000, 0x7F80, 0x0001, 0x4049], np.uint16)
    v = O.bf16_bits_to_f64(bits)
    assert v[0] == 1.0 and v[1] == -2.0
    assert v[2] == 1.0 + 2.0 ** -7
    assert v[3] == 0.0 and np.signbit(v[4])
    assert np.isinf(v[5])
    assert v[6] == 2.0 ** -133
    assert v[7] == 3.140625


# --------------------------------------------------------------------------- #
# RoPE (rotate-half reading)
# --------------------------------------------------------------------------- #
def test_rope_hand_values_fix_pairing_and_frequencies():
    # hd = 4, theta = 100: inv_freq = [1, 100^(-1/2)] = [1, 0.1]; pairs (0,2) and (1,3).
    for pos in (0.0, 1.0, 3.0, 11.0):
        e0 = O.rope(np.array([1.0, 0, 0, 0]), pos, 100.0)
        e1 = O.rope(np.array([0, 1.0, 0, 0]), pos, 100.0)
        e2 = O.rope(np.array([0, 0, 1.0, 0]), pos, 100.0)
        np.testing.assert_allclose(e0, [math.cos(pos), 0, math.sin(pos), 0], atol=1e-15)
        np.testing.assert_allclose(e1, [0, math.cos(0.1 * pos), 0, math.sin(0.1 * pos)], atol=1e-15)
        np.testing.assert_allclose(e2, [-math.sin(pos), 0, math.cos(pos), 0], atol=1e-15)


def test_rope_matches_complex_exponential():
    hd, theta = 64, 5.0e5
    x = RNG.standard_normal((7, hd))
    pos = np.arange(7) * 1000.0 + 3
    z = x[:, :hd // 2] + 1j * x[:, hd // 2:]
    w = np.exp(1j * pos[:, None] * np.exp(-np.log(theta) * np.arange(0, hd, 2) / hd))
    zr = z * w
    np.testing.assert_allclose(O.rope(x, pos, theta),
                               np.concatenate([zr.real, zr.imag], axis=1), rtol=0, atol=1e-11)


def test_rope_group_and_relative_position_properties():
    hd, theta = 128, 1.0e6
    q, k = RNG.standard_normal((2, hd))
    np.testing.assert_allclose(O.rope(q, 0.0, theta), q, atol=0)
    np.testing.assert_allclose(O.rope(O.rope(q, 17.0, theta), 25.0, theta), O.rope(q, 42.0, theta), atol=1e-12)
    np.testing.assert_allclose(O.rope(O.rope(q, 300.0, theta), 300.0, theta, inverse=True), q, atol=1e-12)
    assert abs(np.linalg.norm(O.rope(q, 12345.0, theta)) - np.linalg.norm(q)) < 1e-12
    s1 = O.rope(q, 40.0, theta) @ O.rope(k, 9.0, theta)
    s2 = O.rope(q, 1040.0, theta) @ O.rope(k, 1009.0, theta)
    assert abs(s1 - s2) < 1e-10


# --------------------------------------------------------------------------- #
# RMSNorm
# --------------------------------------------------------------------------- #
def test_rms_norm_invariants():
    x = RNG.standard_normal((5, 96)) * 3.0
    y = O.rms_norm(x, np.ones(96), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, atol=1e-14)
    np.testing.assert_allclose(O.rms_norm(7.5 * x, np.ones(96), 0.0), y, atol=1e-14)
    g = RNG.standard_normal(96)
    np.testing.assert_allclose(O.rms_norm(x, g, 0.0), g * y, atol=1e-14)
    assert np.all(O.rms_norm(np.zeros((1, 8)), np.ones(8), 1e-5) == 0)
    # eps enters inside the square root: x = [a, a], mean(x^2) = a^2
    a, eps = 0.01, 1e-4
    np.testing.assert_allclose(O.rms_norm(np.array([a, a]), np.ones(2), eps), a / math.sqrt(a * a + eps), rtol=1e-15)


# --------------------------------------------------------------------------- #
# Bookkeeping: the pages' worked example
# --------------------------------------------------------------------------- #
def _read_golden(golden_dir, name):
    out = {}
    with open(os.path.join(golden_dir, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            out[k] = [int(t) for t in v]
    return out


def test_worked_example_partition(golden_dir):
    g = _read_golden(golden_dir, "toy_bookkeeping.txt")
    L, N, S, T = g["L"][0], g["N"][0], g["S"][0], g["T"][0]
    mask = np.zeros(N - T, np.uint8)
    mask[g["exact_rows"]] = 1
    assert O.prefix_partition(N, T, mask).tolist() == g["filled_rows"]
    # whole-cache fill touches exactly filled_rows x filled_layers
    d, H, hd = 16, 1, 4
    P = L - S
    kc = np.full((L, N, H, hd), np.nan)
    vc = np.full((L, N, H, hd), np.nan)
    A = np.stack([np.eye(d)] * P)
    b = np.zeros((P, d))
    gain = np.ones((P, d))
    W = RNG.standard_normal((P, H * hd, d))
    x = RNG.standard_normal((N, d))
    k2, v2, idx = O.fill_kv(kc, vc, x, mask, A, b, gain, W, W, L=L, S=S, N=N, T=T,
                            n_kv_heads=H, head_dim=hd, rope_theta=5e5, rms_eps=1e-5)
    written = ~np.isnan(k2[..., 0, 0])
    assert sorted(set(np.nonzero(written)[0].tolist())) == g["filled_layers"]
    assert sorted(set(np.nonzero(written)[1].tolist())) == g["filled_rows"]
    assert written.sum() == len(g["filled_layers"]) * len(g["filled_rows"])
    assert np.array_equal(written, ~np.isnan(v2[..., 0, 0]))
    for t in g["tail_rows"]:
        assert not written[:, t].any()
    for l in g["exact_layers_for_all_rows"]:
        assert not written[l].any()


@pytest.mark.parametrize("case", ["all_fill", "no_fill", "tail_is_all", "one_layer"])
def test_partition_special_arms(case):
    L, N, T, S = 6, 20, 5, 2
    mask = None
    if case == "no_fill":
        mask = np.ones(N - T, np.uint8)       # every prefix row exact: nothing written
    if case == "tail_is_all":
        T = N
    if case == "one_layer":
        S = L - 1
    d, H, hd = 8, 1, 4
    P = L - S
    kc = np.full((L, N, H, hd), np.nan)
    rng = np.random.default_rng(3)
    args = (rng.standard_normal((N, d)), mask, rng.standard_normal((P, d, d)),
            rng.standard_normal((P, d)), np.ones((P, d)), rng.standard_normal((P, H * hd, d)),
            rng.standard_normal((P, H * hd, d)))
    k2, _, idx = O.fill_kv(kc, kc, *args, L=L, S=S, N=N, T=T, n_kv_heads=H, head_dim=hd,
                           rope_theta=1e4, rms_eps=1e-5)
    written = ~np.isnan(k2[..., 0, 0])
    if case == "all_fill":
        assert idx.tolist() == list(range(N - T)) and written[S:, :N - T].all()
        assert not written[:S].any() and not written[:, N - T:].any()
    elif case in ("no_fill", "tail_is_all"):
        assert idx.size == 0 and not written.any()
    else:
        assert written[L - 1, :N - T].all() and written.sum() == N - T


# --------------------------------------------------------------------------- #
# Fill arithmetic
# --------------------------------------------------------------------------- #
def _tiny_fill_problem(seed=7, d=8, H=2, hd=4, P=2, n=3):
    rng = np.random.default_rng(seed)
    return dict(x=rng.standard_normal((n, d)), A=rng.standard_normal((P, d, d)),
                b=rng.standard_normal((P, d)), g=1.0 + 0.1 * rng.standard_normal((P, d)),
                Wk=rng.standard_normal((P, H * hd, d)), Wv=rng.standard_normal((P, H * hd, d)),
                pos=np.array([0, 5, 9]), H=H, hd=hd, P=P, n=n, d=d)


def test_fill_rows_brute_force_scalar_loops():
    """Brute force: every scalar of the definition written as explicit loops."""
    pr = _tiny_fill_problem()
    theta, eps = 1.0e4, 1e-5
    K, V = O.fill_rows(pr["x"], pr["pos"], pr["A"], pr["b"], pr["g"], pr["Wk"], pr["Wv"],
                       pr["H"], pr["hd"], theta, eps)
    d, H, hd = pr["d"], pr["H"], pr["hd"]
    for p in range(pr["P"]):
        for r in range(pr["n"]):
            xh = [sum(pr["A"][p][o][i] * pr["x"][r][i] for i in range(d)) + pr["b"][p][o] for o in range(d)]
            ms = sum(v * v for v in xh) / d
            y = [pr["g"][p][i] * xh[i] / math.sqrt(ms + eps) for i in range(d)]
            for h in range(H):
                kk = [sum(pr["Wk"][p][h * hd + c][i] * y[i] for i in range(d)) for c in range(hd)]
                vv = [sum(pr["Wv"][p][h * hd + c][i] * y[i] for i in range(d)) for c in range(hd)]
                for c in range(hd // 2):
                    ang = pr["pos"][r] * theta ** (-2.0 * c / hd)
                    k1, k2 = kk[c], kk[c + hd // 2]
                    assert abs(K[p, r, h, c] - (k1 * math.cos(ang) - k2 * math.sin(ang))) < 1e-10
                    assert abs(K[p, r, h, c + hd // 2] - (k2 * math.cos(ang) + k1 * math.sin(ang))) < 1e-10
                for c in range(hd):
                    assert abs(V[p, r, h, c] - vv[c]) < 1e-10


def test_identity_fill_arm_gives_same_cache_in_every_layer():
    """Table 3, identity arm: x̂_l = x_S for every l, so with equal layer weights every
    upper layer receives the same approximation (A = I, b = 0)."""
    pr = _tiny_fill_problem(d=16, P=3)
    P, d = pr["P"], pr["d"]
    A = np.stack([np.eye(d)] * P)
    b = np.zeros((P, d))
    g = np.stack([pr["g"][0]] * P)
    Wk = np.stack([pr["Wk"][0]] * P)
    Wv = np.stack([pr["Wv"][0]] * P)
    K, V = O.fill_rows(pr["x"], pr["pos"], A, b, g, Wk, Wv, pr["H"], pr["hd"], 1e4, 1e-5)
    for p in range(1, P):
        np.testing.assert_array_equal(K[p], K[0])
        np.testing.assert_array_equal(V[p], V[0])
    # and x̂ is x_S itself
    np.testing.assert_array_equal(O.map_predict(pr["x"], A[0], b[0]), pr["x"])


def test_constant_map_gives_rotated_constant_key():
    """A = 0, b = c: every row's pre-RoPE key is the same vector k0, so
    unroping K[l][t] at its position recovers k0 for every t, and V is constant."""
    pr = _tiny_fill_problem(d=16, n=3)
    P, d = pr["P"], pr["d"]
    A = np.zeros((P, d, d))
    pos = np.array([0, 7, 1000])
    K, V = O.fill_rows(pr["x"], pos, A, pr["b"], pr["g"], pr["Wk"], pr["Wv"], pr["H"], pr["hd"], 1e4, 1e-5)
    unr = O.rope(K, pos[None, :, None], 1e4, inverse=True)
    for p in range(P):
        np.testing.assert_allclose(unr[p], np.broadcast_to(unr[p, 0], unr[p].shape), atol=1e-12)
        np.testing.assert_allclose(V[p], np.broadcast_to(V[p, 0], V[p].shape), atol=1e-12)
        assert np.abs(unr[p, 0]).max() > 0.1     # the offset b was not dropped


def test_fill_is_scale_invariant_through_the_norm():
    """With eps = 0, scaling x_S and b by c leaves K and V unchanged (the norm sits
    between the map and the projections)."""
    pr = _tiny_fill_problem(d=16)
    K1, V1 = O.fill_rows(pr["x"], pr["pos"], pr["A"], pr["b"], pr["g"], pr["Wk"], pr["Wv"], pr["H"], pr["hd"], 1e4, 0.0)
    K2, V2 = O.fill_rows(3.5 * pr["x"], pr["pos"], pr["A"], 3.5 * pr["b"], pr["g"], pr["Wk"], pr["Wv"], pr["H"], pr["hd"], 1e4, 0.0)
    np.testing.assert_allclose(K1, K2, atol=1e-12)
    np.testing.assert_allclose(V1, V2, atol=1e-12)
    K3, _ = O.fill_rows(pr["x"], pr["pos"], pr["A"], pr["b"], 2.0 * pr["g"], pr["Wk"], pr["Wv"], pr["H"], pr["hd"], 1e4, 0.0)
    np.testing.assert_allclose(K3, 2.0 * K1, atol=1e-12)


def test_position_offset_is_an_extra_rotation():
    L, S, N, T, d, H, hd = 4, 2, 10, 2, 8, 2, 4
    rng = np.random.default_rng(11)
    P = L - S
    args = (rng.standard_normal((N, d)), None, rng.standard_normal((P, d, d)), rng.standard_normal((P, d)),
            np.ones((P, d)), rng.standard_normal((P, H * hd, d)), rng.standard_normal((P, H * hd, d)))
    c0 = np.zeros((L, N, H, hd))
    k0, _, idx = O.fill_kv(c0, c0, *args, L=L, S=S, N=N, T=T, n_kv_heads=H, head_dim=hd, rope_theta=1e4, rms_eps=1e-5)
    k5, _, _ = O.fill_kv(c0, c0, *args, L=L, S=S, N=N, T=T, n_kv_heads=H, head_dim=hd, rope_theta=1e4,
                         rms_eps=1e-5, pos_offset=5)
    np.testing.assert_allclose(k5[S:, idx], O.rope(k0[S:, idx], 5.0, 1e4), atol=1e-12)


def test_map_size_arithmetic(golden_dir):
    """A map is d_out x d_in per layer: the page's printed sizes follow."""
    unit = {"MiB": 2 ** 20, "GiB": 2 ** 30}
    with open(os.path.join(golden_dir, "map_sizes.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for din, dout, nm, eb, val, u in rows:
        A = np.zeros((1, int(dout), int(din)), dtype=np.uint8 if eb == "1" else np.uint16)
        total = A.nbytes * int(nm) / unit[u]
        prec = 10 ** -(len(val.split(".")[1]) if "." in val else 0)
        assert abs(total - float(val)) <= 0.5 * prec + 0.05 * float(val), (din, dout, total, val)


# --------------------------------------------------------------------------- #
# Calibration statistics and the ridge solve
# --------------------------------------------------------------------------- #
def _planted(n=400, din=12, dout=10, P=2, noise=0.0, seed=5, shift=0.0):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((n, din)) + shift
    At = rng.standard_normal((P, dout, din))
    bt = rng.standard_normal((P, dout))
    Y = np.stack([X @ At[p].T + bt[p] + noise * rng.standard_normal((n, dout)) for p in range(P)])
    return X, Y, At, bt


def test_calib_stats_brute_force_and_resume():
    X, Y, _, _ = _planted(n=6, din=3, dout=2, P=2)
    st = O.calib_stats(X, Y)
    for i in range(3):
        for j in range(3):
            assert abs(st["G"][i, j] - sum(X[t, i] * X[t, j] for t in range(6))) < 1e-12
        for p in range(2):
            for j in range(2):
                assert abs(st["C"][p, i, j] - sum(X[t, i] * Y[p, t, j] for t in range(6))) < 1e-12
    assert st["n"] == 6
    np.testing.assert_allclose(st["sx"], [sum(X[t, i] for t in range(6)) for i in range(3)], atol=1e-12)
    both = O.add_stats(O.calib_stats(X[:2], Y[:, :2]), O.calib_stats(X[2:], Y[:, 2:]))
    for k in ("G", "C", "sx", "sy"):
        np.testing.assert_allclose(both[k], st[k], atol=1e-12)
    assert both["n"] == 6


def test_centring_matches_two_pass():
    X, Y, _, _ = _planted(shift=3.0)
    Gc, Cc, mx, my = O.centre_stats(O.calib_stats(X, Y))
    Xc = X - X.mean(0)
    np.testing.assert_allclose(Gc, Xc.T @ Xc, rtol=1e-10, atol=1e-9)
    for p in range(Y.shape[0]):
        np.testing.assert_allclose(Cc[p], Xc.T @ (Y[p] - Y[p].mean(0)), rtol=1e-10, atol=1e-9)


@pytest.mark.parametrize("lam", [0.03, 0.3, 1e-4])
def test_normal_equations_gradient_is_zero(lam):
    """The solved (A, b) zeroes the gradient of Σ_t ||y_t - (A x_t + b)||^2 + alpha ||A||_F^2,
    evaluated from the raw rows, with alpha = lambda tr(XᵀX)/d_in on centred X."""
    X, Y, _, _ = _planted(noise=0.3, shift=0.7)
    A, b, alpha = O.ridge_solve(O.calib_stats(X, Y), lam)
    Xc = X - X.mean(0)
    assert abs(alpha - lam * np.trace(Xc.T @ Xc) / X.shape[1]) < 1e-9 * alpha
    for p in range(Y.shape[0]):
        R = Y[p] - (X @ A[p].T + b[p])
        gA = -2.0 * R.T @ X + 2.0 * alpha * A[p]
        gb = -2.0 * R.sum(0)
        scale = np.abs(Y[p].T @ X).max()
        assert np.abs(gA).max() < 1e-10 * scale
        assert np.abs(gb).max() < 1e-10 * np.abs(Y[p]).sum(0).max()


def test_ridge_equals_augmented_least_squares():
    """Textbook identity: ridge = ordinary least squares on [Xc; sqrt(alpha) I]."""
    X, Y, _, _ = _planted(noise=0.5)
    A, b, alpha = O.ridge_solve(O.calib_stats(X, Y), 0.05)
    Xc = X - X.mean(0)
    for p in range(Y.shape[0]):
        Yc = Y[p] - Y[p].mean(0)
        Xa = np.vstack([Xc, math.sqrt(alpha) * np.eye(X.shape[1])])
        Ya = np.vstack([Yc, np.zeros((X.shape[1], Y.shape[2]))])
        W = np.linalg.lstsq(Xa, Ya, rcond=None)[0]
        np.testing.assert_allclose(A[p], W.T, rtol=1e-9, atol=1e-11)


def test_planted_noiseless_recovery():
    X, Y, At, bt = _planted(noise=0.0, shift=1.5)
    A, b, _ = O.ridge_solve(O.calib_stats(X, Y), 0.0, "absolute")
    np.testing.assert_allclose(A, At, atol=1e-10)
    np.testing.assert_allclose(b, bt, atol=1e-10)
    x_new = np.random.default_rng(99).standard_normal((4, X.shape[1]))
    for p in range(A.shape[0]):
        np.testing.assert_allclose(O.map_predict(x_new, A[p], b[p]), x_new @ At[p].T + bt[p], atol=1e-9)


def test_planted_noise_error_matches_theory():
    """E||Â - A||_F^2 ≈ sigma^2 d_out tr(Gc^-1) for lambda -> 0."""
    sig = 0.05
    errs, preds = [], []
    for seed in range(6):
        X, Y, At, bt = _planted(n=2048, din=32, dout=32, P=1, noise=sig, seed=seed)
        A, b, _ = O.ridge_solve(O.calib_stats(X, Y), 0.0, "absolute")
        Gc, _, _, _ = O.centre_stats(O.calib_stats(X, Y))
        errs.append(np.sum((A[0] - At[0]) ** 2))
        preds.append(sig ** 2 * 32 * np.trace(np.linalg.inv(Gc)))
    ratio = np.mean(errs) / np.mean(preds)
    assert 0.67 < ratio < 1.5, ratio


def test_shift_invariance_of_A():
    X, Y, _, _ = _planted(noise=0.2)
    A1, b1, _ = O.ridge_solve(O.calib_stats(X, Y), 0.03)
    c = np.linspace(-2, 3, X.shape[1])
    A2, b2, _ = O.ridge_solve(O.calib_stats(X + c, Y), 0.03)
    np.testing.assert_allclose(A2, A1, atol=1e-10)
    for p in range(A1.shape[0]):
        np.testing.assert_allclose(b2[p], b1[p] - A1[p] @ c, atol=1e-9)


def test_trace_scaled_alpha_makes_lambda_scale_free():
    X, Y, _, _ = _planted(noise=0.2)
    A1, _, a1 = O.ridge_solve(O.calib_stats(X, Y), 0.03)
    A2, _, a2 = O.ridge_solve(O.calib_stats(4.0 * X, Y), 0.03)
    np.testing.assert_allclose(A2, A1 / 4.0, rtol=1e-10, atol=1e-12)
    assert abs(a2 / a1 - 16.0) < 1e-9


def test_self_map_spectrum():
    """Y = X: A = Gc (Gc + alpha I)^-1 has eigenvalues s / (s + alpha)."""
    X, _, _, _ = _planted(n=300, din=10)
    A, b, alpha = O.ridge_solve(O.calib_stats(X, X[None]), 0.1)
    Gc, _, _, _ = O.centre_stats(O.calib_stats(X, X[None]))
    s = np.linalg.eigvalsh(Gc)
    ev = np.sort(np.linalg.eigvals(A[0]).real)
    np.testing.assert_allclose(ev, np.sort(s / (s + alpha)), atol=1e-12)


def test_resolve_from_same_statistics():
    X, Y, _, _ = _planted(noise=0.2)
    st = O.calib_stats(X, Y)
    O.ridge_solve(st, 0.5)
    A2, b2, _ = O.ridge_solve(st, 0.01)
    A3, b3, _ = O.ridge_solve(O.calib_stats(X, Y), 0.01)
    np.testing.assert_array_equal(A2, A3)
    np.testing.assert_array_equal(b2, b3)


# --------------------------------------------------------------------------- #
# Cross-model mapper
# --------------------------------------------------------------------------- #
def _xm_problem(Ls=5, n=6, H=2, hd=8, k=3, seed=21):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((Ls, n, H, hd)), rng.standard_normal((Ls, n, H, hd)), [1, 3, 4], np.arange(n) * 37.0


def test_xmodel_identity_on_one_source_layer():
    ks, vs, src, pos = _xm_problem()
    H, hd, k = 2, 8, 3
    KV = H * hd
    for j in range(k):
        W = np.zeros((KV, k * KV))
        W[:, j * KV:(j + 1) * KV] = np.eye(KV)
        z = np.zeros(KV)
        Kh, Vh = O.xmodel_map_layer(ks, vs, src, W, z, W, z, pos, 1e6, 1e6, H, hd)
        np.testing.assert_allclose(Kh, ks[src[j]], atol=1e-12)
        np.testing.assert_allclose(Vh, vs[src[j]], atol=1e-12)
        # different target theta: K re-rotated with the target's frequencies, V untouched
        Kh2, Vh2 = O.xmodel_map_layer(ks, vs, src, W, z, W, z, pos, 1e6, 1e4, H, hd)
        unr = O.rope(Kh2, pos[:, None], 1e4, inverse=True)
        np.testing.assert_allclose(O.rope(unr, pos[:, None], 1e6), ks[src[j]], atol=1e-10)
        np.testing.assert_allclose(Vh2, vs[src[j]], atol=1e-12)
        np.testing.assert_allclose(np.linalg.norm(Kh2, axis=-1), np.linalg.norm(ks[src[j]], axis=-1), rtol=1e-12)


def test_xmodel_feature_order_layer_head_dim():
    ks, vs, src, pos = _xm_problem()
    F = O.xmodel_features(vs, src, pos, None)
    j, h, c = 2, 1, 5
    assert F[3, j * 16 + h * 8 + c] == vs[src[j], 3, h, c]


def test_xmodel_bias_and_content_space():
    """With W = 0 the key is RoPE_tgt(b_K): the bias is added before the target RoPE."""
    ks, vs, src, pos = _xm_problem()
    H, hd, k = 2, 8, 3
    KV = H * hd
    bk = np.arange(KV, dtype=float)
    Kh, Vh = O.xmodel_map_layer(ks, vs, src, np.zeros((KV, k * KV)), bk, np.zeros((KV, k * KV)), bk,
                                pos, 1e6, 1e6, H, hd)
    np.testing.assert_allclose(Kh, O.rope(np.broadcast_to(bk.reshape(H, hd), Kh.shape), pos[:, None], 1e6), atol=1e-12)
    np.testing.assert_allclose(Vh, np.broadcast_to(bk.reshape(H, hd), Vh.shape), atol=0)


def test_per_head_solve_equals_multi_output_solve():
    """The per-head ridge of the digest equals the head blocks of one multi-output
    solve when the heads share X (columns of a ridge problem decouple)."""
    rng = np.random.default_rng(8)
    n, din, H, hd = 500, 24, 3, 4
    X = rng.standard_normal((n, din))
    Y = X @ rng.standard_normal((din, H * hd)) + 0.3 * rng.standard_normal((n, H * hd))
    A, b, _ = O.ridge_solve(O.calib_stats(X, Y[None]), 0.01, "absolute")
    for h in range(H):
        Ah, bh, _ = O.ridge_solve(O.calib_stats(X, Y[None, :, h * hd:(h + 1) * hd]), 0.01, "absolute")
        np.testing.assert_allclose(A[0, h * hd:(h + 1) * hd], Ah[0], atol=1e-12)
        np.testing.assert_allclose(b[0, h * hd:(h + 1) * hd], bh[0], atol=1e-12)


def test_flops_per_row_layer():
    # map 2 d^2 plus K and V projections 2 * d * (2 H hd); 8B shape: 11,059 rows x 20 layers.
    f = O.fill_flops_per_row_layer(4096, 8, 128)
    assert f == 2 * 4096 * 4096 + 2 * 4096 * 2048
    assert abs(f * 11059 * 20 / 1e12 - 11.13) < 0.01


# --------------------------------------------------------------------------- #
# Value rescale (RidgeFill review, "Hybrid layers and two corrections")
# --------------------------------------------------------------------------- #
def _rescale_problem(P=2, c=6, d=32, H=2, hd=8, seed=7):
    rng = np.random.default_rng(seed)
    KV = H * hd
    return {"P": P, "c": c, "d": d, "H": H, "hd": hd,
            "x": rng.normal(size=(c, d)), "A": np.eye(d)[None] + 0.1 * rng.normal(size=(P, d, d)),
            "b": 0.1 * rng.normal(size=(P, d)), "g": 1.0 + 0.1 * rng.normal(size=(P, d)),
            "Wv": rng.normal(size=(P, KV, d)) / math.sqrt(d)}


def test_value_scale_is_one_when_the_map_predicts_exactly():
    pr = _rescale_problem()
    x_exact = np.stack([pr["x"] @ pr["A"][p].T + pr["b"][p] for p in range(pr["P"])])
    s = O.value_scale(pr["x"], x_exact, pr["A"], pr["b"], pr["g"], pr["Wv"], pr["H"], pr["hd"], 1e-5)
    assert s.shape == (pr["P"], pr["H"])
    np.testing.assert_allclose(s, 1.0, rtol=0, atol=1e-12)


def test_value_scale_closed_form_for_a_scaled_subspace():
    """W_v reads only coordinates [0, k). If the exact input equals the prediction
    with those coordinates multiplied by beta, every head's exact value is the
    predicted one times beta * rms(x̂) / rms(x_exact), rms including eps, so the
    scale is the row mean of that factor, the same for every head."""
    pr = _rescale_problem(P=2, c=5, d=32, H=3, hd=8)
    k, beta, eps = 12, 2.5, 1e-3
    Wv = pr["Wv"].copy()
    Wv[:, :, k:] = 0.0
    xhat = np.stack([pr["x"] @ pr["A"][p].T + pr["b"][p] for p in range(pr["P"])])
    x_exact = xhat.copy()
    x_exact[:, :, :k] *= beta
    s = O.value_scale(pr["x"], x_exact, pr["A"], pr["b"], pr["g"], Wv, pr["H"], pr["hd"], eps)
    for p in range(pr["P"]):
        rms_pred = np.sqrt((xhat[p] ** 2).mean(axis=1) + eps)
        rms_exact = np.sqrt((x_exact[p] ** 2).mean(axis=1) + eps)
        want = np.mean(beta * rms_pred / rms_exact)
        np.testing.assert_allclose(s[p], want, rtol=1e-12)


def test_value_scale_invariants_and_direction():
    pr = _rescale_problem(P=1, c=7, d=24, H=2, hd=6, seed=11)
    rng = np.random.default_rng(3)
    x_exact = rng.normal(size=(1, pr["c"], pr["d"]))
    args = (pr["A"], pr["b"], pr["g"])
    s = O.value_scale(pr["x"], x_exact, *args, pr["Wv"], pr["H"], pr["hd"], 1e-5)
    # order of the c rows does not matter
    perm = rng.permutation(pr["c"])
    s_perm = O.value_scale(pr["x"][perm], x_exact[:, perm], *args, pr["Wv"], pr["H"], pr["hd"], 1e-5)
    np.testing.assert_allclose(s_perm, s, rtol=1e-12)
    # a head's W_v rows scaled by any factor cancel in its ratio and leave the other head alone
    W2 = pr["Wv"].copy()
    W2[:, 0:pr["hd"]] *= 7.0
    np.testing.assert_allclose(O.value_scale(pr["x"], x_exact, *args, W2, pr["H"], pr["hd"], 1e-5), s, rtol=1e-12)
    # the ratio is exact over predicted: with one row, swapping the two inputs inverts it
    xhat0 = pr["x"][:1] @ pr["A"][0].T + pr["b"][0]
    eye = (np.eye(pr["d"])[None], np.zeros((1, pr["d"])))
    s1 = O.value_scale(xhat0, x_exact[:, :1], *eye, pr["g"], pr["Wv"], pr["H"], pr["hd"], 1e-5)
    s2 = O.value_scale(x_exact[0, :1], xhat0[None], *eye, pr["g"], pr["Wv"], pr["H"], pr["hd"], 1e-5)
    np.testing.assert_allclose(s1 * s2, 1.0, rtol=1e-12)
    assert not np.allclose(s1, 1.0)


def test_value_scale_skips_rows_with_a_zero_prediction():
    pr = _rescale_problem(P=1, c=4, d=16, H=2, hd=4, seed=5)
    rng = np.random.default_rng(9)
    x_exact = rng.normal(size=(1, 4, 16))
    b = pr["b"].copy()
    x = pr["x"].copy()
    x[2] = 0.0
    b[0] = 0.0            # row 2 predicts x̂ = 0, so every head's v_pred is 0 there
    s_all = O.value_scale(x, x_exact, pr["A"], b, pr["g"], pr["Wv"], 2, 4, 1e-5)
    keep = [0, 1, 3]
    s_kept = O.value_scale(x[keep], x_exact[:, keep], pr["A"], b, pr["g"], pr["Wv"], 2, 4, 1e-5)
    np.testing.assert_allclose(s_all, s_kept, rtol=1e-12)
    only_zero = O.value_scale(x[2:3], x_exact[:, 2:3], pr["A"], b, pr["g"], pr["Wv"], 2, 4, 1e-5)
    np.testing.assert_array_equal(only_zero, 1.0)


def test_fill_rows_value_scale_multiplies_values_only():
    pr = _rescale_problem(P=2, c=3, d=16, H=2, hd=4, seed=21)
    rng = np.random.default_rng(1)
    Wk = rng.normal(size=(2, 8, 16))
    vs = np.array([[1.5, 0.25], [2.0, -1.0]])
    pos = np.arange(3) + 10
    K0, V0 = O.fill_rows(pr["x"], pos, pr["A"], pr["b"], pr["g"], Wk, pr["Wv"], 2, 4, 1e4, 1e-5)
    K1, V1 = O.fill_rows(pr["x"], pos, pr["A"], pr["b"], pr["g"], Wk, pr["Wv"], 2, 4, 1e4, 1e-5, v_scale=vs)
    np.testing.assert_array_equal(K1, K0)
    for p in range(2):
        for h in range(2):
            np.testing.assert_allclose(V1[p, :, h], vs[p, h] * V0[p, :, h], rtol=1e-14)


# --------------------------------------------------------------------------- #
# Key normalisation ("Qwen models normalize keys")
# --------------------------------------------------------------------------- #
def _knorm_args(pr, gk, eps=0.0, Wk=None):
    return (pr["x"], pr["pos"], pr["A"], pr["b"], pr["g"], pr["Wk"] if Wk is None else Wk, pr["Wv"],
            pr["H"], pr["hd"], 1.0e4, eps)


def test_key_norm_fixes_every_key_magnitude():
    """eps = 0 and g_k = 1: each key head has RMS 1 before RoPE, and RoPE keeps
    norms, so every filled key head has norm sqrt(hd) exactly; with a general g_k
    the un-rotated key divided by g_k has RMS 1."""
    pr = _tiny_fill_problem()
    P, hd = pr["P"], pr["hd"]
    K, V = O.fill_rows(*_knorm_args(pr, None), k_norm_gain=np.ones((P, hd)))
    np.testing.assert_allclose(np.linalg.norm(K, axis=-1), math.sqrt(hd), rtol=1e-12)
    gk = 1.0 + 0.5 * RNG.uniform(size=(P, hd))
    K2, V2 = O.fill_rows(*_knorm_args(pr, None), k_norm_gain=gk)
    for p in range(P):
        raw = O.rope(K2[p], np.asarray(pr["pos"], np.float64)[:, None], 1.0e4, inverse=True) / gk[p]
        np.testing.assert_allclose(np.sqrt(np.mean(raw ** 2, axis=-1)), 1.0, rtol=1e-12)
    _, V0 = O.fill_rows(*_knorm_args(pr, None))
    np.testing.assert_array_equal(V, V0)      # values are not normalised


def test_key_norm_removes_the_key_projection_scale():
    pr = _tiny_fill_problem()
    gk = 1.0 + 0.1 * RNG.normal(size=(pr["P"], pr["hd"]))
    K1, _ = O.fill_rows(*_knorm_args(pr, None), k_norm_gain=gk)
    K2, _ = O.fill_rows(*_knorm_args(pr, None, Wk=3.5 * np.asarray(pr["Wk"])), k_norm_gain=gk)
    np.testing.assert_allclose(K2, K1, rtol=1e-12, atol=1e-12)
    K3, _ = O.fill_rows(*_knorm_args(pr, None, Wk=3.5 * np.asarray(pr["Wk"])))
    K4, _ = O.fill_rows(*_knorm_args(pr, None))
    np.testing.assert_allclose(K3, 3.5 * K4, rtol=1e-12)   # without the norm the scale stays


def test_key_norm_brute_force_scalar_loops():
    pr = _tiny_fill_problem()
    theta, eps = 1.0e4, 1e-3
    gk = 1.0 + 0.2 * RNG.normal(size=(pr["P"], pr["hd"]))
    K, _ = O.fill_rows(pr["x"], pr["pos"], pr["A"], pr["b"], pr["g"], pr["Wk"], pr["Wv"], pr["H"], pr["hd"],
                       theta, eps, k_norm_gain=gk)
    d, H, hd = pr["d"], pr["H"], pr["hd"]
    for p in range(pr["P"]):
        for r in range(pr["n"]):
            xh = [sum(pr["A"][p][o][i] * pr["x"][r][i] for i in range(d)) + pr["b"][p][o] for o in range(d)]
            ms = sum(v * v for v in xh) / d
            y = [pr["g"][p][i] * xh[i] / math.sqrt(ms + eps) for i in range(d)]
            for h in range(H):
                kk = [sum(pr["Wk"][p][h * hd + c][i] * y[i] for i in range(d)) for c in range(hd)]
                km = sum(v * v for v in kk) / hd
                kn = [gk[p][c] * kk[c] / math.sqrt(km + eps) for c in range(hd)]
                for c in range(hd // 2):
                    ang = pr["pos"][r] * theta ** (-2.0 * c / hd)
                    k1, k2 = kn[c], kn[c + hd // 2]
                    assert abs(K[p, r, h, c] - (k1 * math.cos(ang) - k2 * math.sin(ang))) < 1e-10
                    assert abs(K[p, r, h, c + hd // 2] - (k2 * math.cos(ang) + k1 * math.sin(ang))) < 1e-10


# --------------------------------------------------------------------------- #
# Non-square maps (RidgeFill review, "Ridge map": 10,240 -> 2,560 for Flash-Next)
# --------------------------------------------------------------------------- #
def test_stream_mean_map_reduces_to_the_square_identity_fill():
    """x_S made of 4 identical streams of width d, A = [I I I I] / 4, b = 0: x̂ = x,
    so the fill equals the square identity fill of x."""
    pr = _tiny_fill_problem()
    d, P = pr["d"], pr["P"]
    x4 = np.concatenate([pr["x"]] * 4, axis=1)
    A4 = np.stack([np.concatenate([np.eye(d)] * 4, axis=1) / 4.0] * P)
    b0 = np.zeros((P, d))
    K1, V1 = O.fill_rows(x4, pr["pos"], A4, b0, pr["g"], pr["Wk"], pr["Wv"], pr["H"], pr["hd"], 1e4, 1e-5)
    K2, V2 = O.fill_rows(pr["x"], pr["pos"], np.stack([np.eye(d)] * P), b0, pr["g"], pr["Wk"], pr["Wv"],
                         pr["H"], pr["hd"], 1e4, 1e-5)
    np.testing.assert_allclose(K1, K2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(V1, V2, rtol=1e-12, atol=1e-12)


def test_rectangular_map_brute_force():
    rng = np.random.default_rng(17)
    d_in, d, H, hd, P, n = 6, 4, 1, 4, 2, 2
    x = rng.standard_normal((n, d_in))
    A = rng.standard_normal((P, d, d_in))
    b = rng.standard_normal((P, d))
    g = 1.0 + 0.1 * rng.standard_normal((P, d))
    Wk = rng.standard_normal((P, H * hd, d))
    Wv = rng.standard_normal((P, H * hd, d))
    pos = np.array([2, 7])
    K, V = O.fill_rows(x, pos, A, b, g, Wk, Wv, H, hd, 1e4, 1e-5)
    for p in range(P):
        for r in range(n):
            xh = [sum(A[p][o][i] * x[r][i] for i in range(d_in)) + b[p][o] for o in range(d)]
            ms = sum(v * v for v in xh) / d
            y = [g[p][i] * xh[i] / math.sqrt(ms + 1e-5) for i in range(d)]
            vv = [sum(Wv[p][c][i] * y[i] for i in range(d)) for c in range(hd)]
            for c in range(hd):
                assert abs(V[p, r, 0, c] - vv[c]) < 1e-10


# --------------------------------------------------------------------------- #
# int8 maps (symmetric per output row)
# --------------------------------------------------------------------------- #
def test_int8_rows_hit_full_range_and_the_rounding_bound():
    rng = np.random.default_rng(23)
    A = (rng.standard_normal((3, 16, 40)) * rng.uniform(0.01, 3.0, size=(3, 16, 1))).astype(np.float32)
    q, s = O.quantize_rows_int8(A)
    assert q.dtype == np.int8 and s.dtype == np.float32
    assert np.all(np.abs(q.astype(int)).max(axis=-1) == 127)            # every row uses the full range
    err = np.abs(A.astype(np.float64) - O.dequantize_rows_int8(q, s))
    assert np.all(err <= 0.5 * s.astype(np.float64)[..., None] * (1 + 1e-6))   # half a step, up to fp32 division
    # exact for rows that are integers times a power of two
    B = np.zeros((1, 2, 8), np.float32)
    B[0, 0] = np.arange(-3, 5) * 0.25
    B[0, 1] = np.array([127, -127, 0, 1, -1, 64, 2, 3]) * 2.0 ** -5
    qb, sb = O.quantize_rows_int8(B)
    np.testing.assert_array_equal(O.dequantize_rows_int8(qb, sb)[0, 1], B[0, 1].astype(np.float64))


def test_int8_zero_row_power_of_two_scaling_and_half_even_ties():
    A = np.zeros((2, 4), np.float32)
    A[1] = [127.0, 0.5, 1.5, -2.5]                 # s = 1: ties at .5 go to the even neighbour
    q, s = O.quantize_rows_int8(A)
    np.testing.assert_array_equal(s, [0.0, 1.0])
    np.testing.assert_array_equal(q[0], 0)
    np.testing.assert_array_equal(q[1], [127, 0, 2, -2])
    q2, s2 = O.quantize_rows_int8(A * np.float32(8.0))
    np.testing.assert_array_equal(q2, q)
    np.testing.assert_array_equal(s2, s * 8)


# --------------------------------------------------------------------------- #
# Cross-layer source selection (greedy forward selection by head-mean R²)
# --------------------------------------------------------------------------- #
def _layered_rows(n, L_src, F, P, Ft, seed, noise=0.3):
    """Tiny raw calibration rows: source features [n, L_src*F] from a random walk
    over layers, targets [P, n, Ft] as noisy linear functions of two layers."""
    rng = np.random.default_rng(seed)
    R = 3
    r = [rng.standard_normal((n, R))]
    for _ in range(1, L_src):
        r.append(r[-1] + 0.7 * rng.standard_normal((n, R)))
    X = np.concatenate([r[s] @ rng.standard_normal((R, F)) + noise * rng.standard_normal((n, F))
                        for s in range(L_src)], axis=1) + 0.5
    Ys = np.stack([r[p % L_src] @ rng.standard_normal((R, Ft)) + r[(p + 2) % L_src] @ rng.standard_normal((R, Ft))
                   + noise * rng.standard_normal((n, Ft)) - 1.0 for p in range(P)])
    return X, Ys


def _head_r2_from_fit(Y, Yhat, head_dim, penalty=None):
    """Head-mean R² straight from rows: 1 - (‖Y_h - Ŷ_h‖² + penalty_h) / ‖Y_h - Ȳ_h‖²."""
    res = ((Y - Yhat) ** 2).sum(axis=0)
    if penalty is not None:
        res = res + penalty
    tot = ((Y - Y.mean(axis=0)) ** 2).sum(axis=0)
    rh = 1.0 - res.reshape(-1, head_dim).sum(axis=1) / tot.reshape(-1, head_dim).sum(axis=1)
    return rh.mean()


def _cols(layers, F):
    return np.concatenate([np.arange(s * F, (s + 1) * F) for s in layers])


def test_selection_score_is_least_squares_r2_of_the_rows():
    # lambda = 0: the score of a set is the head-mean R² of an ordinary least-squares
    # fit with an intercept column, solved by lstsq from the raw rows.
    n, L, F, P, Ft, hd = 300, 4, 3, 2, 4, 2
    X, Ys = _layered_rows(n, L, F, P, Ft, seed=7)
    st = O.calib_stats(X, Ys)
    for layers in ([1], [3, 0], [2, 1, 3]):
        got = O.selection_scores([st], layers, F, hd, 0.0, "absolute")[0]
        Z = np.concatenate([X[:, _cols(layers, F)], np.ones((n, 1))], axis=1)
        for p in range(P):
            w, *_ = np.linalg.lstsq(Z, Ys[p], rcond=None)
            assert abs(got[p] - _head_r2_from_fit(Ys[p], Z @ w, hd)) < 1e-10


@pytest.mark.parametrize("mode", ["absolute", "trace"])
def test_selection_score_is_one_minus_ridge_objective_over_tss(mode):
    # lambda > 0: with alpha from the centred Gram of ALL source features (trace mode)
    # or alpha = lambda, the score is 1 - (RSS + alpha |w|²)/TSS per head, w being the
    # ridge solution of the centred rows, solved as the augmented least-squares
    # problem [Xc; sqrt(alpha) I] w = [Yc; 0] (a textbook identity).
    n, L, F, P, Ft, hd = 250, 4, 3, 2, 4, 2
    X, Ys = _layered_rows(n, L, F, P, Ft, seed=8)
    st = O.calib_stats(X, Ys)
    lam = 0.3
    Xc = X - X.mean(axis=0)
    alpha = lam * np.trace(Xc.T @ Xc) / Xc.shape[1] if mode == "trace" else lam
    layers = [2, 0]
    got = O.selection_scores([st], layers, F, hd, lam, mode)[0]
    Xs = Xc[:, _cols(layers, F)]
    aug = np.concatenate([Xs, math.sqrt(alpha) * np.eye(Xs.shape[1])], axis=0)
    for p in range(P):
        Yc = Ys[p] - Ys[p].mean(axis=0)
        w, *_ = np.linalg.lstsq(aug, np.concatenate([Yc, np.zeros((Xs.shape[1], Ft))]), rcond=None)
        want = _head_r2_from_fit(Yc, Xs @ w, hd, penalty=alpha * (w ** 2).sum(axis=0))
        assert abs(got[p] - want) < 1e-10


def test_single_feature_score_is_squared_correlation():
    # One feature per layer, one column per head, lambda = 0: R² = Pearson r².
    rng = np.random.default_rng(9)
    n = 500
    X = rng.standard_normal((n, 3))
    X[:, 1] += 0.8 * X[:, 0]
    Y = (0.6 * X[:, 0] - 0.3 * X[:, 2] + rng.standard_normal(n))[None, :, None]
    st = O.calib_stats(X, Y)
    for s in range(3):
        got = O.selection_scores([st], [s], 1, 1, 0.0, "absolute")[0, 0]
        assert abs(got - np.corrcoef(X[:, s], Y[0, :, 0])[0, 1] ** 2) < 1e-12


def test_greedy_path_is_the_argmax_of_least_squares_r2_at_every_step():
    # Brute force: at every step, fit every remaining layer added to the chosen ones
    # by lstsq from the rows; the oracle's table must hold those scores and its
    # choice must be their argmax.
    n, L, F, P, Ft, hd, k = 400, 5, 2, 3, 4, 2, 4
    X, Ys = _layered_rows(n, L, F, P, Ft, seed=10)
    st = O.calib_stats(X, Ys)
    sel, table = O.select_sources([st], L, F, hd, k, 0.0, "absolute")
    for p in range(P):
        chosen = []
        for j in range(k):
            scores = np.full(L, -np.inf)
            for s in range(L):
                if s in chosen:
                    assert np.isnan(table[0, p, j, s])
                    continue
                Z = np.concatenate([X[:, _cols(chosen + [s], F)], np.ones((n, 1))], axis=1)
                w, *_ = np.linalg.lstsq(Z, Ys[p], rcond=None)
                scores[s] = _head_r2_from_fit(Ys[p], Z @ w, hd)
                assert abs(table[0, p, j, s] - scores[s]) < 1e-10
            assert sel[p, j] == int(np.argmax(scores))
            chosen.append(int(sel[p, j]))
        assert sorted(chosen) == sorted(set(chosen))


def test_planted_source_layers_are_found_and_explain_everything():
    # A noise-free target built from layers 3 (larger weight) and 1 is explained
    # exactly by them: the path starts [3, 1] and the step-2 score is 1.
    rng = np.random.default_rng(11)
    n, L, F = 600, 5, 4
    X = rng.standard_normal((n, L * F))
    Y = (3.0 * X[:, 12:16] @ rng.standard_normal((4, 4)) + X[:, 4:8] @ rng.standard_normal((4, 4)))[None]
    st = O.calib_stats(X, Y)
    sel, table = O.select_sources([st], L, F, 2, 3, 0.0, "absolute")
    assert list(sel[0, :2]) == [3, 1]
    assert abs(table[0, 0, 1, 1] - 1.0) < 1e-10
    assert np.all(table[0, 0, 0, [0, 1, 2, 4]] < table[0, 0, 0, 3])


def test_selection_is_equivariant_under_layer_permutation():
    n, L, F, P, Ft, hd, k = 300, 5, 2, 2, 4, 2, 3
    X, Ys = _layered_rows(n, L, F, P, Ft, seed=12)
    perm = np.array([3, 0, 4, 1, 2])          # new layer i is old layer perm[i]
    Xp = np.concatenate([X[:, perm[i] * F:(perm[i] + 1) * F] for i in range(L)], axis=1)
    s0, t0 = O.select_sources([O.calib_stats(X, Ys)], L, F, hd, k, 0.05)
    s1, t1 = O.select_sources([O.calib_stats(Xp, Ys)], L, F, hd, k, 0.05)
    np.testing.assert_array_equal(perm[s1], s0)
    np.testing.assert_allclose(t1, t0[..., perm], atol=1e-10)


def test_joint_selection_averages_the_kinds():
    # Two identical kinds select like one. With two different kinds, each kind's table
    # entry is that kind's own score of the set, and each step takes the argmax of
    # the mean of the two tables.
    n, L, F, P, Ft, hd, k = 300, 4, 2, 2, 4, 2, 3
    X, Ys = _layered_rows(n, L, F, P, Ft, seed=13)
    X2, Ys2 = _layered_rows(n, L, F, P, Ft, seed=14)
    a, b = O.calib_stats(X, Ys), O.calib_stats(X2, Ys2)
    s1, t1 = O.select_sources([a], L, F, hd, k, 0.01)
    s2, t2 = O.select_sources([a, a], L, F, hd, k, 0.01)
    np.testing.assert_array_equal(s1, s2)
    np.testing.assert_allclose(t2[1], t1[0], atol=0)
    sj, tj = O.select_sources([a, b], L, F, hd, k, 0.01)
    for p in range(P):
        chosen = []
        for j in range(k):
            sa = O.selection_scores([a], chosen + [int(sj[p, j])], F, hd, 0.01)[0, p]
            sb = O.selection_scores([b], chosen + [int(sj[p, j])], F, hd, 0.01)[0, p]
            assert abs(tj[0, p, j, sj[p, j]] - sa) < 1e-12 and abs(tj[1, p, j, sj[p, j]] - sb) < 1e-12
            assert sj[p, j] == int(np.nanargmax(tj[:, p, j].mean(axis=0)))
            chosen.append(int(sj[p, j]))


def test_calibration_sum_of_squares_gives_total_variance():
    rng = np.random.default_rng(15)
    X = rng.standard_normal((100, 4))
    Y = rng.standard_normal((2, 100, 3)) * 2 + 1
    st = O.add_stats(O.calib_stats(X[:60], Y[:, :60]), O.calib_stats(X[60:], Y[:, 60:]))
    tss = st["syy"] - st["n"] * (st["sy"] / st["n"]) ** 2
    np.testing.assert_allclose(tss, Y.var(axis=1) * 100, rtol=1e-12)


def test_replayed_path_reproduces_the_greedy_run_and_scores_its_prefixes():
    # Replaying the oracle's own greedy choices must give back its selection and its
    # whole score table exactly. Replaying a hand-chosen path (not the greedy one)
    # must record, at each step, every remaining layer's score as the head-mean R²
    # of a least-squares fit (lstsq with an intercept column, from the raw rows) on
    # the path's prefix plus that layer, NaN for the prefix's own layers, and must
    # return the path itself as the selection.
    n, L, F, P, Ft, hd, k = 400, 5, 2, 2, 4, 2, 4
    X, Ys = _layered_rows(n, L, F, P, Ft, seed=16)
    st = O.calib_stats(X, Ys)
    sel, table = O.select_sources([st], L, F, hd, k, 0.0, "absolute")
    sel2, table2 = O.select_sources([st], L, F, hd, k, 0.0, "absolute", path=sel)
    np.testing.assert_array_equal(sel2, sel)
    np.testing.assert_array_equal(table2, table)          # NaNs in the same places
    path = np.array([[4, 0, 2, 1], [1, 3, 0, 4]])
    assert not np.array_equal(path, sel)
    selp, tablep = O.select_sources([st], L, F, hd, k, 0.0, "absolute", path=path)
    np.testing.assert_array_equal(selp, path)
    for p in range(P):
        for j in range(k):
            prefix = [int(c) for c in path[p, :j]]
            for s in range(L):
                if s in prefix:
                    assert np.isnan(tablep[0, p, j, s])
                    continue
                Z = np.concatenate([X[:, _cols(prefix + [s], F)], np.ones((n, 1))], axis=1)
                w, *_ = np.linalg.lstsq(Z, Ys[p], rcond=None)
                assert abs(tablep[0, p, j, s] - _head_r2_from_fit(Ys[p], Z @ w, hd)) < 1e-10
