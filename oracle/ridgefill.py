"""Plain float64 CPU oracle for the RidgeFill upper-layer KV fill, its calibration
statistics and closed-form ridge solve, and the cross-model per-head ridge mapper.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or links this
module: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
use it. It shares no code with the CUDA library (no kernels, headers, tables or
helpers); the two meet only through the seeded input generators in ``synth/``.

Every function restates one definition from the pages, in float64, with numpy's
matmul, ``linalg.solve`` and elementwise math as the only library steps. There is no
blocking, fusion or reordering beyond what the definition states. Inputs arrive as
the same bf16 bit patterns the GPU receives and are decoded exactly.

Sources (cited by page and section):
  [RF] RidgeFill review, jaehun.me, English edition ("Paper: RidgeFill" review of
       arXiv 2611.09709). Sections "Two numbers set the skip range", "Ridge map:
       predict the input, and the original projection runs unchanged", Table 2
       (notation), Table 3 (the four arms), the worked example "A small example:
       how one row lands in the cache", and "Hybrid layers and two corrections"
       (value rescale).
  [XM] "Cross-Model KV Cache Transfer in LLM Families: A Closed-Form Linear Mapping
       for Prefill Reuse" (digest, seosoyoung.eiaserinnys.me). Sections "헤드별 리지
       회귀" (per-head ridge regression), "층 교차 소스 선택" (cross-layer source
       selection), "RoPE를 제거한 내용 공간 매핑" (content-space mapping, equation
       for K̂_t).

Readings where the pages leave a step open:
  * x_S is the residual stream entering layer S; one map per layer l in [S, L).
  * RMSNorm is y = g * x / sqrt(mean(x^2) + eps); K/V projections have no bias.
  * RoPE is the rotate-half form: pair (i, i + hd/2), inv_freq_i = theta^(-2i/hd),
    angle = position * inv_freq_i, position = row index + pos_offset.
  * Calibration sums are raw one-pass sums; they are centred at solve time.
  * alpha = lambda * tr(Gc) / d_in by default ("trace" mode), or alpha = lambda.
  * The cross-model bias is b = mu_Y - W mu_X (centred-ridge identity).
  * Value rescale: "the first c rows of the tail" are rows N-T .. N-T+c-1; the
    value projection includes the layer's RMSNorm (the same path as the fill);
    a head's "magnitude" is the L2 norm of its hd-vector; rows whose predicted
    norm is 0 carry no ratio and are left out of the mean (scale 1 if none is left).
  * Key normalisation ("Qwen models normalize keys", same section): an RMSNorm of
    each key head over its hd values, k_h <- g_k * k_h / sqrt(mean(k_h^2) + eps)
    with one gain vector g_k of length hd per layer and the layer's eps, applied
    after the K projection and before RoPE.
  * int8 maps ([RF] "Ridge map": 27B's 48 maps "in int8 total 1.2 GiB"; the scheme
    is unstated): symmetric per output row, s[o] = max_i |A[o][i]| / 127 and
    q[o][i] = rint(A[o][i] / s[o]) (round half to even), both in float32 (the
    precision that decides the integers); a zero row has s = 0, q = 0. The map
    used is then A'[o][i] = s[o] q[o][i].
  * Source selection ([XM] greedy forward selection by head-mean R²): a head's R²
    is the share of its total centred variance (over its head_dim columns) that
    the fit explains; the fit is the ridge regression with the mapper's lambda and
    one alpha per kind from the Gram of all source features, and its explained
    energy c_oᵀ(Gc_SS + alpha I)⁻¹c_o makes R² = 1 - (RSS + alpha|w|²)/TSS, the
    least-squares R² at lambda = 0; keys and values share one set per target
    layer, chosen by the mean of their head-mean R²; ties go to the lower layer
    index; a head with zero variance has R² = 0.

Parity status: every public function here is pinned by tests/test_oracle_pins.py
against closed forms, invariants, textbook routines or brute force; none is
"parity unpinned".
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_bits_to_f64", "rope_inv_freq", "rope", "rms_norm", "prefix_partition",
    "map_predict", "fill_rows", "fill_kv", "calib_stats", "centre_stats",
    "ridge_alpha", "ridge_solve", "xmodel_features", "xmodel_map_layer",
    "fill_flops_per_row_layer", "value_scale", "quantize_rows_int8", "dequantize_rows_int8",
    "selection_scores", "select_sources",
]


# --------------------------------------------------------------------------- #
# Number format
# --------------------------------------------------------------------------- #
def bf16_bits_to_f64(bits) -> np.ndarray:
    """Decode bfloat16 bit patterns (uint16 / int16 arrays) exactly to float64.

    A bf16 value is the upper 16 bits of an IEEE binary32, so widening the bit
    pattern by 16 zero bits and reinterpreting as float32 is exact.
    """
    u = np.asarray(bits).view(np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------- #
# RoPE and RMSNorm: the layer's own operations that run unchanged on the
# predicted input ([RF] "Ridge map ... the original projection runs unchanged").
# --------------------------------------------------------------------------- #
def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """Rotary inverse frequencies theta^(-2i/hd), i = 0 .. hd/2 - 1 (float64)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * i / head_dim)


def rope(x: np.ndarray, positions, theta: float, inverse: bool = False) -> np.ndarray:
    """Rotate-half RoPE over the last axis of ``x`` (length hd).

    Pair (i, i + hd/2) is rotated by angle pos * inv_freq_i. ``positions`` must
    broadcast against ``x.shape[:-1]``. ``inverse=True`` applies R^-1 (the
    "unrope" of [XM] content-space mapping).
    """
    x = np.asarray(x, dtype=np.float64)
    hd = x.shape[-1]
    half = hd // 2
    pos = np.asarray(positions, dtype=np.float64)[..., None]
    ang = pos * rope_inv_freq(hd, theta)
    c, s = np.cos(ang), np.sin(ang)
    if inverse:
        s = -s
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rms_norm(x: np.ndarray, gain: np.ndarray, eps: float) -> np.ndarray:
    """y = g * x / sqrt(mean(x^2) + eps) over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return np.asarray(gain, dtype=np.float64) * x / np.sqrt(ms + eps)


# --------------------------------------------------------------------------- #
# Bookkeeping: which rows are filled ([RF] "Two numbers set the skip range")
# --------------------------------------------------------------------------- #
def prefix_partition(N: int, T: int, exact_mask=None) -> np.ndarray:
    """Rows filled by the map: prefix rows t < N - T that are not exact rows.

    Layers < S run for every row, the last T rows run every layer, and an exact
    prefix row runs every layer; the rest of the prefix is filled. Returned in
    ascending order (int64).
    """
    n_prefix = N - T
    if exact_mask is None:
        return np.arange(n_prefix, dtype=np.int64)
    m = np.asarray(exact_mask).astype(bool)
    assert m.shape == (n_prefix,)
    return np.nonzero(~m)[0].astype(np.int64)


# --------------------------------------------------------------------------- #
# The fill ([RF] "Ridge map", equation x̂_l = A_l x_S + b_l, and Fig. 2)
# --------------------------------------------------------------------------- #
def map_predict(x_S: np.ndarray, A_l: np.ndarray, b_l: np.ndarray) -> np.ndarray:
    """x̂_l = A_l x_S + b_l for each row of ``x_S`` ([n, d_in] -> [n, d_out])."""
    return np.asarray(x_S, np.float64) @ np.asarray(A_l, np.float64).T + np.asarray(b_l, np.float64)


def fill_rows(x_S_rows, positions, A, b, gain, Wk, Wv, n_kv_heads, head_dim,
              rope_theta, rms_eps, v_scale=None, k_norm_gain=None):
    """Filled keys and values for a set of rows and every upper layer.

    For each row t and upper layer l (index p = l - S):
        x̂ = A_p x_S[t] + b_p
        y  = g_p * x̂ / sqrt(mean(x̂^2) + eps)
        k  = Wk_p y,  v = Wv_p y          (the layer's own projections)
        k_h <- RoPE(k_h, position_t)      (per KV head)

    Shapes: x_S_rows [n, d]; positions [n]; A [P, d, d]; b [P, d]; gain [P, d];
    Wk, Wv [P, H*hd, d]. Returns K, V as [P, n, H, hd] float64.
    With ``v_scale`` [P, H] (the value rescale), V_p[:, h] is multiplied by v_scale[p, h].
    With ``k_norm_gain`` [P, hd] (key normalisation), each key head is RMS-normalised
    with that layer's gain before RoPE.
    """
    x = np.asarray(x_S_rows, np.float64)
    n = x.shape[0]
    P = A.shape[0]
    K = np.empty((P, n, n_kv_heads, head_dim))
    V = np.empty((P, n, n_kv_heads, head_dim))
    pos = np.asarray(positions, np.float64)
    for p in range(P):
        xhat = map_predict(x, A[p], b[p])
        y = rms_norm(xhat, gain[p], rms_eps)
        k = (y @ np.asarray(Wk[p], np.float64).T).reshape(n, n_kv_heads, head_dim)
        v = (y @ np.asarray(Wv[p], np.float64).T).reshape(n, n_kv_heads, head_dim)
        if k_norm_gain is not None:
            k = rms_norm(k, np.asarray(k_norm_gain, np.float64)[p], rms_eps)
        K[p] = rope(k, pos[:, None], rope_theta)
        V[p] = v if v_scale is None else v * np.asarray(v_scale, np.float64)[p][None, :, None]
    return K, V


def fill_kv(k_cache, v_cache, x_S, exact_mask, A, b, gain, Wk, Wv, *, L, S, N, T,
            n_kv_heads, head_dim, rope_theta, rms_eps, pos_offset=0, v_scale=None, k_norm_gain=None):
    """Whole-cache fill: returns (new_k_cache, new_v_cache, fill_idx).

    Caches are [L, N_cap, H, hd] arrays (float64 copies of the input caches).
    Only cache[l][t] for l in [S, L) and t in fill_idx is replaced; every other
    entry keeps its input value ([RF] Table 3: exact rows and the tail run the
    real layers, the no-fill arm writes nothing).
    """
    assert A.shape[0] == L - S
    idx = prefix_partition(N, T, exact_mask)
    kc = np.array(k_cache, dtype=np.float64, copy=True)
    vc = np.array(v_cache, dtype=np.float64, copy=True)
    if idx.size and L > S:
        K, V = fill_rows(np.asarray(x_S, np.float64)[idx], idx + pos_offset, A, b, gain,
                         Wk, Wv, n_kv_heads, head_dim, rope_theta, rms_eps, v_scale, k_norm_gain)
        for p in range(L - S):
            kc[S + p][idx] = K[p]
            vc[S + p][idx] = V[p]
    return kc, vc, idx


def value_scale(x_S_tail, x_exact_tail, A, b, gain, Wv, n_kv_heads, head_dim, rms_eps):
    """Value rescale ([RF] "Hybrid layers and two corrections", value rescale).

    In each upper layer p, each of the first c tail rows passes through the
    layer's value projection twice, with the exact input and with the map's
    prediction:
        v_pred  = Wv_p RMSNorm_g(A_p x_S[t] + b_p)
        v_exact = Wv_p RMSNorm_g(x_exact[p, t])
    and per KV head h the scale is the mean over the rows of
    ||v_exact_h|| / ||v_pred_h|| (rows with ||v_pred_h|| = 0 left out; 1 if none).

    Shapes: x_S_tail [c, d] (x_S at rows N-T .. N-T+c-1); x_exact_tail [P, c, d]
    (the exact inputs of layers S .. L-1 at those rows); A [P, d, d]; b, gain [P, d];
    Wv [P, H*hd, d]. Returns [P, H] float64.
    """
    x = np.asarray(x_S_tail, np.float64)
    c = x.shape[0]
    P = A.shape[0]
    out = np.ones((P, n_kv_heads))
    for p in range(P):
        W = np.asarray(Wv[p], np.float64)
        y_pred = rms_norm(map_predict(x, A[p], b[p]), gain[p], rms_eps)
        y_exact = rms_norm(np.asarray(x_exact_tail[p], np.float64), gain[p], rms_eps)
        n_pred = np.linalg.norm((y_pred @ W.T).reshape(c, n_kv_heads, head_dim), axis=-1)
        n_exact = np.linalg.norm((y_exact @ W.T).reshape(c, n_kv_heads, head_dim), axis=-1)
        for h in range(n_kv_heads):
            ok = n_pred[:, h] > 0
            if ok.any():
                out[p, h] = np.mean(n_exact[ok, h] / n_pred[ok, h])
    return out


def quantize_rows_int8(A):
    """Symmetric per-row int8 code of maps A [..., d_out, d_in] (see the module
    header): returns (q int8 [..., d_out, d_in], s float32 [..., d_out]). The
    scale and the rounding decisions are taken in float32."""
    a = np.asarray(A, np.float32)
    amax = np.max(np.abs(a), axis=-1)
    s = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
    q = np.rint((a / safe[..., None]).astype(np.float32))
    q = np.where(s[..., None] > 0, q, np.float32(0.0))
    return np.clip(q, -127, 127).astype(np.int8), s


def dequantize_rows_int8(q, s) -> np.ndarray:
    """A'[o][i] = s[o] q[o][i] in float64."""
    return np.asarray(s, np.float64)[..., None] * np.asarray(q, np.float64)


def fill_flops_per_row_layer(d: int, n_kv_heads: int, head_dim: int) -> int:
    """Algorithmic flops for one filled (row, layer): the map (2 d^2) plus the
    K and V projections (2 * d * 2 * H * hd). Norm, RoPE and bias are O(d)."""
    kv = n_kv_heads * head_dim
    return 2 * d * d + 2 * d * (2 * kv)


# --------------------------------------------------------------------------- #
# Calibration and the closed-form ridge solve ([RF] "Ridge map": objective,
# closed form, alpha = lambda tr(XᵀX)/d_in, one-pass statistics)
# --------------------------------------------------------------------------- #
def calib_stats(X, Ys) -> dict:
    """Raw one-pass sums over the rows of X [n, d_in] and Ys [P, n, d_out].

    G = Σ_t x_t x_tᵀ,  C_p = Σ_t x_t y_{p,t}ᵀ,  sx = Σ_t x_t,  sy_p = Σ_t y_{p,t},
    syy_p = Σ_t y_{p,t}² (per column; the total sum of squares of R²),  n.
    """
    X = np.asarray(X, np.float64)
    Ys = np.asarray(Ys, np.float64)
    return {
        "G": X.T @ X,
        "C": np.stack([X.T @ Ys[p] for p in range(Ys.shape[0])]),
        "sx": X.sum(axis=0),
        "sy": Ys.sum(axis=1),
        "syy": (Ys * Ys).sum(axis=1),
        "n": int(X.shape[0]),
    }


def add_stats(a: dict, b: dict) -> dict:
    """Sum of two sets of raw statistics (calibration is resumable by adding)."""
    return {k: a[k] + b[k] for k in ("G", "C", "sx", "sy", "syy", "n") if k in a}


def centre_stats(st: dict):
    """Centred Gram and cross terms from raw sums.

    mu_x = sx/n, mu_p = sy_p/n, Gc = G - n mu_x mu_xᵀ, Cc_p = C_p - n mu_x mu_pᵀ.
    These equal Σ (x - mu_x)(x - mu_x)ᵀ and Σ (x - mu_x)(y_p - mu_p)ᵀ.
    """
    n = float(st["n"])
    mu_x = st["sx"] / n
    mu_y = st["sy"] / n
    Gc = st["G"] - n * np.outer(mu_x, mu_x)
    Cc = st["C"] - n * np.einsum("i,pj->pij", mu_x, mu_y)
    return Gc, Cc, mu_x, mu_y


def ridge_alpha(Gc: np.ndarray, lam: float, mode: str = "trace") -> float:
    """alpha = lambda * tr(XᵀX)/d_in (centred X) in "trace" mode, else alpha = lambda."""
    if mode == "trace":
        return float(lam) * float(np.trace(Gc)) / Gc.shape[0]
    if mode == "absolute":
        return float(lam)
    raise ValueError(mode)


def ridge_solve(st: dict, lam: float, alpha_mode: str = "trace"):
    """A_p = Y_pᵀX (XᵀX + alpha I)^-1 and b_p = mu_p - A_p mu_x for every map p.

    With centred data, Y_pᵀX = Cc_pᵀ and XᵀX = Gc, so A_pᵀ solves
    (Gc + alpha I) A_pᵀ = Cc_p. Returns A [P, d_out, d_in], b [P, d_out], alpha.
    """
    Gc, Cc, mu_x, mu_y = centre_stats(st)
    alpha = ridge_alpha(Gc, lam, alpha_mode)
    H = Gc + alpha * np.eye(Gc.shape[0])
    P = Cc.shape[0]
    A = np.empty((P, Cc.shape[2], Cc.shape[1]))
    b = np.empty((P, Cc.shape[2]))
    for p in range(P):
        A[p] = np.linalg.solve(H, Cc[p]).T
        b[p] = mu_y[p] - A[p] @ mu_x
    return A, b, alpha


# --------------------------------------------------------------------------- #
# Cross-model mapper ([XM] content-space mapping K̂_t = (K_s R_s^-1(t) W_K + b_K) R_t(t);
# V is mapped without RoPE; source layers of a target layer are concatenated)
# --------------------------------------------------------------------------- #
def xmodel_features(src_cache, src_layers, positions, theta_src=None):
    """Concatenated features of the selected source layers for each row.

    ``src_cache`` is [L_src, n, H, hd]. With ``theta_src`` given (keys), each
    selected layer is un-roped at the row's position first; with None (values)
    the cache is used as is. Feature order: selected layer j, then head h, then
    dim c. Returns [n, k*H*hd].
    """
    parts = []
    for s in src_layers:
        blk = np.asarray(src_cache[s], np.float64)
        if theta_src is not None:
            blk = rope(blk, np.asarray(positions, np.float64)[:, None], theta_src, inverse=True)
        parts.append(blk.reshape(blk.shape[0], -1))
    return np.concatenate(parts, axis=1)


def xmodel_map_layer(k_src, v_src, src_layers, Wk, bk, Wv, bv, positions,
                     theta_src, theta_tgt, n_kv_heads, head_dim):
    """One target layer of the cross-model mapper.

    K̂ = RoPE_tgt(F_K Wkᵀ + bk) with F_K the un-roped source keys; V̂ = F_V Wvᵀ + bv.
    Wk, Wv are [H*hd, k*H*hd] (output x input). Returns K̂, V̂ as [n, H, hd].
    """
    FK = xmodel_features(k_src, src_layers, positions, theta_src)
    FV = xmodel_features(v_src, src_layers, positions, None)
    n = FK.shape[0]
    kc = (FK @ np.asarray(Wk, np.float64).T + np.asarray(bk, np.float64)).reshape(n, n_kv_heads, head_dim)
    vh = (FV @ np.asarray(Wv, np.float64).T + np.asarray(bv, np.float64)).reshape(n, n_kv_heads, head_dim)
    kh = rope(kc, np.asarray(positions, np.float64)[:, None], theta_tgt)
    return kh, vh


# --------------------------------------------------------------------------- #
# Cross-layer source selection ([XM] "소스 층은 몇 개가 필요한가": greedy forward
# selection that adds, one at a time, the source layer raising the head-mean R²
# most; "층 교차 소스 선택": the k layers are chosen per target layer by the
# head-mean R² of the un-roped keys and of the values, and all heads of a target
# layer share them; "헤드별 리지 회귀": the fit is the ridge regression of the
# centred target on the concatenated features of the chosen layers)
# --------------------------------------------------------------------------- #
def _selection_system(st: dict, lam: float, alpha_mode: str):
    """Centred Gram, cross terms and per-column total sums of squares of one kind.

    TSS_p[o] = Σ_t (y_{p,t,o} - mu_p[o])² = syy_p[o] - n mu_p[o]²; alpha is taken
    once from the Gram of ALL source features (reading: every candidate set of the
    selection is scored under the same penalty).
    """
    Gc, Cc, _, mu_y = centre_stats(st)
    tss = st["syy"] - float(st["n"]) * mu_y * mu_y
    return Gc, Cc, tss, ridge_alpha(Gc, lam, alpha_mode)


def _head_mean_r2(explained: np.ndarray, tss: np.ndarray, head_dim: int) -> float:
    """Mean over heads of R²_h = Σ_{o in h} explained[o] / Σ_{o in h} TSS[o].

    A head is its head_dim columns: its R² is the share of its total centred
    variance that the fit explains. A head with zero variance counts as R²_h = 0.
    """
    e = explained.reshape(-1, head_dim).sum(axis=1)
    t = tss.reshape(-1, head_dim).sum(axis=1)
    r = np.where(t > 0, e / np.where(t > 0, t, 1.0), 0.0)
    return float(r.mean())


def selection_scores(stats, layers, F: int, head_dim: int, lam: float, alpha_mode: str = "trace"):
    """Head-mean R² of every target map fitted on the features of ``layers``.

    ``stats`` is one statistics dict per kind (keys, values), each with d_in = L_src*F
    and n_maps target layers. For each kind and map p the fit is the ridge
    regression on the columns of the chosen layers (in the listed order); with
    H = Gc_SS + alpha I and c_o the cross terms of output column o, the explained
    energy is c_oᵀ H⁻¹ c_o, so R² = 1 - (RSS + alpha |w|²) / TSS (the least-squares
    R² when alpha = 0). Returns [n_kinds, n_maps].
    """
    idx = np.concatenate([np.arange(s * F, (s + 1) * F) for s in layers])
    out = []
    for st in stats:
        Gc, Cc, tss, alpha = _selection_system(st, lam, alpha_mode)
        H = Gc[np.ix_(idx, idx)] + alpha * np.eye(idx.size)
        row = []
        for p in range(Cc.shape[0]):
            c = Cc[p][idx, :]
            explained = (c * np.linalg.solve(H, c)).sum(axis=0)
            row.append(_head_mean_r2(explained, tss[p], head_dim))
        out.append(row)
    return np.asarray(out)


def select_sources(stats, L_src: int, F: int, head_dim: int, k: int, lam: float,
                   alpha_mode: str = "trace", path=None):
    """Greedy forward selection of k source layers for every target layer.

    Step j scores every layer s not yet chosen by the head-mean R² of the fit on
    the chosen layers plus s (``selection_scores``), for each kind; the joint score
    is the mean over kinds, and the layer with the highest joint score is added
    (the lowest index among equal scores). ``path`` [n_maps, k] replays given
    choices instead, and the scores are then those along that path.

    Returns (sel [n_maps, k] int, table [n_kinds, n_maps, k, L_src]) where table
    holds each candidate's score at each step and NaN for layers already chosen.
    """
    systems = [_selection_system(st, lam, alpha_mode) for st in stats]
    n_maps = systems[0][1].shape[0]
    sel = np.zeros((n_maps, k), np.int64)
    table = np.full((len(stats), n_maps, k, L_src), np.nan)
    for p in range(n_maps):
        chosen = []
        for j in range(k):
            for s in range(L_src):
                if s in chosen:
                    continue
                idx = np.concatenate([np.arange(c * F, (c + 1) * F) for c in chosen + [s]])
                for kind, (Gc, Cc, tss, alpha) in enumerate(systems):
                    H = Gc[np.ix_(idx, idx)] + alpha * np.eye(idx.size)
                    c = Cc[p][idx, :]
                    explained = (c * np.linalg.solve(H, c)).sum(axis=0)
                    table[kind, p, j, s] = _head_mean_r2(explained, tss[p], head_dim)
            joint = table[:, p, j, :].mean(axis=0)      # NaN for layers already chosen
            if path is None:
                b = int(np.nanargmax(joint))
            else:
                b = int(path[p][j])
            chosen.append(b)
            sel[p, j] = b
    return sel, table
