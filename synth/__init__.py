"""Seeded synthetic inputs shaped like the pages' deployments.

This module holds workload shapes and random-number recipes only; it contains
none of the method's arithmetic (no map, norm, projection, RoPE or solve). Both
the fp64 oracle and the CUDA library receive the bf16 tensors made here, so the
two sides see identical bit patterns.

Recipe (one per workload):
  * x_S ~ N(0, 1); maps A = I + N(0, 0.02^2/d) and offsets b ~ N(0, 0.1^2), one
    per upper layer; RMSNorm gains 1 + 0.1 N(0, 1); W_k, W_v ~ N(0, 1/d); all cast
    to bf16 (b stays fp32).
  * calibration rows: x ~ N(0, 1), y_l = A_true,l x + b_true,l + 0.05 N(0, 1).
  * exact-row masks: the toy's rows {4, 5, 6, 7}; "uniform 10%": exactly
    round(0.10 (N - T)) rows by a seeded permutation; "blocks of 16, 5%":
    round(0.05 (N - T)/16) aligned 16-row blocks chosen without replacement.
  * cross-model: source K, V ~ N(0, 1), W ~ N(0, 1/(k H hd)), b ~ N(0, 0.1^2);
    target layer j reads the k consecutive source layers starting at
    clamp(round(j (L_src - 1)/(L_tgt - 1)) - k/2 + 1, 0, L_src - k).
  * source selection: a latent random walk over source depth, r_0 ~ N(0, I_R),
    r_s = r_{s-1} + 0.5 N(0, I_R); source layer s's features (un-roped keys, or
    values) are r_s P_s + 0.3 N(0, 1) + mu_x with P_s ~ N(0, 1/R); target layer t
    at depth a = floor(t (L_src - 1)/(L_tgt - 1)) is r_a M_1 + 0.6 r_{a+1} M_2 +
    0.3 r_c M_3 + 0.3 N(0, 1) + mu_y (c = a + L_src/2 mod L_src, M ~ N(0, 1/R)),
    so nearby layers carry most of a target and far ones a little; keys and values
    share the walk and draw their own loadings. Raw rows are drawn from this
    model; the full-size case uses its exact population sums instead.
  * mapper fit (6 -> 3 layers): source K, V ~ N(0, 1); each target layer's K (V)
    is a sum over k planted source layers (disjoint sets from a seeded
    permutation) of the source cache rows times w_j M, M ~ N(0, 1/KV), w_j from 1
    to 0.6, plus 0.1 N(0, 1).
Seeds: base = 20261202 + workload index; one sub-seed per named tensor.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

BASE_SEED = 20261202


@dataclasses.dataclass(frozen=True)
class FillConfig:
    name: str
    index: int
    d: int
    L: int
    S: int
    N: int
    T: int
    H: int
    hd: int
    rope_theta: float
    exact: object            # tuple of rows, "uniform10", "blocks16_5", or None
    lam: float
    calib_n: int
    rms_eps: float = 1e-5
    pos_offset: int = 0
    d_in: int = 0            # width of x_S and of the maps' input; 0 = d (square maps)

    @property
    def D_in(self) -> int:
        return self.d_in if self.d_in > 0 else self.d

    @property
    def P(self) -> int:
        return self.L - self.S

    @property
    def KV(self) -> int:
        return self.H * self.hd

    def with_layers(self, n_upper: int) -> "FillConfig":
        """Same shapes with only the top ``n_upper`` layers filled (S = L - n_upper)."""
        return dataclasses.replace(self, S=self.L - n_upper)

    def with_rows(self, N: int, T: int) -> "FillConfig":
        return dataclasses.replace(self, N=N, T=T)


@dataclasses.dataclass(frozen=True)
class XModelConfig:
    name: str
    index: int
    L_src: int
    L_tgt: int
    k: int
    H: int
    hd: int
    N: int
    theta_src: float
    theta_tgt: float
    calib_n: int
    lam: float
    pos_offset: int = 0

    @property
    def KV(self) -> int:
        return self.H * self.hd

    @property
    def d_in(self) -> int:
        return self.k * self.H * self.hd


TOY = FillConfig("toy-8layer d256", 0, d=256, L=8, S=4, N=12, T=3, H=2, hd=64,
                 rope_theta=5.0e5, exact=(4, 5, 6, 7), lam=0.03, calib_n=2048)
LLAMA8B = FillConfig("llama3.1-8b-shaped d4096 L32 S12 N16384 T4096", 1, d=4096, L=32, S=12,
                     N=16384, T=4096, H=8, hd=128, rope_theta=5.0e5, exact="uniform10",
                     lam=0.03, calib_n=8192)
QWEN3_8B = FillConfig("qwen3-8b-shaped d4096 L36 S13 N32768 T4096", 2, d=4096, L=36, S=13,
                      N=32768, T=4096, H=8, hd=128, rope_theta=1.0e6, exact=None,
                      lam=0.01, calib_n=8192)
DENSE27B = FillConfig("27b-shaped d5120 L64 S16 N32768 T4096", 3, d=5120, L=64, S=16,
                      N=32768, T=4096, H=8, hd=128, rope_theta=1.0e6, exact="blocks16_5",
                      lam=0.03, calib_n=16384)
XMODEL = XModelConfig("xmodel 40->64 layers 8x128 k8 N32768", 4, L_src=40, L_tgt=64, k=8,
                      H=8, hd=128, N=32768, theta_src=1.0e6, theta_tgt=1.0e6,
                      calib_n=131072, lam=0.01)

# Non-square maps shaped like the pages' Flash-Next deployment ([RF] "Ridge map":
# four parallel residual streams of width 2,560 read through gates, so each map is
# 10,240 -> 2,560; split 24/48, tail 2,048, "Two numbers set the skip range"). The
# pages give neither its KV heads nor an exact-row rate: 2 x 128 heads, none exact.
FLASH_NEXT = FillConfig("flash-next-shaped maps d_in10240 d2560 L48 S24 N32768 T2048", 5, d=2560, L=48, S=24,
                        N=32768, T=2048, H=2, hd=128, rope_theta=1.0e6, exact=None, lam=0.03, calib_n=0,
                        d_in=10240)


@dataclasses.dataclass(frozen=True)
class SelectConfig:
    """Greedy source-layer selection: L_src candidate layers of H x hd features,
    L_tgt target layers of H x hd columns, k layers chosen per target."""
    name: str
    index: int
    L_src: int
    L_tgt: int
    k: int
    H: int
    hd: int
    n: int                   # calibration rows
    R: int                   # latent width of the random walk
    lam: float
    sigma: float = 0.3

    @property
    def F(self) -> int:
        return self.H * self.hd

    @property
    def D(self) -> int:
        return self.L_src * self.F


# Small case the oracle finishes in seconds; the pages' 40 -> 64 layer pair with
# k = 8, 8 x 128 heads and ~128K calibration rows ([XM] calibration setup).
SELECT_SMALL = SelectConfig("selection 6->4 layers 2x128 k3", 6, L_src=6, L_tgt=4, k=3, H=2, hd=128,
                            n=4096, R=32, lam=0.01)
SELECT_XMODEL = SelectConfig("selection 40->64 layers 8x128 k8 n131072", 7, L_src=40, L_tgt=64, k=8, H=8,
                             hd=128, n=131072, R=64, lam=0.01)
FILL_CONFIGS = {"toy": TOY, "llama8b": LLAMA8B, "qwen3_8b": QWEN3_8B, "dense27b": DENSE27B,
                "flash_next": FLASH_NEXT}

_TENSOR_IDS = {name: i for i, name in enumerate(
    ["x_S", "mask", "A", "b", "gain", "Wk", "Wv", "calib_X", "calib_Atrue", "calib_btrue",
     "calib_noise", "k_src", "v_src", "xWk", "xWv", "xbk", "xbv", "cache", "extra",
     "rescale_scale", "rescale_noise", "key_norm_gain", "sel_P", "sel_M", "sel_mu", "sel_latent",
     "sel_noise", "fit_perm", "fit_Mk", "fit_Mv", "fit_noise"])}


def sub_seed(index: int, tensor: str, salt: int = 0) -> int:
    return (BASE_SEED + index) * 1009 + _TENSOR_IDS[tensor] * 101 + salt


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, seed, device, std=1.0, mean=0.0, dtype=torch.bfloat16, chunk_rows=None):
    """N(mean, std^2) in float32, then cast to ``dtype``; generated in slabs along
    dim 0 so that large tensors never need a full float32 copy."""
    shape = tuple(int(s) for s in shape)
    out = torch.empty(shape, dtype=dtype, device=device)
    g = _gen(device, seed)
    if len(shape) == 0 or shape[0] == 0:
        return out
    per = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    step = chunk_rows or max(1, (1 << 26) // max(per, 1))
    for i in range(0, shape[0], step):
        j = min(shape[0], i + step)
        t = torch.randn((j - i,) + shape[1:], generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        if mean != 0.0:
            t.add_(mean)
        out[i:j] = t.to(dtype)
    return out


def exact_mask(cfg: FillConfig, device="cpu", seed: Optional[int] = None) -> Optional[torch.Tensor]:
    """uint8 [N - T] mask, 1 = exact prefix row (never filled); None = no exact rows."""
    n_prefix = cfg.N - cfg.T
    if cfg.exact is None:
        return None
    m = torch.zeros(n_prefix, dtype=torch.uint8)
    seed = sub_seed(cfg.index, "mask") if seed is None else seed
    g = _gen("cpu", seed)
    if isinstance(cfg.exact, (tuple, list)):
        rows = [r for r in cfg.exact if r < n_prefix]
        m[list(rows)] = 1
    elif cfg.exact == "uniform10":
        k = int(round(0.10 * n_prefix))
        m[torch.randperm(n_prefix, generator=g)[:k]] = 1
    elif cfg.exact == "blocks16_5":
        nb = n_prefix // 16
        k = int(round(0.05 * nb))
        for blk in torch.randperm(nb, generator=g)[:k].tolist():
            m[blk * 16:(blk + 1) * 16] = 1
    else:
        raise ValueError(cfg.exact)
    return m.to(device)


def fill_inputs(cfg: FillConfig, device="cpu", with_mask=True) -> dict:
    """Inputs of one fill: x_S [N, d_in], mask [N-T] (or None), maps A [P, d, d_in],
    offsets b [P, d] (fp32), gains [P, d], W_k and W_v [P, H*hd, d]."""
    P, d, KV, di = cfg.P, cfg.d, cfg.KV, cfg.D_in
    ix = cfg.index
    A = _randn((P, d, di), sub_seed(ix, "A"), device, std=0.02 / math.sqrt(di))
    # Square maps are I + noise. A wider input (di = s * d, s parallel streams of
    # width d) maps to the mean of the streams + noise: [I ... I] / s.
    eye = torch.eye(d, dtype=torch.float32, device=device)
    streams = di // d if di % d == 0 else 0
    for p in range(P):
        if streams:
            A[p] = (A[p].float() + eye.repeat(1, streams) / streams).to(torch.bfloat16)
        elif di == d:
            A[p] = (A[p].float() + eye).to(torch.bfloat16)
    return {
        "x_S": _randn((cfg.N, di), sub_seed(ix, "x_S"), device),
        "mask": exact_mask(cfg, device) if with_mask else None,
        "A": A,
        "b": _randn((P, d), sub_seed(ix, "b"), device, std=0.1, dtype=torch.float32),
        "gain": _randn((P, d), sub_seed(ix, "gain"), device, std=0.1, mean=1.0),
        "Wk": _randn((P, KV, d), sub_seed(ix, "Wk"), device, std=1.0 / math.sqrt(d)),
        "Wv": _randn((P, KV, d), sub_seed(ix, "Wv"), device, std=1.0 / math.sqrt(d)),
    }


def key_norm_gain(cfg: FillConfig, device="cpu") -> torch.Tensor:
    """Per-layer key-normalisation gains [P, hd] (bf16), 1 + 0.1 * N(0, 1)."""
    return _randn((cfg.P, cfg.hd), sub_seed(cfg.index, "key_norm_gain"), device, std=0.1, mean=1.0)


def rescale_inputs(cfg: FillConfig, x_S: torch.Tensor, c: int, device="cpu") -> torch.Tensor:
    """Exact inputs of the upper layers at the first c tail rows, x_exact [P, c, d]
    (bf16): per layer, the tail's residual stream with the first d/2 channels
    scaled by about 0.5 and the others by about 1.5 (each factor times U[0.9, 1.1]),
    plus 0.1 * N(0, 1). With value weights that read both halves alike the norm
    ratio stays near 1 (the layer norm removes the overall magnitude); weights
    that favour one half move it well away from 1."""
    P, d = cfg.P, cfg.d
    g = _gen(device, sub_seed(cfg.index, "rescale_scale"))
    half = torch.cat([torch.full((d // 2,), 0.5), torch.full((d - d // 2,), 1.5)]).to(device)
    s = half.view(1, 1, d) * (0.9 + 0.2 * torch.rand((P, 1, d), generator=g, device=device, dtype=torch.float32))
    tail = x_S[cfg.N - cfg.T: cfg.N - cfg.T + c, :d].to(device).float()   # first d channels if d_in > d
    noise = _randn((P, c, d), sub_seed(cfg.index, "rescale_noise"), device, std=0.1, dtype=torch.float32)
    return (s * tail[None] + noise).to(torch.bfloat16)


def calib_inputs(d_in: int, d_out: int, n_maps: int, n_rows: int, index: int, device="cpu",
                 noise: float = 0.05, salt: int = 0) -> dict:
    """Planted calibration rows: X [n, d_in] ~ N(0,1); Y [P, n, d_out] with
    y_p = A_true,p x + b_true,p + noise * N(0,1), everything rounded to bf16."""
    X = _randn((n_rows, d_in), sub_seed(index, "calib_X", salt), device)
    At = _randn((n_maps, d_out, d_in), sub_seed(index, "calib_Atrue", salt), device,
                std=0.02 / math.sqrt(d_in), dtype=torch.float32)
    for p in range(n_maps):
        if d_out == d_in:
            At[p].diagonal().add_(1.0)
    bt = _randn((n_maps, d_out), sub_seed(index, "calib_btrue", salt), device, std=0.1,
                dtype=torch.float32)
    Y = torch.empty((n_maps, n_rows, d_out), dtype=torch.bfloat16, device=device)
    gn = _gen(device, sub_seed(index, "calib_noise", salt))
    Xf = X.float()
    for p in range(n_maps):
        e = torch.randn((n_rows, d_out), generator=gn, device=device, dtype=torch.float32)
        Y[p] = (Xf @ At[p].T + bt[p] + noise * e).to(torch.bfloat16)
    return {"X": X, "Y": Y, "A_true": At, "b_true": bt}


def source_table(L_src: int, L_tgt: int, k: int) -> np.ndarray:
    """int32 [L_tgt, k]: the k consecutive source layers each target layer reads."""
    tab = np.empty((L_tgt, k), dtype=np.int32)
    for j in range(L_tgt):
        c = int(round(j * (L_src - 1) / max(L_tgt - 1, 1)))
        s0 = min(max(c - k // 2 + 1, 0), L_src - k)
        tab[j] = np.arange(s0, s0 + k, dtype=np.int32)
    return tab


def xmodel_inputs(cfg: XModelConfig, device="cpu", L_tgt: Optional[int] = None,
                  N: Optional[int] = None) -> dict:
    """Source caches [L_src, N, H, hd], mapper weights [L_tgt, KV, k*KV], biases."""
    L_t = cfg.L_tgt if L_tgt is None else L_tgt
    n = cfg.N if N is None else N
    KV, din, ix = cfg.KV, cfg.d_in, cfg.index
    return {
        "k_src": _randn((cfg.L_src, n, cfg.H, cfg.hd), sub_seed(ix, "k_src"), device),
        "v_src": _randn((cfg.L_src, n, cfg.H, cfg.hd), sub_seed(ix, "v_src"), device),
        "Wk": _randn((L_t, KV, din), sub_seed(ix, "xWk"), device, std=1.0 / math.sqrt(din)),
        "Wv": _randn((L_t, KV, din), sub_seed(ix, "xWv"), device, std=1.0 / math.sqrt(din)),
        "bk": _randn((L_t, KV), sub_seed(ix, "xbk"), device, std=0.1, dtype=torch.float32),
        "bv": _randn((L_t, KV), sub_seed(ix, "xbv"), device, std=0.1, dtype=torch.float32),
        "src": source_table(cfg.L_src, cfg.L_tgt, cfg.k)[:L_t].copy(),
    }


# A model pair for an end-to-end mapper fit: 6 source and 3 target layers of 2 x 128
# heads, k = 2, 4,096 rows, different RoPE bases on the two sides.
MAPPER_FIT = XModelConfig("mapper fit 6->3 layers 2x128 k2 N4096", 8, L_src=6, L_tgt=3, k=2, H=2, hd=128, N=4096,
                          theta_src=1.0e6, theta_tgt=5.0e5, calib_n=4096, lam=0.01)


def mapper_fit_caches(cfg: XModelConfig, device="cpu") -> dict:
    """Source and target caches [L, N, H, hd] bf16 for a mapper fit with planted
    sources: source K, V ~ N(0, 1); target layer t's K (V) is the sum over its
    planted source layers j = 0..k-1 of the source cache rows times w_j M_{t,j},
    M ~ N(0, 1/KV) and w_j falling from 1 to 0.6 (so every greedy step has a clear
    best layer), plus 0.1 N(0, 1). The planted sets (disjoint, k layers each, in
    order of weight, from a seeded permutation of the source layers; needs
    L_tgt k <= L_src) are returned too."""
    L, T, k, KV, ix = cfg.L_src, cfg.L_tgt, cfg.k, cfg.KV, cfg.index
    assert T * k <= L
    g = _gen("cpu", sub_seed(ix, "fit_perm"))
    perm = torch.randperm(L, generator=g).numpy()
    plant = perm[:T * k].reshape(T, k).astype(np.int32)
    ks = _randn((L, cfg.N, cfg.H, cfg.hd), sub_seed(ix, "k_src"), device)
    vs = _randn((L, cfg.N, cfg.H, cfg.hd), sub_seed(ix, "v_src"), device)
    out = {"k_src": ks, "v_src": vs, "plant": plant}
    for name, src, mix in (("k_tgt", ks, "fit_Mk"), ("v_tgt", vs, "fit_Mv")):
        M = _randn((T, k, KV, KV), sub_seed(ix, mix), device, std=1.0 / math.sqrt(KV), dtype=torch.float32)
        tgt = _randn((T, cfg.N, KV), sub_seed(ix, "fit_noise", 0 if name == "k_tgt" else 1), device, std=0.1,
                     dtype=torch.float32)
        for t in range(T):
            for j in range(k):
                w = 1.0 - 0.4 * j / max(k - 1, 1)
                tgt[t] += src[int(plant[t, j])].reshape(cfg.N, KV).float() @ (w * M[t, j])
        out[name] = tgt.to(torch.bfloat16).reshape(T, cfg.N, cfg.H, cfg.hd)
    return out


def canary_cache(L: int, N_cap: int, H: int, hd: int, kind: int, device="cpu") -> torch.Tensor:
    """bf16 cache filled with NaN canaries whose payload encodes (kind, l, t, h, c)
    modulo the 6 free mantissa bits, so any stray write is visible bit for bit."""
    out = torch.empty((L, N_cap, H, hd), dtype=torch.int16, device=device)
    t = torch.arange(N_cap, dtype=torch.int32, device=device).view(N_cap, 1, 1)
    h = torch.arange(H, dtype=torch.int32, device=device).view(1, H, 1)
    c = torch.arange(hd, dtype=torch.int32, device=device).view(1, 1, hd)
    for l in range(L):
        payload = (kind * 31 + l * 7 + t * 13 + h * 5 + c) % 63 + 1     # 1..63, never 0
        out[l] = (0x7F80 | payload).to(torch.int16)                     # NaN bit patterns
    return out.view(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    """Host numpy uint16 view of a bf16 tensor's bit patterns (no arithmetic)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().numpy()


# --------------------------------------------------------------------------- #
# Source selection inputs (latent random-walk model; see the recipe above)
# --------------------------------------------------------------------------- #
def _walk_scale(l: int) -> float:
    return 1.0 if l == 0 else 0.5


def selection_loadings(cfg: SelectConfig, kind: int, device="cpu") -> dict:
    """Loadings of the model on the independent standard walk steps e_0..e_{L_src-1}
    (r_s = sum_{l <= s} c_l e_l): Z [L_src R, D] for the source features and
    W [L_tgt, L_src R, F] for the targets, plus the means (float32)."""
    L, R, F = cfg.L_src, cfg.R, cfg.F
    P = _randn((L, R, F), sub_seed(cfg.index, "sel_P", kind), device, std=1 / math.sqrt(R), dtype=torch.float32)
    M = _randn((cfg.L_tgt, 3, R, F), sub_seed(cfg.index, "sel_M", kind), device, std=1 / math.sqrt(R),
               dtype=torch.float32)
    Z = torch.zeros((L * R, L * F), dtype=torch.float32, device=device)
    for s in range(L):
        for l in range(s + 1):
            Z[l * R:(l + 1) * R, s * F:(s + 1) * F] = _walk_scale(l) * P[s]
    W = torch.zeros((cfg.L_tgt, L * R, F), dtype=torch.float32, device=device)
    for t in range(cfg.L_tgt):
        a = (t * (L - 1)) // max(cfg.L_tgt - 1, 1)
        for depth, m, wgt in ((a, 0, 1.0), (min(a + 1, L - 1), 1, 0.6), ((a + L // 2) % L, 2, 0.3)):
            for l in range(depth + 1):
                W[t, l * R:(l + 1) * R] += (wgt * _walk_scale(l)) * M[t, m]
    mu = _randn((L * F + cfg.L_tgt * F,), sub_seed(cfg.index, "sel_mu", kind), device, std=0.1,
                dtype=torch.float32)
    return {"Z": Z, "W": W, "mu_x": mu[:L * F], "mu_y": mu[L * F:].view(cfg.L_tgt, F)}


def selection_rows(cfg: SelectConfig, kind: int, rows: int, chunk: int = 0, device="cpu",
                   loadings: Optional[dict] = None) -> dict:
    """One chunk of calibration rows: X [rows, D] bf16 (all source layers side by
    side) and Y [L_tgt, rows, F] bf16. The walk steps depend on the chunk only, so
    keys (kind 0) and values (kind 1) of a chunk come from the same walk."""
    ld = selection_loadings(cfg, kind, device) if loadings is None else loadings
    e = _randn((rows, cfg.L_src * cfg.R), sub_seed(cfg.index, "sel_latent", chunk), device, dtype=torch.float32)
    X = e @ ld["Z"]
    X += _randn((rows, cfg.D), sub_seed(cfg.index, "sel_noise", 2 * chunk + 64 * kind), device,
                std=cfg.sigma, dtype=torch.float32)
    X += ld["mu_x"]
    Y = torch.empty((cfg.L_tgt, rows, cfg.F), dtype=torch.bfloat16, device=device)
    noise = _randn((cfg.L_tgt, rows, cfg.F), sub_seed(cfg.index, "sel_noise", 2 * chunk + 1 + 64 * kind), device,
                   std=cfg.sigma, dtype=torch.float32)
    for t in range(cfg.L_tgt):
        Y[t] = (e @ ld["W"][t] + noise[t] + ld["mu_y"][t]).to(torch.bfloat16)
    return {"X": X.to(torch.bfloat16), "Y": Y}


def selection_population_stats(cfg: SelectConfig, kind: int, device="cpu", loadings: Optional[dict] = None) -> dict:
    """The model's exact sums over cfg.n rows, as float64 tensors:
    G = n (ZᵀZ + sigma² I + mu_x mu_xᵀ), C_t = n (Zᵀ W_t + mu_x mu_tᵀ), sx = n mu_x,
    sy_t = n mu_t, syy_t = n (diag(W_tᵀW_t) + sigma² + mu_t²). Products in float32."""
    ld = selection_loadings(cfg, kind, device) if loadings is None else loadings
    n = float(cfg.n)
    Z, W, mx, my = ld["Z"], ld["W"], ld["mu_x"], ld["mu_y"]
    G = (Z.T @ Z).to(torch.float64)
    G.diagonal().add_(cfg.sigma ** 2)
    G += torch.outer(mx.double(), mx.double())
    G *= n
    C = torch.empty((cfg.L_tgt, cfg.D, cfg.F), dtype=torch.float64, device=device)
    for t in range(cfg.L_tgt):
        C[t] = (Z.T @ W[t]).double() + torch.outer(mx.double(), my[t].double())
    C *= n
    syy = ((W * W).sum(dim=1).double() + cfg.sigma ** 2 + my.double() ** 2) * n
    return {"G": G, "C": C, "sx": mx.double() * n, "sy": my.double() * n, "syy": syy,
            "n": torch.tensor([cfg.n], dtype=torch.int64, device=device)}
