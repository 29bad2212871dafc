"""GPU parity of the value rescale (rf_value_scale) and of the fill with a value
scale (rf_fill_desc.v_scale) against the fp64 oracle.

Value rescale: RidgeFill review, "Hybrid layers and two corrections". Scales are
compared per (layer, KV head) within 2e-3 relative: each norm carries the bf16
roundings of the fill path (x̂, the folded W_v), which mostly cancel in the ratio
of the exact to the predicted norm and average over the c rows. The fill with a
scale is checked with the same per-head tolerance as the fill itself, the oracle
taking the same scale values; K must be bit-identical to the unscaled fill.
"""
import numpy as np
import pytest
import torch

import oracle as O
import ridge_map_kv_gb300 as rf
import synth
from fillcheck import assert_bookkeeping, assert_values, desc_of, fold, run_fill

pytestmark = pytest.mark.gpu
DEV = "cuda"
KERNELS = pytest.mark.parametrize("flags", [rf.RF_FLAG_SINGLE_CTA, rf.RF_FLAG_CTA_PAIR], ids=["single-cta", "cta-pair"])


def _small(name, **kw):
    base = dict(name=name, index=95, d=512, L=5, S=2, N=400, T=300, H=2, hd=128, rope_theta=5e5,
                exact="uniform10", lam=0.03, calib_n=0)
    base.update(kw)
    return synth.FillConfig(**base)


def _f64(t):
    return O.bf16_bits_to_f64(synth.bits(t))


def _gpu_scale(cfg, inp, x_exact, c, flags=0, prefolded=False):
    """rf_value_scale with the gain folded in the call, or (``prefolded``) with the V
    projection folded beforehand by rf_fold_kv_weights."""
    desc = desc_of(cfg, flags | (rf.RF_WEIGHTS_PREFOLDED if prefolded else 0))
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    gain, Wv = (None, fold(desc, g)[1]) if prefolded else (g["gain"], g["Wv"])
    vs = torch.full((cfg.P, cfg.H), float("nan"), dtype=torch.float32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    wsb = rf.rf_value_scale_workspace_bytes(desc, c)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    rf.rf_value_scale(desc, c, g["x_S"], cfg.D_in, x_exact.to(DEV), cfg.d, g["A"], g["b"], gain, Wv, vs, status, ws,
                      wsb)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return vs


def _oracle_scale(cfg, inp, x_exact, c, layers):
    t0 = cfg.N - cfg.T
    lt = torch.as_tensor(list(layers), device=inp["A"].device)
    return O.value_scale(_f64(inp["x_S"][t0:t0 + c]), _f64(x_exact[lt.to(x_exact.device)]),
                         _f64(inp["A"].index_select(0, lt)), synth.f32(inp["b"].index_select(0, lt)).astype(np.float64),
                         _f64(inp["gain"].index_select(0, lt)), _f64(inp["Wv"].index_select(0, lt)),
                         cfg.H, cfg.hd, cfg.rms_eps)


def _favour_first_half(inp, cfg):
    """Value weights that read mostly the first d/2 channels (the rest x 0.1)."""
    Wv = inp["Wv"].float()
    Wv[:, :, cfg.d // 2:] *= 0.1
    inp["Wv"] = Wv.to(torch.bfloat16)
    return inp


def _assert_scales(got, ref):
    rel = np.abs(got - ref) / np.abs(ref)
    assert np.all(np.isfinite(got)) and rel.max() <= 2e-3, (rel.max(), got, ref)


@pytest.mark.parametrize("cfg,c", [
    (_small("hd128 2 heads, c = 64"), 64),
    (_small("hd128 2 heads, c = T (300 rows, 2 M-tiles)"), 300),
    (_small("hd64 2 heads (KV = 128), c = 1", hd=64), 1),
    (_small("hd64 4 heads, 4 layers, c = 37", d=768, L=6, S=2, H=4, hd=64, T=37), 37),
    (_small("non-square maps d_in 1024 -> d 512, c = 100", d_in=1024), 100),
], ids=lambda x: x.name if hasattr(x, "name") else str(x))
@KERNELS
def test_value_scale_matches_oracle(cfg, c, flags):
    inp = _favour_first_half(synth.fill_inputs(cfg), cfg)
    x_exact = synth.rescale_inputs(cfg, inp["x_S"], c)
    vs = _gpu_scale(cfg, inp, x_exact, c, flags).cpu().numpy().astype(np.float64)
    ref = _oracle_scale(cfg, inp, x_exact, c, range(cfg.P))
    assert np.abs(ref - 1.0).max() > 0.05          # the inputs move the scale away from 1
    _assert_scales(vs, ref)
    # the V projection folded beforehand gives the same scales, bit for bit
    pre = _gpu_scale(cfg, inp, x_exact, c, flags, prefolded=True).cpu().numpy().astype(np.float64)
    np.testing.assert_array_equal(pre, vs)


def test_value_scale_is_near_one_when_the_exact_rows_are_the_predictions():
    """x_exact = the oracle's x̂ (rounded to bf16): the two value norms differ only
    by roundings, so every scale is 1 within the tolerance."""
    cfg = _small("self")
    c = 48
    inp = synth.fill_inputs(cfg)
    t0 = cfg.N - cfg.T
    x = _f64(inp["x_S"][t0:t0 + c])
    xh = np.stack([O.map_predict(x, _f64(inp["A"][p]), synth.f32(inp["b"][p]).astype(np.float64))
                   for p in range(cfg.P)])
    x_exact = torch.as_tensor(xh, dtype=torch.float32).to(torch.bfloat16)
    vs = _gpu_scale(cfg, inp, x_exact, c).cpu().numpy()
    assert np.abs(vs - 1.0).max() <= 2e-3


@KERNELS
def test_fill_with_value_scale_matches_oracle(flags):
    cfg = _small("fill with scale", T=37, d=512, L=5, S=2, N=400)
    inp = synth.fill_inputs(cfg)
    vs = torch.tensor([[1.25, 0.5], [0.8, 2.0], [1.1, 0.9]], dtype=torch.float32, device=DEV)
    res = run_fill(cfg, inp, flags=flags, v_scale=vs)
    base = run_fill(cfg, inp, flags=flags)
    assert res["status"] == 0 and base["status"] == 0
    mnp = inp["mask"].cpu().numpy()
    idx = O.prefix_partition(cfg.N, cfg.T, mnp)
    assert_bookkeeping(cfg, res, mnp)
    assert torch.equal(res["kc"].view(torch.int16), base["kc"].view(torch.int16))   # K untouched
    assert_values(cfg, inp, res, idx, v_scale=vs.cpu().numpy())


@pytest.mark.slow
def test_value_scale_27b_shape_sampled_layers():
    """27B deployment shape with its rescale setting (c = 512): d = 5120, 48 upper
    layers, 8 KV heads x 128; the oracle checks three layers."""
    cfg = synth.DENSE27B
    c = 512
    inp = _favour_first_half(synth.fill_inputs(cfg, device=DEV), cfg)
    x_exact = synth.rescale_inputs(cfg, inp["x_S"], c, device=DEV)
    vs = _gpu_scale(cfg, inp, x_exact, c).cpu().numpy().astype(np.float64)
    layers = [0, 23, cfg.P - 1]
    ref = _oracle_scale(cfg, inp, x_exact, c, layers)
    _assert_scales(vs[layers], ref)
