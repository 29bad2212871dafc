"""GPU parity of rf_xmodel_map and rf_rope_rows against the fp64 oracle.

Small cases compare every mapped head; the full 40 -> 64 layer, N = 32768 case
compares sampled rows of sampled target layers. Tolerance: per-head relative
error max <= 2e-2, mean <= 3e-3.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
import ridge_map_kv_gb300 as rf
import synth
from fillcheck import TOL_MAX, TOL_MEAN, head_errors

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(cfg, inp, L_tgt, N, flags=0):
    desc = rf.rf_xmodel_desc(L_src=cfg.L_src, L_tgt=L_tgt, k=cfg.k, n_kv_heads=cfg.H, head_dim=cfg.hd, N=N,
                             theta_src=cfg.theta_src, theta_tgt=cfg.theta_tgt, pos_offset=cfg.pos_offset,
                             flags=flags)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    kt = torch.full((L_tgt, N, cfg.H, cfg.hd), float("nan"), dtype=torch.bfloat16, device=DEV)
    vt = torch.full_like(kt, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    wsb = rf.rf_xmodel_workspace_bytes(desc)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    src = torch.as_tensor(np.asarray(g["src"], np.int32), device=DEV)     # the device table the call takes
    rf.rf_xmodel_map(desc, src, g["k_src"], g["v_src"], g["Wk"], g["bk"], g["Wv"], g["bv"], kt, vt, status,
                     ws, wsb)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return kt, vt


def _oracle_layer(cfg, inp, l, rows):
    f64 = O.bf16_bits_to_f64
    rt = torch.as_tensor(rows, device=inp["k_src"].device)
    ks = f64(synth.bits(inp["k_src"].index_select(1, rt)))
    vs = f64(synth.bits(inp["v_src"].index_select(1, rt)))
    return O.xmodel_map_layer(ks, vs, list(inp["src"][l]), f64(synth.bits(inp["Wk"][l])),
                              synth.f32(inp["bk"][l]).astype(np.float64), f64(synth.bits(inp["Wv"][l])),
                              synth.f32(inp["bv"][l]).astype(np.float64), rows + cfg.pos_offset, cfg.theta_src,
                              cfg.theta_tgt, cfg.H, cfg.hd)


def _check(cfg, inp, kt, vt, layers, rows):
    errs = []
    rt = torch.as_tensor(rows, device=kt.device)
    for l in layers:
        K, V = _oracle_layer(cfg, inp, l, rows)
        errs.append(head_errors(synth.bits(kt[l].index_select(0, rt)), K).ravel())
        errs.append(head_errors(synth.bits(vt[l].index_select(0, rt)), V).ravel())
    e = np.concatenate(errs)
    assert np.all(np.isfinite(e)) and e.max() <= TOL_MAX and e.mean() <= TOL_MEAN, (e.max(), e.mean())


SMALL = synth.XModelConfig("xmodel small", 94, L_src=5, L_tgt=3, k=2, H=2, hd=128, N=300, theta_src=1.0e6,
                           theta_tgt=5.0e5, calib_n=0, lam=0.01)


@pytest.mark.parametrize("cfg", [SMALL,
                                 dataclasses.replace(SMALL, name="hd64 4 heads offset", H=4, hd=64, k=3, N=131,
                                                     pos_offset=700, theta_tgt=1.0e6),
                                 dataclasses.replace(SMALL, name="positions near 2^25", pos_offset=(1 << 25) + 321)],
                         ids=lambda c: c.name)
@pytest.mark.parametrize("flags", [rf.RF_FLAG_SINGLE_CTA, rf.RF_FLAG_CTA_PAIR], ids=["single-cta", "cta-pair"])
def test_xmodel_small_matches_oracle(cfg, flags):
    inp = synth.xmodel_inputs(cfg)
    rng = np.random.default_rng(4)
    inp["src"] = rng.integers(0, cfg.L_src, size=(cfg.L_tgt, cfg.k)).astype(np.int32)
    kt, vt = _run(cfg, inp, cfg.L_tgt, cfg.N, flags)
    _check(cfg, inp, kt, vt, range(cfg.L_tgt), np.arange(cfg.N))


def test_xmodel_identity_on_one_source_layer():
    cfg = dataclasses.replace(SMALL, theta_tgt=SMALL.theta_src)
    inp = synth.xmodel_inputs(cfg)
    KV = cfg.KV
    for l in range(cfg.L_tgt):
        j = l % cfg.k
        W = torch.zeros((KV, cfg.k * KV))
        W[:, j * KV:(j + 1) * KV] = torch.eye(KV)
        inp["Wk"][l] = W.to(torch.bfloat16)
        inp["Wv"][l] = W.to(torch.bfloat16)
    inp["bk"].zero_()
    inp["bv"].zero_()
    kt, vt = _run(cfg, inp, cfg.L_tgt, cfg.N)
    for l in range(cfg.L_tgt):
        s = int(inp["src"][l][l % cfg.k])
        assert torch.equal(vt[l].cpu(), inp["v_src"][s])             # V: exact copy
        e = head_errors(synth.bits(kt[l]), O.bf16_bits_to_f64(synth.bits(inp["k_src"][s])))
        assert e.max() <= 1e-2 and e.mean() <= 3e-3                  # K: unrope, bf16, re-rope


@pytest.mark.slow
@pytest.mark.parametrize("flags", [rf.RF_FLAG_SINGLE_CTA, rf.RF_FLAG_CTA_PAIR], ids=["single-cta", "cta-pair"])
def test_xmodel_full_size_sampled(flags):
    cfg = synth.XMODEL
    inp = synth.xmodel_inputs(cfg, device=DEV)
    kt, vt = _run(cfg, inp, cfg.L_tgt, cfg.N, flags)
    # every target entry was written: no NaN canary is left anywhere (checked on the device)
    assert not bool(torch.isnan(kt).any()) and not bool(torch.isnan(vt).any())
    rows = np.unique(np.concatenate([[0, 1, 127, 128, cfg.N - 1],
                                     np.random.default_rng(3).choice(cfg.N, 59, replace=False)]))
    _check(cfg, inp, kt, vt, [0, 21, 40, 63], rows)


@pytest.mark.parametrize("bad", [-1, 5, 1 << 30], ids=["negative", "L_src", "huge"])
def test_xmodel_table_out_of_range_is_reported_on_the_device_and_writes_nothing(bad):
    """The source-layer table lives on the device, so its range is checked there: an
    entry outside [0, L_src) sets RF_ERR_INVALID_ARG in the status word and the call
    writes no target entry (the NaN canaries stay); the context stays usable and a
    valid table afterwards maps as usual."""
    cfg = SMALL
    inp = synth.xmodel_inputs(cfg)
    desc = rf.rf_xmodel_desc(L_src=cfg.L_src, L_tgt=cfg.L_tgt, k=cfg.k, n_kv_heads=cfg.H, head_dim=cfg.hd, N=cfg.N,
                             theta_src=cfg.theta_src, theta_tgt=cfg.theta_tgt, pos_offset=0)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    tab = np.asarray(inp["src"], np.int32).copy()
    tab[1, 0] = bad
    kt = torch.full((cfg.L_tgt, cfg.N, cfg.H, cfg.hd), float("nan"), dtype=torch.bfloat16, device=DEV)
    vt = torch.full_like(kt, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    wsb = rf.rf_xmodel_workspace_bytes(desc)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    rf.rf_xmodel_map(desc, torch.as_tensor(tab, device=DEV), g["k_src"], g["v_src"], g["Wk"], g["bk"], g["Wv"],
                     g["bv"], kt, vt, status, ws, wsb)
    torch.cuda.synchronize()
    assert int(status.item()) == rf.RF_ERR_INVALID_ARG
    assert bool(torch.isnan(kt).all()) and bool(torch.isnan(vt).all())
    kt2, vt2 = _run(cfg, inp, cfg.L_tgt, cfg.N)
    _check(cfg, inp, kt2, vt2, range(cfg.L_tgt), np.arange(cfg.N))


@pytest.mark.parametrize("hd,theta,off", [(128, 1.0e6, 0), (64, 5.0e5, 12345), (128, 1.0e6, (1 << 27) + 12345),
                                          (64, 1.0e4, -4096)])
def test_rope_rows_matches_oracle_and_inverts(hd, theta, off):
    """RoPE at positions off .. off + 512 against the fp64 oracle, and its inverse: the
    angle is reduced mod 2π in 64-bit fixed point, so positions near 2^27 and negative
    ones are as accurate as small ones."""
    n, H = 513, 3
    ld = H * hd + 8
    x = synth._randn((n, ld), 77, DEV)
    y = torch.empty_like(x)
    rf.rf_rope_rows(x, y, n, ld, H, hd, theta, off, False)
    z = torch.empty_like(x)
    rf.rf_rope_rows(y, z, n, ld, H, hd, theta, off, True)
    torch.cuda.synchronize()
    xs = O.bf16_bits_to_f64(synth.bits(x[:, :H * hd])).reshape(n, H, hd)
    ref = O.rope(xs, (np.arange(n) + off)[:, None], theta)
    e = head_errors(synth.bits(y[:, :H * hd]).reshape(n, H, hd), ref)
    assert e.max() <= 1e-2 and e.mean() <= 2e-3
    e2 = head_errors(synth.bits(z[:, :H * hd]).reshape(n, H, hd), xs)
    assert e2.max() <= 1e-2 and e2.mean() <= 3e-3
