"""Helpers shared by the fill tests: run rf_fill_kv on seeded inputs and compare
with the fp64 oracle (bookkeeping bit for bit, values by the per-head error)."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import ridge_map_kv_gb300 as rf
import synth

TOL_MAX = 2e-2     # max over (layer, row, head, K|V) of ||gpu - ref|| / ||ref||
TOL_MEAN = 3e-3    # mean of the same


def desc_of(cfg, flags: int = 0, v_scale=None, k_norm_gain=None) -> rf.rf_fill_desc:
    return rf.rf_fill_desc(d=cfg.d, L=cfg.L, S=cfg.S, N=cfg.N, T=cfg.T, n_kv_heads=cfg.H, head_dim=cfg.hd,
                           rope_theta=cfg.rope_theta, rms_eps=cfg.rms_eps, pos_offset=cfg.pos_offset, flags=flags,
                           d_in=cfg.d_in,
                           v_scale=None if v_scale is None else v_scale.data_ptr(),
                           k_norm_gain=None if k_norm_gain is None else k_norm_gain.data_ptr())


def fold(desc, g):
    """Gain-folded K and V projections of the device inputs ``g`` (rf_fold_kv_weights)."""
    Wkf, Wvf = torch.empty_like(g["Wk"]), torch.empty_like(g["Wv"])
    rf.rf_fold_kv_weights(desc, g["gain"], g["Wk"], g["Wv"], Wkf, Wvf)
    return Wkf, Wvf


def run_fill(cfg, inp: dict, dev="cuda", mask="inp", canary=True, flags: int = 0, v_scale=None,
             k_norm_gain=None, prefolded=False):
    """Runs the fill on device copies of ``inp``. Returns a dict with the caches
    before/after, n_fill and the device status. ``flags`` selects the GEMM kernels
    (rf.RF_FLAG_SINGLE_CTA or rf.RF_FLAG_CTA_PAIR; 0 = library default). The fill
    folds the RMSNorm gain into its workspace, or with ``prefolded`` it gets
    projections folded beforehand by rf_fold_kv_weights (RF_WEIGHTS_PREFOLDED)."""
    dev = torch.device(dev)
    kng = None if k_norm_gain is None else k_norm_gain.to(dev)   # alive until the fill is done
    desc = desc_of(cfg, flags | (rf.RF_WEIGHTS_PREFOLDED if prefolded else 0), v_scale, kng)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    m = g["mask"] if mask == "inp" else (mask.to(dev) if mask is not None else None)
    P, KV = cfg.P, cfg.KV
    gain, Wk, Wv = (g["gain"], g["Wk"], g["Wv"]) if P > 0 else (None, None, None)
    if prefolded and P > 0:
        Wk, Wv = fold(desc, g)
        gain = None
    if canary:
        kc = synth.canary_cache(cfg.L, cfg.N, cfg.H, cfg.hd, 0, dev)
        vc = synth.canary_cache(cfg.L, cfg.N, cfg.H, cfg.hd, 1, dev)
    else:
        kc = torch.zeros((cfg.L, cfg.N, cfg.H, cfg.hd), dtype=torch.bfloat16, device=dev)
        vc = torch.zeros_like(kc)
    kc0, vc0 = kc.clone(), vc.clone()
    ws_bytes = rf.rf_fill_workspace_bytes(desc)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    nfill = torch.full((1,), -1, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    rf.rf_fill_kv(desc, g["x_S"], cfg.D_in, m, g["A"] if P > 0 else None, g["b"] if P > 0 else None,
                  gain, Wk, Wv, kc, vc, cfg.N * KV, KV, nfill, status, ws, ws_bytes)
    torch.cuda.synchronize()
    return {"kc": kc, "vc": vc, "kc0": kc0, "vc0": vc0, "n_fill": int(nfill.item()),
            "status": int(status.item()), "ws": ws}


def _f64_of(t) -> np.ndarray:
    """float64 copy of a bf16 tensor (exact decode) or of a float tensor."""
    if t.dtype == torch.bfloat16:
        return O.bf16_bits_to_f64(synth.bits(t))
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_rows(cfg, inp: dict, rows: np.ndarray, v_scale=None, k_norm_gain=None):
    """fp64 oracle K, V [P, n, H, hd] for the given filled rows (V scaled by
    v_scale [P, H] when given)."""
    f64 = O.bf16_bits_to_f64
    x = f64(synth.bits(inp["x_S"][torch.as_tensor(rows, device=inp["x_S"].device)]))
    Ks, Vs = [], []
    for p in range(cfg.P):          # one layer at a time keeps the fp64 copies small
        K, V = O.fill_rows(x, rows + cfg.pos_offset, _f64_of(inp["A"][p:p + 1]),
                           synth.f32(inp["b"][p:p + 1]).astype(np.float64), f64(synth.bits(inp["gain"][p:p + 1])),
                           f64(synth.bits(inp["Wk"][p:p + 1])), f64(synth.bits(inp["Wv"][p:p + 1])),
                           cfg.H, cfg.hd, cfg.rope_theta, cfg.rms_eps,
                           None if v_scale is None else np.asarray(v_scale, np.float64)[p:p + 1],
                           None if k_norm_gain is None else f64(synth.bits(k_norm_gain[p:p + 1])))
        Ks.append(K[0])
        Vs.append(V[0])
    return np.stack(Ks), np.stack(Vs)


def head_errors(got_bits: np.ndarray, ref: np.ndarray) -> np.ndarray:
    got = O.bf16_bits_to_f64(got_bits)
    return np.linalg.norm(got - ref, axis=-1) / np.maximum(np.linalg.norm(ref, axis=-1), 1e-6)


def check_values(cfg, inp, res, rows: np.ndarray, v_scale=None, k_norm_gain=None):
    """Per-head relative errors of the filled K and V at ``rows`` (all layers)."""
    K, V = oracle_rows(cfg, inp, rows, v_scale, k_norm_gain)
    rt = torch.as_tensor(rows, device=res["kc"].device)
    kb = synth.bits(res["kc"][cfg.S:].index_select(1, rt))
    vb = synth.bits(res["vc"][cfg.S:].index_select(1, rt))
    ek = head_errors(kb, K)
    ev = head_errors(vb, V)
    e = np.concatenate([ek.ravel(), ev.ravel()])
    return e


def assert_values(cfg, inp, res, rows, v_scale=None, k_norm_gain=None):
    e = check_values(cfg, inp, res, rows, v_scale, k_norm_gain)
    assert np.all(np.isfinite(e)), "non-finite filled values"
    assert e.max() <= TOL_MAX and e.mean() <= TOL_MEAN, f"max {e.max():.3e} mean {e.mean():.3e}"
    return e


def expected_written(cfg, mask_np) -> np.ndarray:
    """bool [L, N]: which (layer, row) entries the fill owns."""
    w = np.zeros((cfg.L, cfg.N), bool)
    idx = O.prefix_partition(cfg.N, cfg.T, mask_np)
    if cfg.P > 0:
        w[cfg.S:, idx] = True
    return w


def assert_bookkeeping(cfg, res, mask_np):
    """Bit-exact: entries outside the filled set keep their canaries; every entry
    of the filled set changed (canaries are NaN, the fill is finite)."""
    w = torch.as_tensor(expected_written(cfg, mask_np), device=res["kc"].device)
    for cur, old in ((res["kc"], res["kc0"]), (res["vc"], res["vc0"])):
        ci = cur.view(torch.int16)
        oi = old.view(torch.int16)
        same = (ci == oi).all(dim=-1).all(dim=-1)      # [L, N]
        assert bool(same[~w].all()), "a cache entry outside the filled set was written"
        if bool(w.any()):
            assert not bool(same[w].any()), "a filled entry kept its canary"
            assert bool(torch.isfinite(cur[w].float()).all()), "non-finite filled value"
