"""GPU tests of map storage: the int8 code (rf_quantize_maps_int8) and the
layer-by-layer fill from device or host maps, bf16 or int8 (rf_fill_kv_layered).

RidgeFill review, "Ridge map": the 27B maps in int8; maps "kept resident in GPU
memory or streamed from host memory one layer at a time".
- The int8 codes and row scales must equal the oracle's bit for bit (both take
  the rounding decisions in fp32).
- A layered fill from the same bf16 maps must equal rf_fill_kv bit for bit, in
  every cache entry, with the maps on the device or the host (same kernels, same
  summation order; only the launch granularity differs).
- A layered fill from int8 maps is checked against the oracle fill with the
  dequantized maps s[o] q[o][i], with the fill's per-head tolerance.
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
    base = dict(name=name, index=97, d=512, L=5, S=2, N=400, T=37, H=2, hd=128, rope_theta=5e5,
                exact="uniform10", lam=0.03, calib_n=0)
    base.update(kw)
    return synth.FillConfig(**base)


def _quantize(cfg, A):
    desc = desc_of(cfg)
    q = torch.empty(A.shape, dtype=torch.int8, device=DEV)
    s = torch.empty(A.shape[:2], dtype=torch.float32, device=DEV)
    rf.rf_quantize_maps_int8(desc, A.to(DEV), q, s)
    torch.cuda.synchronize()
    return q, s


def _run_layered(cfg, inp, maps, flags=0, v_scale=None, k_norm_gain=None, prefolded=False):
    desc = desc_of(cfg, flags | (rf.RF_WEIGHTS_PREFOLDED if prefolded else 0), v_scale, k_norm_gain)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    P, KV = cfg.P, cfg.KV
    W = (None, *fold(desc, g)) if prefolded else (g["gain"], g["Wk"], g["Wv"])
    kc = synth.canary_cache(cfg.L, cfg.N, cfg.H, cfg.hd, 0, DEV)
    vc = synth.canary_cache(cfg.L, cfg.N, cfg.H, cfg.hd, 1, DEV)
    kc0, vc0 = kc.clone(), vc.clone()
    wsb = rf.rf_fill_layered_workspace_bytes(desc, maps)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=DEV)
    nf = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    rf.rf_fill_kv_layered(desc, g["x_S"], cfg.D_in, g["mask"], maps, g["b"], *W, kc, vc, cfg.N * KV, KV, nf, status,
                          ws, wsb)
    torch.cuda.synchronize()
    return {"kc": kc, "vc": vc, "kc0": kc0, "vc0": vc0, "n_fill": int(nf.item()), "status": int(status.item()),
            "ws_bytes": wsb}


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_int8_codes_match_the_oracle_bit_for_bit():
    cfg = _small("quantize", d=256, d_in=768, L=5, S=2)
    A = synth.fill_inputs(cfg)["A"].float()
    A[1, 7] = 0.0                                   # a zero row
    A[2, 3] *= 1e-3                                 # a small row
    A = A.to(torch.bfloat16)
    q, s = _quantize(cfg, A)
    qr, sr = O.quantize_rows_int8(O.bf16_bits_to_f64(synth.bits(A)).astype(np.float32))
    np.testing.assert_array_equal(q.cpu().numpy(), qr)
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), sr.view(np.uint32))


@pytest.mark.parametrize("cfg", [
    _small("hd128 ragged"),
    _small("non-square d_in 1024 -> 256, hd64", d=256, d_in=1024, L=4, S=1, N=300, T=20, H=2, hd=64),
], ids=lambda c: c.name)
@KERNELS
def test_layered_bf16_fill_equals_the_resident_fill(cfg, flags):
    inp = synth.fill_inputs(cfg)
    ref = run_fill(cfg, inp, flags=flags)
    assert ref["status"] == 0
    A_host = inp["A"].pin_memory()
    # device maps with the gain folded in the call; host maps with prefolded projections
    for maps, pre in ((rf.map_source(rf.RF_MAPS_BF16, inp["A"].to(DEV)), False),
                      (rf.map_source(rf.RF_MAPS_BF16, A_host, on_host=True), True)):
        res = _run_layered(cfg, inp, maps, flags, prefolded=pre)
        assert res["status"] == 0 and res["n_fill"] == ref["n_fill"]
        assert _same_bits(res["kc"], ref["kc"]) and _same_bits(res["vc"], ref["vc"])


def test_layered_fill_applies_value_scale_and_key_norm_per_layer():
    cfg = _small("layered with corrections", L=6, S=2)
    inp = synth.fill_inputs(cfg)
    vs = torch.rand((cfg.P, cfg.H), dtype=torch.float32, device=DEV) + 0.5
    kg = synth.key_norm_gain(cfg)
    ref = run_fill(cfg, inp, v_scale=vs, k_norm_gain=kg)
    res = _run_layered(cfg, inp, rf.map_source(rf.RF_MAPS_BF16, inp["A"].pin_memory(), on_host=True),
                       v_scale=vs, k_norm_gain=kg.to(DEV))
    assert ref["status"] == 0 and res["status"] == 0
    assert _same_bits(res["kc"], ref["kc"]) and _same_bits(res["vc"], ref["vc"])


@KERNELS
def test_layered_int8_fill_matches_the_oracle_with_dequantized_maps(flags):
    cfg = _small("int8 maps", L=6, S=2)
    inp = synth.fill_inputs(cfg)
    q, s = _quantize(cfg, inp["A"])
    dev = _run_layered(cfg, inp, rf.map_source(rf.RF_MAPS_INT8, q, row_scale=s), flags)
    host = _run_layered(cfg, inp, rf.map_source(rf.RF_MAPS_INT8, q.cpu().pin_memory(), on_host=True, row_scale=s),
                        flags)
    assert dev["status"] == 0 and host["status"] == 0
    assert _same_bits(dev["kc"], host["kc"]) and _same_bits(dev["vc"], host["vc"])
    mnp = inp["mask"].cpu().numpy()
    idx = O.prefix_partition(cfg.N, cfg.T, mnp)
    assert_bookkeeping(cfg, dev, mnp)
    deq = O.dequantize_rows_int8(q.cpu().numpy(), s.cpu().numpy())
    inp_deq = dict(inp)
    inp_deq["A"] = torch.as_tensor(deq, dtype=torch.float32)       # exact: s[o] q is representable in fp32
    assert_values(cfg, inp_deq, dev, idx)


@pytest.mark.slow
def test_layered_8b_shape_host_bf16_equals_resident_and_int8_sampled():
    cfg = synth.LLAMA8B
    inp = synth.fill_inputs(cfg, device=DEV)
    ref = run_fill(cfg, inp, canary=False)
    A_host = inp["A"].cpu().pin_memory()
    res = _run_layered(cfg, inp, rf.map_source(rf.RF_MAPS_BF16, A_host, on_host=True))
    assert ref["status"] == 0 and res["status"] == 0
    fill = torch.as_tensor(O.prefix_partition(cfg.N, cfg.T, inp["mask"].cpu().numpy()), device=DEV)
    for a, b in ((res["kc"], ref["kc"]), (res["vc"], ref["vc"])):
        assert _same_bits(a[cfg.S:].index_select(1, fill), b[cfg.S:].index_select(1, fill))
    q, s = _quantize(cfg, inp["A"])
    del A_host
    r8 = _run_layered(cfg, inp, rf.map_source(rf.RF_MAPS_INT8, q.cpu().pin_memory(), on_host=True, row_scale=s))
    assert r8["status"] == 0
    mnp = inp["mask"].cpu().numpy()
    idx = O.prefix_partition(cfg.N, cfg.T, mnp)
    rows = np.sort(np.random.default_rng(2).choice(idx, 96, replace=False))
    deq = O.dequantize_rows_int8(q.cpu().numpy(), s.cpu().numpy())
    inp_deq = dict(inp)
    inp_deq["A"] = torch.as_tensor(deq, dtype=torch.float32)
    assert_values(cfg, inp_deq, r8, rows)
