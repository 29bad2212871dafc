"""rf_fill_kv_static: the fill for callers that cannot allocate device memory.

A plugin inside a serving engine that owns all device memory through its own
pool, or a latency-critical path where a cudaMalloc would synchronise the device,
cannot hand the library a workspace. rf_fill_kv_static keeps its scratch in a
fixed array inside the library instead. These tests call it twice in a row
through the C ABI, on two different fills, and check each result against
rf_fill_kv run with a caller workspace on the same inputs. Both calls run the
same kernels in the same order on the same workspace layout, so the caches must
agree bit for bit. The first fill then runs once more after the second and must
reproduce its own first result bit for bit: nothing may depend on what the
previous call left in the shared array. Last, a fill too large for the fixed
array is refused before anything runs.

This file is collected last on purpose, and it needs nothing from the other
tests: it passes alone in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

import oracle as O
import ridge_map_kv_gb300 as rf
import synth
from fillcheck import desc_of, fold

pytestmark = pytest.mark.gpu


def _cfg(name, **kw):
    base = dict(name=name, index=91, d=512, L=5, S=2, N=400, T=37, H=2, hd=128, rope_theta=5e5,
                exact="uniform10", lam=0.03, calib_n=0)
    base.update(kw)
    return synth.FillConfig(**base)


def _prepare(cfg, prefolded):
    """Device inputs and the weights the fill takes: projections folded beforehand
    (RF_WEIGHTS_PREFOLDED), or gain and projections for the call to fold in its scratch."""
    dev = torch.device("cuda")
    inp = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in synth.fill_inputs(cfg).items()}
    desc = desc_of(cfg, rf.RF_WEIGHTS_PREFOLDED if prefolded else 0)
    W = (None, *fold(desc, inp)) if prefolded else (inp["gain"], inp["Wk"], inp["Wv"])
    return desc, inp, W


def _caches(cfg):
    return (synth.canary_cache(cfg.L, cfg.N, cfg.H, cfg.hd, 0, "cuda"),
            synth.canary_cache(cfg.L, cfg.N, cfg.H, cfg.hd, 1, "cuda"))


def _out():
    return torch.full((1,), -1, dtype=torch.int32, device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda")


def _compare(cfg, inp, got_k, got_v, ref_k, ref_v):
    """Bit-for-bit equality of the whole caches (written and untouched entries)."""
    mask = None if inp["mask"] is None else inp["mask"].cpu().numpy()
    idx = O.prefix_partition(cfg.N, cfg.T, mask)
    written = np.zeros((cfg.L, cfg.N), bool)
    written[cfg.S:, idx] = True
    for got, ref in ((got_k, ref_k), (got_v, ref_v)):
        gb, rb = synth.bits(got), synth.bits(ref)
        assert np.array_equal(gb[~written], rb[~written]), "entries outside the filled set differ"
        assert np.array_equal(gb[written], rb[written]), "filled entries differ from the workspace fill"


def _static_fill(cfg, prepared):
    desc, inp, W = prepared
    kc, vc = _caches(cfg)
    nf, st = _out()
    rf.rf_fill_kv_static(desc, inp["x_S"], cfg.d, inp["mask"], inp["A"], inp["b"], *W, kc, vc,
                         cfg.N * cfg.KV, cfg.KV, nf, st)
    return kc, vc, nf, st


def test_static_fill_matches_workspace_fill_on_two_calls_in_a_row():
    cfgs = [_cfg("static fill A"),
            _cfg("static fill B", index=92, d=768, L=4, S=2, N=300, T=20, H=4, hd=64, exact="blocks16_5")]
    prepared = [_prepare(cfgs[0], True), _prepare(cfgs[1], False)]

    # references through rf_fill_kv with a caller workspace
    refs = []
    for cfg, (desc, inp, W) in zip(cfgs, prepared):
        kc, vc = _caches(cfg)
        nf, st = _out()
        ws_bytes = rf.rf_fill_workspace_bytes(desc)
        assert ws_bytes <= rf.RF_STATIC_SCRATCH_BYTES
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        rf.rf_fill_kv(desc, inp["x_S"], cfg.d, inp["mask"], inp["A"], inp["b"], *W, kc, vc, cfg.N * cfg.KV, cfg.KV,
                      nf, st, ws, ws_bytes)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        refs.append((kc, vc, int(nf.item())))

    # the two static-scratch calls, back to back on one stream, then the first again
    outs = [_static_fill(cfg, pr) for cfg, pr in zip(cfgs, prepared)]
    again = _static_fill(cfgs[0], prepared[0])
    torch.cuda.synchronize()

    for cfg, (desc, inp, W), (rk, rv, rn), (kc, vc, nf, st) in zip(cfgs, prepared, refs, outs):
        assert int(st.item()) == 0
        assert int(nf.item()) == rn
        _compare(cfg, inp, kc, vc, rk, rv)
    kc, vc, nf, st = again
    assert int(st.item()) == 0 and int(nf.item()) == refs[0][2]
    _compare(cfgs[0], prepared[0][1], kc, vc, outs[0][0], outs[0][1])


def test_static_fill_refuses_fills_larger_than_its_scratch():
    desc = desc_of(synth.LLAMA8B)
    assert rf.rf_fill_workspace_bytes(desc) > rf.RF_STATIC_SCRATCH_BYTES
    with pytest.raises(rf.RFError) as ei:
        rf.rf_fill_kv_static(desc, None, synth.LLAMA8B.d, None, None, None, None, None, None, None, None, 0, 0)
    assert ei.value.status == rf.RF_ERR_WORKSPACE
    assert "static scratch" in str(ei.value)
