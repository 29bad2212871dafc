"""CPU-only checks of the C ABI: librf.so loads without a GPU, exports every
function include/rf.h declares, and rejects bad arguments on the host (before any
launch, so no GPU is touched)."""
import ctypes
import os
import re

import pytest

import ridge_map_kv_gb300 as rf
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built_library():
    if not os.path.exists(rf.LIB_PATH):
        from ridge_map_kv_gb300 import build
        build.build()
    rf.lib()


def _declared_functions():
    txt = open(os.path.join(ROOT, "include", "rf.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(rf_[a-z0-9_]+)\s*\(", txt)))


def test_library_exports_every_declared_function():
    names = _declared_functions()
    assert len(names) >= 19
    L = ctypes.CDLL(rf.LIB_PATH)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


def test_binding_covers_every_declared_function():
    from ridge_map_kv_gb300 import _binding
    assert set(_declared_functions()) <= set(_binding._SIGS)


def test_status_strings_and_version():
    assert rf.rf_version() >= 100
    assert rf.rf_status_string(rf.RF_OK) == "ok"
    assert "timed out" in rf.rf_status_string(rf.RF_ERR_TIMEOUT)
    assert rf.rf_status_string(999) == "unknown status"
    for s in ("compact", "map_gemm", "kv_gemm", "calib_gemm", "xmodel_gemm"):
        assert s in [rf.rf_stage_name(i) for i in range(1, 13)]
    assert rf.rf_stage_name(12) == "value_rescale"
    assert [rf.rf_stage_name(i) for i in (18, 19, 20, 21)] == ["select_gemm", "select_factor", "select_score",
                                                               "select_split"]


def _fill_desc(**kw):
    c = synth.TOY
    d = dict(d=c.d, L=c.L, S=c.S, N=c.N, T=c.T, n_kv_heads=c.H, head_dim=c.hd, rope_theta=c.rope_theta,
             rms_eps=c.rms_eps, pos_offset=0)
    d.update(kw)
    return rf.rf_fill_desc(**d)


def test_fill_workspace_size_follows_the_layout():
    desc = _fill_desc(flags=rf.RF_WEIGHTS_PREFOLDED)
    # fill_idx, n_fill, the GEMMs' unit counter, Xf [M x d], x̂ [P x M x d], ss partials [P x d/256 x M],
    # with M = the prefix rows padded to a whole 256-row unit (RoPE angles are computed in the kernel: no table)
    r = lambda x: (x + 255) // 256 * 256
    n_prefix, M, P, d, KV = 9, 256, 4, 256, 128
    want = r(n_prefix * 4) + r(4) + r(4) + r(M * d * 2) + r(P * M * d * 2) + r(P * (d // 256) * M * 4)
    assert rf.rf_fill_workspace_bytes(desc) == want
    # without RF_WEIGHTS_PREFOLDED the call folds the gain into two [P][KV][d] bf16 arrays of its own
    assert rf.rf_fill_workspace_bytes(_fill_desc()) == want + 2 * r(P * KV * d * 2)


@pytest.mark.parametrize("bad", [dict(d=100), dict(head_dim=96), dict(S=9), dict(T=13), dict(n_kv_heads=1),
                                 dict(rope_theta=0.0)])
def test_fill_rejects_bad_descriptors_on_the_host(bad):
    desc = _fill_desc(**bad)
    assert rf.rf_fill_workspace_bytes(desc) == 0
    with pytest.raises(rf.RFError) as ei:
        rf.rf_fill_kv(desc, 16, 256, None, 16, 16, 16, 16, 16, 16, 16, 0, 128, None, None, 256, 1 << 30, stream=0)
    assert ei.value.status in (rf.RF_ERR_INVALID_ARG, rf.RF_ERR_SHAPE)


def test_fill_row_limit_is_the_documented_one():
    """rf.h: N − T may be at most 2^24 (row indices, tile and unit counts are 32-bit in
    the kernels). The limit itself is accepted, one row past it is refused on the host."""
    at = _fill_desc(N=(1 << 24) + 3, T=3)
    assert rf.rf_fill_workspace_bytes(at) > 0
    past = _fill_desc(N=(1 << 24) + 4, T=3)
    assert rf.rf_fill_workspace_bytes(past) == 0
    with pytest.raises(rf.RFError) as ei:
        _fill_call(past)
    assert ei.value.status == rf.RF_ERR_SHAPE and "2^24" in rf.rf_last_error()


@pytest.mark.parametrize("d_in,d_out,P,ok", [(32768, 256, 1, True), (33024, 256, 1, False), (256, 256, 65535, True),
                                            (256, 256, 65536, False), (384, 256, 1, False), (256, 320, 1, False),
                                            (256, 256, 0, False)],
                         ids=["d_in at its limit", "d_in past it", "maps at their limit", "maps past it",
                              "d_in not a multiple of 256", "d_out not a multiple of 256", "no maps"])
def test_solve_shape_limits(d_in, d_out, P, ok):
    """rf.h: d_in and d_out multiples of 256, d_in <= 32768, 1 <= n_maps <= 65535; the
    workspace query answers 0 outside them and the call refuses with RF_ERR_SHAPE or
    RF_ERR_INVALID_ARG before any launch."""
    desc = rf.rf_calib_desc(d_in=d_in, d_out=d_out, n_maps=P)
    wsb = rf.rf_solve_workspace_bytes(desc)
    assert (wsb > 0) == ok
    if not ok:
        with pytest.raises(rf.RFError) as ei:
            rf.rf_solve(desc, rf.calib_stats_struct(256, 256, 256, 256, 256), 0.03, rf.RF_ALPHA_TRACE, 0, 256, 256,
                        workspace=256, workspace_bytes=1 << 40, stream=0)
        assert ei.value.status in (rf.RF_ERR_SHAPE, rf.RF_ERR_INVALID_ARG)


@pytest.mark.parametrize("lam,refine", [(-1.0, 0), (float("nan"), 0), (0.03, -1), (0.03, 9)],
                         ids=["negative lambda", "NaN lambda", "negative sweeps", "more than 8 sweeps"])
def test_solve_rejects_bad_lambda_and_sweep_counts(lam, refine):
    desc = rf.rf_calib_desc(d_in=256, d_out=256, n_maps=1)
    with pytest.raises(rf.RFError) as ei:
        rf.rf_solve(desc, rf.calib_stats_struct(256, 256, 256, 256, 256), lam, rf.RF_ALPHA_TRACE, refine, 256, 256,
                    workspace=256, workspace_bytes=1 << 40, stream=0)
    assert ei.value.status == rf.RF_ERR_INVALID_ARG


def _fill_call(desc, **kw):
    """rf_fill_kv with valid-looking (aligned, non-NULL, never dereferenced) arguments,
    some replaced by ``kw``; the host checks reject before any launch."""
    a = dict(x_S=256, ld_x=256, mask=None, A=256, b=256, gain=256, Wk=256, Wv=256, kc=256, vc=256, ls=0, rs=128,
             ws=256, wsb=1 << 30)
    a.update(kw)
    rf.rf_fill_kv(desc, a["x_S"], a["ld_x"], a["mask"], a["A"], a["b"], a["gain"], a["Wk"], a["Wv"], a["kc"],
                  a["vc"], a["ls"], a["rs"], None, None, a["ws"], a["wsb"], stream=0)


@pytest.mark.parametrize("kw,status", [
    (dict(A=None), rf.RF_ERR_INVALID_ARG),
    (dict(Wk=None), rf.RF_ERR_INVALID_ARG),
    (dict(Wv=None), rf.RF_ERR_INVALID_ARG),
    (dict(gain=None), rf.RF_ERR_INVALID_ARG),           # the call must fold, so it needs the gain
    (dict(x_S=258), rf.RF_ERR_ALIGN),
    (dict(gain=264), rf.RF_ERR_ALIGN),
    (dict(Wv=264), rf.RF_ERR_ALIGN),
    (dict(rs=100), rf.RF_ERR_ALIGN),
    (dict(wsb=1024), rf.RF_ERR_WORKSPACE),
], ids=["A NULL", "Wk NULL", "Wv NULL", "gain NULL", "x_S misaligned", "gain misaligned", "Wv misaligned",
        "row stride", "small workspace"])
def test_fill_rejects_null_and_misaligned_pointers_and_small_workspace(kw, status):
    with pytest.raises(rf.RFError) as ei:
        _fill_call(_fill_desc(), **kw)
    assert ei.value.status == status
    if status == rf.RF_ERR_WORKSPACE:
        assert "workspace" in rf.rf_last_error()


def test_prefolded_fill_needs_no_gain_and_a_smaller_workspace():
    pre = _fill_desc(flags=rf.RF_WEIGHTS_PREFOLDED)
    need = rf.rf_fill_workspace_bytes(pre)
    assert need < rf.rf_fill_workspace_bytes(_fill_desc())
    # gain NULL is accepted with the flag: the first complaint is about the workspace
    with pytest.raises(rf.RFError) as ei:
        _fill_call(pre, gain=None, wsb=need - 1)
    assert ei.value.status == rf.RF_ERR_WORKSPACE
    with pytest.raises(rf.RFError) as ei:
        _fill_call(pre, gain=None, Wk=None)
    assert ei.value.status == rf.RF_ERR_INVALID_ARG


def test_fold_validates_on_the_host():
    desc = _fill_desc()
    for args, status in (((None, 256, 256, 256, 256), rf.RF_ERR_INVALID_ARG),
                         ((256, 256, 256, None, 256), rf.RF_ERR_INVALID_ARG),
                         ((256, 256, 256, 256, 264), rf.RF_ERR_ALIGN)):
        with pytest.raises(rf.RFError) as ei:
            rf.rf_fold_kv_weights(desc, *args, stream=0)
        assert ei.value.status == status
    rf.rf_fold_kv_weights(_fill_desc(S=8), None, None, None, None, None, stream=0)   # no upper layer: nothing to do


def test_calib_and_xmodel_and_solve_validate_on_the_host():
    with pytest.raises(rf.RFError) as ei:
        rf.rf_calib_accumulate(rf.rf_calib_desc(d_in=100, d_out=256, n_maps=1), 256, 256, 256, 256, 0, 8,
                               rf.calib_stats_struct(256, 256, 256, 256, 256), stream=0)
    assert ei.value.status == rf.RF_ERR_SHAPE
    with pytest.raises(rf.RFError) as ei:
        rf.rf_solve(rf.rf_calib_desc(d_in=256, d_out=256, n_maps=1), rf.calib_stats_struct(256, 256, 256, 256, 256),
                    0.03, 7, 0, 256, 256, workspace=256, workspace_bytes=1 << 30, stream=0)
    assert ei.value.status == rf.RF_ERR_INVALID_ARG
    xd = rf.rf_xmodel_desc(L_src=4, L_tgt=2, k=2, n_kv_heads=2, head_dim=128, N=64, theta_src=1e6, theta_tgt=1e6,
                           pos_offset=0)
    # the source-layer table is a device pointer (its range is checked on the device)
    with pytest.raises(rf.RFError) as ei:
        rf.rf_xmodel_map(xd, None, 256, 256, 256, 256, 256, 256, 256, 256, workspace=256,
                         workspace_bytes=1 << 34, stream=0)
    assert ei.value.status == rf.RF_ERR_INVALID_ARG
    assert "src_layers" in rf.rf_last_error()
    with pytest.raises(rf.RFError) as ei:
        rf.rf_xmodel_map(xd, 256, 256, 256, 256, 256, 256, 256, 264, 256, workspace=256,
                         workspace_bytes=1 << 34, stream=0)
    assert ei.value.status == rf.RF_ERR_ALIGN
    big = rf.rf_xmodel_desc(L_src=4, L_tgt=1 << 13, k=1 << 12, n_kv_heads=2, head_dim=128, N=64, theta_src=1e6,
                            theta_tgt=1e6, pos_offset=0)
    with pytest.raises(rf.RFError) as ei:
        rf.rf_xmodel_map(big, 256, 256, 256, 256, 256, 256, 256, 256, 256, workspace=256, workspace_bytes=1 << 40,
                         stream=0)
    assert ei.value.status == rf.RF_ERR_SHAPE


def test_calib_workspace_is_optional_but_checked_when_given():
    desc = rf.rf_calib_desc(d_in=256, d_out=256, n_maps=1)
    assert rf.rf_calib_workspace_bytes(desc, 1024) == 256
    stats = rf.calib_stats_struct(256, 256, 256, 256, 256)
    with pytest.raises(rf.RFError) as ei:     # too small
        rf.rf_calib_accumulate(desc, 256, 256, 256, 256, 1024 * 256, 1024, stats, None, 256, 128, stream=0)
    assert ei.value.status == rf.RF_ERR_WORKSPACE
    with pytest.raises(rf.RFError) as ei:     # not 256-byte aligned
        rf.rf_calib_accumulate(desc, 256, 256, 256, 256, 1024 * 256, 1024, stats, None, 272, 256, stream=0)
    assert ei.value.status == rf.RF_ERR_WORKSPACE


def test_selftest_mode_is_checked_on_the_host():
    for mode in (-1, 4):
        with pytest.raises(rf.RFError) as ei:
            rf.rf_selftest_wait_timeout(mode, 256, stream=0)
        assert ei.value.status == rf.RF_ERR_INVALID_ARG


def test_value_scale_validates_on_the_host():
    desc = _fill_desc()                       # toy: T = 3
    assert rf.rf_value_scale_workspace_bytes(desc, 0) == 0
    assert rf.rf_value_scale_workspace_bytes(desc, 4) == 0
    assert rf.rf_value_scale_workspace_bytes(desc, 3) > 0
    for c in (0, 4):
        with pytest.raises(rf.RFError) as ei:
            rf.rf_value_scale(desc, c, 256, 256, 256, 256, 256, 256, 256, 256, 256, workspace=256,
                              workspace_bytes=1 << 30, stream=0)
        assert ei.value.status == rf.RF_ERR_INVALID_ARG
    with pytest.raises(rf.RFError) as ei:
        rf.rf_value_scale(desc, 2, 256, 256, None, 256, 256, 256, 256, 256, 256, workspace=256,
                          workspace_bytes=1 << 30, stream=0)
    assert ei.value.status == rf.RF_ERR_INVALID_ARG
    with pytest.raises(rf.RFError) as ei:              # the call folds the gain, so it needs it
        rf.rf_value_scale(desc, 2, 256, 256, 256, 256, 256, 256, None, 256, 256, workspace=256,
                          workspace_bytes=1 << 30, stream=0)
    assert ei.value.status == rf.RF_ERR_INVALID_ARG
    with pytest.raises(rf.RFError) as ei:
        rf.rf_value_scale(desc, 2, 256, 256, 256, 256, 256, 256, 256, 256, 256, workspace=256, workspace_bytes=64,
                          stream=0)
    assert ei.value.status == rf.RF_ERR_WORKSPACE
    pre = _fill_desc(flags=rf.RF_WEIGHTS_PREFOLDED)
    assert rf.rf_value_scale_workspace_bytes(pre, 3) < rf.rf_value_scale_workspace_bytes(desc, 3)
    with pytest.raises(rf.RFError) as ei:              # prefolded: no gain needed, the workspace is checked next
        rf.rf_value_scale(pre, 2, 256, 256, 256, 256, 256, 256, None, 256, 256, workspace=256, workspace_bytes=64,
                          stream=0)
    assert ei.value.status == rf.RF_ERR_WORKSPACE


def test_layered_fill_workspace_and_host_checks():
    desc = _fill_desc(L=10)                         # 6 upper layers
    bf = rf.map_source(rf.RF_MAPS_BF16, 256)
    resident = rf.rf_fill_workspace_bytes(desc)
    inplace = rf.rf_fill_layered_workspace_bytes(desc, bf)
    staged = rf.rf_fill_layered_workspace_bytes(desc, rf.map_source(rf.RF_MAPS_BF16, 256, on_host=True))
    int8_host = rf.rf_fill_layered_workspace_bytes(desc, rf.map_source(rf.RF_MAPS_INT8, 256, on_host=True,
                                                                        row_scale=256))
    assert 0 < inplace < resident                   # x̂ for 4 layers at a time instead of all 6
    r = lambda x: (x + 255) // 256 * 256
    assert staged == inplace + 2 * r(4 * 256 * 256 * 2)  # two bf16 map slots of 4 layers
    assert int8_host == staged + 2 * r(4 * 256 * 256)    # plus two int8 landing slots
    assert rf.rf_fill_layered_workspace_bytes(desc, rf.map_source(7, 256)) == 0
    with pytest.raises(rf.RFError) as ei:
        rf.rf_fill_kv_layered(desc, 256, 256, None, rf.map_source(rf.RF_MAPS_INT8, 256), 256, 256, 256, 256, 256,
                              256, 0, 128, workspace=256, workspace_bytes=1 << 30, stream=0)
    assert ei.value.status == rf.RF_ERR_INVALID_ARG and "row_scale" in rf.rf_last_error()


def test_flag_and_mode_constants_match_header():
    txt = open(os.path.join(ROOT, "include", "rf.h")).read()
    defs = dict(re.findall(r"#define (RF_(?:FLAG|WEIGHTS|SOLVE|MAPS)_\w+) (\d+)u?\b", txt))
    assert {"RF_FLAG_SINGLE_CTA", "RF_FLAG_CTA_PAIR", "RF_WEIGHTS_PREFOLDED", "RF_SOLVE_DIGITS7",
            "RF_MAPS_BF16", "RF_MAPS_INT8"} <= set(defs)
    for name, val in defs.items():
        assert getattr(rf, name) == int(val), name
    flags = [int(defs[n]) for n in defs if not n.startswith("RF_MAPS_")]
    assert all(f & (f - 1) == 0 for f in flags) and len(set(flags)) == len(flags)   # distinct single bits


def test_static_fill_scratch_constant_matches_header():
    txt = open(os.path.join(ROOT, "include", "rf.h")).read()
    assert "RF_STATIC_SCRATCH_BYTES (64u * 1024u * 1024u)" in txt
    assert rf.RF_STATIC_SCRATCH_BYTES == 64 * 1024 * 1024


def _select_desc(**kw):
    d = dict(L_src=6, F=256, n_targets=4, d_out=256, head_dim=128, k=3, n_kinds=2, group=0)
    d.update(kw)
    return rf.rf_select_desc(**d)


def test_select_workspace_size_follows_the_layout():
    base = rf.rf_select_workspace_bytes(_select_desc())
    assert base > 0
    # per-pass buffers scale with the targets per pass; the per-kind Gram does not
    one = rf.rf_select_workspace_bytes(_select_desc(group=1))
    two = rf.rf_select_workspace_bytes(_select_desc(group=2))
    assert 0 < one < two < base
    assert rf.rf_select_workspace_bytes(_select_desc(group=4)) == base
    for bad in (dict(F=100), dict(d_out=300), dict(k=7), dict(n_kinds=3), dict(head_dim=96),
                dict(L_src=300), dict(k=0)):
        assert rf.rf_select_workspace_bytes(_select_desc(**bad)) == 0, bad


def test_select_and_concat_validate_on_the_host():
    st = rf.calib_stats_struct(256, 256, 256, 256, 256, 256)
    no_syy = rf.calib_stats_struct(256, 256, 256, 256, 256)
    d = _select_desc(n_kinds=1)
    wsb = rf.rf_select_workspace_bytes(d)
    cases = [
        (dict(desc=_select_desc(F=100), stats=[st]), rf.RF_ERR_SHAPE),
        (dict(desc=_select_desc(k=9), stats=[st]), rf.RF_ERR_INVALID_ARG),
        (dict(desc=d, stats=[no_syy]), rf.RF_ERR_INVALID_ARG),
        (dict(desc=d, stats=[st], alpha_mode=5), rf.RF_ERR_INVALID_ARG),
        (dict(desc=d, stats=[st], lam=-1.0), rf.RF_ERR_INVALID_ARG),
        (dict(desc=d, stats=[st], workspace_bytes=wsb - 1), rf.RF_ERR_WORKSPACE),
    ]
    for kw, want in cases:
        args = dict(lam=0.01, alpha_mode=rf.RF_ALPHA_TRACE, workspace_bytes=wsb)
        args.update(kw)
        with pytest.raises(rf.RFError) as ei:
            rf.rf_select_sources(args["desc"], args["stats"], args["lam"], args["alpha_mode"], 256, None, None, 256,
                                 args["workspace_bytes"], stream=0)
        assert ei.value.status == want, kw
    with pytest.raises(rf.RFError) as ei:
        rf.rf_concat_layers(256, 3, 1024 * 10, 10, 1024, 8, 128, 1e6, 0, 256, 2048, stream=0)
    assert ei.value.status == rf.RF_ERR_ALIGN
    with pytest.raises(rf.RFError) as ei:
        rf.rf_concat_layers(256, 3, 768 * 10, 10, 768, 8, 96, 1e6, 0, 256, 3 * 768, stream=0)
    assert ei.value.status == rf.RF_ERR_SHAPE
    rf.rf_concat_layers(256, 3, 768 * 10, 0, 768, 8, 96, 0.0, 0, 256, 3 * 768, stream=0)   # no rows: nothing to do
