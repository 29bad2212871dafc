"""ctypes binding of librf.so (include/rf.h). Argument marshalling only.

Functions keep the C names and argument order. Tensor arguments may be torch
tensors (their data_ptr() is passed), plain integers (device addresses) or None
(NULL). ``stream=None`` means torch's current CUDA stream. A status other than
RF_OK raises RFError carrying the status and the library's error text. There is
no fallback: if librf.so has not been built, loading raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_double, c_int, c_int32, c_int64, c_size_t, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "librf.so")

RF_OK = 0
RF_ERR_INVALID_ARG = 1
RF_ERR_SHAPE = 2
RF_ERR_ALIGN = 3
RF_ERR_CUDA = 4
RF_ERR_NOT_SPD = 5
RF_ERR_TIMEOUT = 6
RF_ERR_UNSUPPORTED = 7
RF_ERR_WORKSPACE = 8
RF_ALPHA_TRACE = 0
RF_ALPHA_ABSOLUTE = 1


class RFError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


RF_FLAG_SINGLE_CTA = 1
RF_FLAG_CTA_PAIR = 2
RF_WEIGHTS_PREFOLDED = 4
RF_SOLVE_DIGITS7 = 8


RF_MAPS_BF16 = 0
RF_MAPS_INT8 = 1


class rf_map_source(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("on_host", ctypes.c_int32), ("A", c_void_p), ("row_scale", c_void_p)]


class rf_fill_desc(ctypes.Structure):
    _fields_ = [("d", c_int64), ("L", c_int64), ("S", c_int64), ("N", c_int64), ("T", c_int64),
                ("n_kv_heads", c_int64), ("head_dim", c_int64), ("rope_theta", c_double),
                ("rms_eps", c_double), ("pos_offset", c_int64), ("flags", ctypes.c_uint64),
                ("v_scale", ctypes.c_void_p), ("k_norm_gain", ctypes.c_void_p), ("d_in", c_int64)]


class rf_calib_desc(ctypes.Structure):
    _fields_ = [("d_in", c_int64), ("d_out", c_int64), ("n_maps", c_int64), ("flags", ctypes.c_uint64)]


class rf_calib_stats(ctypes.Structure):
    _fields_ = [("G", c_void_p), ("C", c_void_p), ("sx", c_void_p), ("sy", c_void_p), ("n", c_void_p),
                ("syy", c_void_p)]


class rf_select_desc(ctypes.Structure):
    _fields_ = [("L_src", c_int64), ("F", c_int64), ("n_targets", c_int64), ("d_out", c_int64),
                ("head_dim", c_int64), ("k", c_int64), ("n_kinds", c_int64), ("group", c_int64),
                ("flags", ctypes.c_uint64)]


class rf_xmodel_desc(ctypes.Structure):
    _fields_ = [("L_src", c_int64), ("L_tgt", c_int64), ("k", c_int64), ("n_kv_heads", c_int64),
                ("head_dim", c_int64), ("N", c_int64), ("theta_src", c_double), ("theta_tgt", c_double),
                ("pos_offset", c_int64), ("flags", ctypes.c_uint64)]


_SIGS = {
    "rf_version": (c_int, []),
    "rf_status_string": (c_char_p, [c_int]),
    "rf_last_error": (c_char_p, []),
    "rf_device_supported": (c_int, [c_int]),
    "rf_set_wait_timeout_ms": (None, [c_int64]),
    "rf_profile_start": (c_int, [c_int]),
    "rf_profile_stop": (c_int, [POINTER(c_int32), POINTER(ctypes.c_float), c_int]),
    "rf_stage_name": (c_char_p, [c_int]),
    "rf_fill_workspace_bytes": (c_size_t, [POINTER(rf_fill_desc)]),
    "rf_fold_kv_weights": (c_int, [POINTER(rf_fill_desc), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                   c_void_p]),
    "rf_fill_kv": (c_int, [POINTER(rf_fill_desc), c_void_p, c_int64, c_void_p, c_void_p, c_void_p, c_void_p,
                           c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_void_p, c_void_p, c_void_p,
                           c_size_t, c_void_p]),
    "rf_fill_kv_static": (c_int, [POINTER(rf_fill_desc), c_void_p, c_int64, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_void_p,
                                  c_void_p, c_void_p]),
    "rf_selftest_wait_timeout": (c_int, [c_int, c_void_p, c_void_p]),
    "rf_quantize_maps_int8": (c_int, [POINTER(rf_fill_desc), c_void_p, c_void_p, c_void_p, c_void_p]),
    "rf_fill_layered_workspace_bytes": (c_size_t, [POINTER(rf_fill_desc), POINTER(rf_map_source)]),
    "rf_fill_kv_layered": (c_int, [POINTER(rf_fill_desc), c_void_p, c_int64, c_void_p, POINTER(rf_map_source),
                                   c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int64,
                                   c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "rf_value_scale_workspace_bytes": (c_size_t, [POINTER(rf_fill_desc), c_int64]),
    "rf_value_scale": (c_int, [POINTER(rf_fill_desc), c_int64, c_void_p, c_int64, c_void_p, c_int64, c_void_p,
                               c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "rf_calib_workspace_bytes": (c_size_t, [POINTER(rf_calib_desc), c_int64]),
    "rf_calib_accumulate": (c_int, [POINTER(rf_calib_desc), c_void_p, c_int64, c_void_p, c_int64, c_int64,
                                    c_int64, POINTER(rf_calib_stats), c_void_p, c_void_p, c_size_t, c_void_p]),
    "rf_solve_workspace_bytes": (c_size_t, [POINTER(rf_calib_desc)]),
    "rf_solve": (c_int, [POINTER(rf_calib_desc), POINTER(rf_calib_stats), c_double, c_int, c_int, c_void_p,
                         c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "rf_xmodel_workspace_bytes": (c_size_t, [POINTER(rf_xmodel_desc)]),
    "rf_xmodel_map": (c_int, [POINTER(rf_xmodel_desc), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                              c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "rf_rope_rows": (c_int, [c_void_p, c_void_p, c_int64, c_int64, c_int64, c_int64, c_double, c_int64, c_int,
                             c_void_p]),
    "rf_concat_layers": (c_int, [c_void_p, c_int64, c_int64, c_int64, c_int64, c_int64, c_int64, c_double,
                                 c_int64, c_void_p, c_int64, c_void_p]),
    "rf_select_workspace_bytes": (c_size_t, [POINTER(rf_select_desc)]),
    "rf_select_sources": (c_int, [POINTER(rf_select_desc), POINTER(rf_calib_stats), c_double, c_int, c_void_p,
                                  c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Loads librf.so once. Raises if it is missing or lacks a declared symbol."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"librf.so is not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name, None)
            if f is None:
                continue
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _p(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, fn: str):
    if st != RF_OK:
        L = lib()
        raise RFError(st, f"{fn}: {L.rf_status_string(st).decode()}: {L.rf_last_error().decode()}")


# ---------------------------------------------------------------- library-wide
def rf_version() -> int:
    return lib().rf_version()


def rf_status_string(status: int) -> str:
    return lib().rf_status_string(status).decode()


def rf_last_error() -> str:
    return lib().rf_last_error().decode()


def rf_device_supported(device: int = 0) -> bool:
    return bool(lib().rf_device_supported(device))


def rf_set_wait_timeout_ms(ms: int) -> None:
    lib().rf_set_wait_timeout_ms(int(ms))


def rf_profile_start(max_records: int) -> None:
    _check(lib().rf_profile_start(int(max_records)), "rf_profile_start")


def rf_profile_stop(capacity: int = 1 << 16):
    """Returns a list of (stage name, milliseconds) in launch order."""
    ids = (c_int32 * capacity)()
    ms = (ctypes.c_float * capacity)()
    n = lib().rf_profile_stop(ids, ms, capacity)
    if n < 0:
        raise RFError(RF_ERR_CUDA, "rf_profile_stop: CUDA error while reading events")
    L = lib()
    return [(L.rf_stage_name(ids[i]).decode(), float(ms[i])) for i in range(n)]


def rf_stage_name(stage_id: int) -> str:
    return lib().rf_stage_name(int(stage_id)).decode()


# ------------------------------------------------------------------------ fill
def rf_fill_workspace_bytes(desc: rf_fill_desc) -> int:
    return int(lib().rf_fill_workspace_bytes(ctypes.byref(desc)))


def rf_fold_kv_weights(desc, gain, Wk, Wv, Wk_folded, Wv_folded, stream=None):
    _check(lib().rf_fold_kv_weights(ctypes.byref(desc), _p(gain), _p(Wk), _p(Wv), _p(Wk_folded), _p(Wv_folded),
                                    _s(stream)), "rf_fold_kv_weights")


def rf_fill_kv(desc, x_S, ld_x, exact_mask, A, b, gain, Wk, Wv, k_cache, v_cache, layer_stride, row_stride,
               n_fill_out=None, dev_status=None, workspace=None, workspace_bytes=0, stream=None):
    """The fill; with RF_WEIGHTS_PREFOLDED in desc.flags, Wk and Wv hold the gain and ``gain`` may be None."""
    _check(lib().rf_fill_kv(ctypes.byref(desc), _p(x_S), int(ld_x), _p(exact_mask), _p(A), _p(b), _p(gain), _p(Wk),
                            _p(Wv), _p(k_cache), _p(v_cache), int(layer_stride), int(row_stride), _p(n_fill_out),
                            _p(dev_status), _p(workspace), int(workspace_bytes), _s(stream)), "rf_fill_kv")


RF_STATIC_SCRATCH_BYTES = 64 * 1024 * 1024


def rf_fill_kv_static(desc, x_S, ld_x, exact_mask, A, b, gain, Wk, Wv, k_cache, v_cache, layer_stride, row_stride,
                      n_fill_out=None, dev_status=None, stream=None):
    """rf_fill_kv for callers that cannot allocate device memory: the library's own
    fixed 64 MiB device array serves as scratch (see include/rf.h)."""
    _check(lib().rf_fill_kv_static(ctypes.byref(desc), _p(x_S), int(ld_x), _p(exact_mask), _p(A), _p(b), _p(gain),
                                   _p(Wk), _p(Wv), _p(k_cache), _p(v_cache), int(layer_stride), int(row_stride),
                                   _p(n_fill_out), _p(dev_status), _s(stream)), "rf_fill_kv_static")


def rf_selftest_wait_timeout(mode, dev_status, stream=None):
    """Runs the GEMM core on a problem whose copies never arrive: *dev_status becomes
    RF_ERR_TIMEOUT after the wait limit. mode bit 0: CTA pair; bit 1: dynamic unit order."""
    _check(lib().rf_selftest_wait_timeout(int(mode), _p(dev_status), _s(stream)), "rf_selftest_wait_timeout")


def rf_quantize_maps_int8(desc, A, q, s, stream=None):
    """Symmetric per-row int8 code of the maps: q [P][d][d_in] int8, s [P][d] fp32."""
    _check(lib().rf_quantize_maps_int8(ctypes.byref(desc), _p(A), _p(q), _p(s), _s(stream)), "rf_quantize_maps_int8")


def map_source(kind, A, on_host=False, row_scale=None) -> rf_map_source:
    """rf_map_source for maps A (a device or host tensor, or an address)."""
    return rf_map_source(int(kind), int(bool(on_host)), _p(A), _p(row_scale))


def rf_fill_layered_workspace_bytes(desc, maps) -> int:
    return int(lib().rf_fill_layered_workspace_bytes(ctypes.byref(desc), ctypes.byref(maps)))


def rf_fill_kv_layered(desc, x_S, ld_x, exact_mask, maps, b, gain, Wk, Wv, k_cache, v_cache, layer_stride,
                       row_stride, n_fill_out=None, dev_status=None, workspace=None, workspace_bytes=0, stream=None):
    """rf_fill_kv one layer at a time, maps from the device or the host, bf16 or int8 (see include/rf.h)."""
    _check(lib().rf_fill_kv_layered(ctypes.byref(desc), _p(x_S), int(ld_x), _p(exact_mask), ctypes.byref(maps),
                                    _p(b), _p(gain), _p(Wk), _p(Wv), _p(k_cache), _p(v_cache), int(layer_stride),
                                    int(row_stride),
                                    _p(n_fill_out), _p(dev_status), _p(workspace), int(workspace_bytes),
                                    _s(stream)), "rf_fill_kv_layered")


def rf_value_scale_workspace_bytes(desc: rf_fill_desc, c: int) -> int:
    return int(lib().rf_value_scale_workspace_bytes(ctypes.byref(desc), int(c)))


def rf_value_scale(desc, c, x_S, ld_x, x_exact, ld_e, A, b, gain, Wv, v_scale, dev_status=None, workspace=None,
                   workspace_bytes=0, stream=None):
    """Per-(layer, KV head) value-rescale factors into v_scale [P][H] fp32 (see include/rf.h)."""
    _check(lib().rf_value_scale(ctypes.byref(desc), int(c), _p(x_S), int(ld_x), _p(x_exact), int(ld_e), _p(A), _p(b),
                                _p(gain), _p(Wv), _p(v_scale), _p(dev_status), _p(workspace), int(workspace_bytes),
                                _s(stream)), "rf_value_scale")


# ----------------------------------------------------------------- calibration
def rf_calib_workspace_bytes(desc: rf_calib_desc, n_rows: int) -> int:
    return int(lib().rf_calib_workspace_bytes(ctypes.byref(desc), int(n_rows)))


def calib_stats_struct(G, C, sx, sy, n, syy=None) -> rf_calib_stats:
    return rf_calib_stats(_p(G), _p(C), _p(sx), _p(sy), _p(n), _p(syy))


def rf_calib_accumulate(desc, X, ld_x, Y, ld_y, y_map_stride, n_rows, stats, dev_status=None,
                        workspace=None, workspace_bytes=0, stream=None):
    _check(lib().rf_calib_accumulate(ctypes.byref(desc), _p(X), int(ld_x), _p(Y), int(ld_y), int(y_map_stride),
                                     int(n_rows), ctypes.byref(stats), _p(dev_status), _p(workspace),
                                     int(workspace_bytes), _s(stream)), "rf_calib_accumulate")


# ----------------------------------------------------------------------- solve
def rf_solve_workspace_bytes(desc: rf_calib_desc) -> int:
    return int(lib().rf_solve_workspace_bytes(ctypes.byref(desc)))


def rf_solve(desc, stats, lam, alpha_mode, refine_iters, A, b, A_bf16=None, alpha_out=None, dev_status=None,
             workspace=None, workspace_bytes=0, stream=None):
    _check(lib().rf_solve(ctypes.byref(desc), ctypes.byref(stats), float(lam), int(alpha_mode), int(refine_iters),
                          _p(A), _p(b), _p(A_bf16), _p(alpha_out), _p(dev_status), _p(workspace),
                          int(workspace_bytes), _s(stream)), "rf_solve")


# ------------------------------------------------------------------ cross-model
def rf_xmodel_workspace_bytes(desc: rf_xmodel_desc) -> int:
    return int(lib().rf_xmodel_workspace_bytes(ctypes.byref(desc)))


def rf_xmodel_map(desc, src_layers, k_src, v_src, Wk, bk, Wv, bv, k_tgt, v_tgt, dev_status=None,
                  workspace=None, workspace_bytes=0, stream=None):
    """``src_layers``: device int32 tensor [L_tgt][k] (e.g. rf_select_sources' output)."""
    _check(lib().rf_xmodel_map(ctypes.byref(desc), _p(src_layers), _p(k_src), _p(v_src),
                               _p(Wk), _p(bk), _p(Wv), _p(bv), _p(k_tgt), _p(v_tgt), _p(dev_status),
                               _p(workspace), int(workspace_bytes), _s(stream)), "rf_xmodel_map")


def rf_rope_rows(inp, out, n_rows, ld, n_heads, head_dim, theta, pos_offset=0, inverse=False, stream=None):
    _check(lib().rf_rope_rows(_p(inp), _p(out), int(n_rows), int(ld), int(n_heads), int(head_dim), float(theta),
                              int(pos_offset), 1 if inverse else 0, _s(stream)), "rf_rope_rows")


def rf_concat_layers(src, n_layers, layer_stride, n_rows, ld_src, n_heads, head_dim, theta, pos_offset, out, ld_out,
                     stream=None):
    """out[t][l*W + j] = (inverse RoPE if theta > 0 else identity)(src[l][t][j]); see include/rf.h."""
    _check(lib().rf_concat_layers(_p(src), int(n_layers), int(layer_stride), int(n_rows), int(ld_src), int(n_heads),
                                  int(head_dim), float(theta), int(pos_offset), _p(out), int(ld_out), _s(stream)),
           "rf_concat_layers")


def rf_select_workspace_bytes(desc: rf_select_desc) -> int:
    return int(lib().rf_select_workspace_bytes(ctypes.byref(desc)))


def rf_select_sources(desc, stats, lam, alpha_mode, src_layers, r2=None, dev_status=None, workspace=None,
                      workspace_bytes=0, stream=None):
    """Greedy source-layer selection; ``stats`` is a sequence of n_kinds rf_calib_stats."""
    arr = (rf_calib_stats * len(stats))(*stats)
    _check(lib().rf_select_sources(ctypes.byref(desc), arr, float(lam), int(alpha_mode), _p(src_layers), _p(r2),
                                   _p(dev_status), _p(workspace), int(workspace_bytes), _s(stream)),
           "rf_select_sources")
