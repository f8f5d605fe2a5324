"""CPU oracle of the deterministic MoE layer (fp64) -- test infrastructure.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg may import
this module. It loads `liboracle.so`, compiled from `oracle.c` with gcc, and wraps its
functions for numpy arrays. It shares no code with the CUDA path.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRC = [os.path.join(_HERE, "oracle.c"), os.path.join(_HERE, "oracle.h")]
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so (plain C, OpenMP) if it is missing or older than its sources."""
    stale = force or not os.path.exists(_SO) or any(
        os.path.getmtime(s) > os.path.getmtime(_SO) for s in _SRC)
    if stale:
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC[0], "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        i64, i32, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        L.oracle_route.argtypes = [i64, i32, i32, p, p, p]
        L.oracle_schedule.argtypes = [i64, i32, i64, p, p, p, p, p, p, i64, p]
        L.oracle_schedule.restype = ctypes.c_int
        L.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        L.oracle_e4m3_encode.restype = ctypes.c_uint8
        L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_decode.restype = ctypes.c_double
        L.oracle_mxfp8_quantize.argtypes = [i64, i64, p, p, p]
        L.oracle_mxfp8_dequantize.argtypes = [i64, i64, p, p, p]
        L.oracle_mxfp8_quantize_bf16.argtypes = [i64, i64, p, p, p]
        L.oracle_forward.argtypes = [i64, i32, i32, i32, i32, p, p, p, i32, p, p, p, p, i32,
                                     i32, p, p, p]
        L.oracle_backward.argtypes = [i64, i32, i32, i32, i32, p, p, p, i32, p, p, p, p, i32,
                                      i32, p, p, p, p, p, p, p, p, p, p, p, p]
        L.oracle_mxfp8_qdq_slack.argtypes = [i64, p, p, p, p, p, p]
        L.oracle_bf16_slack.argtypes = [ctypes.c_double, ctypes.c_double]
        L.oracle_bf16_slack.restype = ctypes.c_double
        L.oracle_round_bf16.argtypes = [ctypes.c_double]
        L.oracle_round_bf16.restype = ctypes.c_double
        L.oracle_dot_rel_rows.argtypes = [i64]
        L.oracle_dot_rel_rows.restype = ctypes.c_double
        L.oracle_router_grad.argtypes = [i64, i32, i32, p, p, p, p]
        L.oracle_router_grad_slack.argtypes = [i64, i32, i32, p, p, p, p]
        _lib = L
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def bf16_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# ------------------------------------------------------------------------- steps

def route(logits, K):
    """Top-k routing: (idx int32 [T,K], w float64 [T,K])."""
    lg = _f64(logits)
    T, E = lg.shape
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float64)
    lib().oracle_route(T, E, K, _p(lg), _p(idx), _p(w))
    return idx, w


def schedule(idx, E, MB, seg_cap=None):
    """Stable expert schedule: dict of counts, offsets, perm, inv, segs [n,3]."""
    f = _i32(idx).reshape(-1)
    R = f.size
    if seg_cap is None:
        seg_cap = E + (R + MB - 1) // MB if R > 0 else 1
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(max(R, 1), np.int32)
    inv = np.empty(max(R, 1), np.int32)
    segs = np.empty((max(seg_cap, 1), 3), np.int32)
    n = np.zeros(1, np.int32)
    rc = lib().oracle_schedule(R, E, MB, _p(f), _p(counts), _p(offsets), _p(perm), _p(inv),
                               _p(segs), seg_cap, _p(n))
    if rc != 0:
        raise ValueError("segment capacity exceeded")
    return dict(counts=counts, offsets=offsets, perm=perm[:R], inv=inv[:R],
                segs=segs[: int(n[0])].copy())


def e4m3_encode(v: float) -> int:
    return int(lib().oracle_e4m3_encode(float(v)))


def e4m3_decode(code: int) -> float:
    return float(lib().oracle_e4m3_decode(int(code)))


def mxfp8_quantize(src):
    """MXFP8 along the last axis: (q uint8 [rows,cols], scale uint8 [rows,cols/32])."""
    s = _f64(src)
    rows, cols = s.reshape(-1, s.shape[-1]).shape
    assert cols % 32 == 0
    q = np.empty((rows, cols), np.uint8)
    sc = np.empty((rows, cols // 32), np.uint8)
    lib().oracle_mxfp8_quantize(rows, cols, _p(s), _p(q), _p(sc))
    return q.reshape(s.shape), sc.reshape(s.shape[:-1] + (cols // 32,))


def mxfp8_dequantize(q, scale):
    q = np.ascontiguousarray(q, np.uint8)
    sc = np.ascontiguousarray(scale, np.uint8)
    cols = q.shape[-1]
    rows = q.size // cols
    out = np.empty(q.shape, np.float64)
    lib().oracle_mxfp8_dequantize(rows, cols, _p(q), _p(sc), _p(out))
    return out


W_F64, W_BF16, W_MXFP8 = 0, 1, 2
EXACT, BF16, MXFP8 = 0, 1, 2  # operand precision modes
STORE_F32, STORE_BF16 = 0, 1  # storage of the values that are only stored (oracle.h)
DOT_REL = 2.0 ** -19          # ORACLE_DOT_REL: fp32 dot-product error bound / sum|terms|
SLACK_REL = 2.0 ** -20        # ORACLE_SLACK_REL: elementwise fp32 error bound / |value|
SUM_ULP = 2.0 ** -24          # ORACLE_SUM_ULP: fp32 unit roundoff


class _Rows(ctypes.Structure):
    """oracle_rows: optional per-routed-row intermediates (oracle.h)."""
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "a", "a_mag", "a_slack", "h", "h_slack", "h_q", "h_scale", "da", "da_slack", "sh",
        "sh_slack", "da_q", "da_scale", "daq_slack", "dtopk_slack", "h_in", "a_in", "da_in",
        "sh_in", "daq_in", "y_in", "dx_in")]


_INPUTS = ("h_in", "a_in", "da_in", "sh_in", "daq_in", "y_in", "dx_in")


def _rows(R, I, names, mx, given=None):
    """numpy arrays for the requested intermediates and the struct pointing at them; `given`
    maps *_in names to arrays of given intermediates (kept alive in the returned dict)."""
    shapes = dict(a=(R, 2 * I, np.float64), a_mag=(R, 2 * I, np.float64),
                  a_slack=(R, 2 * I, np.float64), h=(R, I, np.float64),
                  h_slack=(R, I, np.float64), h_q=(R, I, np.uint8),
                  h_scale=(R, I // 32, np.uint8), da=(R, 2 * I, np.float64),
                  da_slack=(R, 2 * I, np.float64), sh=(R, I, np.float64),
                  sh_slack=(R, I, np.float64), da_q=(R, 2 * I, np.uint8),
                  da_scale=(R, 2 * I // 32, np.uint8), daq_slack=(R, 2 * I, np.float64),
                  dtopk_slack=(R, 1, np.float64))
    out = {}
    st = _Rows()
    for n in names:
        r, c, dt = shapes[n]
        a = np.zeros((max(r, 1), c), dt)
        out[n] = a
        setattr(st, n, a.ctypes.data)
    keep = {}
    for n, v in (given or {}).items():
        assert n in _INPUTS, n
        if n in ("y_in", "dx_in"):  # [T][H], per token
            a = np.ascontiguousarray(v, np.float64)
            keep[n] = a
            setattr(st, n, a.ctypes.data)
            continue
        want = 2 * I if n in ("a_in", "da_in", "daq_in") else I
        a = np.ascontiguousarray(v, np.float64).reshape(R, want)
        keep[n] = a
        setattr(st, n, a.ctypes.data)
    return (out, keep), st


def mxfp8_qdq_slack(v, err):
    """MXFP8 quantize-dequantize along the last axis of v, each value known to within err:
    (dequantized, slack, q, scale) -- oracle_mxfp8_qdq_slack row by row."""
    v = _f64(v)
    err = np.broadcast_to(_f64(err), v.shape).copy()
    n = v.shape[-1]
    assert n % 32 == 0
    rows = v.size // n
    out = np.empty(v.shape, np.float64)
    sl = np.empty(v.shape, np.float64)
    q = np.empty(v.shape, np.uint8)
    sc = np.empty(v.shape[:-1] + (n // 32,), np.uint8)
    for r in range(rows):
        o = r * n
        lib().oracle_mxfp8_qdq_slack(
            n, v.ctypes.data + 8 * o, err.ctypes.data + 8 * o, out.ctypes.data + 8 * o,
            sl.ctypes.data + 8 * o, q.ctypes.data + o, sc.ctypes.data + (o // 32))
    return out, sl, q, sc


def round_bf16(v: float) -> float:
    return float(lib().oracle_round_bf16(float(v)))


def dot_rel_rows(n: int) -> float:
    """The oracle's fp32 error bound, relative to sum|terms|, of a weight gradient summed
    over n rows (oracle_dot_rel_rows)."""
    return float(lib().oracle_dot_rel_rows(int(n)))


def _weights(w):
    """(kind, data, scale) of a weight tensor: float arrays are widened to float64, uint16
    arrays are bf16 bit patterns, a (q, scale) pair of uint8 arrays is MXFP8."""
    if isinstance(w, tuple):
        q, s = np.ascontiguousarray(w[0], np.uint8), np.ascontiguousarray(w[1], np.uint8)
        return W_MXFP8, q, s, q.shape
    if w.dtype == np.uint16:
        w = np.ascontiguousarray(w)
        return W_BF16, w, None, w.shape
    w = _f64(w)
    return W_F64, w, None, w.shape


def bf16_slack(v: float, err: float = 0.0) -> float:
    """Slack of rounding v to bf16 when the value is only known to within err."""
    return float(lib().oracle_bf16_slack(float(v), float(err)))


def forward(x, idx, w, w13, w2, mode=EXACT, with_slack=False, store=STORE_F32, rows=(),
            given=None):
    """Layer forward in fp64: y [T,H], with the operand rounding of `mode` (EXACT, BF16 or
    MXFP8) and the storage rounding of `store` (STORE_F32 or STORE_BF16). Weights as
    described in _weights (both of the same kind). With with_slack, returns (y, slack): the
    per-element bound on how far a correct result may lie from y because of rounding
    decisions taken on values within fp32 error of a midpoint. `rows` names per-routed-row
    intermediates (oracle_rows fields: a, a_mag, h, h_slack, h_q, h_scale) to return as a
    dict after the other results; `given` = {"h_in": [T*K, I]} feeds the down GEMM the
    given h (rows in flat id order t*K + k) instead of the oracle's own, and {"y_in": [T, H]}
    adds the expert outputs to y_in (see oracle_rows)."""
    x, w = _f64(x), _f64(w)
    idx = _i32(idx)
    k13, d13, s13, sh13 = _weights(w13)
    k2, d2, s2, _ = _weights(w2)
    assert k13 == k2
    T, H = x.shape
    E, I2, _ = sh13
    K = idx.shape[1]
    y = np.empty((T, H), np.float64)
    sl = np.empty((T, H), np.float64) if with_slack else None
    (rv, _keep), rs = _rows(T * K, I2 // 2, rows, mode == MXFP8, given)
    lib().oracle_forward(T, H, I2 // 2, E, K, _p(x), _p(idx), _p(w), k13, _p(d13),
                         None if s13 is None else _p(s13), _p(d2),
                         None if s2 is None else _p(s2), int(mode), int(store), _p(y),
                         None if sl is None else _p(sl),
                         ctypes.addressof(rs) if (rows or given) else None)
    out = (y, sl) if with_slack else (y,)
    if rows:
        out = out + (rv,)
    return out if len(out) > 1 else out[0]


def quantize_transposed_bf16(bits):
    """MXFP8 codes and scales of the transpose of each [rows][cols] matrix of `bits` (bf16
    patterns [E][rows][cols]), quantized along its rows: (q [E][cols][rows],
    scale [E][cols][rows/32]) -- the oracle's row quantizer on an explicit transpose."""
    return mxfp8_quantize_bf16(np.ascontiguousarray(np.swapaxes(bits, -1, -2)))


def backward(x, idx, w, w13, w2, dy, weight_grads=True, mode=EXACT, with_slack=False,
             store=STORE_F32, rows=(), given=None, mx_weights=None):
    """Layer backward in fp64: (dx, dw13, dw2, dtopk), with the operand rounding of `mode`
    (EXACT, BF16 or MXFP8) and the storage rounding of `store`; dw13/dw2 are None when
    weight_grads is False. With with_slack, also the slacks of dx, dw13, dw2 (see forward).
    `rows` names per-routed-row intermediates (a, a_slack, da, da_slack, sh, sh_slack,
    da_q, da_scale, daq_slack) to return as a dict after the other results; `given` maps
    a_in, da_in, sh_in, daq_in to arrays ([T*K, 2I] or [T*K, I], flat id order) that replace
    the oracle's own values where they enter the next step, and dx_in [T, H] to a dx that
    the results are added to (see oracle_rows).

    In MXFP8 mode w13 and w2 are the bf16 weights (uint16 bit patterns). A is recomputed
    with the forward's operands (x and W13 quantized along H); G uses dy and W2 quantized
    along H; dgrad uses dA and W13 quantized along 2I; the weight gradients use bf16 dA
    and w*h. mx_weights may give those three quantizations, as made by this module
    (mxfp8_quantize_bf16(w13), quantize_transposed_bf16(w13), quantize_transposed_bf16(w2)),
    so that a caller running many backward calls on the same weights computes them once."""
    x, w, dy = _f64(x), _f64(w), _f64(dy)
    idx = _i32(idx)
    mxw = (None,) * 4
    s13 = None
    if mode == MXFP8:
        assert w13.dtype == np.uint16 and w2.dtype == np.uint16
        if mx_weights is None:
            mx_weights = (mxfp8_quantize_bf16(w13), quantize_transposed_bf16(w13),
                          quantize_transposed_bf16(w2))
        w13, w13t, w2t = mx_weights               # W13 along H; W13 along 2I; W2 along H
        mxw = tuple(np.ascontiguousarray(a, np.uint8) for a in (*w13t, *w2t))
    k13, d13, s13, sh13 = _weights(w13)
    k2, d2, _, sh2 = _weights(w2)
    assert k2 != W_MXFP8 and (k13 != W_MXFP8 or mode == MXFP8)
    T, H = x.shape
    E, I2, _ = sh13
    K = idx.shape[1]
    dx = np.empty((T, H), np.float64)
    dw13 = np.empty(sh13, np.float64) if weight_grads else None
    dw2 = np.empty(sh2, np.float64) if weight_grads else None
    dtopk = np.empty((T, K), np.float64)
    sdx = np.empty((T, H), np.float64) if with_slack else None
    sdw13 = np.empty(sh13, np.float64) if (with_slack and weight_grads) else None
    sdw2 = np.empty(sh2, np.float64) if (with_slack and weight_grads) else None
    (rv, _keep), rs = _rows(T * K, I2 // 2, rows, mode == MXFP8, given)
    n = lambda a: None if a is None else _p(a)  # noqa: E731
    lib().oracle_backward(T, H, I2 // 2, E, K, _p(x), _p(idx), _p(w), k13, _p(d13), n(s13),
                          _p(d2), _p(dy), int(mode), int(store), *(n(a) for a in mxw), _p(dx),
                          n(dw13), n(dw2), _p(dtopk), n(sdx), n(sdw13), n(sdw2),
                          ctypes.addressof(rs) if (rows or given) else None)
    out = (dx, dw13, dw2, dtopk)
    if with_slack:
        out = out + (sdx, sdw13, sdw2)
    if rows:
        out = out + (rv,)
    return out


def mxfp8_qdq_axis_bf16(bits, axis):
    """MXFP8 quantize-dequantize of bf16 bit patterns in 32-element blocks along `axis`
    (the oracle's row quantizer applied to that axis moved last): float64, same shape."""
    b = np.moveaxis(np.asarray(bits, np.uint16), axis, -1)
    q, sc = mxfp8_quantize_bf16(np.ascontiguousarray(b))
    return np.ascontiguousarray(np.moveaxis(mxfp8_dequantize(q, sc), -1, axis))


def mxfp8_quantize_bf16(bits):
    """MXFP8 of bf16 bit patterns along the last axis: (q, scale)."""
    b = np.ascontiguousarray(bits, np.uint16)
    cols = b.shape[-1]
    rows = b.size // cols
    q = np.empty(b.shape, np.uint8)
    sc = np.empty(b.shape[:-1] + (cols // 32,), np.uint8)
    lib().oracle_mxfp8_quantize_bf16(rows, cols, _p(b), _p(q), _p(sc))
    return q, sc


def router_grad(idx, w, dtopk, E):
    idx, w, dtopk = _i32(idx), _f64(w), _f64(dtopk)
    T, K = idx.shape
    dl = np.empty((T, E), np.float64)
    lib().oracle_router_grad(T, E, K, _p(idx), _p(w), _p(dtopk), _p(dl))
    return dl



def router_grad_slack(idx, w, sdtopk, E):
    """Slack of router_grad's logit gradients given the slack of each dS (oracle.h)."""
    idx, w, sdtopk = _i32(idx), _f64(w), _f64(sdtopk)
    T, K = idx.shape
    sl = np.empty((T, E), np.float64)
    lib().oracle_router_grad_slack(T, E, K, _p(idx), _p(w), _p(sdtopk), _p(sl))
    return sl
