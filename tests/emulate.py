"""A numpy/torch stand-in for a kernel that is allowed to err within the oracle's fp32 bounds.

Test infrastructure for the slack pins: it recomputes the layer with its own code (numpy
matmuls, torch's bf16 and float8 conversions, a quantizer written here), and perturbs every
value that a GPU kernel computes in fp32 by a random amount inside the bound the oracle
assumes for it (oracle.h): dot products by up to DOT_REL * sum|terms|, elementwise results
by up to SLACK_REL * |value|, the fp32 k-sums by fp32 arithmetic itself. Every rounding
happens where the layer's definition puts it. Each draw is therefore one result that a
correct kernel could produce; the oracle's slack must cover all of them.
"""
import numpy as np
import torch

import oracle

DOT_REL, SLACK_REL = oracle.DOT_REL, oracle.SLACK_REL


def bf16(v):
    """fp32 value -> bf16 (round to nearest even), as a float64 array; the input is first
    rounded to fp32, as a kernel holds it."""
    t = torch.from_numpy(np.ascontiguousarray(v, np.float64)).float().to(torch.bfloat16)
    return t.double().numpy()


def mx_qdq_rows(v):
    """MXFP8 quantize-dequantize along the last axis, written from the OCP MX rule: scale
    2^(floor(log2 amax) - 8) per 32 elements (clamped to [2^-127, 2^127]), E4M3 codes by
    torch's float8_e4m3fn conversion of values clipped to +-448."""
    v = np.asarray(v, np.float64)
    blk = v.reshape(v.shape[:-1] + (v.shape[-1] // 32, 32))
    amax = np.abs(blk).max(-1, keepdims=True)
    _, ex = np.frexp(amax)
    s = np.where(amax > 0, np.clip(ex - 1 - 8, -127, 127), -127)
    u = np.clip(np.ldexp(blk, -s), -448.0, 448.0)
    q = torch.from_numpy(u).float().to(torch.float8_e4m3fn).double().numpy()
    return np.ldexp(q, s).reshape(v.shape)


def _silu(z):
    return z / (1.0 + np.exp(-z))


def _dsilu(z):
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def _dot(rng, A, B):
    """A @ B with each result moved by up to DOT_REL * sum|terms| (the tensor-core bound)."""
    exact = A @ B
    mag = np.abs(A) @ np.abs(B)
    return exact + DOT_REL * mag * rng.uniform(-1.0, 1.0, exact.shape)


def _elem(rng, v):
    return v * (1.0 + 0.9 * SLACK_REL * rng.uniform(-1.0, 1.0, np.shape(v)))


def forward(rng, x, idx, w, w13, w2, mode, h_in=None, y_in=None):
    """One possible kernel result of the forward with bf16 storage: (y [T, H], h [T*K, I]),
    h as it entered the down GEMM (rows in flat id order t*K + k). With h_in, that h is
    used instead of computing one; with y_in, the weighted expert outputs are added to y_in
    in fp32 with no bf16 slot in between (an expert added to an existing output)."""
    T, H = x.shape
    K = idx.shape[1]
    I = w13.shape[1] // 2
    xa = mx_qdq_rows(x) if mode == oracle.MXFP8 else x
    y = np.zeros((T, H), np.float32) if y_in is None else np.asarray(y_in, np.float32)
    hs = np.zeros((T * K, I))
    for k in range(K):
        o = np.empty((T, H))
        for t in range(T):
            e = idx[t, k]
            if h_in is None:
                a = _dot(rng, w13[e], xa[t])
                h = _elem(rng, _silu(a[:I]) * a[I:])
                h = mx_qdq_rows(h) if mode == oracle.MXFP8 else bf16(h)
            else:
                h = h_in[t * K + k]
            hs[t * K + k] = h
            o[t] = _dot(rng, w2[e], h)
            if y_in is None:
                o[t] = bf16(o[t])                       # the (token, k) slot
        y = y + (w[:, k:k + 1].astype(np.float32) * o.astype(np.float32))  # fp32, k ascending
    return bf16(y), hs


def backward(rng, x, idx, w, w13, w2, dy, mode, given=None, dx_in=None):
    """One possible kernel result of the backward with bf16 storage: dx, dw13, dw2 and a
    dict of the intermediates (rows in flat id order): a (saved A), da, sh (bf16), daq
    (MXFP8: dequantized dgrad operand), slot (each slot's bf16 dgrad result). `given` may hold a_in, da_in, sh_in, daq_in to use
    instead of computing them. With dx_in, each dgrad result is added to dx_in in fp32 with
    no bf16 slot in between."""
    given = given or {}
    T, H = x.shape
    K = idx.shape[1]
    E, I2, _ = w13.shape
    I = I2 // 2
    mx = mode == oracle.MXFP8
    qcols = lambda m: np.swapaxes(mx_qdq_rows(np.swapaxes(m, -1, -2)), -1, -2)  # noqa: E731
    w13a = mx_qdq_rows(w13) if mx else w13       # the forward's W13 (along H)
    w13d = qcols(w13) if mx else w13             # dgrad's W13 (along 2I)
    w2g = qcols(w2) if mx else w2                # G's W2 (along H)
    xa = mx_qdq_rows(x) if mx else x
    dyg = mx_qdq_rows(dy) if mx else dy
    dx = np.zeros((T, H), np.float32) if dx_in is None else np.asarray(dx_in, np.float32)
    rows = dict(a=np.zeros((T * K, I2)), da=np.zeros((T * K, I2)), sh=np.zeros((T * K, I)),
                daq=np.zeros((T * K, I2)), slot=np.zeros((T * K, H)))
    for k in range(K):
        xs = np.empty((T, H))
        for t in range(T):
            f = t * K + k
            e, s = idx[t, k], w[t, k]
            if "a_in" in given:
                a = given["a_in"][f]
            else:
                a = bf16(_dot(rng, w13a[e], xa[t]))    # saved A, bf16
            ag, au = a[:I], a[I:]
            g = _dot(rng, w2g[e].T, dyg[t])
            sig = 1.0 / (1.0 + np.exp(-ag))
            # silu'(a_g) = sig (1 + a_g (1 - sig)) evaluated in fp32 cancels near its root:
            # its error is a few ulps of the terms (1, |a_g|), not of the result
            d1 = _dsilu(ag) + 0.9 * SLACK_REL * sig * (1.0 + np.abs(ag)) * \
                rng.uniform(-1.0, 1.0, ag.shape)
            da = np.concatenate([_elem(rng, s * g * au * d1), _elem(rng, s * g * ag * sig)])
            sh = bf16(_elem(rng, s * ag * sig * au))
            daq = mx_qdq_rows(da) if mx else None
            da = bf16(da)
            if "da_in" in given:
                da = given["da_in"][f]
            if "sh_in" in given:
                sh = given["sh_in"][f]
            if mx and "daq_in" in given:
                daq = given["daq_in"][f]
            rows["a"][f], rows["da"][f], rows["sh"][f] = a, da, sh
            if mx:
                rows["daq"][f] = daq
            xs[t] = _dot(rng, w13d[e].T, daq if mx else da)
            if dx_in is None:
                xs[t] = bf16(xs[t])                    # the slot's dgrad result
            rows["slot"][f] = xs[t]
        dx = dx + xs.astype(np.float32)
    dw13 = np.zeros(w13.shape)
    dw2 = np.zeros(w2.shape)
    for e in range(E):
        t_e, k_e = np.nonzero(idx == e)
        f_e = np.sort(t_e * K + k_e)
        t_e = f_e // K
        dw13[e] = bf16(_dot(rng, rows["da"][f_e].T, x[t_e]))
        dw2[e] = bf16(_dot(rng, dy[t_e].T, rows["sh"][f_e]))
    return bf16(dx), dw13, dw2, rows
