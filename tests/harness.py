"""Shared helpers of the GPU parity tests: device transfer, error measures, cached inputs.

Inputs come from `workloads` (seeded, shared with the oracle side); expected values come
from `oracle` only.
"""
import functools

import numpy as np

import oracle
from workloads import synth


def torch():
    import torch as _t
    return _t


def to_dev(a, dtype=None):
    """numpy -> CUDA tensor; uint16 arrays are bf16 bit patterns."""
    T = torch()
    if a.dtype == np.uint16:
        t = T.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(T.bfloat16)
    else:
        t = T.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.view(dtype)


def bf16_dev_to_np(t):
    """CUDA bf16 tensor -> uint16 bit patterns."""
    T = torch()
    return t.contiguous().view(T.int16).cpu().numpy().view(np.uint16)


def bf16_dev_to_f64(t):
    return oracle.bf16_to_f64(bf16_dev_to_np(t))


def rel_err(got, ref, slack=None):
    """max |got - ref| / rms(ref): the parity measure of the float outputs.

    With `slack` (the oracle's per-element bound on how far a correct result may lie from
    its own because of rounding decisions taken within fp32 error of a midpoint), each
    element's error is first reduced by its slack: max((|got - ref| - slack)+) / rms(ref)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    if slack is not None:
        err = np.maximum(err - np.asarray(slack, np.float64).reshape(err.shape), 0.0)
    rms = np.sqrt(np.mean(ref ** 2))
    if rms == 0:
        return float(err.max()) if err.size else 0.0
    return float(err.max() / rms)


TOL_BF16 = 1e-2   # max|err| / rms(ref), BF16 path
TOL_MXFP8 = 3e-2  # max|err| / rms(ref), MXFP8 path


@functools.lru_cache(maxsize=4)
def inputs(cfg, weights=True):
    """Seeded host inputs of a configuration (cached per test session)."""
    d = dict(x=synth.make_x(cfg), logits=synth.make_logits(cfg))
    if weights:
        d["w13"] = synth.make_w13(cfg)
        d["w2"] = synth.make_w2(cfg)
    if cfg.passes == "bwd":
        d["dy"] = synth.make_dy(cfg)
    return d


def sample_tokens(T, n, seed=0):
    r = np.random.default_rng(1000 + seed)
    n = min(n, T)
    return np.sort(r.choice(T, size=n, replace=False))


def oracle_forward_tokens(tokens, x_bits, idx, w, w13, w2, mode):
    """Oracle (y, slack) for a subset of tokens, with the experts they use only (remapped)."""
    idx_s = idx[tokens]
    used = np.unique(idx_s)
    remap = np.full(int(idx.max()) + 1 if idx.size else 1, -1, np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    if isinstance(w13, tuple):
        w13s = (w13[0][used], w13[1][used])
        w2s = (w2[0][used], w2[1][used])
    else:
        w13s, w2s = w13[used], w2[used]
    return oracle.forward(oracle.bf16_to_f64(x_bits[tokens]), remap[idx_s], w[tokens], w13s,
                          w2s, mode=mode, with_slack=True)
