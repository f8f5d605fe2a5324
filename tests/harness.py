"""Shared helpers of the GPU parity tests: device transfer, the two parity measures, slack
statistics, the mapping between the layer's row orders, cached inputs.

Inputs come from `workloads` (seeded, shared with the oracle side); expected values come
from `oracle` only.

Two measures, both against the oracle's value and its per-element slack (the distance
within which another correct result lies, because a rounding decision was taken on a value
within fp32 error of its threshold):
  * check_exact: bit-exact wherever the oracle flags no decision, within the slack
    elsewhere, nothing else allowed. Used step by step: each step is fed the intermediates
    the GPU actually produced (the oracle's `given` inputs), so its slack is that step's own
    decisions only (a bf16 step or two of its output).
  * check_tol: max((|got - ref| - slack)+) / rms(ref) <= tol (1e-2 BF16, 3e-2 MXFP8),
    end to end from the layer's inputs, where slack carries every upstream decision.
Each call records the fraction of elements with a flagged decision and max(slack)/rms(ref)
and fails when they exceed the bound given for that check (slack must not quietly grow);
conftest prints the records at the end of the session.
"""
import functools

import numpy as np

import oracle
from workloads import synth

SLACK_RECORDS = []


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


def host(t):
    """A CUDA tensor (bf16 or fp32) as float64 numpy, exactly."""
    T = torch()
    if t.dtype == T.bfloat16:
        return bf16_dev_to_f64(t)
    return t.cpu().numpy().astype(np.float64)


def preact_rows(a):
    """Saved pre-activations [n, 2I] in the layer's layout ((gate, up) pairs per feature)
    -> the plain [n, 2I] order (gate features 0..I-1, then up)."""
    a = np.asarray(a)
    n, i2 = a.shape
    pr = a.reshape(n, i2 // 2, 2)
    return np.concatenate([pr[:, :, 0], pr[:, :, 1]], axis=1)


def same_bits(a, b):
    T = torch()
    u8 = lambda t: t.contiguous().view(T.uint8) if t.dtype != T.uint8 else t  # noqa: E731
    return a.shape == b.shape and T.equal(u8(a), u8(b))


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
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    if rms == 0:
        return float(err.max()) if err.size else 0.0
    return float(err.max() / rms)


TOL_BF16 = 1e-2   # max|err| / rms(ref), BF16 path
TOL_MXFP8 = 3e-2  # max|err| / rms(ref), MXFP8 path


def _record(name, ref, slack, moved, max_flagged, max_slack_rms):
    ref = np.asarray(ref, np.float64)
    slack = np.zeros_like(ref) if slack is None else np.asarray(slack, np.float64).reshape(
        ref.shape)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    # a flagged decision: the slack reaches half a bf16 step of the value (smaller slack is
    # an upstream flip too small to move this value's own rounding)
    step = np.ldexp(1.0, np.frexp(np.maximum(np.abs(ref), 1e-300))[1] - 8)
    flagged = float(np.mean(slack >= 0.5 * step)) if ref.size else 0.0
    srms = float(slack.max() / rms) if (ref.size and rms > 0) else 0.0
    SLACK_RECORDS.append(dict(name=name, n=int(ref.size), flagged=flagged,
                              max_slack_rms=srms, moved=int(moved)))
    assert flagged <= max_flagged, (name, "flagged fraction", flagged, max_flagged)
    assert srms <= max_slack_rms, (name, "max slack / rms", srms, max_slack_rms)


def check_exact(name, got, ref, slack, max_flagged=0.35, max_slack_rms=0.25):
    """Bit-exact where the oracle flags nothing, within the slack elsewhere."""
    got = np.asarray(got, np.float64).reshape(np.shape(ref))
    ref = np.asarray(ref, np.float64)
    slack = np.asarray(slack, np.float64).reshape(ref.shape)
    d = np.abs(got - ref)
    bad_exact = int(np.sum(d[slack == 0] != 0))
    bad_slack = int(np.sum(d > slack * (1 + 1e-9)))
    assert bad_exact == 0 and bad_slack == 0, (
        name, "unflagged mismatches", bad_exact, "beyond slack", bad_slack,
        "worst", float(np.max(d - slack)) if d.size else 0.0)
    _record(name, ref, slack, np.sum(d > 0), max_flagged, max_slack_rms)


def check_tol(name, got, ref, slack, tol, max_flagged=1.0, max_slack_rms=1.0):
    """max((|got - ref| - slack)+) / rms(ref) <= tol, with bounded slack statistics."""
    got = np.asarray(got, np.float64).reshape(np.shape(ref))
    err = rel_err(got, ref, slack)
    assert err <= tol, (name, err, rel_err(got, ref))
    _record(name, ref, slack, np.sum(np.abs(got - np.asarray(ref)) > 0), max_flagged,
            max_slack_rms)


def check_codes(name, q_gpu, s_gpu, q_ref, s_ref, slack):
    """MXFP8 codes and scales: bit-exact in every 32-element block where the oracle flags no
    decision; in a flagged block the dequantized values must lie within the slack."""
    q_gpu, q_ref = np.asarray(q_gpu, np.uint8), np.asarray(q_ref, np.uint8)
    s_gpu, s_ref = np.asarray(s_gpu, np.uint8), np.asarray(s_ref, np.uint8)
    n = q_ref.shape[-1]
    slack = np.asarray(slack, np.float64).reshape(q_ref.shape)
    blk_flag = (slack.reshape(-1, n // 32, 32) > 0).any(-1).reshape(s_ref.shape)
    assert np.array_equal(s_gpu[~blk_flag], s_ref[~blk_flag]), name
    qb_g = q_gpu.reshape(-1, n // 32, 32)[~blk_flag.reshape(-1, n // 32)]
    qb_r = q_ref.reshape(-1, n // 32, 32)[~blk_flag.reshape(-1, n // 32)]
    assert np.array_equal(qb_g, qb_r), (name, int((qb_g != qb_r).sum()))
    dg = oracle.mxfp8_dequantize(q_gpu, s_gpu)
    dr = oracle.mxfp8_dequantize(q_ref, s_ref)
    d = np.abs(dg - dr)
    assert np.all(d <= slack * (1 + 1e-9)), (name, float(np.max(d - slack)))
    SLACK_RECORDS.append(dict(name=name, n=int(q_ref.size), flagged=float(blk_flag.mean()),
                              max_slack_rms=0.0, moved=int(np.sum(q_gpu != q_ref))))


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


def remap_experts(idx_s):
    """Experts used by a token sample, renumbered 0..n-1: (used ids, remapped idx)."""
    used = np.unique(idx_s)
    remap = np.full(int(idx_s.max()) + 1 if idx_s.size else 1, -1, np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    return used, remap[idx_s]


def sorted_rows(inv, tokens, K):
    """Sorted rows (schedule order) of the flat ids of `tokens`, in flat id order."""
    f = (np.asarray(tokens)[:, None] * K + np.arange(K)[None, :]).reshape(-1)
    return np.asarray(inv)[f]


def padded_rows(rows, offsets, poff):
    """Padded row of each sorted row: poff[e] + r - offsets[e] for the expert e owning r."""
    rows = np.asarray(rows, np.int64)
    e = np.searchsorted(np.asarray(offsets), rows, side="right") - 1
    return np.asarray(poff)[e] + rows - np.asarray(offsets)[e]


def oracle_forward_tokens(tokens, x_bits, idx, w, w13, w2, mode, store=oracle.STORE_BF16,
                          rows=(), given=None):
    """Oracle forward for a subset of tokens, with the experts they use only (remapped)."""
    used, idx_r = remap_experts(idx[tokens])
    if isinstance(w13, tuple):
        w13s = (w13[0][used], w13[1][used])
        w2s = (w2[0][used], w2[1][used])
    else:
        w13s, w2s = w13[used], w2[used]
    return oracle.forward(oracle.bf16_to_f64(x_bits[tokens]), idx_r, w[tokens], w13s, w2s,
                          mode=mode, with_slack=True, store=store, rows=rows, given=given)
