"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test ties one oracle function to something independent: a hand-worked example
(tests/golden, with its derivation), a library routine (numpy stable sort, scipy softmax,
torch's float8 conversion, numpy matmul for the dense special cases), brute force over a
finite set, a closed form, an invariant, or central finite differences. A plausible
mistake in the oracle (a dropped term, a wrong sign, a swapped gate/up half, a transposed
weight, an unstable sort, a wrong rounding direction) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(12345)


def _silu(z):
    return z / (1.0 + np.exp(-z))


# ------------------------------------------------------------------ routing

def test_route_matches_stable_lexsort_with_ties():
    T, E, K = 64, 16, 5
    # few distinct values -> many ties; include both zeros
    vals = np.array([-1.5, -0.0, 0.0, 0.25, 0.25, 2.0])
    logits = rng.choice(vals, size=(T, E))
    idx, w = oracle.route(logits, K)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t]))  # by logit desc, then id asc
        assert list(idx[t]) == list(order[:K])


def test_route_weights_are_renormalised_full_softmax():
    T, E, K = 50, 32, 6
    logits = rng.standard_normal((T, E)) * 3
    idx, w = oracle.route(logits, K)
    p = scipy.special.softmax(logits, axis=1)
    sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-12, atol=0)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-12)
    assert np.all(np.diff(w, axis=1) <= 0)  # descending logits give descending weights


def test_route_one_hot_and_k_equals_e():
    E = 8
    lg = np.zeros((E, E)) - 5.0
    lg[np.arange(E), np.arange(E)] = 5.0
    idx, w = oracle.route(lg, 1)
    assert list(idx[:, 0]) == list(range(E)) and np.all(w == 1.0)
    logits = rng.standard_normal((4, E))
    idx, w = oracle.route(logits, E)
    full = scipy.special.softmax(logits, axis=1)
    np.testing.assert_allclose(np.take_along_axis(full, idx.astype(np.int64), 1), w,
                               rtol=1e-12)


# ------------------------------------------------------------------ schedule

def test_schedule_hand_example():
    g = json.load(open(os.path.join(GOLDEN, "schedule_hand.json")))
    s = oracle.schedule(np.array(g["idx"]), g["E"], g["MB"])
    for key in ("counts", "offsets", "perm", "inv"):
        assert list(s[key]) == g[key], key
    assert s["segs"].tolist() == g["segs"]


@pytest.mark.parametrize("T,E,K,MB", [(200, 16, 4, 37), (64, 64, 8, 1000), (300, 5, 2, 1),
                                      (1, 4, 1, 3), (0, 8, 2, 16)])
def test_schedule_matches_stable_sort_and_run_lengths(T, E, K, MB):
    idx = rng.integers(0, E, size=(T, K)).astype(np.int32)
    if T > 3:
        idx[: T // 3] = 0  # a hot expert and some empty ones
    s = oracle.schedule(idx, E, MB)
    f = idx.reshape(-1)
    R = f.size
    np.testing.assert_array_equal(s["perm"], np.argsort(f, kind="stable"))
    np.testing.assert_array_equal(s["counts"], np.bincount(f, minlength=E))
    assert s["counts"].sum() == R  # no routed row is dropped
    if R:
        np.testing.assert_array_equal(s["inv"][s["perm"]], np.arange(R))
    # segments: maximal runs of rows sharing (expert, minibatch)
    key_e = f[s["perm"]] if R else np.zeros(0, np.int64)
    key_m = np.arange(R) // MB
    runs = []
    for r in range(R):
        if r == 0 or key_e[r] != key_e[r - 1] or key_m[r] != key_m[r - 1]:
            runs.append([int(key_e[r]), r, r + 1])
        else:
            runs[-1][2] = r + 1
    assert s["segs"].tolist() == runs


# ------------------------------------------------------------------ MXFP8

def _torch_e4m3(v):
    t = torch.tensor(np.asarray(v, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_matches_torch_table():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3_decode(int(c)) for c in codes])
    finite = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[finite], ref[finite])
    assert np.all(np.isnan(ours[~finite]))


@pytest.mark.parametrize("shift", [-9, 0, 6])
def test_e4m3_encode_all_bf16_patterns(shift):
    bits = np.arange(65536, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    f = f[np.isfinite(f)].astype(np.float64) * 2.0 ** shift
    f = f[np.isfinite(f)]
    ours = np.array([oracle.e4m3_encode(v) for v in f], dtype=np.uint8)
    sat = np.abs(f) >= 448.0
    # saturation by definition; torch's conversion does not saturate
    assert np.all(ours[sat] & 0x7F == 0x7E)
    assert np.all((ours[sat] >> 7) == np.signbit(f[sat]))
    small = ~sat & (np.abs(f) < 3.0e38)
    ref = _torch_e4m3(f[small])
    np.testing.assert_array_equal(ours[small], ref)


def test_e4m3_encode_bruteforce_nearest_even():
    mags = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])  # 0 .. 448
    vals = np.concatenate([rng.uniform(0, 460, 3000), rng.uniform(0, 2.0 ** -5, 3000),
                           (mags[:-1] + mags[1:]) / 2])  # exact midpoints
    for v in vals:
        d = np.abs(mags - v)
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        if v >= 448:
            want = 0x7E
        assert oracle.e4m3_encode(v) == want, v
        assert oracle.e4m3_encode(-v) == want | 0x80, v


def test_mxfp8_hand_vectors():
    g = json.load(open(os.path.join(GOLDEN, "mxfp8_hand.json")))
    for case in g["cases"]:
        blk = np.full(32, case["fill"])
        first = np.array(case["block_first"], dtype=np.float64)
        blk[: len(first)] = first
        q, s = oracle.mxfp8_quantize(blk[None, :])
        assert int(s[0, 0]) == case["scale_byte"], case["what"]
        assert list(q[0, : len(first)]) == case["codes_first"], case["what"]


def test_mxfp8_scale_rule_and_roundtrip_bound():
    x = rng.standard_normal((40, 256)) * np.exp(rng.uniform(-20, 20, size=(40, 1)))
    x[3, :32] = 0.0
    q, s = oracle.mxfp8_quantize(x)
    blocks = np.abs(x).reshape(40, 8, 32).max(-1)
    m, e = np.frexp(blocks)  # blocks = m * 2**e, m in [0.5, 1)
    want = np.where(blocks > 0, np.clip(e - 1 - 8, -127, 127) + 127, 0)
    np.testing.assert_array_equal(s, want)
    dq = oracle.mxfp8_dequantize(q, s)
    # error per element: at most half a step of amax's binade (2^(e-4), e = floor(log2 amax)),
    # or the clipping of the block's top values to 448 * 2^(e-8)
    err = np.abs(dq - x).reshape(40, 8, 32).max(-1)
    ef = e - 1
    bound = np.maximum(np.ldexp(1.0, ef - 4), blocks - 448.0 * np.ldexp(1.0, ef - 8))
    assert np.all(err <= np.where(blocks > 0, bound, 0.0))
    # quantize-dequantize is idempotent
    q2, s2 = oracle.mxfp8_quantize(dq)
    np.testing.assert_array_equal(q2, q)
    np.testing.assert_array_equal(s2, s)


# ------------------------------------------------------------------ forward

def _rand_layer(T, H, I, E, K, scale=0.3, seed=0):
    r = np.random.default_rng(seed)
    x = r.standard_normal((T, H))
    logits = r.standard_normal((T, E))
    w13 = r.standard_normal((E, 2 * I, H)) * scale
    w2 = r.standard_normal((E, H, I)) * scale
    return x, logits, w13, w2


def test_forward_hand_example():
    g = json.load(open(os.path.join(GOLDEN, "forward_hand.json")))
    idx, w = oracle.route(np.array(g["logits"]), 2)
    assert idx.tolist() == g["idx"]
    np.testing.assert_allclose(w[0], g["w"], rtol=1e-15)
    y = oracle.forward(np.array(g["x"]), idx, w, np.array(g["w13"]), np.array(g["w2"]))
    np.testing.assert_allclose(y[0], g["y"], rtol=1e-14)
    # closed form, recomputed from the definition of silu
    h0, h1 = 2.0 / (1 + math.exp(-2.0)), 2.0 / (1 + math.exp(-1.0))
    np.testing.assert_allclose(y[0], [0.75 * h1 + 0.5 * h0, -0.75 * h1], rtol=1e-14)


def test_forward_single_expert_is_dense_swiglu_ffn():
    T, H, I = 7, 24, 10
    x, _, w13, w2 = _rand_layer(T, H, I, 1, 1)
    idx = np.zeros((T, 1), np.int32)
    w = np.ones((T, 1))
    y = oracle.forward(x, idx, w, w13, w2)
    a = x @ w13[0].T
    ref = (_silu(a[:, :I]) * a[:, I:]) @ w2[0].T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_forward_k_equals_e_is_dense_softmax_mixture():
    T, H, I, E = 5, 16, 6, 4
    x, logits, w13, w2 = _rand_layer(T, H, I, E, E)
    idx, w = oracle.route(logits, E)
    y = oracle.forward(x, idx, w, w13, w2)
    p = scipy.special.softmax(logits, axis=1)
    ref = np.zeros_like(y)
    for e in range(E):
        a = x @ w13[e].T
        ref += p[:, e: e + 1] * ((_silu(a[:, :I]) * a[:, I:]) @ w2[e].T)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_forward_equivariance_and_linearity():
    T, H, I, E, K = 12, 16, 8, 6, 3
    x, logits, w13, w2 = _rand_layer(T, H, I, E, K, seed=3)
    idx, w = oracle.route(logits, K)
    y = oracle.forward(x, idx, w, w13, w2)
    # permuting tokens permutes outputs
    p = rng.permutation(T)
    idx_p, w_p = oracle.route(logits[p], K)
    np.testing.assert_array_equal(oracle.forward(x[p], idx_p, w_p, w13, w2), y[p])
    # relabelling experts (weights and logit columns together) leaves y unchanged
    q = rng.permutation(E)
    idx_q, w_q = oracle.route(logits[:, q], K)
    np.testing.assert_allclose(oracle.forward(x, idx_q, w_q, w13[q], w2[q]), y, rtol=1e-13,
                               atol=1e-15)
    # y is linear in W2 and in the routing weights
    np.testing.assert_allclose(oracle.forward(x, idx, w, w13, 2.0 * w2), 2.0 * y, rtol=1e-15)
    np.testing.assert_allclose(oracle.forward(x, idx, 0.5 * w, w13, w2), 0.5 * y, rtol=1e-15)


def test_round_bf16_matches_single_rounding_of_fp32_values():
    """For values exactly representable in fp32, rounding to bf16 is the library's fp32 ->
    bf16 conversion (torch) and the workload generator's bit rounding."""
    r = np.random.default_rng(8)
    f = (r.standard_normal(20000) * np.exp(r.uniform(-90, 80, 20000))).astype(np.float32)
    u = f.view(np.uint32)
    ties = ((u & ~np.uint32(0xFFFF)) | np.uint32(0x8000)).view(np.float32)[:2000]  # halfway
    f = np.concatenate([f, ties, np.array([1e-40, -3e-39, 0.0, -0.0], np.float32)])
    ours = np.array([oracle.round_bf16(float(v)) for v in f])
    lib_ref = torch.from_numpy(f).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, lib_ref)
    np.testing.assert_array_equal(np.signbit(ours), np.signbit(lib_ref))


def test_forward_bf16_mode_rounds_h_before_the_down_gemm():
    """With one expert, K=1 and W2 = identity (H = I), y is exactly bf16(h)."""
    T, H, I = 6, 32, 32
    r = np.random.default_rng(6)
    x = r.standard_normal((T, H))
    w13 = r.standard_normal((1, 2 * I, H)) * 0.2
    w2 = np.eye(H)[None]
    idx = np.zeros((T, 1), np.int32)
    w = np.ones((T, 1))
    y = oracle.forward(x, idx, w, w13, w2, mode=oracle.BF16)
    a = x @ w13[0].T
    h = _silu(a[:, :I]) * a[:, I:]
    rb = np.array([oracle.round_bf16(v) for v in h.reshape(-1)]).reshape(h.shape)
    # h here and inside the oracle may differ in the last bits; that can only change the
    # rounding of values within a hair of a midpoint between bf16 neighbours
    ulp = np.ldexp(1.0, np.frexp(np.abs(h))[1] - 8)
    frac = np.abs(h) / ulp - np.floor(np.abs(h) / ulp)
    near_mid = np.abs(frac - 0.5) < 1e-6
    np.testing.assert_array_equal(y[~near_mid], rb[~near_mid])
    assert np.all(np.abs(y - rb)[near_mid] <= ulp[near_mid])
    assert not np.allclose(y, h, rtol=1e-6)
    # exact mode does not round
    np.testing.assert_allclose(oracle.forward(x, idx, w, w13, w2), h, rtol=1e-12, atol=1e-15)


def test_backward_bf16_mode_rounds_da_and_sh():
    """dtopk does not depend on the operand rounding; with W13 = [I; I] stacked identities
    (H = I) and one row, dx is the sum of the rounded gate and up gradients."""
    T, H, I = 4, 32, 32
    r = np.random.default_rng(10)
    x = r.standard_normal((T, H))
    w13 = np.concatenate([np.eye(I), np.eye(I)])[None]  # a_g = a_u = x
    w2 = r.standard_normal((1, H, I)) * 0.3
    dy = r.standard_normal((T, H))
    idx = np.zeros((T, 1), np.int32)
    w = np.full((T, 1), 0.75)
    dx0, _, _, dt0 = oracle.backward(x, idx, w, w13, w2, dy)
    dx1, dw13, dw2, dt1 = oracle.backward(x, idx, w, w13, w2, dy, mode=oracle.BF16)
    np.testing.assert_array_equal(dt0, dt1)
    g = dy @ w2[0]
    sig = 1 / (1 + np.exp(-x))
    dag = 0.75 * g * x * sig * (1 + x * (1 - sig))
    dau = 0.75 * g * x * sig
    rb = np.vectorize(oracle.round_bf16)
    np.testing.assert_allclose(dx1, rb(dag) + rb(dau), rtol=1e-12)
    np.testing.assert_allclose(dx0, dag + dau, rtol=1e-12)
    sh = rb(0.75 * x * sig * x)
    np.testing.assert_allclose(dw2[0], dy.T @ sh, rtol=1e-12)


def test_forward_mxfp8_quantizes_x_and_h_at_the_right_places():
    """With one expert, K=1 and W2 = identity (H = I = 32), y is exactly the dequantized
    MXFP8 image of h computed from the dequantized MXFP8 image of x."""
    T, H, I = 6, 32, 32
    r = np.random.default_rng(5)
    x = r.standard_normal((T, H))
    w13 = r.standard_normal((1, 2 * I, H)) * 0.2
    w2 = np.eye(H)[None]
    idx = np.zeros((T, 1), np.int32)
    w = np.ones((T, 1))
    y = oracle.forward(x, idx, w, w13, w2, mode=oracle.MXFP8)
    xq = oracle.mxfp8_dequantize(*oracle.mxfp8_quantize(x))
    a = xq @ w13[0].T
    h = _silu(a[:, :I]) * a[:, I:]
    hq = oracle.mxfp8_dequantize(*oracle.mxfp8_quantize(h))
    np.testing.assert_allclose(y, hq, rtol=1e-12, atol=0)
    assert not np.allclose(y, h, rtol=1e-6)  # quantization really happened


# ------------------------------------------------------------------ backward

def _loss(x, logits, w13, w2, dy, K):
    idx, w = oracle.route(logits, K)
    return float((oracle.forward(x, idx, w, w13, w2) * dy).sum())


def _fd_check(f, arr, grad, n=40, eps=1e-6, seed=0):
    r = np.random.default_rng(seed)
    flat = arr.reshape(-1)
    picks = r.choice(flat.size, size=min(n, flat.size), replace=False)
    for i in picks:
        old = flat[i]
        flat[i] = old + eps
        lp = f()
        flat[i] = old - eps
        lm = f()
        flat[i] = old
        fd = (lp - lm) / (2 * eps)
        g = grad.reshape(-1)[i]
        assert abs(fd - g) <= 1e-6 * max(1.0, abs(g)), (i, fd, g)


def test_backward_hand_example():
    g = json.load(open(os.path.join(GOLDEN, "forward_hand.json")))
    x, w13, w2, dy = (np.array(g[k]) for k in ("x", "w13", "w2", "dy"))
    idx, w = oracle.route(np.array(g["logits"]), 2)
    dx, dw13, dw2, dtopk = oracle.backward(x, idx, w, w13, w2, dy)
    np.testing.assert_allclose(dtopk[0], g["dtopk"], rtol=1e-14)
    sig = lambda z: 1 / (1 + math.exp(-z))  # noqa: E731
    dsilu = lambda z: sig(z) * (1 + z * (1 - sig(z)))  # noqa: E731
    silu = lambda z: z * sig(z)  # noqa: E731
    # expert 1 (w=3/4, g=1): da = (3/4 * 2 * silu'(1), 3/4 * silu(1)); W13[1] = identity
    # expert 0 (w=1/4, g=2): da = (1/2 * silu'(2), 1/2 * silu(2)); W13[0] swaps the inputs
    dx_ref = [0.75 * 2 * dsilu(1.0) + 0.5 * silu(2.0), 0.75 * silu(1.0) + 0.5 * dsilu(2.0)]
    np.testing.assert_allclose(dx[0], dx_ref, rtol=1e-14)
    h0, h1 = 2 / (1 + math.exp(-2.0)), 2 / (1 + math.exp(-1.0))
    dl = oracle.router_grad(idx, w, dtopk, 2)
    np.testing.assert_allclose(dl[0], [3 / 16 * (2 * h0 - h1), 3 / 16 * (h1 - 2 * h0)],
                               rtol=1e-13)


def test_backward_finite_differences():
    T, H, I, E, K = 6, 16, 8, 4, 2
    r = np.random.default_rng(7)
    for _ in range(100):
        logits = r.standard_normal((T, E))
        s = -np.sort(-logits, axis=1)
        if np.all(s[:, K - 1] - s[:, K] > 1e-2):
            break
    x = r.standard_normal((T, H))
    w13 = r.standard_normal((E, 2 * I, H)) * 0.3
    w2 = r.standard_normal((E, H, I)) * 0.3
    dy = r.standard_normal((T, H))
    idx, w = oracle.route(logits, K)
    dx, dw13, dw2, dtopk = oracle.backward(x, idx, w, w13, w2, dy)
    dlogits = oracle.router_grad(idx, w, dtopk, E)
    f = lambda: _loss(x, logits, w13, w2, dy, K)  # noqa: E731
    _fd_check(f, x, dx, seed=1)
    _fd_check(f, w13, dw13, seed=2)
    _fd_check(f, w2, dw2, seed=3)
    _fd_check(f, logits, dlogits, seed=4)
    # dS is the derivative with respect to the routing weights themselves
    wv = w.copy()
    g = lambda: float((oracle.forward(x, idx, wv, w13, w2) * dy).sum())  # noqa: E731
    _fd_check(g, wv, dtopk, seed=5)
    # unrouted experts get zero weight gradients
    used = np.zeros(E, bool)
    used[np.unique(idx)] = True
    assert np.all(dw13[~used] == 0) and np.all(dw2[~used] == 0)


def test_weight_storage_kinds_agree_exactly():
    """bf16 bit patterns and MXFP8 bytes are read as their exact values."""
    from workloads.synth import f32_to_bf16_bits
    T, H, I, E, K = 5, 64, 32, 3, 2
    x, logits, w13, w2 = _rand_layer(T, H, I, E, K, seed=9)
    b13 = f32_to_bf16_bits(w13.astype(np.float32))
    b2 = f32_to_bf16_bits(w2.astype(np.float32))
    idx, w = oracle.route(logits, K)
    y_bits = oracle.forward(x, idx, w, b13, b2)
    y_wide = oracle.forward(x, idx, w, oracle.bf16_to_f64(b13), oracle.bf16_to_f64(b2))
    np.testing.assert_array_equal(y_bits, y_wide)
    q13, s13 = oracle.mxfp8_quantize_bf16(b13)
    q2, s2 = oracle.mxfp8_quantize_bf16(b2)
    r13 = oracle.mxfp8_quantize(oracle.bf16_to_f64(b13))
    np.testing.assert_array_equal(q13, r13[0])
    np.testing.assert_array_equal(s13, r13[1])
    y_q = oracle.forward(x, idx, w, (q13, s13), (q2, s2), mode=oracle.MXFP8)
    y_d = oracle.forward(x, idx, w, oracle.mxfp8_dequantize(q13, s13),
                         oracle.mxfp8_dequantize(q2, s2), mode=oracle.MXFP8)
    np.testing.assert_array_equal(y_q, y_d)
    dy = np.random.default_rng(1).standard_normal((T, H))
    g_bits = oracle.backward(x, idx, w, b13, b2, dy)
    g_wide = oracle.backward(x, idx, w, oracle.bf16_to_f64(b13), oracle.bf16_to_f64(b2), dy)
    for a, b in zip(g_bits, g_wide):
        np.testing.assert_array_equal(a, b)


def test_bf16_slack_marks_exactly_the_decisions_a_small_error_can_flip():
    r = np.random.default_rng(21)
    f = (r.standard_normal(3000) * np.exp(r.uniform(-30, 30, 3000))).astype(np.float32)
    u = f.view(np.uint32) & ~np.uint32(0xFFFF)
    lo = u.view(np.float32).astype(np.float64)
    hi = (u + np.uint32(0x10000)).view(np.float32).astype(np.float64)
    mid = (lo + hi) / 2  # exact midpoints between bf16 neighbours
    for m, a, b in zip(mid[:500], lo[:500], hi[:500]):
        err = abs(m) * 2.0 ** -16  # a value known to within err
        for v in (m, m + err / 2, m - err / 2):
            # values within err of v on either side round to different neighbours
            down = torch.tensor(v - err * 0.9).float().to(torch.bfloat16).double().item()
            up = torch.tensor(v + err * 0.9).float().to(torch.bfloat16).double().item()
            assert oracle.bf16_slack(v, err) == abs(b - a) >= abs(up - down)
        # with no error beyond the elementwise margin, points a bit off the midpoint are
        # unambiguous
        assert oracle.bf16_slack(m * (1 + 2.0 ** -12), 0.0) == 0.0
        assert oracle.bf16_slack(m, 0.0) == abs(b - a)
    for v in lo[:500]:  # representable values are far from every midpoint
        assert oracle.bf16_slack(v, abs(v) * 2.0 ** -16) == 0.0


def test_forward_slack_in_the_identity_structure():
    """With one expert, K=1, weight 1 and W2 = identity, y = bf16(h) and the slack of y_c is
    the slack of the single decision h_c."""
    T, H, I = 64, 32, 32
    r = np.random.default_rng(22)
    x = r.standard_normal((T, H))
    w13 = r.standard_normal((1, 2 * I, H)) * 0.2
    idx = np.zeros((T, 1), np.int32)
    y, sl = oracle.forward(x, idx, np.ones((T, 1)), w13, np.eye(H)[None], mode=oracle.BF16,
                           with_slack=True)
    a = x @ w13[0].T
    h = _silu(a[:, :I]) * a[:, I:]
    # the h error bound: dot-product bounds through the partial derivatives of silu(g)*u
    mag = np.abs(x) @ np.abs(w13[0]).T * oracle.DOT_REL
    sig = 1 / (1 + np.exp(-a[:, :I]))
    dsl = sig * (1 + a[:, :I] * (1 - sig))
    err = np.abs(dsl * a[:, I:]) * mag[:, :I] + np.abs(_silu(a[:, :I])) * mag[:, I:]
    want = np.array([oracle.bf16_slack(v, e) for v, e in zip(h.reshape(-1), err.reshape(-1))])
    np.testing.assert_allclose(sl, want.reshape(h.shape), rtol=0, atol=0)
    _, sl0 = oracle.forward(x, idx, np.ones((T, 1)), w13, np.eye(H)[None], with_slack=True)
    assert np.all(sl0 == 0.0)  # exact mode rounds nothing


def test_backward_slack_zero_in_exact_mode():
    T, H, I, E, K = 16, 32, 32, 2, 2
    x, logits, w13, w2 = _rand_layer(T, H, I, E, K, seed=23)
    dy = np.random.default_rng(24).standard_normal((T, H))
    idx, w = oracle.route(logits, K)
    for store in (oracle.STORE_F32, oracle.STORE_BF16):
        out0 = oracle.backward(x, idx, w, w13, w2, dy, with_slack=True, store=store)
        assert all(np.all(s == 0) for s in out0[4:])
        ref = oracle.backward(x, idx, w, w13, w2, dy)
        for a, b in zip(out0[:4], ref):  # nothing is rounded in exact mode
            np.testing.assert_array_equal(a, b)


# ---------------------------------------------------------------- MXFP8 backward
from workloads.synth import f32_to_bf16_bits  # noqa: E402  (seeded input helper only)
# [arex] "Cursor 放出 MoK", section "pull 代替 push": MXFP8 with pre-quantized weights and
# activations quantized where they enter a GEMM. The backward's G GEMM contracts over H
# (dy and W2 quantized along H), dgrad over 2I (dA and W13 quantized along 2I).

def test_mxfp8_axis_quantization_is_per_column_quantization():
    r = np.random.default_rng(41)
    w = f32_to_bf16_bits((r.standard_normal((2, 64, 96)) * 0.1).astype(np.float32))
    got = oracle.mxfp8_qdq_axis_bf16(w, axis=1)
    for e in range(2):
        for col in range(96):
            q, s = oracle.mxfp8_quantize_bf16(w[e, :, col][None, :].copy())
            np.testing.assert_array_equal(got[e, :, col], oracle.mxfp8_dequantize(q, s)[0])


def _exact_case():
    """Every MXFP8 quantization in the backward is exact and so is every bf16 rounding.
    K = 1 (weight 1); x[t] and dy[t] are one-hot (+-1 at column c_t, d_t); the weights
    take values in {0, +-1, +-2}, with W13's gate rows zero in the columns c_t, so
    a_g = 0 (silu(0) = 0, silu'(0) = 1/2), a_u and G = W2^T dy are single weight entries,
    and dA_g = G a_u / 2 lies in {0, +-1/2, +-1, +-2}, while dx = W13_g^T dA_g is not
    zero."""
    T, H, I, E = 3, 64, 32, 2
    r = np.random.default_rng(43)
    pick = lambda *s: r.choice([-2.0, -1.0, 0.0, 1.0, 2.0], size=s).astype(np.float64)  # noqa
    c = np.array([5, 17, 40]); d = np.array([3, 33, 60])
    sign = np.array([1.0, -1.0, 1.0])
    x = np.zeros((T, H)); x[np.arange(T), c] = sign
    dy = np.zeros((T, H)); dy[np.arange(T), d] = -sign
    w13 = np.concatenate([pick(E, I, H), pick(E, I, H)], axis=1)
    w13[:, :I, c] = 0.0  # a_g = 0 for every token
    w2 = pick(E, H, I)
    idx = np.array([[0], [1], [1]], np.int32)
    w = np.ones((T, 1))
    b = lambda a: f32_to_bf16_bits(a.astype(np.float32))  # noqa: E731
    return b(x), idx, w, b(w13), b(w2), b(dy)


def test_mxfp8_backward_equals_exact_when_every_quantization_is_exact():
    x, idx, w, w13, w2, dy = _exact_case()
    xf, dyf = oracle.bf16_to_f64(x), oracle.bf16_to_f64(dy)
    ref = oracle.backward(xf, idx, w, w13, w2, dyf, mode=oracle.EXACT)
    assert np.abs(ref[0]).max() > 0 and np.abs(ref[1]).max() > 0  # dx, dW13 not trivial
    for mode in (oracle.BF16, oracle.MXFP8):
        got = oracle.backward(xf, idx, w, w13, w2, dyf, mode=mode)
        for a, b in zip(got, ref):
            np.testing.assert_array_equal(a, b)


def test_mxfp8_backward_g_uses_the_quantized_operands():
    """dS = <G, h> with G = W2q^T Q(dy) and h from A = W13q Q(x): equal to the BF16-mode
    backward run on those operands already quantized (W13 along H, W2 along H, x and dy
    along H), where nothing else touches dS."""
    r = np.random.default_rng(47)
    T, H, I, E, K = 5, 64, 32, 3, 2
    x = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    dy = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    w13 = f32_to_bf16_bits((r.standard_normal((E, 2 * I, H)) * 0.2).astype(np.float32))
    w2 = f32_to_bf16_bits((r.standard_normal((E, H, I)) * 0.2).astype(np.float32))
    idx, w = oracle.route(r.standard_normal((T, E)).astype(np.float32), K)
    _, _, _, dtk = oracle.backward(oracle.bf16_to_f64(x), idx, w, w13, w2,
                                   oracle.bf16_to_f64(dy), mode=oracle.MXFP8)
    # references built without the along-axis helper: the row quantizer on rows that run
    # along H (x, dy, W13 rows), and on an explicit transpose for W2 (its H axis is not last)
    rowq = lambda b: oracle.mxfp8_dequantize(*oracle.mxfp8_quantize_bf16(b))  # noqa: E731
    xq, dyq, w13q = rowq(x), rowq(dy), rowq(w13)
    w2q = rowq(np.ascontiguousarray(w2.transpose(0, 2, 1))).transpose(0, 2, 1)
    _, _, _, dtk_ref = oracle.backward(xq, idx, w, w13q, w2q, dyq, mode=oracle.BF16)
    np.testing.assert_array_equal(dtk, dtk_ref)
    # and differs from the unquantized BF16 backward (the quantization is not skipped)
    _, _, _, dtk_b = oracle.backward(oracle.bf16_to_f64(x), idx, w, w13, w2,
                                     oracle.bf16_to_f64(dy), mode=oracle.BF16)
    assert not np.array_equal(dtk, dtk_b)


# ---------------------------------------------------------------- rounding slack
# The slack of a rounding decision is pinned against a stand-in kernel (tests/emulate.py)
# that recomputes the layer with numpy and torch and errs, at random, anywhere inside the
# fp32 bounds the oracle assumes. Each draw is a result a correct kernel could give; the
# oracle's value must equal it wherever the oracle flags no decision, and lie within the
# slack of it everywhere. A dropped propagation term, a wrong exponent direction or a
# missing storage rounding lets some draw escape its slack.
import emulate  # noqa: E402


def _bf16_case(T, H, I, E, K, seed):
    r = np.random.default_rng(seed)
    b = lambda a: oracle.bf16_to_f64(f32_to_bf16_bits(a.astype(np.float32)))  # noqa: E731
    x = b(r.standard_normal((T, H)))
    w13 = b(r.standard_normal((E, 2 * I, H)) / np.sqrt(H))
    w2 = b(r.standard_normal((E, H, I)) / np.sqrt(I))
    dy = b(r.standard_normal((T, H)))
    idx, w = oracle.route(r.standard_normal((T, E)), K)
    # routing weights as a kernel holds them (fp32)
    return x, idx, w.astype(np.float32).astype(np.float64), w13, w2, dy


def _covers(draw, ref, slack, what):
    d = np.abs(draw - ref)
    # where nothing is flagged the draw is the oracle's value itself
    assert np.all(d[slack == 0] == 0), (what, int((d[slack == 0] > 0).sum()))
    assert np.all(d <= slack * (1 + 1e-9)), (what, float((d - slack).max()))
    return int((d > 0).sum())


def _step(v):
    """bf16 step (ulp) at each value"""
    return np.ldexp(1.0, np.frexp(np.maximum(np.abs(v), 1e-300))[1] - 8)


def _fwd_case(mode):
    T, H, I, E, K = 24, 64, 64, 4, 2
    x, idx, w, w13, w2, _ = _bf16_case(T, H, I, E, K, seed=60 + mode)
    if mode == oracle.MXFP8:  # pre-quantized weights: both sides read the same values
        w13, w2 = emulate.mx_qdq_rows(w13), emulate.mx_qdq_rows(w2)
    return x, idx, w, w13, w2


@pytest.mark.parametrize("mode", [oracle.BF16, oracle.MXFP8])
def test_forward_slack_covers_every_kernel_draw(mode):
    """End to end: the slack of y covers every draw of the stand-in kernel, and the slack
    of each h decision covers the draw's h."""
    x, idx, w, w13, w2 = _fwd_case(mode)
    y, sl, rows = oracle.forward(x, idx, w, w13, w2, mode=mode, with_slack=True,
                                 store=oracle.STORE_BF16, rows=("h", "h_slack"))
    np.testing.assert_array_equal(y, emulate.bf16(y))  # y is stored as bf16
    r = np.random.default_rng(1)
    moved = 0
    for _ in range(12):
        gy, gh = emulate.forward(r, x, idx, w, w13, w2, mode)
        moved += _covers(gy, y, sl, "y") + _covers(gh, rows["h"], rows["h_slack"], "h")
    assert moved > 0  # some draws really took the other neighbour


@pytest.mark.parametrize("mode", [oracle.BF16, oracle.MXFP8])
def test_forward_slack_given_h_is_the_down_steps_own(mode):
    """Given the h a kernel fed its down GEMM, the slack of y is that of the slot and
    output roundings alone: it covers every draw and is at most two bf16 steps of each
    weighted slot plus two of y."""
    x, idx, w, w13, w2 = _fwd_case(mode)
    r = np.random.default_rng(3)
    T, K = idx.shape
    moved = 0
    for _ in range(6):
        _, gh = emulate.forward(r, x, idx, w, w13, w2, mode)
        y, sl = oracle.forward(x, idx, w, w13, w2, mode=mode, with_slack=True,
                               store=oracle.STORE_BF16, given={"h_in": gh})
        gy, _ = emulate.forward(r, x, idx, w, w13, w2, mode, h_in=gh)
        moved += _covers(gy, y, sl, "y")
        o = np.stack([np.stack([w2[idx[t, k]] @ gh[t * K + k] for k in range(K)])
                      for t in range(T)])                    # [T, K, H]
        bound = 2 * (np.abs(w)[:, :, None] * _step(o)).sum(1) + 2 * _step(y)
        assert np.all(sl <= bound)
    assert moved > 0


@pytest.mark.parametrize("mode", [oracle.BF16, oracle.MXFP8])
def test_backward_slack_covers_every_kernel_draw(mode):
    T, H, I, E, K = 16, 64, 64, 3, 2
    x, idx, w, w13, w2, dy = _bf16_case(T, H, I, E, K, seed=70 + mode)
    bits = lambda a: f32_to_bf16_bits(a.astype(np.float32))  # noqa: E731
    w13b, w2b = (bits(w13), bits(w2)) if mode == oracle.MXFP8 else (w13, w2)
    names = ("a", "a_slack", "da", "da_slack", "sh", "sh_slack")
    dx, dw13, dw2, _, sdx, s13, s2, rows = oracle.backward(
        x, idx, w, w13b, w2b, dy, mode=mode, with_slack=True, store=oracle.STORE_BF16,
        rows=names)
    r = np.random.default_rng(2)
    moved = 0
    for _ in range(6):
        gx, g13, g2, gr = emulate.backward(r, x, idx, w, w13, w2, dy, mode)
        moved += _covers(gx, dx, sdx, "dx") + _covers(g13, dw13, s13, "dw13") + \
            _covers(g2, dw2, s2, "dw2") + _covers(gr["a"], rows["a"], rows["a_slack"], "a")
    assert moved > 0


@pytest.mark.parametrize("mode", [oracle.BF16, oracle.MXFP8])
def test_backward_slack_given_each_steps_inputs(mode):
    """Step by step: given the kernel's A, the slacks of dA and w*h cover every draw of its
    dA and w*h; given also its dA and w*h (and MXFP8 dgrad operand), the slacks of dx, dW13
    and dW2 cover every draw of its results. Each slack is at most twice the spread the
    draws reach plus two bf16 steps: no wider than the decisions the kernel can take."""
    T, H, I, E, K = 16, 64, 64, 3, 2
    x, idx, w, w13, w2, dy = _bf16_case(T, H, I, E, K, seed=74 + mode)
    bits = lambda a: f32_to_bf16_bits(a.astype(np.float32))  # noqa: E731
    w13b, w2b = (bits(w13), bits(w2)) if mode == oracle.MXFP8 else (w13, w2)
    r = np.random.default_rng(4)

    def tight(sl, ref, spread, what):
        assert np.all(sl <= 2 * spread + 2 * _step(ref)), what

    _, _, _, g0 = emulate.backward(r, x, idx, w, w13, w2, dy, mode)
    *_, rows = oracle.backward(x, idx, w, w13b, w2b, dy, mode=mode, store=oracle.STORE_BF16,
                               given={"a_in": g0["a"]},
                               rows=("da", "da_slack", "sh", "sh_slack"))
    sp_da = np.zeros_like(rows["da"])
    sp_sh = np.zeros_like(rows["sh"])
    moved = 0
    for _ in range(10):
        _, _, _, gr = emulate.backward(r, x, idx, w, w13, w2, dy, mode, given={"a_in": g0["a"]})
        moved += _covers(gr["da"], rows["da"], rows["da_slack"], "da")
        moved += _covers(gr["sh"], rows["sh"], rows["sh_slack"], "sh")
        sp_da = np.maximum(sp_da, np.abs(gr["da"] - rows["da"]))
        sp_sh = np.maximum(sp_sh, np.abs(gr["sh"] - rows["sh"]))
    tight(rows["da_slack"], rows["da"], sp_da, "da")
    tight(rows["sh_slack"], rows["sh"], sp_sh, "sh")
    # dx, dW given every operand the kernel fed its dgrad and weight-gradient GEMMs
    given = {"a_in": gr["a"], "da_in": gr["da"], "sh_in": gr["sh"]}
    if mode == oracle.MXFP8:
        given["daq_in"] = gr["daq"]
    dx, dw13, dw2, _, sdx, s13, s2 = oracle.backward(
        x, idx, w, w13b, w2b, dy, mode=mode, with_slack=True, store=oracle.STORE_BF16,
        given=given)
    sp = [np.zeros_like(dx), np.zeros_like(dw13), np.zeros_like(dw2)]
    slot_steps = np.zeros_like(dx)
    for _ in range(10):
        *outs, gr = emulate.backward(r, x, idx, w, w13, w2, dy, mode, given=given)
        for i, (g, ref, sl, nm) in enumerate(zip(outs, (dx, dw13, dw2), (sdx, s13, s2),
                                                 ("dx", "dw13", "dw2"))):
            moved += _covers(g, ref, sl, nm)
            sp[i] = np.maximum(sp[i], np.abs(g - ref))
        slot_steps = np.maximum(slot_steps, _step(gr["slot"]).reshape(T, K, H).sum(1))
    # dx sums K rounded slots: each may be a step or two off, whatever the size of dx
    tight(sdx, dx, sp[0] + slot_steps, "dx")
    tight(s13, dw13, sp[1], "dw13")
    tight(s2, dw2, sp[2], "dw2")
    assert moved > 0


def test_storage_rounding_is_where_the_definition_puts_it():
    """With one expert, K=1, weight 1, W2 = identity (H = I): the slot is bf16(h), which is
    already bf16, and y = bf16(h); with two experts at weights 1/2, y = bf16(o_0/2 + o_1/2)
    of the two rounded slots. A missing or extra rounding changes these values."""
    T, H, I = 32, 32, 32
    r = np.random.default_rng(80)
    x = r.standard_normal((T, H))
    w13 = r.standard_normal((2, 2 * I, H)) * 0.3
    w2 = np.stack([np.eye(H), np.eye(H) * 1.5])
    _, rows = oracle.forward(x, np.zeros((T, 1), np.int32), np.ones((T, 1)), w13[:1], w2[:1],
                             mode=oracle.BF16, store=oracle.STORE_BF16, rows=("h",))
    y1 = oracle.forward(x, np.zeros((T, 1), np.int32), np.ones((T, 1)), w13[:1], w2[:1],
                        mode=oracle.BF16, store=oracle.STORE_BF16)
    np.testing.assert_array_equal(y1, rows["h"])
    idx = np.tile(np.array([[0, 1]], np.int32), (T, 1))
    y2, rows2 = oracle.forward(x, idx, np.full((T, 2), 0.5), w13, w2, mode=oracle.BF16,
                               store=oracle.STORE_BF16, rows=("h",))
    h = rows2["h"].reshape(T, 2, I)
    o1 = emulate.bf16(1.5 * h[:, 1])  # slot of expert 1: bf16 of 1.5 h
    np.testing.assert_array_equal(y2, emulate.bf16(0.5 * h[:, 0] + 0.5 * o1))
    assert not np.array_equal(o1, 1.5 * h[:, 1])  # that slot rounding is not a no-op


def test_backward_reads_the_saved_pre_activations_in_bf16():
    """Under bf16 storage the backward's A is bf16(W13 x), and dS = <G, silu(A_g) A_u>
    uses it; under fp32 storage A is exact."""
    T, H, I, E, K = 8, 64, 32, 2, 1
    x, idx, w, w13, w2, dy = _bf16_case(T, H, I, E, K, seed=81)
    for store in (oracle.STORE_F32, oracle.STORE_BF16):
        *_, dtk, rows = oracle.backward(x, idx, w, w13, w2, dy, mode=oracle.BF16,
                                        store=store, rows=("a",))
        a = np.stack([w13[idx[t, 0]] @ x[t] for t in range(T)])
        want = emulate.bf16(a) if store == oracle.STORE_BF16 else a
        near = np.abs(rows["a"] - want) > 0
        assert near.mean() < 0.01  # only values within fp32 error of a bf16 midpoint
        ag, au = rows["a"][:, :I], rows["a"][:, I:]
        g = np.stack([w2[idx[t, 0]].T @ dy[t] for t in range(T)])
        np.testing.assert_allclose(dtk[:, 0], (g * _silu(ag) * au).sum(1), rtol=1e-12)


def _mx_block_exp(v):
    return int(np.frexp(np.abs(v).max())[1] - 1 - 8)


def _e4m3_torch(u):
    return torch.tensor(np.clip(u, -448, 448)).float().to(torch.float8_e4m3fn).double().numpy()


def test_mxfp8_slack_near_a_power_of_two_is_the_other_exponents_result():
    r = np.random.default_rng(90)
    blk = r.uniform(-0.9, 0.9, 32)
    blk[7] = 1.0 - 2.0 ** -20            # amax just below 1: exponent -9, or -8 above 1
    err = np.full(32, 2.0 ** -18)        # the error reaches across 1.0
    out, sl, q, sc = oracle.mxfp8_qdq_slack(blk[None], err[None])
    s = _mx_block_exp(blk)
    assert s == -9 and sc[0, 0] == 127 - 9
    chosen = np.ldexp(_e4m3_torch(np.ldexp(blk, -s)), s)
    alt = np.ldexp(_e4m3_torch(np.ldexp(blk, -(s + 1))), s + 1)
    np.testing.assert_array_equal(out[0], chosen)
    # no code decision is near a midpoint here, so the slack is the exponent alternative
    u = np.ldexp(blk, -s)
    sp = np.ldexp(1.0, np.maximum(np.frexp(np.abs(u))[1] - 1, -6) - 3)
    frac = np.abs(u) / sp - np.floor(np.abs(u) / sp)
    assert np.all(np.abs(frac - 0.5) * sp > np.ldexp(err, -s) + 2.0 ** -20 * np.abs(u))
    ua = np.ldexp(blk, -(s + 1))
    spa = np.ldexp(1.0, np.maximum(np.frexp(np.abs(ua))[1] - 1, -6) - 3)
    fa = np.abs(ua) / spa - np.floor(np.abs(ua) / spa)
    clear = np.abs(fa - 0.5) * spa > np.ldexp(err, -(s + 1)) + 2.0 ** -20 * np.abs(ua)
    np.testing.assert_array_equal(sl[0][clear], np.abs(alt - chosen)[clear])
    assert np.all(sl[0] >= np.abs(alt - chosen))
    assert np.abs(alt - chosen).max() > 0


def test_mxfp8_slack_zero_far_from_every_decision_and_one_step_at_a_midpoint():
    s = -8  # amax in [1, 2)
    codes = np.array([1.0, 1.125, 1.25, 1.5, -1.75, 0.5, 0.625, -0.25] * 4)
    blk = np.ldexp(codes, s + 8) * 1.0  # exactly representable: far from every midpoint
    blk[0] = 1.5 * 1.0                  # amax 1.5: exponent -8, not near a power of two
    err = np.full(32, 2.0 ** -30)
    out, sl, _, _ = oracle.mxfp8_qdq_slack(blk[None], err[None])
    np.testing.assert_array_equal(out[0], blk)
    assert np.all(sl == 0)
    mid = blk.copy()
    mid[3] = (1.5 + 1.625) / 2           # a code midpoint (ties to even: 1.5)
    out, sl, _, _ = oracle.mxfp8_qdq_slack(mid[None], err[None])
    assert out[0, 3] == 1.5 and sl[0, 3] == 0.125
    assert np.all(np.delete(sl[0], 3) == 0)


def test_mxfp8_slack_covers_random_perturbations():
    r = np.random.default_rng(91)
    v = r.standard_normal((400, 64)) * np.exp(r.uniform(-5, 5, (400, 1)))
    # push some block maxima onto powers of two and some values onto code midpoints
    v[::7, 0] = np.ldexp(1.0, r.integers(-5, 5, v[::7, 0].shape)) * (1 - 2.0 ** -22)
    err = np.abs(v) * 2.0 ** -19
    out, sl, _, _ = oracle.mxfp8_qdq_slack(v, err)
    moved = 0
    for _ in range(20):
        p = v + err * r.uniform(-1, 1, v.shape)
        d = np.abs(emulate.mx_qdq_rows(p) - out)
        assert np.all(d[sl == 0] == 0)
        assert np.all(d <= sl * (1 + 1e-12))
        moved += int((d > 0).sum())
    assert moved > 0


def test_mxfp8_dgrad_reads_da_quantized_along_2i():
    """dx of the MXFP8 backward (fp32 storage, nothing else rounded on its path) is
    sum_k W13q^T Q(dA) with W13 quantized along 2I (an explicit transpose fed to the row
    quantizer) and dA quantized in 32-blocks along 2I, dA computed here from the forward's
    quantized operands; the same sum with unquantized dA is far from it."""
    T, H, I, E, K = 6, 64, 64, 2, 2
    x, idx, w, w13, w2, dy = _bf16_case(T, H, I, E, K, seed=92)
    bits = lambda a: f32_to_bf16_bits(a.astype(np.float32))  # noqa: E731
    dx, *_ = oracle.backward(x, idx, w, bits(w13), bits(w2), dy, mode=oracle.MXFP8)
    rowq = lambda m: oracle.mxfp8_dequantize(*oracle.mxfp8_quantize(m))  # noqa: E731
    tq = lambda m: np.swapaxes(rowq(np.ascontiguousarray(np.swapaxes(m, -1, -2))), -1, -2)  # noqa
    xq, dyq, w13h = rowq(x), rowq(dy), rowq(w13)
    w13i, w2h = tq(w13), tq(w2)
    ref = np.zeros_like(dx)
    ref_plain = np.zeros_like(dx)
    for t in range(T):
        for k in range(K):
            e, s = idx[t, k], w[t, k]
            a = w13h[e] @ xq[t]
            ag, au = a[:I], a[I:]
            g = w2h[e].T @ dyq[t]
            sig = 1 / (1 + np.exp(-ag))
            da = np.concatenate([s * g * au * sig * (1 + ag * (1 - sig)), s * g * ag * sig])
            ref[t] += w13i[e].T @ rowq(da[None])[0]
            ref_plain[t] += w13i[e].T @ da
    np.testing.assert_allclose(dx, ref, rtol=1e-11, atol=1e-13)
    assert np.abs(ref - ref_plain).max() > 1e-3 * np.abs(ref).max()


@pytest.mark.parametrize("mode", [oracle.BF16, oracle.MXFP8])
def test_added_expert_slack_covers_every_kernel_draw(mode):
    """An expert whose output is added to an existing bf16 output (a shared expert, K=1,
    weight one): y = bf16(y_in + o) and dx = bf16(dx_in + W13^T dA) with no slot between;
    given the kernel's h (forward) or A, dA and w*h (backward), every draw lies within the
    slack, equal to the oracle where nothing is flagged."""
    T, H, I = 24, 64, 64
    x, _, _, w13, w2, dy = _bf16_case(T, H, I, 1, 1, seed=95 + mode)
    idx, w = np.zeros((T, 1), np.int32), np.ones((T, 1))
    r = np.random.default_rng(7)
    y_in = emulate.bf16(r.standard_normal((T, H)) * 0.5)
    wq = (emulate.mx_qdq_rows(w13), emulate.mx_qdq_rows(w2)) if mode == oracle.MXFP8 \
        else (w13, w2)
    moved = 0
    for _ in range(6):
        _, gh = emulate.forward(r, x, idx, w, wq[0], wq[1], mode)
        y, sl = oracle.forward(x, idx, w, wq[0], wq[1], mode=mode, with_slack=True,
                               store=oracle.STORE_BF16, given={"h_in": gh, "y_in": y_in})
        gy, _ = emulate.forward(r, x, idx, w, wq[0], wq[1], mode, h_in=gh, y_in=y_in)
        moved += _covers(gy, y, sl, "y added")
        assert np.all(sl <= 2 * _step(y) + 2 * _step(y - y_in))
    bits = lambda a: f32_to_bf16_bits(a.astype(np.float32))  # noqa: E731
    w13b, w2b = (bits(w13), bits(w2)) if mode == oracle.MXFP8 else (w13, w2)
    dx_in = emulate.bf16(r.standard_normal((T, H)) * 0.5)
    for _ in range(4):
        _, _, _, gr = emulate.backward(r, x, idx, w, w13, w2, dy, mode)
        given = {"a_in": gr["a"], "da_in": gr["da"], "sh_in": gr["sh"], "dx_in": dx_in}
        if mode == oracle.MXFP8:
            given["daq_in"] = gr["daq"]
        dx, _, _, _, sdx, _, _ = oracle.backward(x, idx, w, w13b, w2b, dy, mode=mode,
                                                 with_slack=True, store=oracle.STORE_BF16,
                                                 given=given)
        gx, _, _, _ = emulate.backward(r, x, idx, w, w13, w2, dy, mode, given=given,
                                       dx_in=dx_in)
        moved += _covers(gx, dx, sdx, "dx added")
    assert moved > 0


def test_router_gradient_slack_covers_the_saved_a_decisions():
    """dS = <G, h> moves with the stored A's rounding decisions (h is recomputed from A):
    with G exact, dS from each draw's A lies within dtopk_slack, and the logit gradients
    from it within router_grad_slack."""
    T, H, I, E, K = 16, 64, 64, 3, 2
    x, idx, w, w13, w2, dy = _bf16_case(T, H, I, E, K, seed=97)
    *_, dtk, sdx, _, _, ro = oracle.backward(x, idx, w, w13, w2, dy, mode=oracle.BF16,
                                             store=oracle.STORE_BF16, with_slack=True,
                                             rows=("dtopk_slack",))
    sdtk = ro["dtopk_slack"].reshape(T, K)
    sdl = oracle.router_grad_slack(idx, w, sdtk, E)
    dl = oracle.router_grad(idx, w, dtk, E)
    assert sdtk.max() > 0
    r = np.random.default_rng(5)
    moved = 0
    for _ in range(8):
        _, _, _, gr = emulate.backward(r, x, idx, w, w13, w2, dy, oracle.BF16)
        a = gr["a"].reshape(T, K, 2 * I)
        ds = np.empty((T, K))
        for t in range(T):
            for k in range(K):
                g = w2[idx[t, k]].T @ dy[t]
                ds[t, k] = g @ (_silu(a[t, k, :I]) * a[t, k, I:])
        d = np.abs(ds - dtk)
        assert np.all(d <= sdtk * (1 + 1e-9) + 1e-12 * np.abs(dtk)), float((d - sdtk).max())
        dld = np.abs(oracle.router_grad(idx, w, ds, E) - dl)
        assert np.all(dld <= sdl * (1 + 1e-9) + 1e-12 * np.abs(dl).max())
        moved += int((d > 1e-12 * np.abs(dtk)).sum())
    assert moved > 0


def test_backward_weight_gradients_restrict_to_features():
    """A feature's dW13 rows (gate, up) and dW2 column depend only on its own weights: the
    oracle's expert restricted to a feature subset (its gate and up rows of W13, its W2
    columns) gives the full expert's rows and columns bit for bit, slack included. The
    full-size GPU check of hot experts' weight gradients rests on this."""
    r = np.random.default_rng(1)
    n, H, I = 300, 256, 128
    x = oracle.bf16_to_f64(f32_to_bf16_bits(r.standard_normal((n, H)).astype(np.float32)))
    dy = oracle.bf16_to_f64(f32_to_bf16_bits(r.standard_normal((n, H)).astype(np.float32)))
    w13 = f32_to_bf16_bits((r.standard_normal((1, 2 * I, H)) / 16).astype(np.float32))
    w2 = f32_to_bf16_bits((r.standard_normal((1, H, I)) / 16).astype(np.float32))
    w = r.random((n, 1))
    one = np.zeros((n, 1), np.int32)
    run = lambda a, b: oracle.backward(x, one, w, a, b, dy, mode=oracle.BF16,  # noqa: E731
                                       store=oracle.STORE_BF16, with_slack=True)
    full = run(w13, w2)
    feats = np.sort(r.choice(I, 16, replace=False))
    cols = np.concatenate([feats, I + feats])
    sub = run(w13[:, cols], w2[:, :, feats])
    assert np.array_equal(full[1][0][cols], sub[1][0])           # dW13 rows
    assert np.array_equal(full[2][0][:, feats], sub[2][0])       # dW2 columns
    assert np.array_equal(full[5][0][cols], sub[5][0])           # their slack
    assert np.array_equal(full[6][0][:, feats], sub[6][0])
    # and not trivially: another subset's rows differ
    other = np.setdiff1d(np.arange(I), feats)[:16]
    assert not np.array_equal(full[1][0][other], sub[1][0])


def test_weight_gradient_window_grows_with_the_expert_rows():
    """A weight gradient over n rows may round either way when its exact value lies within
    2^-19 max(1, sqrt(n / 2048)) sum|terms| (+ 2^-20 of the value) of a rounding midpoint:
    the tensor cores' fp32 error grows with the length of the sum (measured on GB300 up to
    65535 rows). One dW13 element is built to lie 0.0029296875 above the midpoint
    1.00390625 of the bf16 values 1 and 1.0078125, with sum|terms| = 1199.0068 from 1200
    nonzero rows and the rest zero: over 2048 rows the window is 0.00229 and the rounding is
    certain (slack 0); over 8192 rows (the same nonzero rows) it is 0.00457 and the element
    is flagged with the slack of one bf16 step."""
    H, I = 8, 2
    target = 1.0 + 0.0068359375
    col = np.zeros(8192)
    col[:1198:2], col[1:1198:2] = 1.0, -1.0                # sum 0, sum|.| 1198
    col[1198], col[1199] = 1.0, 0.0068359375               # both exact in bf16
    out = {}
    for n in (2048, 8192):
        # dW13[0][c] = sum_r dA[r][0] x[r][c] with x = 1; dW2[c][0] = sum_r dy[r][c] (w*h)[r][0]
        # with dy = 1: both equal the sum of `col` over the first n rows
        da = np.zeros((n, 2 * I))
        sh = np.zeros((n, I))
        da[:, 0] = sh[:, 0] = col[:n]
        _, d13, d2, _, _, s13, s2 = oracle.backward(
            np.ones((n, H)), np.zeros((n, 1), np.int32), np.ones((n, 1)),
            np.zeros((1, 2 * I, H)), np.zeros((1, H, I)), np.ones((n, H)), mode=oracle.BF16,
            store=oracle.STORE_BF16, with_slack=True, given={"da_in": da, "sh_in": sh})
        assert np.all(d13[0, 0] == oracle.round_bf16(target)), d13[0, 0]  # 1.0078125
        assert np.all(d2[0][:, 0] == oracle.round_bf16(target)), d2[0][:, 0]
        out[n] = (s13[0, 0], s2[0][:, 0])
    for s in out[2048]:
        assert np.all(s == 0.0), s
    for s in out[8192]:
        assert np.all(s == 2.0 ** -7), s
