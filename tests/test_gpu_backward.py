"""GPU parity of the layer backward (BF16) against the oracle, step by step and end to end
(tests/bwd_checks.py): the saved A, dA, w*h, dx, dW13, dW2, the router-weight gradient and
the logit gradient; bitwise run to run; the recompute path equal to the saved-A path bit for
bit; full size on sampled tokens and experts (including the hottest)."""
import numpy as np
import pytest

import oracle
from bwd_checks import check_expert, check_expert_features, check_tokens, gpu_state
from harness import inputs, same_bits, sample_tokens, to_dev
from mixture_experts_layer_deterministic_gb300 import binding as B
from mixture_experts_layer_deterministic_gb300.buffers import MoELayer
from workloads import CONFIGS
from workloads.synth import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


def gpu_backward(dims, x, logits, w13, w2, dy, MB, reps=1, recompute=False, flags=0):
    import torch
    T, H, I, E, K = dims
    L = MoELayer(T, H, I, E, K, MB, 0, B.MOK_BF16, backward=True, flags=flags)
    xd, w13d, w2d, dyd = to_dev(x), to_dev(w13), to_dev(w2), to_dev(dy)
    L.route(to_dev(logits))
    L.schedule()
    R = T * K
    st = dict(dtype=L.dtype, device="cuda")
    pre = torch.empty(max(R, 1), 2 * I, **st)
    y = torch.empty(max(T, 1), H, **st)
    L.forward(xd, w13d, w2d, y, saved_preact=pre)
    outs = []
    for _ in range(reps):
        dx = torch.empty(xd.shape, **st)
        dw13 = torch.empty(w13d.shape, **st)
        dw2 = torch.empty(w2d.shape, **st)
        dtk = torch.empty(max(R, 1), dtype=torch.float32, device="cuda")
        dlg = torch.empty(max(T, 1), E, dtype=torch.float32, device="cuda")
        L.backward(xd, None if recompute else pre, w13d, w2d, dyd, dx, dw13, dw2, dtk, dlg)
        outs.append(dict(dx=dx, dw13=dw13, dw2=dw2, dtk=dtk[:R].view(T, K), dlg=dlg[:T]))
    torch.cuda.synchronize()
    s, dev = B.mok_read_device_status()
    assert s == B.MOK_OK and dev == B.MOK_OK
    g = dict(idx=L.idx[:R].view(T, K).cpu().numpy(),
             w=L.w[:R].view(T, K).cpu().numpy().astype(np.float64), T=T, K=K, E=E)
    which = B.MOK_WS_BACKWARD_RECOMPUTE if recompute else B.MOK_WS_BACKWARD
    ws = L.ws_r if recompute else L.ws_b
    # the recompute path's A lives in its workspace; the saved-A path's is `pre`
    return outs, g, L, (ws, which, pre)


def small_case(T, H, I, E, K, seed, scale=0.05, skew=0.0):
    r = np.random.default_rng(seed)
    x = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    lg = (r.standard_normal((T, E)) - skew * np.log1p(np.arange(E))).astype(np.float32)
    w13 = f32_to_bf16_bits((r.standard_normal((E, 2 * I, H)) * scale).astype(np.float32))
    w2 = f32_to_bf16_bits((r.standard_normal((E, H, I)) * scale).astype(np.float32))
    dy = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    return x, lg, w13, w2, dy


def check_all(outs, g, L, wsinfo, x, w13, w2, dy, tokens=None, experts=None, tag=""):
    ws, which, pre = wsinfo
    st = gpu_state(L, ws, which, pre)
    gg = dict(g, **outs[0])
    tokens = np.arange(L.T) if tokens is None else tokens
    check_tokens(gg, st, x, w13, w2, dy, False, tokens, tag=tag)
    for e in (range(L.E) if experts is None else experts):
        check_expert(gg, st, x, w13, w2, dy, False, int(e), tag=tag)


def test_tiny_config():
    cfg = CONFIGS["tiny"]
    d = inputs(cfg)
    r = np.random.default_rng(77)
    dy = f32_to_bf16_bits(r.standard_normal((cfg.T, cfg.H)).astype(np.float32))
    outs, g, L, wsi = gpu_backward((cfg.T, cfg.H, cfg.I, cfg.E, cfg.K), d["x"], d["logits"],
                                   d["w13"], d["w2"], dy, cfg.minibatch, reps=2)
    check_all(outs, g, L, wsi, d["x"], d["w13"], d["w2"], dy)
    for k in outs[0]:
        assert same_bits(outs[0][k], outs[1][k]), k  # bitwise run to run


@pytest.mark.parametrize("dims,skew", [((600, 256, 256, 16, 4), 0.0),
                                       ((333, 384, 128, 24, 3), 3.0),
                                       ((50, 128, 128, 8, 8), 0.0)])
def test_ragged_and_empty_experts(dims, skew):
    x, lg, w13, w2, dy = small_case(*dims, seed=dims[0], skew=skew)
    outs, g, L, wsi = gpu_backward(dims, x, lg, w13, w2, dy, 100)
    if skew:
        assert len(np.unique(g["idx"])) < dims[3]  # some experts get no rows
    check_all(outs, g, L, wsi, x, w13, w2, dy)


def test_large_experts_and_a_partial_column_block():
    """Skewed routing gives two experts about 3x the rows of an even split (their weight
    gradients run K over 1000 and 880 rows) and leaves three experts empty; I=384 makes the
    last 256-wide column block of dW2 half past the end of its rows."""
    dims = (1000, 256, 384, 8, 2)
    x, lg, w13, w2, dy = small_case(*dims, seed=5, skew=4.0)
    outs, g, L, wsi = gpu_backward(dims, x, lg, w13, w2, dy, 2368, reps=2)
    counts = np.bincount(g["idx"].reshape(-1), minlength=dims[3])
    assert counts.max() > 2 * 352, counts
    check_all(outs, g, L, wsi, x, w13, w2, dy)
    for k in outs[0]:
        assert same_bits(outs[0][k], outs[1][k]), k  # bitwise run to run


@pytest.mark.parametrize("dims,MB", [((256, 256, 128, 8, 2), 64),
                                     ((600, 256, 256, 16, 4), 100),
                                     ((333, 384, 128, 24, 3), 2368)])
def test_recompute_matches_saved_preact(dims, MB):
    """Without saved pre-activations the backward recomputes the gate/up GEMM with the
    forward's tiles and K order and stores A as the forward would, so every output equals
    the saved-A path bit for bit."""
    x, lg, w13, w2, dy = small_case(*dims, seed=11)
    a, _, _, _ = gpu_backward(dims, x, lg, w13, w2, dy, MB)
    b, _, _, _ = gpu_backward(dims, x, lg, w13, w2, dy, MB, recompute=True)
    for k in a[0]:
        assert same_bits(a[0][k], b[0][k]), k


@pytest.mark.parametrize("dims,skew,flags", [
    ((600, 256, 256, 16, 4), 0.0, B.MOK_FLAG_SM_PAIR_GEMMS),
    ((333, 384, 128, 24, 3), 3.0, B.MOK_FLAG_SM_PAIR_GEMMS),
    ((1000, 256, 384, 8, 2), 4.0, B.MOK_FLAG_SM_PAIR_GEMMS),
    ((40, 128, 128, 4, 2), 0.0, B.MOK_FLAG_SM_PAIR_GEMMS),
    ((2048, 256, 128, 4, 2), 0.0, 0)])
def test_pair_gemms_equal_one_sm(dims, skew, flags):
    """The weight gradients and the dx GEMM on SM pairs equal the one-SM kernels' results
    bit for bit: the same fixed-order dot products. The shapes give 256-wide and 128-wide
    last M blocks (in the latter rank 1's A half lies wholly past the end), 128-column N
    blocks of dW, token tiles from 16 to 256 rows, empty experts and experts with 3x the
    rows of an even split; the last shape (1024 rows per expert) takes the pairs by
    default, the others are forced onto them."""
    x, lg, w13, w2, dy = small_case(*dims, seed=dims[0] + 1, skew=skew)
    a, _, _, _ = gpu_backward(dims, x, lg, w13, w2, dy, 100, flags=flags)
    b, _, _, _ = gpu_backward(dims, x, lg, w13, w2, dy, 100, flags=B.MOK_FLAG_ONE_SM_GEMMS)
    for k in a[0]:
        assert same_bits(a[0][k], b[0][k]), k


def test_fp32_storage_backward():
    """Under MOK_FLAG_FP32_STORAGE (fp32 A, dx slots, dx and dW) the outputs stay within
    tolerance of the oracle's fp32-storage backward."""
    from harness import TOL_BF16, check_tol, host
    dims = (300, 256, 256, 8, 2)
    T, H, I, E, K = dims
    x, lg, w13, w2, dy = small_case(*dims, seed=21)
    outs, g, L, _ = gpu_backward(dims, x, lg, w13, w2, dy, 64, flags=B.MOK_FLAG_FP32_STORAGE)
    dx_o, d13, d2, dtk_o, sdx, s13, s2 = oracle.backward(
        oracle.bf16_to_f64(x), g["idx"], g["w"], w13, w2, oracle.bf16_to_f64(dy),
        mode=oracle.BF16, store=oracle.STORE_F32, with_slack=True)
    o = outs[0]
    check_tol("bwd dx e2e fp32 storage", host(o["dx"]), dx_o, sdx, TOL_BF16)
    check_tol("bwd dW13 e2e fp32 storage", host(o["dw13"]), d13, s13, TOL_BF16)
    check_tol("bwd dW2 e2e fp32 storage", host(o["dw2"]), d2, s2, TOL_BF16)
    check_tol("bwd d_topk_w e2e fp32 storage", host(o["dtk"]), dtk_o, None, TOL_BF16)


def test_full_size_bwd():
    cfg = CONFIGS["bwd_bf16"]
    d = inputs(cfg)
    dims = (cfg.T, cfg.H, cfg.I, cfg.E, cfg.K)
    outs, g, L, wsi = gpu_backward(dims, d["x"], d["logits"], d["w13"], d["w2"], d["dy"],
                                   cfg.minibatch, reps=2)
    for k in outs[0]:
        assert same_bits(outs[0][k], outs[1][k]), k
    rc, _, _, _ = gpu_backward(dims, d["x"], d["logits"], d["w13"], d["w2"], d["dy"],
                               cfg.minibatch, recompute=True)
    for k in outs[0]:
        assert same_bits(outs[0][k], rc[0][k]), ("recompute", k)
    del rc
    # the weight gradients on SM pairs equal those of the one-SM kernel (the default here)
    pr, _, _, _ = gpu_backward(dims, d["x"], d["logits"], d["w13"], d["w2"], d["dy"],
                               cfg.minibatch, flags=B.MOK_FLAG_SM_PAIR_GEMMS)
    for k in outs[0]:
        assert same_bits(outs[0][k], pr[0][k]), ("SM pairs", k)
    del pr
    # token-local outputs on 128 sampled tokens; weight gradients of 8 sampled experts,
    # the hottest among them
    toks = sample_tokens(cfg.T, 128, seed=cfg.seed)
    counts = np.bincount(g["idx"].reshape(-1), minlength=cfg.E)
    r = np.random.default_rng(5)
    experts = list(r.choice(np.flatnonzero(counts > 0), 7, replace=False)) + \
        [int(np.argmax(counts))]
    check_all(outs, g, L, wsi, d["x"], d["w13"], d["w2"], d["dy"], tokens=toks,
              experts=experts, tag=" full")


@pytest.mark.parametrize("name", ["ring_bf16_e64", "imbalanced_bf16"])
def test_full_size_imbalanced_bwd(name):
    """The backward of the Zipf-routed workloads (8192 tokens over 64 experts; 65536 over
    512): 1280 rows per expert on average, the hottest experts taking every token, some
    none; their dx and weight gradients run on SM pairs by default. Token-local outputs on
    64 sampled tokens; the weight gradients of the hottest expert, a mid-sized one and an
    empty one on 32 sampled features each (a feature's dW13 rows and dW2 column are the
    oracle's expert restricted to that feature)."""
    cfg = CONFIGS[name].with_(passes="bwd", ring_capacity=0)
    d = inputs(cfg)
    dims = (cfg.T, cfg.H, cfg.I, cfg.E, cfg.K)
    outs, g, L, wsi = gpu_backward(dims, d["x"], d["logits"], d["w13"], d["w2"], d["dy"],
                                   cfg.minibatch)
    counts = np.bincount(g["idx"].reshape(-1), minlength=cfg.E)
    assert counts.max() >= cfg.T // 2 and counts.min() == 0, counts  # the skew this test wants
    ws, which, pre = wsi
    st = gpu_state(L, ws, which, pre)
    gg = dict(g, **outs[0])
    check_tokens(gg, st, d["x"], d["w13"], d["w2"], d["dy"], False,
                 sample_tokens(cfg.T, 64, seed=cfg.seed), tag=" zipf")
    nz = np.flatnonzero(counts > 0)
    mid = int(nz[np.argsort(counts[nz], kind="stable")[len(nz) // 2]])
    r = np.random.default_rng(8)
    for e in (int(np.argmax(counts)), mid, int(np.argmin(counts))):
        feats = np.sort(r.choice(cfg.I, 32, replace=False))
        check_expert_features(gg, st, d["x"], d["w13"], d["w2"], d["dy"], e, feats,
                              tag=" zipf")


def test_weight_gradient_fp32_error_within_the_oracle_bound():
    """The oracle's error window of a weight gradient (oracle.dot_rel_rows: 2^-19 times
    max(1, sqrt(n / 2048)) of sum|terms| for a sum over n rows) holds on this GPU: dW13
    stored in fp32 against the exact sums of the GPU's own bf16 dA and x, for experts of
    about 300 to 65535 rows of the Zipf-routed 65536-token workload (64 dW13 rows each; the
    fp64 sums of exact bf16 products are within 2^-37 of exact)."""
    import torch
    cfg = CONFIGS["imbalanced_bf16"].with_(passes="bwd", ring_capacity=0)
    d = inputs(cfg)
    dims = (cfg.T, cfg.H, cfg.I, cfg.E, cfg.K)
    outs, g, L, wsi = gpu_backward(dims, d["x"], d["logits"], d["w13"], d["w2"], d["dy"],
                                   cfg.minibatch, flags=B.MOK_FLAG_FP32_STORAGE)
    ws, which, pre = wsi
    st = gpu_state(L, ws, which, pre)
    counts = np.diff(st["offsets"])
    nz = np.flatnonzero(counts > 0)
    r = np.random.default_rng(4)
    x = to_dev(d["x"])
    for target in (300, 2000, 8000, 16000, 65536):
        e = int(nz[np.argmin(np.abs(counts[nz] - target))])
        n, r0 = int(counts[e]), int(st["offsets"][e])
        t_e = torch.from_numpy((st["perm"][r0:r0 + n] // cfg.K).astype(np.int64)).cuda()
        prow = torch.from_numpy((st["poff"][e] + np.arange(n)).astype(np.int64)).cuda()
        j = torch.from_numpy(np.sort(r.choice(2 * cfg.I, 64, replace=False))).cuda()
        a = st["dA"][prow][:, j].double()
        xe = x[t_e].double()
        exact, mag = a.T @ xe, a.abs().T @ xe.abs()
        got = outs[0]["dw13"][e][j].double()
        ok = mag > 0
        ratio = float(((got - exact).abs()[ok] / mag[ok]).max())
        assert ratio <= oracle.dot_rel_rows(n), (e, n, ratio, oracle.dot_rel_rows(n))
