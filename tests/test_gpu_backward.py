"""GPU parity of the layer backward (BF16) against the oracle: dx, dW13, dW2, the
router-weight gradient and the logit gradient; run to run; full size on samples."""
import numpy as np
import pytest

import oracle
from harness import TOL_BF16, bf16_dev_to_f64, inputs, rel_err, sample_tokens, to_dev
from mixture_experts_layer_deterministic_gb300 import binding as B
from mixture_experts_layer_deterministic_gb300.buffers import MoELayer
from workloads import CONFIGS
from workloads.synth import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


def gpu_backward(dims, x, logits, w13, w2, dy, MB, reps=1, recompute=False):
    import torch
    T, H, I, E, K = dims
    L = MoELayer(T, H, I, E, K, MB, 0, B.MOK_BF16, backward=True)
    xd, w13d, w2d, dyd = to_dev(x), to_dev(w13), to_dev(w2), to_dev(dy)
    L.route(to_dev(logits))
    L.schedule()
    R = T * K
    pre = torch.empty(max(R, 1), 2 * I, dtype=torch.float32, device="cuda")
    y = torch.empty(max(T, 1), H, dtype=torch.float32, device="cuda")
    L.forward(xd, w13d, w2d, y, saved_preact=pre)
    outs = []
    for _ in range(reps):
        dx = torch.empty(xd.shape, dtype=torch.float32, device="cuda")
        dw13 = torch.empty(w13d.shape, dtype=torch.float32, device="cuda")
        dw2 = torch.empty(w2d.shape, dtype=torch.float32, device="cuda")
        dtk = torch.empty(max(R, 1), dtype=torch.float32, device="cuda")
        dlg = torch.empty(max(T, 1), E, dtype=torch.float32, device="cuda")
        L.backward(xd, None if recompute else pre, w13d, w2d, dyd, dx, dw13, dw2, dtk, dlg)
        outs.append((dx, dw13, dw2, dtk, dlg))
    torch.cuda.synchronize()
    st, dev = B.mok_read_device_status()
    assert st == B.MOK_OK and dev == B.MOK_OK
    res = [dict(dx=dx, dw13=dw13, dw2=dw2, dtk=dtk[:R].view(T, K), dlg=dlg[:T])
           for dx, dw13, dw2, dtk, dlg in outs]
    idx = L.idx[:R].view(T, K).cpu().numpy()
    w = L.w[:R].view(T, K).cpu().numpy().astype(np.float64)
    return res, idx, w


def small_case(T, H, I, E, K, seed, scale=0.05, skew=0.0):
    r = np.random.default_rng(seed)
    x = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    lg = (r.standard_normal((T, E)) - skew * np.log1p(np.arange(E))).astype(np.float32)
    w13 = f32_to_bf16_bits((r.standard_normal((E, 2 * I, H)) * scale).astype(np.float32))
    w2 = f32_to_bf16_bits((r.standard_normal((E, H, I)) * scale).astype(np.float32))
    dy = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    return x, lg, w13, w2, dy


def host(t):
    import torch
    return bf16_dev_to_f64(t) if t.dtype == torch.bfloat16 else t.cpu().numpy()


def same_bits(a, b):
    import torch
    return torch.equal(a.view(torch.uint8) if a.dtype != torch.uint8 else a,
                       b.view(torch.uint8) if b.dtype != torch.uint8 else b)


def check_all(g, idx, w, x, w13, w2, dy, E):
    dx_o, dw13_o, dw2_o, dtk_o, sdx, sdw13, sdw2 = oracle.backward(
        oracle.bf16_to_f64(x), idx, w, w13, w2, oracle.bf16_to_f64(dy), mode=oracle.BF16,
        with_slack=True)
    dl_o = oracle.router_grad(idx, w, dtk_o, E)
    for name, got, want, sl in (("dx", g["dx"], dx_o, sdx), ("dw13", g["dw13"], dw13_o, sdw13),
                                ("dw2", g["dw2"], dw2_o, sdw2), ("d_topk_w", g["dtk"], dtk_o, None),
                                ("d_logits", g["dlg"], dl_o, None)):
        err = rel_err(host(got).reshape(want.shape), want, sl)
        assert err <= TOL_BF16, (name, err, rel_err(host(got).reshape(want.shape), want))


def test_tiny_config():
    cfg = CONFIGS["tiny"]
    d = inputs(cfg)
    r = np.random.default_rng(77)
    dy = f32_to_bf16_bits(r.standard_normal((cfg.T, cfg.H)).astype(np.float32))
    res, idx, w = gpu_backward((cfg.T, cfg.H, cfg.I, cfg.E, cfg.K), d["x"], d["logits"],
                               d["w13"], d["w2"], dy, cfg.minibatch, reps=2)
    check_all(res[0], idx, w, d["x"], d["w13"], d["w2"], dy, cfg.E)
    for k in res[0]:
        assert same_bits(res[0][k], res[1][k]), k  # bitwise run to run


@pytest.mark.parametrize("dims,skew", [((600, 256, 256, 16, 4), 0.0),
                                       ((333, 384, 128, 24, 3), 3.0),
                                       ((50, 128, 128, 8, 8), 0.0)])
def test_ragged_and_empty_experts(dims, skew):
    x, lg, w13, w2, dy = small_case(*dims, seed=dims[0], skew=skew)
    res, idx, w = gpu_backward(dims, x, lg, w13, w2, dy, 100)
    if skew:
        assert len(np.unique(idx)) < dims[3]  # some experts get no rows
    check_all(res[0], idx, w, x, w13, w2, dy, dims[3])


def test_large_experts_and_a_partial_column_block():
    """Skewed routing gives two experts about 3x the rows of an even split (their weight
    gradients run K over 1000 and 880 rows) and leaves three experts empty; I=384 makes the
    last 256-wide column block of dW2 half past the end of its rows."""
    dims = (1000, 256, 384, 8, 2)
    x, lg, w13, w2, dy = small_case(*dims, seed=5, skew=4.0)
    res, idx, w = gpu_backward(dims, x, lg, w13, w2, dy, 2368, reps=2)
    counts = np.bincount(idx.reshape(-1), minlength=dims[3])
    assert counts.max() > 2 * 352, counts
    check_all(res[0], idx, w, x, w13, w2, dy, dims[3])
    for k in res[0]:
        assert same_bits(res[0][k], res[1][k]), k  # bitwise run to run


@pytest.mark.parametrize("dims,MB", [((256, 256, 128, 8, 2), 64),
                                     ((600, 256, 256, 16, 4), 100),
                                     ((333, 384, 128, 24, 3), 2368)])
def test_recompute_matches_saved_preact(dims, MB):
    """Without saved pre-activations the backward recomputes the gate/up GEMM with the
    forward's tiles and K order, so every output equals the saved-A path bit for bit (the
    forward here runs in several ring passes when MB < R)."""
    x, lg, w13, w2, dy = small_case(*dims, seed=11)
    a, _, _ = gpu_backward(dims, x, lg, w13, w2, dy, MB)
    b, _, _ = gpu_backward(dims, x, lg, w13, w2, dy, MB, recompute=True)
    for k in a[0]:
        assert same_bits(a[0][k], b[0][k]), k


def test_full_size_bwd():
    cfg = CONFIGS["bwd_bf16"]
    d = inputs(cfg)
    dims = (cfg.T, cfg.H, cfg.I, cfg.E, cfg.K)
    res, idx, w = gpu_backward(dims, d["x"], d["logits"], d["w13"], d["w2"], d["dy"],
                               cfg.minibatch, reps=2)
    g = res[0]
    for k in g:
        assert same_bits(g[k], res[1][k]), k
    rc, _, _ = gpu_backward(dims, d["x"], d["logits"], d["w13"], d["w2"], d["dy"],
                            cfg.minibatch, recompute=True)
    for k in g:
        assert same_bits(g[k], rc[0][k]), ("recompute", k)
    # token-local outputs on sampled tokens
    toks = sample_tokens(cfg.T, 128, seed=cfg.seed)
    idx_s = idx[toks]
    used = np.unique(idx_s)
    remap = np.full(cfg.E, -1, np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    xs = oracle.bf16_to_f64(d["x"][toks])
    dys = oracle.bf16_to_f64(d["dy"][toks])
    dx_o, _, _, dtk_o, sdx, _, _ = oracle.backward(xs, remap[idx_s], w[toks], d["w13"][used],
                                                   d["w2"][used], dys, weight_grads=False,
                                                   mode=oracle.BF16, with_slack=True)
    import torch
    tk = torch.from_numpy(toks).cuda()
    assert rel_err(host(g["dx"][tk]), dx_o, sdx) <= TOL_BF16
    assert rel_err(host(g["dtk"][tk]), dtk_o) <= TOL_BF16
    dl_o = oracle.router_grad(idx_s, w[toks], dtk_o, cfg.E)
    assert rel_err(host(g["dlg"][tk]), dl_o) <= TOL_BF16
    # per-expert weight gradients on sampled experts: the expert's own rows only
    r = np.random.default_rng(5)
    counts = np.bincount(idx.reshape(-1), minlength=cfg.E)
    for e in list(r.choice(np.flatnonzero(counts > 0), 3, replace=False)) + \
            [int(np.argmax(counts))]:
        t_e, k_e = np.nonzero(idx == e)
        order = np.argsort(t_e * cfg.K + k_e, kind="stable")
        t_e, k_e = t_e[order], k_e[order]
        _, dw13_o, dw2_o, _, _, s13, s2 = oracle.backward(
            oracle.bf16_to_f64(d["x"][t_e]), np.zeros((len(t_e), 1), np.int32),
            w[t_e, k_e][:, None], d["w13"][e:e + 1], d["w2"][e:e + 1],
            oracle.bf16_to_f64(d["dy"][t_e]), mode=oracle.BF16, with_slack=True)
        g13 = host(g["dw13"][e]).reshape(-1)
        g2 = host(g["dw2"][e]).reshape(-1)
        assert rel_err(g13, dw13_o.reshape(-1), s13) <= TOL_BF16, (e, rel_err(g13, dw13_o.reshape(-1)))
        assert rel_err(g2, dw2_o.reshape(-1), s2) <= TOL_BF16, (e, rel_err(g2, dw2_o.reshape(-1)))
