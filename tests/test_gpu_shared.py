"""GPU parity of the shared-expert forward against the oracle: every token also passes
through one SwiGLU expert with weight one, added to the routed output. The oracle of the
shared expert is its own layer forward with one expert and top-1 routing at weight one
(the E=1, K=1 case, pinned on the CPU as a plain SwiGLU FFN)."""
import numpy as np
import pytest

import oracle
from harness import TOL_BF16, TOL_MXFP8, inputs, rel_err, sample_tokens, to_dev
from mixture_experts_layer_deterministic_gb300 import binding as B
from mixture_experts_layer_deterministic_gb300.buffers import (MoELayer, SharedExpert,
                                                                 quantize_mxfp8)
from workloads import CONFIGS
from workloads.synth import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


def shared_weights(H, I, seed, scale):
    r = np.random.default_rng(seed)
    w13s = f32_to_bf16_bits((r.standard_normal((2 * I, H)) * scale).astype(np.float32))
    w2s = f32_to_bf16_bits((r.standard_normal((H, I)) * scale).astype(np.float32))
    return w13s, w2s


def gpu_routed_plus_shared(dims, x, logits, w13, w2, w13s, w2s, MB=2368, reps=1):
    import torch
    T, H, I, E, K = dims
    L = MoELayer(T, H, I, E, K, MB, 0, B.MOK_BF16)
    S = SharedExpert(L)
    xd, w13d, w2d, w13sd, w2sd = to_dev(x), to_dev(w13), to_dev(w2), to_dev(w13s), to_dev(w2s)
    L.route(to_dev(logits))
    L.schedule()
    pre_s = torch.empty(max(T, 1), 2 * I, dtype=torch.float32, device="cuda")
    outs = []
    for _ in range(reps):
        y = torch.empty(max(T, 1), H, dtype=torch.float32, device="cuda")
        L.forward(xd, w13d, w2d, y)
        y_routed = y[:T].clone()
        S.forward(xd, w13sd, w2sd, y, saved_preact=pre_s)
        outs.append((y_routed.cpu().numpy(), y[:T].cpu().numpy()))
    torch.cuda.synchronize()
    st, dev = B.mok_read_device_status()
    assert st == B.MOK_OK and dev == B.MOK_OK
    R = T * K
    idx = L.idx[:R].view(T, K).cpu().numpy()
    w = L.w[:R].view(T, K).cpu().numpy().astype(np.float64)
    return outs, idx, w, pre_s[:T].cpu().numpy()


def oracle_shared(x_bits, w13s, w2s):
    T = x_bits.shape[0]
    return oracle.forward(oracle.bf16_to_f64(x_bits), np.zeros((T, 1), np.int32),
                          np.ones((T, 1)), w13s[None], w2s[None], mode=oracle.BF16,
                          with_slack=True)


def check(outs, idx, w, pre_s, x, w13, w2, w13s, w2s, toks=None):
    y_routed, y_total = outs[0]
    if toks is not None:
        idx_s = idx[toks]
        used = np.unique(idx_s)
        remap = np.full(w13.shape[0], -1, np.int32)
        remap[used] = np.arange(len(used), dtype=np.int32)
        yr, sr = oracle.forward(oracle.bf16_to_f64(x[toks]), remap[idx_s], w[toks], w13[used],
                                w2[used], mode=oracle.BF16, with_slack=True)
        ys, ss = oracle_shared(x[toks], w13s, w2s)
        y_routed, y_total, pre_s, xs = y_routed[toks], y_total[toks], pre_s[toks], x[toks]
    else:
        yr, sr = oracle.forward(oracle.bf16_to_f64(x), idx, w, w13, w2, mode=oracle.BF16,
                                with_slack=True)
        ys, ss = oracle_shared(x, w13s, w2s)
        xs = x
    # the routed part is untouched and the total is the routed plus the shared output
    assert rel_err(y_routed, yr, sr) <= TOL_BF16
    assert rel_err(y_total, yr + ys, sr + ss) <= TOL_BF16
    # the shared output alone, as the GPU's fp32 difference
    assert rel_err(y_total - y_routed, ys, ss) <= TOL_BF16
    # saved pre-activations: fp32 dot products of the bf16 operands, whose products are
    # exact in fp32; n-term fp32 summation stays within n * 2^-24 * sum|terms| of the exact
    # sum (the recursive-summation bound), elementwise
    xf, wf = oracle.bf16_to_f64(xs), oracle.bf16_to_f64(w13s)
    a = xf @ wf.T
    bound = xf.shape[1] * 2.0 ** -24 * (np.abs(xf) @ np.abs(wf).T)
    assert np.all(np.abs(pre_s - a) <= bound)


def test_tiny_config():
    cfg = CONFIGS["tiny"]
    d = inputs(cfg)
    w13s, w2s = shared_weights(cfg.H, cfg.I, 5, 0.05)
    dims = (cfg.T, cfg.H, cfg.I, cfg.E, cfg.K)
    outs, idx, w, pre_s = gpu_routed_plus_shared(dims, d["x"], d["logits"], d["w13"], d["w2"],
                                                 w13s, w2s, cfg.minibatch, reps=2)
    check(outs, idx, w, pre_s, d["x"], d["w13"], d["w2"], w13s, w2s)
    np.testing.assert_array_equal(outs[0][1], outs[1][1])  # bitwise run to run


@pytest.mark.parametrize("dims", [(300, 256, 128, 8, 2), (1, 128, 128, 4, 1),
                                  (517, 384, 256, 16, 4)])
def test_ragged_token_counts(dims):
    T, H, I, E, K = dims
    r = np.random.default_rng(T)
    x = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    lg = r.standard_normal((T, E)).astype(np.float32)
    w13 = f32_to_bf16_bits((r.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32))
    w2 = f32_to_bf16_bits((r.standard_normal((E, H, I)) * 0.05).astype(np.float32))
    w13s, w2s = shared_weights(H, I, T + 1, 0.05)
    outs, idx, w, pre_s = gpu_routed_plus_shared(dims, x, lg, w13, w2, w13s, w2s, 100)
    check(outs, idx, w, pre_s, x, w13, w2, w13s, w2s)


def test_full_size_sampled_tokens():
    cfg = CONFIGS["fwd_bf16"]
    d = inputs(cfg)
    w13s, w2s = shared_weights(cfg.H, cfg.I, 9, cfg.w_std)
    dims = (cfg.T, cfg.H, cfg.I, cfg.E, cfg.K)
    outs, idx, w, pre_s = gpu_routed_plus_shared(dims, d["x"], d["logits"], d["w13"], d["w2"],
                                                 w13s, w2s, cfg.minibatch)
    check(outs, idx, w, pre_s, d["x"], d["w13"], d["w2"], w13s, w2s,
          toks=sample_tokens(cfg.T, 128, seed=3))


def test_mxfp8_config_needs_the_mxfp8_entry():
    import torch
    L = MoELayer(64, 128, 128, 4, 2, 64, 0, B.MOK_MXFP8)
    ws = torch.empty(max(1, B.mok_workspace_size(L.cfg, B.MOK_WS_SHARED)), dtype=torch.uint8,
                     device="cuda")
    x = torch.zeros(64, 128, dtype=torch.bfloat16, device="cuda")
    w13s = torch.zeros(256, 128, dtype=torch.bfloat16, device="cuda")
    w2s = torch.zeros(128, 128, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(64, 128, dtype=torch.float32, device="cuda")
    st = B.mok_shared_expert_forward(L.cfg, x, w13s, w2s, y, None, ws, ws.numel())
    assert st == B.MOK_ERR_UNSUPPORTED
    # and the MXFP8 entry point takes MXFP8 configurations only
    Lb = MoELayer(64, 128, 128, 4, 2, 64, 0, B.MOK_BF16)
    u8 = dict(dtype=torch.uint8, device="cuda")
    st = B.mok_shared_expert_forward_mxfp8(Lb.cfg, x, torch.zeros(256, 128, **u8),
                                           torch.zeros(256, 4, **u8), torch.zeros(128, 128, **u8),
                                           torch.zeros(128, 4, **u8), y, None, ws, ws.numel())
    assert st == B.MOK_ERR_INVALID_ARG
    torch.cuda.synchronize()
    st, dev = B.mok_read_device_status()
    assert st == B.MOK_OK and dev == B.MOK_OK


def gpu_routed_plus_shared_mx(dims, x, logits, w13, w2, w13s, w2s, MB=2368, reps=1):
    """MXFP8 layer: routed forward, then the shared expert added on pre-quantized weights."""
    import torch
    T, H, I, E, K = dims
    L = MoELayer(T, H, I, E, K, MB, 0, B.MOK_MXFP8)
    S = SharedExpert(L)
    xd = to_dev(x)
    q13, s13 = quantize_mxfp8(to_dev(w13))
    q2, s2 = quantize_mxfp8(to_dev(w2))
    ws13, ws2 = quantize_mxfp8(to_dev(w13s)), quantize_mxfp8(to_dev(w2s))
    L.route(to_dev(logits))
    L.schedule()
    pre_s = torch.empty(max(T, 1), 2 * I, dtype=torch.float32, device="cuda")
    outs = []
    for _ in range(reps):
        y = torch.empty(max(T, 1), H, dtype=torch.float32, device="cuda")
        L.forward(xd, q13, q2, y, s13, s2)
        y_routed = y[:T].clone()
        S.forward(xd, ws13, ws2, y, saved_preact=pre_s)
        outs.append((y_routed.cpu().numpy(), y[:T].cpu().numpy()))
    torch.cuda.synchronize()
    st, dev = B.mok_read_device_status()
    assert st == B.MOK_OK and dev == B.MOK_OK
    R = T * K
    idx = L.idx[:R].view(T, K).cpu().numpy()
    w = L.w[:R].view(T, K).cpu().numpy().astype(np.float64)
    return outs, idx, w, pre_s[:T].cpu().numpy()


def check_mx(outs, idx, w, pre_s, x, w13, w2, w13s, w2s, toks=None):
    """The oracle's MXFP8 mode: the routed layer, and the shared expert as its own layer with
    one expert and top-1 routing at weight one."""
    y_routed, y_total = outs[0]
    xs, idx_s, w_s, w13u, w2u = x, idx, w, w13, w2
    if toks is not None:
        used = np.unique(idx[toks])
        remap = np.full(w13.shape[0], -1, np.int32)
        remap[used] = np.arange(len(used), dtype=np.int32)
        xs, idx_s, w_s, w13u, w2u = x[toks], remap[idx[toks]], w[toks], w13[used], w2[used]
        y_routed, y_total, pre_s = y_routed[toks], y_total[toks], pre_s[toks]
    xf = oracle.bf16_to_f64(xs)
    q = lambda a: oracle.mxfp8_quantize_bf16(a)
    yr, sr = oracle.forward(xf, idx_s, w_s, q(w13u), q(w2u), mode=oracle.MXFP8, with_slack=True)
    T = xs.shape[0]
    ys, ss = oracle.forward(xf, np.zeros((T, 1), np.int32), np.ones((T, 1)),
                            q(w13s[None]), q(w2s[None]), mode=oracle.MXFP8, with_slack=True)
    assert rel_err(y_routed, yr, sr) <= TOL_MXFP8
    assert rel_err(y_total - y_routed, ys, ss) <= TOL_MXFP8
    assert rel_err(y_total, yr + ys, sr + ss) <= TOL_MXFP8
    # saved pre-activations: dot products of the dequantized x and W13s blocks (each product
    # exact in fp32), accumulated by the tensor core; allow 2^-12 of the sum of |terms|
    xq = oracle.mxfp8_dequantize(*oracle.mxfp8_quantize_bf16(xs))
    wq = oracle.mxfp8_dequantize(*oracle.mxfp8_quantize_bf16(w13s))
    a = xq @ wq.T
    assert np.all(np.abs(pre_s - a) <= 2.0 ** -12 * (np.abs(xq) @ np.abs(wq).T) + 1e-30)


def test_mxfp8_tiny_config():
    cfg = CONFIGS["tiny"]
    d = inputs(cfg)
    w13s, w2s = shared_weights(cfg.H, cfg.I, 15, 0.05)
    dims = (cfg.T, cfg.H, cfg.I, cfg.E, cfg.K)
    outs, idx, w, pre_s = gpu_routed_plus_shared_mx(dims, d["x"], d["logits"], d["w13"],
                                                    d["w2"], w13s, w2s, cfg.minibatch, reps=2)
    check_mx(outs, idx, w, pre_s, d["x"], d["w13"], d["w2"], w13s, w2s)
    np.testing.assert_array_equal(outs[0][1], outs[1][1])  # bitwise run to run


@pytest.mark.parametrize("dims", [(300, 256, 128, 8, 2), (1, 128, 128, 4, 1),
                                  (517, 384, 256, 16, 4)])
def test_mxfp8_ragged_token_counts(dims):
    T, H, I, E, K = dims
    r = np.random.default_rng(T + 11)
    x = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    lg = r.standard_normal((T, E)).astype(np.float32)
    w13 = f32_to_bf16_bits((r.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32))
    w2 = f32_to_bf16_bits((r.standard_normal((E, H, I)) * 0.05).astype(np.float32))
    w13s, w2s = shared_weights(H, I, T + 12, 0.05)
    outs, idx, w, pre_s = gpu_routed_plus_shared_mx(dims, x, lg, w13, w2, w13s, w2s, 100)
    check_mx(outs, idx, w, pre_s, x, w13, w2, w13s, w2s)


def test_mxfp8_full_size_sampled_tokens():
    cfg = CONFIGS["fwd_mxfp8"]
    d = inputs(cfg)
    w13s, w2s = shared_weights(cfg.H, cfg.I, 19, cfg.w_std)
    dims = (cfg.T, cfg.H, cfg.I, cfg.E, cfg.K)
    outs, idx, w, pre_s = gpu_routed_plus_shared_mx(dims, d["x"], d["logits"], d["w13"],
                                                    d["w2"], w13s, w2s, cfg.minibatch)
    check_mx(outs, idx, w, pre_s, d["x"], d["w13"], d["w2"], w13s, w2s,
             toks=sample_tokens(cfg.T, 24, seed=5))


def gpu_step_with_shared(dims, x, logits, w13, w2, w13s, w2s, dy, MB=2368):
    """Routed forward + shared forward, then routed backward + shared backward (which adds
    into dx); returns dx after the routed part, dx in total, the shared weight gradients."""
    import torch
    T, H, I, E, K = dims
    L = MoELayer(T, H, I, E, K, MB, 0, B.MOK_BF16, backward=True)
    S = SharedExpert(L)
    xd, dyd = to_dev(x), to_dev(dy)
    w13d, w2d, w13sd, w2sd = to_dev(w13), to_dev(w2), to_dev(w13s), to_dev(w2s)
    L.route(to_dev(logits))
    L.schedule()
    R = T * K
    f32 = dict(dtype=torch.float32, device="cuda")
    pre, pre_s = torch.empty(R, 2 * I, **f32), torch.empty(T, 2 * I, **f32)
    y = torch.empty(T, H, **f32)
    L.forward(xd, w13d, w2d, y, saved_preact=pre)
    S.forward(xd, w13sd, w2sd, y, saved_preact=pre_s)
    dx = torch.empty(T, H, **f32)
    dw13, dw2 = torch.empty(E, 2 * I, H, **f32), torch.empty(E, H, I, **f32)
    dtk = torch.empty(R, **f32)
    L.backward(xd, pre, w13d, w2d, dyd, dx, dw13, dw2, dtk)
    dx_routed = dx.clone()
    dw13s, dw2s = torch.empty(2 * I, H, **f32), torch.empty(H, I, **f32)
    S.backward(xd, w13sd, w2sd, pre_s, dyd, dx, dw13s, dw2s)
    torch.cuda.synchronize()
    st, dev = B.mok_read_device_status()
    assert st == B.MOK_OK and dev == B.MOK_OK
    idx = L.idx[:R].view(T, K).cpu().numpy()
    w = L.w[:R].view(T, K).cpu().numpy().astype(np.float64)
    return (dx_routed.cpu().numpy(), dx.cpu().numpy(), dw13s.cpu().numpy(),
            dw2s.cpu().numpy(), idx, w)


@pytest.mark.parametrize("dims", [(256, 256, 128, 8, 2), (300, 256, 128, 8, 2),
                                  (517, 384, 256, 16, 4)])
def test_backward_with_shared_expert(dims):
    T, H, I, E, K = dims
    r = np.random.default_rng(T + 2)
    x = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    lg = r.standard_normal((T, E)).astype(np.float32)
    w13 = f32_to_bf16_bits((r.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32))
    w2 = f32_to_bf16_bits((r.standard_normal((E, H, I)) * 0.05).astype(np.float32))
    dy = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    w13s, w2s = shared_weights(H, I, T + 3, 0.05)
    dx_r, dx, dw13s, dw2s, idx, w = gpu_step_with_shared(dims, x, lg, w13, w2, w13s, w2s, dy)
    xf, dyf = oracle.bf16_to_f64(x), oracle.bf16_to_f64(dy)
    dx_ro, _, _, _, sdx_r, _, _ = oracle.backward(xf, idx, w, w13, w2, dyf, weight_grads=False,
                                                  mode=oracle.BF16, with_slack=True)
    # the shared expert: one expert, top-1 routing at weight one
    dx_so, dw13_so, dw2_so, _, sdx_s, s13, s2 = oracle.backward(
        xf, np.zeros((T, 1), np.int32), np.ones((T, 1)), w13s[None], w2s[None], dyf,
        mode=oracle.BF16, with_slack=True)
    assert rel_err(dx_r, dx_ro, sdx_r) <= TOL_BF16
    assert rel_err(dx, dx_ro + dx_so, sdx_r + sdx_s) <= TOL_BF16
    assert rel_err(dx - dx_r, dx_so, sdx_s) <= TOL_BF16
    assert rel_err(dw13s, dw13_so[0], s13[0]) <= TOL_BF16
    assert rel_err(dw2s, dw2_so[0], s2[0]) <= TOL_BF16


def gpu_step_with_shared_mx(dims, x, logits, w13, w2, w13s, w2s, dy, MB=2368, reps=1):
    """MXFP8 layer: routed and shared forward (both saving pre-activations), then the routed
    MXFP8 backward and the shared MXFP8 backward, which adds into dx."""
    import torch
    from mixture_experts_layer_deterministic_gb300.buffers import (backward_mxfp8,
                                                                     quantize_mxfp8_transposed)
    T, H, I, E, K = dims
    L = MoELayer(T, H, I, E, K, MB, 0, B.MOK_MXFP8, backward=True)
    S = SharedExpert(L)
    xd, dyd = to_dev(x), to_dev(dy)
    w13d, w2d, w13sd, w2sd = to_dev(w13), to_dev(w2), to_dev(w13s), to_dev(w2s)
    q13, s13 = quantize_mxfp8(w13d)
    q2, s2 = quantize_mxfp8(w2d)
    w13t, w2t = quantize_mxfp8_transposed(w13d), quantize_mxfp8_transposed(w2d)
    ws13, ws2 = quantize_mxfp8(w13sd), quantize_mxfp8(w2sd)
    wst13 = quantize_mxfp8_transposed(w13sd[None])
    wst2 = quantize_mxfp8_transposed(w2sd[None])
    L.route(to_dev(logits))
    L.schedule()
    R = T * K
    f32 = dict(dtype=torch.float32, device="cuda")
    pre, pre_s = torch.empty(max(R, 1), 2 * I, **f32), torch.empty(max(T, 1), 2 * I, **f32)
    y = torch.empty(max(T, 1), H, **f32)
    L.forward(xd, q13, q2, y, s13, s2, pre)
    S.forward(xd, ws13, ws2, y, saved_preact=pre_s)
    outs = []
    for _ in range(reps):
        dx = torch.empty(max(T, 1), H, **f32)
        dw13, dw2 = torch.empty(E, 2 * I, H, **f32), torch.empty(E, H, I, **f32)
        dtk = torch.empty(max(R, 1), **f32)
        backward_mxfp8(L, xd, pre, w13t, w2t, dyd, dx, dw13, dw2, dtk)
        dx_routed = dx[:T].clone()
        dw13s, dw2s = torch.empty(2 * I, H, **f32), torch.empty(H, I, **f32)
        S.backward(xd, wst13, wst2, pre_s, dyd, dx, dw13s, dw2s)
        outs.append(dict(dx_r=dx_routed.cpu().numpy(), dx=dx[:T].cpu().numpy(),
                         dw13s=dw13s.cpu().numpy(), dw2s=dw2s.cpu().numpy()))
    torch.cuda.synchronize()
    st, dev = B.mok_read_device_status()
    assert st == B.MOK_OK and dev == B.MOK_OK
    idx = L.idx[:R].view(T, K).cpu().numpy()
    w = L.w[:R].view(T, K).cpu().numpy().astype(np.float64)
    return outs, idx, w


@pytest.mark.parametrize("dims", [(256, 256, 128, 8, 2), (300, 256, 128, 8, 2),
                                  (517, 384, 256, 16, 4), (1, 128, 128, 4, 1)])
def test_mxfp8_backward_with_shared_expert(dims):
    T, H, I, E, K = dims
    r = np.random.default_rng(T + 21)
    x = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    lg = r.standard_normal((T, E)).astype(np.float32)
    w13 = f32_to_bf16_bits((r.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32))
    w2 = f32_to_bf16_bits((r.standard_normal((E, H, I)) * 0.05).astype(np.float32))
    dy = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    w13s, w2s = shared_weights(H, I, T + 23, 0.05)
    outs, idx, w = gpu_step_with_shared_mx(dims, x, lg, w13, w2, w13s, w2s, dy, reps=2)
    g = outs[0]
    xf, dyf = oracle.bf16_to_f64(x), oracle.bf16_to_f64(dy)
    dx_ro, _, _, _, sdx_r, _, _ = oracle.backward(xf, idx, w, w13, w2, dyf, weight_grads=False,
                                                  mode=oracle.MXFP8, with_slack=True)
    # the shared expert in the oracle's MXFP8 mode: one expert, top-1 routing at weight one
    dx_so, dw13_so, dw2_so, _, sdx_s, s13, s2 = oracle.backward(
        xf, np.zeros((T, 1), np.int32), np.ones((T, 1)), w13s[None], w2s[None], dyf,
        mode=oracle.MXFP8, with_slack=True)
    assert rel_err(g["dx_r"], dx_ro, sdx_r) <= TOL_MXFP8
    assert rel_err(g["dx"] - g["dx_r"], dx_so, sdx_s) <= TOL_MXFP8
    assert rel_err(g["dx"], dx_ro + dx_so, sdx_r + sdx_s) <= TOL_MXFP8
    assert rel_err(g["dw13s"], dw13_so[0], s13[0]) <= TOL_MXFP8
    assert rel_err(g["dw2s"], dw2_so[0], s2[0]) <= TOL_MXFP8
    for k in g:  # bitwise run to run
        np.testing.assert_array_equal(g[k], outs[1][k])


def test_mxfp8_shared_backward_argument_errors():
    import torch
    T, H, I = 64, 128, 128
    u8 = dict(dtype=torch.uint8, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    x = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    wt13 = (torch.zeros(H, 2 * I, **u8), torch.zeros(H, 2 * I // 32, **u8))
    wt2 = (torch.zeros(I, H, **u8), torch.zeros(I, H // 32, **u8))
    pre = torch.zeros(T, 2 * I, **f32)
    dx = torch.zeros(T, H, **f32)
    dw13s, dw2s = torch.zeros(2 * I, H, **f32), torch.zeros(H, I, **f32)
    for prec, saved, want in ((B.MOK_MXFP8, None, B.MOK_ERR_INVALID_ARG),  # pre required
                              (B.MOK_BF16, pre, B.MOK_ERR_INVALID_ARG)):   # not MXFP8
        L = MoELayer(T, H, I, 4, 2, 64, 0, prec)
        ws = torch.empty(max(1, B.mok_workspace_size(L.cfg, B.MOK_WS_SHARED_BACKWARD)), **u8)
        st = B.mok_shared_expert_backward_mxfp8(L.cfg, x, wt13[0], wt13[1], wt2[0], wt2[1],
                                                saved, x, dx, dw13s, dw2s, ws, ws.numel())
        assert st == want, (prec, st)
    torch.cuda.synchronize()
    st, dev = B.mok_read_device_status()
    assert st == B.MOK_OK and dev == B.MOK_OK
