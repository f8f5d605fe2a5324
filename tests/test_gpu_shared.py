"""GPU parity of the shared expert against the oracle: every token also passes through one
SwiGLU expert with weight one, whose output is added to the routed output (and, in the
backward, whose input gradient is added to the routed dx). The oracle of the shared expert
is its own layer with one expert and top-1 routing at weight one (the E=1, K=1 case, pinned
on the CPU as a plain SwiGLU FFN), adding to a given output (oracle_rows y_in / dx_in).

Step by step: the shared expert's h (or its MXFP8 codes), its saved pre-activations, y =
bf16(y_routed + o) from the GPU's own routed y and h; in the backward its dA, w*h (and MXFP8
dA codes) from the GPU's own A, dx = bf16(dx_routed + W13s^T dA) and its weight gradients
from the GPU's own dA and w*h. End to end within the stated tolerance."""
import numpy as np
import pytest

import oracle
from harness import (TOL_BF16, TOL_MXFP8, check_codes, check_exact, check_tol, host, inputs,
                     oracle_forward_tokens, preact_rows, same_bits, sample_tokens, to_dev)
from mixture_experts_layer_deterministic_gb300 import binding as B
from mixture_experts_layer_deterministic_gb300.buffers import (MoELayer, SharedExpert,
                                                                 quantize_mxfp8,
                                                                 workspace_item)
from workloads import CONFIGS
from workloads.synth import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


def shared_weights(H, I, seed, scale):
    r = np.random.default_rng(seed)
    w13s = f32_to_bf16_bits((r.standard_normal((2 * I, H)) * scale).astype(np.float32))
    w2s = f32_to_bf16_bits((r.standard_normal((H, I)) * scale).astype(np.float32))
    return w13s, w2s


def _step(v):
    return np.ldexp(1.0, np.frexp(np.maximum(np.abs(v), 1e-300))[1] - 8)


def gpu_routed_plus_shared(dims, x, logits, w13, w2, w13s, w2s, prec, MB=2368, reps=1,
                           flags=0):
    import torch
    T, H, I, E, K = dims
    L = MoELayer(T, H, I, E, K, MB, 0, prec, flags=flags)
    S = SharedExpert(L)
    xd = to_dev(x)
    if prec == B.MOK_MXFP8:
        q13, s13 = quantize_mxfp8(to_dev(w13))
        q2, s2 = quantize_mxfp8(to_dev(w2))
        ws13, ws2 = quantize_mxfp8(to_dev(w13s)), quantize_mxfp8(to_dev(w2s))
    else:
        q13, s13, q2, s2 = to_dev(w13), None, to_dev(w2), None
        ws13, ws2 = to_dev(w13s), to_dev(w2s)
    L.route(to_dev(logits))
    L.schedule()
    pre_s = torch.empty(max(T, 1), 2 * I, dtype=L.dtype, device="cuda")
    outs = []
    for _ in range(reps):
        y = torch.empty(max(T, 1), H, dtype=L.dtype, device="cuda")
        L.forward(xd, q13, q2, y, s13, s2)
        y_routed = y[:T].clone()
        S.forward(xd, ws13, ws2, y, saved_preact=pre_s)
        outs.append((y_routed, y[:T]))
    torch.cuda.synchronize()
    st, dev = B.mok_read_device_status()
    assert st == B.MOK_OK and dev == B.MOK_OK
    R = T * K
    g = dict(idx=L.idx[:R].view(T, K).cpu().numpy(),
             w=L.w[:R].view(T, K).cpu().numpy().astype(np.float64),
             y_routed=host(outs[0][0]), y=host(outs[0][1]),
             pre_s=preact_rows(host(pre_s[:T])), outs=outs)
    if prec == B.MOK_MXFP8:
        g["h_q"] = workspace_item(S.ws, L.cfg, B.MOK_WS_SHARED, B.MOK_ITEM_H_RING).view(
            -1, I)[:T].cpu().numpy()
        g["h_s"] = workspace_item(S.ws, L.cfg, B.MOK_WS_SHARED, B.MOK_ITEM_H_RING_SCALE).view(
            -1, I // 32)[:T].cpu().numpy()
        g["h"] = oracle.mxfp8_dequantize(g["h_q"], g["h_s"])
    else:
        g["h"] = host(workspace_item(S.ws, L.cfg, B.MOK_WS_SHARED, B.MOK_ITEM_H_RING)
                      .view(torch.bfloat16).view(-1, I)[:T])
    return g


def check_forward(g, x, w13, w2, w13s, w2s, mx, toks=None, tag=""):
    T = x.shape[0]
    toks = np.arange(T) if toks is None else toks
    mode, tol = (oracle.MXFP8, TOL_MXFP8) if mx else (oracle.BF16, TOL_BF16)
    q = oracle.mxfp8_quantize_bf16
    w13o, w2o = (q(w13), q(w2)) if mx else (w13, w2)
    w13so, w2so = (q(w13s[None]), q(w2s[None])) if mx else (w13s[None], w2s[None])
    n = len(toks)
    xf = oracle.bf16_to_f64(x[toks])
    one = dict(idx=np.zeros((n, 1), np.int32), w=np.ones((n, 1)))
    # routed part, end to end
    yr, sr = oracle_forward_tokens(toks, x, g["idx"], g["w"], w13o, w2o, mode)
    check_tol("shared: routed y e2e" + tag, g["y_routed"][toks], yr, sr, tol,
              max_slack_rms=1.2 if mx else 0.4)
    # the shared expert's h against its own chain from x
    _, _, ro = oracle.forward(xf, one["idx"], one["w"], w13so, w2so, mode=mode, with_slack=True,
                              store=oracle.STORE_BF16, rows=("h", "h_slack", "h_q", "h_scale"))
    if mx:
        check_codes("shared h codes" + tag, g["h_q"][toks], g["h_s"][toks], ro["h_q"],
                    ro["h_scale"], ro["h_slack"])
    else:
        check_exact("shared h" + tag, g["h"][toks], ro["h"], ro["h_slack"])
    # y = bf16(y_routed + o) from the GPU's own routed y and h
    y_s, sl_s = oracle.forward(xf, one["idx"], one["w"], w13so, w2so, mode=mode, with_slack=True,
                               store=oracle.STORE_BF16,
                               given={"h_in": g["h"][toks], "y_in": g["y_routed"][toks]})
    check_exact("shared y | gpu routed y, h" + tag, g["y"][toks], y_s, sl_s)
    # end to end: the oracle's routed y with the shared output added (its slack widened by
    # the routed slack and one step of the final rounding)
    y_e, sl_e = oracle.forward(xf, one["idx"], one["w"], w13so, w2so, mode=mode,
                               with_slack=True, store=oracle.STORE_BF16, given={"y_in": yr})
    check_tol("shared y e2e" + tag, g["y"][toks], y_e, sl_e + sr + _step(y_e), tol,
              max_slack_rms=0.3)
    # the saved pre-activations: bf16 of the exact gate/up product
    *_, ra = oracle.backward(xf, one["idx"], one["w"], w13s[None] if mx else w13s[None],
                             w2s[None], np.zeros((n, x.shape[1])), weight_grads=False,
                             mode=mode, store=oracle.STORE_BF16, rows=("a", "a_slack"))
    check_exact("shared saved A" + tag, g["pre_s"][toks], ra["a"], ra["a_slack"])


@pytest.mark.parametrize("prec", [B.MOK_BF16, B.MOK_MXFP8])
def test_tiny_config(prec):
    cfg = CONFIGS["tiny"]
    d = inputs(cfg)
    w13s, w2s = shared_weights(cfg.H, cfg.I, 5, 0.05)
    dims = (cfg.T, cfg.H, cfg.I, cfg.E, cfg.K)
    g = gpu_routed_plus_shared(dims, d["x"], d["logits"], d["w13"], d["w2"], w13s, w2s, prec,
                               cfg.minibatch, reps=2)
    check_forward(g, d["x"], d["w13"], d["w2"], w13s, w2s, prec == B.MOK_MXFP8)
    assert same_bits(g["outs"][0][1], g["outs"][1][1])  # bitwise run to run


@pytest.mark.parametrize("prec", [B.MOK_BF16, B.MOK_MXFP8])
@pytest.mark.parametrize("dims", [(300, 256, 128, 8, 2), (1, 128, 128, 4, 1),
                                  (517, 384, 256, 16, 4)])
def test_ragged_token_counts(dims, prec):
    T, H, I, E, K = dims
    r = np.random.default_rng(T + prec)
    x = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    lg = r.standard_normal((T, E)).astype(np.float32)
    w13 = f32_to_bf16_bits((r.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32))
    w2 = f32_to_bf16_bits((r.standard_normal((E, H, I)) * 0.05).astype(np.float32))
    w13s, w2s = shared_weights(H, I, T + 1, 0.05)
    g = gpu_routed_plus_shared(dims, x, lg, w13, w2, w13s, w2s, prec, 100)
    check_forward(g, x, w13, w2, w13s, w2s, prec == B.MOK_MXFP8)


@pytest.mark.parametrize("name", ["fwd_bf16", "fwd_mxfp8"])
def test_full_size_sampled_tokens(name):
    cfg = CONFIGS[name]
    d = inputs(cfg)
    w13s, w2s = shared_weights(cfg.H, cfg.I, 9, cfg.w_std)
    dims = (cfg.T, cfg.H, cfg.I, cfg.E, cfg.K)
    prec = B.MOK_MXFP8 if cfg.prec == "mxfp8" else B.MOK_BF16
    g = gpu_routed_plus_shared(dims, d["x"], d["logits"], d["w13"], d["w2"], w13s, w2s, prec,
                               cfg.minibatch)
    check_forward(g, d["x"], d["w13"], d["w2"], w13s, w2s, prec == B.MOK_MXFP8,
                  toks=sample_tokens(cfg.T, 128, seed=3), tag=" full")


def test_mxfp8_config_needs_the_mxfp8_entry():
    import torch
    L = MoELayer(64, 128, 128, 4, 2, 64, 0, B.MOK_MXFP8)
    ws = torch.empty(max(1, B.mok_workspace_size(L.cfg, B.MOK_WS_SHARED)), dtype=torch.uint8,
                     device="cuda")
    x = torch.zeros(64, 128, dtype=torch.bfloat16, device="cuda")
    w13s = torch.zeros(256, 128, dtype=torch.bfloat16, device="cuda")
    w2s = torch.zeros(128, 128, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(64, 128, dtype=torch.bfloat16, device="cuda")
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


# ---------------------------------------------------------------- backward

def gpu_step_with_shared(dims, x, logits, w13, w2, w13s, w2s, dy, prec, MB=2368, reps=1,
                         flags=0):
    """Routed and shared forward (both saving pre-activations), then the routed backward and
    the shared backward, which adds into dx; dx after the routed part, dx in total and the
    shared weight gradients, with the shared backward's workspace intermediates."""
    import torch
    from mixture_experts_layer_deterministic_gb300.buffers import (backward_mxfp8,
                                                                     quantize_mxfp8_transposed)
    T, H, I, E, K = dims
    L = MoELayer(T, H, I, E, K, MB, 0, prec, backward=True, flags=flags)
    S = SharedExpert(L)
    xd, dyd = to_dev(x), to_dev(dy)
    w13d, w2d, w13sd, w2sd = to_dev(w13), to_dev(w2), to_dev(w13s), to_dev(w2s)
    mx = prec == B.MOK_MXFP8
    if mx:
        q13, s13 = quantize_mxfp8(w13d)
        q2, s2 = quantize_mxfp8(w2d)
        w13t, w2t = quantize_mxfp8_transposed(w13d), quantize_mxfp8_transposed(w2d)
        ws13, ws2 = quantize_mxfp8(w13sd), quantize_mxfp8(w2sd)
        wst13 = quantize_mxfp8_transposed(w13sd[None])
        wst2 = quantize_mxfp8_transposed(w2sd[None])
    L.route(to_dev(logits))
    L.schedule()
    R = T * K
    st = dict(dtype=L.dtype, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    pre, pre_s = torch.empty(max(R, 1), 2 * I, **st), torch.empty(max(T, 1), 2 * I, **st)
    y = torch.empty(max(T, 1), H, **st)
    if mx:
        L.forward(xd, q13, q2, y, s13, s2, pre)
        S.forward(xd, ws13, ws2, y, saved_preact=pre_s)
    else:
        L.forward(xd, w13d, w2d, y, saved_preact=pre)
        S.forward(xd, w13sd, w2sd, y, saved_preact=pre_s)
    outs = []
    for _ in range(reps):
        dx = torch.empty(max(T, 1), H, **st)
        dw13, dw2 = torch.empty(E, 2 * I, H, **st), torch.empty(E, H, I, **st)
        dtk = torch.empty(max(R, 1), **f32)
        if mx:
            backward_mxfp8(L, xd, pre, w13t, w2t, dyd, dx, dw13, dw2, dtk)
        else:
            L.backward(xd, pre, w13d, w2d, dyd, dx, dw13, dw2, dtk)
        dx_routed = dx[:T].clone()
        dw13s, dw2s = torch.empty(2 * I, H, **st), torch.empty(H, I, **st)
        if mx:
            S.backward(xd, wst13, wst2, pre_s, dyd, dx, dw13s, dw2s)
        else:
            S.backward(xd, w13sd, w2sd, pre_s, dyd, dx, dw13s, dw2s)
        outs.append(dict(dx_r=dx_routed, dx=dx[:T], dw13s=dw13s, dw2s=dw2s))
    torch.cuda.synchronize()
    s, dev = B.mok_read_device_status()
    assert s == B.MOK_OK and dev == B.MOK_OK
    item = lambda it: workspace_item(S.ws_b, L.cfg, B.MOK_WS_SHARED_BACKWARD, it)  # noqa
    gi = dict(a=preact_rows(host(pre_s[:T])),
              da=host(item(B.MOK_ITEM_DA).view(torch.bfloat16).view(-1, 2 * I)[:T]),
              sh=host(item(B.MOK_ITEM_WH).view(torch.bfloat16).view(-1, I)[:T]))
    if mx:
        gi["da_q"] = item(B.MOK_ITEM_DA_Q).view(-1, 2 * I)[:T].cpu().numpy()
        gi["da_s"] = item(B.MOK_ITEM_DA_SCALE).view(-1, 2 * I // 32)[:T].cpu().numpy()
        gi["daq"] = oracle.mxfp8_dequantize(gi["da_q"], gi["da_s"])
    idx = L.idx[:R].view(T, K).cpu().numpy()
    w = L.w[:R].view(T, K).cpu().numpy().astype(np.float64)
    return outs, gi, idx, w


def check_backward(outs, gi, idx, w, x, w13, w2, w13s, w2s, dy, mx):
    T, H = x.shape
    mode, tol = (oracle.MXFP8, TOL_MXFP8) if mx else (oracle.BF16, TOL_BF16)
    g = {k: host(v) for k, v in outs[0].items()}
    xf, dyf = oracle.bf16_to_f64(x), oracle.bf16_to_f64(dy)
    one_idx, one_w = np.zeros((T, 1), np.int32), np.ones((T, 1))
    dx_ro, _, _, _, sdx_r, _, _ = oracle.backward(xf, idx, w, w13, w2, dyf, weight_grads=False,
                                                  mode=mode, store=oracle.STORE_BF16,
                                                  with_slack=True)
    check_tol("shared: routed dx e2e", g["dx_r"], dx_ro, sdx_r, tol,
              max_slack_rms=1.2 if mx else 0.4)
    run = lambda **kw: oracle.backward(xf, one_idx, one_w, w13s[None], w2s[None], dyf,  # noqa
                                       mode=mode, store=oracle.STORE_BF16, **kw)
    # dA, w*h (and MXFP8 dA codes) from the GPU's own A
    names = ("da", "da_slack", "sh", "sh_slack") + (("da_q", "da_scale", "daq_slack")
                                                    if mx else ())
    *_, ra = run(weight_grads=False, given={"a_in": gi["a"]}, rows=names)
    check_exact("shared bwd dA | gpu A", gi["da"], ra["da"], ra["da_slack"])
    check_exact("shared bwd w*h | gpu A", gi["sh"], ra["sh"], ra["sh_slack"])
    if mx:
        check_codes("shared bwd dA codes | gpu A", gi["da_q"], gi["da_s"], ra["da_q"],
                    ra["da_scale"], ra["daq_slack"])
    # dx = bf16(dx_routed + W13s^T dA) and the weight gradients from the GPU's operands
    given = {"a_in": gi["a"], "da_in": gi["da"], "sh_in": gi["sh"], "dx_in": g["dx_r"]}
    if mx:
        given["daq_in"] = gi["daq"]
    dx_s, d13, d2, _, sdx_s, s13, s2 = run(with_slack=True, given=given)
    check_exact("shared dx | gpu routed dx, dA", g["dx"], dx_s, sdx_s)
    check_exact("shared dW13 | gpu dA", g["dw13s"], d13[0], s13[0])
    check_exact("shared dW2 | gpu w*h", g["dw2s"], d2[0], s2[0])
    # end to end
    _, d13o, d2o, _, _, s13o, s2o = run(with_slack=True)
    check_tol("shared dW13 e2e", g["dw13s"], d13o[0], s13o[0], tol, max_slack_rms=0.6)
    check_tol("shared dW2 e2e", g["dw2s"], d2o[0], s2o[0], tol, max_slack_rms=0.6)


@pytest.mark.parametrize("prec", [B.MOK_BF16, B.MOK_MXFP8])
@pytest.mark.parametrize("dims", [(256, 256, 128, 8, 2), (300, 256, 128, 8, 2),
                                  (517, 384, 256, 16, 4), (1, 128, 128, 4, 1)])
def test_backward_with_shared_expert(dims, prec):
    T, H, I, E, K = dims
    r = np.random.default_rng(T + 2 + 19 * prec)
    x = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    lg = r.standard_normal((T, E)).astype(np.float32)
    w13 = f32_to_bf16_bits((r.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32))
    w2 = f32_to_bf16_bits((r.standard_normal((E, H, I)) * 0.05).astype(np.float32))
    dy = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    w13s, w2s = shared_weights(H, I, T + 3, 0.05)
    outs, gi, idx, w = gpu_step_with_shared(dims, x, lg, w13, w2, w13s, w2s, dy, prec, reps=2)
    check_backward(outs, gi, idx, w, x, w13, w2, w13s, w2s, dy, prec == B.MOK_MXFP8)
    for k in outs[0]:  # bitwise run to run
        assert same_bits(outs[0][k], outs[1][k]), k


@pytest.mark.parametrize("dims", [(517, 384, 256, 16, 4), (600, 256, 384, 8, 2)])
def test_shared_pair_gemms_equal_one_sm(dims):
    """The shared expert's GEMMs on SM pairs, including the down and dx GEMMs that add into
    y and dx, give the one-SM kernels' bits (y, dx, dW13s, dW2s)."""
    T, H, I, E, K = dims
    r = np.random.default_rng(T + 5)
    x = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    lg = r.standard_normal((T, E)).astype(np.float32)
    w13 = f32_to_bf16_bits((r.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32))
    w2 = f32_to_bf16_bits((r.standard_normal((E, H, I)) * 0.05).astype(np.float32))
    dy = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    w13s, w2s = shared_weights(H, I, T + 6, 0.05)
    runs = [gpu_step_with_shared(dims, x, lg, w13, w2, w13s, w2s, dy, B.MOK_BF16, flags=f)[0]
            for f in (B.MOK_FLAG_SM_PAIR_GEMMS, B.MOK_FLAG_ONE_SM_GEMMS)]
    ys = [gpu_routed_plus_shared(dims, x, lg, w13, w2, w13s, w2s, B.MOK_BF16, flags=f)
          for f in (B.MOK_FLAG_SM_PAIR_GEMMS, B.MOK_FLAG_ONE_SM_GEMMS)]
    for k in runs[0][0]:
        assert same_bits(runs[0][0][k], runs[1][0][k]), k
    assert same_bits(ys[0]["outs"][0][1], ys[1]["outs"][0][1])
    assert np.array_equal(ys[0]["pre_s"], ys[1]["pre_s"])


def test_mxfp8_shared_backward_argument_errors():
    import torch
    T, H, I = 64, 128, 128
    u8 = dict(dtype=torch.uint8, device="cuda")
    bf = dict(dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(T, H, **bf)
    wt13 = (torch.zeros(H, 2 * I, **u8), torch.zeros(H, 2 * I // 32, **u8))
    wt2 = (torch.zeros(I, H, **u8), torch.zeros(I, H // 32, **u8))
    pre = torch.zeros(T, 2 * I, **bf)
    dx = torch.zeros(T, H, **bf)
    dw13s, dw2s = torch.zeros(2 * I, H, **bf), torch.zeros(H, I, **bf)
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
