"""GPU parity of the MXFP8 layer backward against the oracle's MXFP8 backward mode: the G
GEMM on dy and W2 quantized along H, the dgrad GEMM on dA and W13 quantized along 2I, the
weight gradients on bf16 operands. Bit-exact pre-quantized (transposed) weights; dx, dW13,
dW2 and the router gradients within the MXFP8 tolerance; run to run; full size on
samples."""
import numpy as np
import pytest

import oracle
from harness import TOL_MXFP8, inputs, rel_err, sample_tokens, to_dev
from mixture_experts_layer_deterministic_gb300 import binding as B
from mixture_experts_layer_deterministic_gb300.buffers import (MoELayer, backward_mxfp8,
                                                                 quantize_mxfp8,
                                                                 quantize_mxfp8_transposed)
from workloads import CONFIGS
from workloads.synth import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


def test_transposed_weight_quantization_is_bit_exact():
    r = np.random.default_rng(3)
    w = f32_to_bf16_bits((r.standard_normal((3, 256, 384)) *
                          np.exp(r.uniform(-6, 6, (3, 256, 1)))).astype(np.float32))
    q, s = quantize_mxfp8_transposed(to_dev(w))
    qo, so = oracle.mxfp8_quantize_bf16(np.ascontiguousarray(w.transpose(0, 2, 1)))
    np.testing.assert_array_equal(q.cpu().numpy(), qo)
    np.testing.assert_array_equal(s.cpu().numpy(), so)


def gpu_backward_mx(dims, x, logits, w13, w2, dy, MB, reps=1):
    import torch
    T, H, I, E, K = dims
    L = MoELayer(T, H, I, E, K, MB, 0, B.MOK_MXFP8, backward=True)
    xd, dyd, w13d, w2d = to_dev(x), to_dev(dy), to_dev(w13), to_dev(w2)
    q13, s13 = quantize_mxfp8(w13d)
    q2, s2 = quantize_mxfp8(w2d)
    w13t, w2t = quantize_mxfp8_transposed(w13d), quantize_mxfp8_transposed(w2d)
    L.route(to_dev(logits))
    L.schedule()
    R = T * K
    f32 = dict(dtype=torch.float32, device="cuda")
    pre = torch.empty(max(R, 1), 2 * I, **f32)
    y = torch.empty(max(T, 1), H, **f32)
    L.forward(xd, q13, q2, y, s13, s2, pre)
    outs = []
    for _ in range(reps):
        dx = torch.empty(max(T, 1), H, **f32)
        dw13 = torch.empty(E, 2 * I, H, **f32)
        dw2 = torch.empty(E, H, I, **f32)
        dtk = torch.empty(max(R, 1), **f32)
        dlg = torch.empty(max(T, 1), E, **f32)
        backward_mxfp8(L, xd, pre, w13t, w2t, dyd, dx, dw13, dw2, dtk, dlg)
        outs.append(dict(dx=dx[:T], dw13=dw13, dw2=dw2, dtk=dtk[:R].view(T, K), dlg=dlg[:T]))
    torch.cuda.synchronize()
    st, dev = B.mok_read_device_status()
    assert st == B.MOK_OK and dev == B.MOK_OK
    idx = L.idx[:R].view(T, K).cpu().numpy()
    w = L.w[:R].view(T, K).cpu().numpy().astype(np.float64)
    return outs, idx, w


def host(t):
    return t.cpu().numpy()


def check_all(g, idx, w, x, w13, w2, dy, E):
    dx_o, dw13_o, dw2_o, dtk_o, sdx, sdw13, sdw2 = oracle.backward(
        oracle.bf16_to_f64(x), idx, w, w13, w2, oracle.bf16_to_f64(dy), mode=oracle.MXFP8,
        with_slack=True)
    dl_o = oracle.router_grad(idx, w, dtk_o, E)
    for name, got, want, sl in (("dx", g["dx"], dx_o, sdx), ("dw13", g["dw13"], dw13_o, sdw13),
                                ("dw2", g["dw2"], dw2_o, sdw2), ("d_topk_w", g["dtk"], dtk_o, None),
                                ("d_logits", g["dlg"], dl_o, None)):
        err = rel_err(host(got).reshape(want.shape), want, sl)
        assert err <= TOL_MXFP8, (name, err, rel_err(host(got).reshape(want.shape), want))


def small_case(T, H, I, E, K, seed, scale=0.05, skew=0.0):
    r = np.random.default_rng(seed)
    x = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    lg = (r.standard_normal((T, E)) - skew * np.log1p(np.arange(E))).astype(np.float32)
    w13 = f32_to_bf16_bits((r.standard_normal((E, 2 * I, H)) * scale).astype(np.float32))
    w2 = f32_to_bf16_bits((r.standard_normal((E, H, I)) * scale).astype(np.float32))
    dy = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    return x, lg, w13, w2, dy


def test_tiny_config():
    cfg = CONFIGS["tiny"]
    d = inputs(cfg)
    r = np.random.default_rng(78)
    dy = f32_to_bf16_bits(r.standard_normal((cfg.T, cfg.H)).astype(np.float32))
    dims = (cfg.T, cfg.H, cfg.I, cfg.E, cfg.K)
    outs, idx, w = gpu_backward_mx(dims, d["x"], d["logits"], d["w13"], d["w2"], dy,
                                   cfg.minibatch, reps=2)
    check_all(outs[0], idx, w, d["x"], d["w13"], d["w2"], dy, cfg.E)
    import torch
    for k in outs[0]:  # bitwise run to run
        assert torch.equal(outs[0][k].view(torch.int32), outs[1][k].view(torch.int32)), k


@pytest.mark.parametrize("dims,skew", [((600, 256, 256, 16, 4), 0.0),
                                       ((333, 384, 128, 24, 3), 3.0)])
def test_ragged_and_empty_experts(dims, skew):
    x, lg, w13, w2, dy = small_case(*dims, seed=dims[0] + 1, skew=skew)
    outs, idx, w = gpu_backward_mx(dims, x, lg, w13, w2, dy, 100)
    if skew:
        assert len(np.unique(idx)) < dims[3]  # some experts get no rows
    check_all(outs[0], idx, w, x, w13, w2, dy, dims[3])


def test_full_size_sampled():
    cfg = CONFIGS["bwd_bf16"]
    d = inputs(cfg)
    dims = (cfg.T, cfg.H, cfg.I, cfg.E, cfg.K)
    outs, idx, w = gpu_backward_mx(dims, d["x"], d["logits"], d["w13"], d["w2"], d["dy"],
                                   cfg.minibatch)
    g = outs[0]
    # few tokens: the oracle's MXFP8 mode holds the used experts' weights in float64
    toks = sample_tokens(cfg.T, 6, seed=cfg.seed + 7)
    idx_s = idx[toks]
    used = np.unique(idx_s)
    remap = np.full(cfg.E, -1, np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    dx_o, _, _, dtk_o, sdx, _, _ = oracle.backward(
        oracle.bf16_to_f64(d["x"][toks]), remap[idx_s], w[toks], d["w13"][used],
        d["w2"][used], oracle.bf16_to_f64(d["dy"][toks]), weight_grads=False,
        mode=oracle.MXFP8, with_slack=True)
    assert rel_err(host(g["dx"])[toks], dx_o, sdx) <= TOL_MXFP8
    assert rel_err(host(g["dtk"])[toks], dtk_o) <= TOL_MXFP8
    # weight gradients of a sampled expert: its own rows only
    r = np.random.default_rng(9)
    counts = np.bincount(idx.reshape(-1), minlength=cfg.E)
    for e in r.choice(np.nonzero(counts)[0], size=1, replace=False):
        rows = np.argwhere(idx == e)
        t_e = rows[:, 0]
        idx_e = np.zeros((len(t_e), 1), np.int32)
        w_e = w[rows[:, 0], rows[:, 1]][:, None]
        _, dw13_o, dw2_o, _, _, s13, s2 = oracle.backward(
            oracle.bf16_to_f64(d["x"][t_e]), idx_e, w_e, d["w13"][[e]], d["w2"][[e]],
            oracle.bf16_to_f64(d["dy"][t_e]), mode=oracle.MXFP8, with_slack=True)
        assert rel_err(host(g["dw13"][e]), dw13_o[0], s13[0]) <= TOL_MXFP8
        assert rel_err(host(g["dw2"][e]), dw2_o[0], s2[0]) <= TOL_MXFP8


def test_argument_errors_are_reported():
    import torch
    T, H, I, E, K = 64, 128, 128, 4, 2
    u8 = dict(dtype=torch.uint8, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    x = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    dy = torch.zeros_like(x)
    w13t = (torch.zeros(E, H, 2 * I, **u8), torch.zeros(E, H, 2 * I // 32, **u8))
    w2t = (torch.zeros(E, I, H, **u8), torch.zeros(E, I, H // 32, **u8))
    dx = torch.zeros(T, H, **f32)
    dw13, dw2 = torch.zeros(E, 2 * I, H, **f32), torch.zeros(E, H, I, **f32)
    dtk = torch.zeros(T * K, **f32)
    pre = torch.zeros(T * K, 2 * I, **f32)
    for prec, saved, want in ((B.MOK_MXFP8, None, B.MOK_ERR_INVALID_ARG),   # A is required
                              (B.MOK_BF16, pre, B.MOK_ERR_INVALID_ARG)):    # not an MXFP8 layer
        L = MoELayer(T, H, I, E, K, 64, 0, prec, backward=True)
        L.route(torch.zeros(T, E, **f32))
        L.schedule()
        st = B.mok_backward_mxfp8(L.cfg, x, L.sched.struct, L.w, saved, w13t[0], w13t[1],
                                  w2t[0], w2t[1], dy, dx, dw13, dw2, dtk, None, L.ws_b,
                                  L.ws_b_n)
        assert st == want, (prec, st)
    # the shared expert's BF16 backward refuses MXFP8 configurations
    Lm = MoELayer(T, H, I, E, K, 64, 0, B.MOK_MXFP8)
    ws = torch.empty(max(1, B.mok_workspace_size(Lm.cfg, B.MOK_WS_SHARED_BACKWARD)), **u8)
    st = B.mok_shared_expert_backward(Lm.cfg, x, torch.zeros(2 * I, H, dtype=torch.bfloat16,
                                                             device="cuda"),
                                      torch.zeros(H, I, dtype=torch.bfloat16, device="cuda"),
                                      torch.zeros(T, 2 * I, **f32), dy, dx,
                                      torch.zeros(2 * I, H, **f32), torch.zeros(H, I, **f32),
                                      ws, ws.numel())
    assert st == B.MOK_ERR_UNSUPPORTED
    # rows of a transposed quantization come in blocks of 32
    st = B.mok_quantize_mxfp8_transposed(torch.zeros(1, 48, 64, dtype=torch.bfloat16,
                                                     device="cuda"), 1, 48, 64,
                                         torch.zeros(64 * 48, **u8), torch.zeros(64 * 2, **u8))
    assert st == B.MOK_ERR_INVALID_ARG
    torch.cuda.synchronize()
    st, dev = B.mok_read_device_status()
    assert st == B.MOK_OK and dev == B.MOK_OK
