"""GPU parity of the MXFP8 layer backward against the oracle's MXFP8 backward mode: the G
GEMM on dy and W2 quantized along H, the dgrad GEMM on dA and W13 quantized along 2I, the
weight gradients on bf16 operands. Bit-exact pre-quantized (transposed) weights; step by
step (tests/bwd_checks.py: the saved A, dA and its MXFP8 codes and scales, w*h, dx, dW13,
dW2, d_topk_w, d_logits) and end to end within the MXFP8 tolerance; run to run; full size
on 128 sampled tokens and 4 experts."""
import numpy as np
import pytest

import oracle
from bwd_checks import check_expert, check_tokens, gpu_state
from harness import inputs, same_bits, sample_tokens, to_dev
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


def gpu_backward_mx(dims, x, logits, w13, w2, dy, MB, reps=1, flags=0):
    import torch
    T, H, I, E, K = dims
    L = MoELayer(T, H, I, E, K, MB, 0, B.MOK_MXFP8, backward=True, flags=flags)
    xd, dyd, w13d, w2d = to_dev(x), to_dev(dy), to_dev(w13), to_dev(w2)
    q13, s13 = quantize_mxfp8(w13d)
    q2, s2 = quantize_mxfp8(w2d)
    w13t, w2t = quantize_mxfp8_transposed(w13d), quantize_mxfp8_transposed(w2d)
    del w13d, w2d
    L.route(to_dev(logits))
    L.schedule()
    R = T * K
    st = dict(dtype=L.dtype, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    pre = torch.empty(max(R, 1), 2 * I, **st)
    y = torch.empty(max(T, 1), H, **st)
    L.forward(xd, q13, q2, y, s13, s2, pre)
    outs = []
    for _ in range(reps):
        dx = torch.empty(max(T, 1), H, **st)
        dw13 = torch.empty(E, 2 * I, H, **st)
        dw2 = torch.empty(E, H, I, **st)
        dtk = torch.empty(max(R, 1), **f32)
        dlg = torch.empty(max(T, 1), E, **f32)
        backward_mxfp8(L, xd, pre, w13t, w2t, dyd, dx, dw13, dw2, dtk, dlg)
        outs.append(dict(dx=dx[:T], dw13=dw13, dw2=dw2, dtk=dtk[:R].view(T, K), dlg=dlg[:T]))
    torch.cuda.synchronize()
    s, dev = B.mok_read_device_status()
    assert s == B.MOK_OK and dev == B.MOK_OK
    g = dict(idx=L.idx[:R].view(T, K).cpu().numpy(),
             w=L.w[:R].view(T, K).cpu().numpy().astype(np.float64), T=T, K=K, E=E)
    return outs, g, L, pre


def small_case(T, H, I, E, K, seed, scale=0.05, skew=0.0):
    r = np.random.default_rng(seed)
    x = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    lg = (r.standard_normal((T, E)) - skew * np.log1p(np.arange(E))).astype(np.float32)
    w13 = f32_to_bf16_bits((r.standard_normal((E, 2 * I, H)) * scale).astype(np.float32))
    w2 = f32_to_bf16_bits((r.standard_normal((E, H, I)) * scale).astype(np.float32))
    dy = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    return x, lg, w13, w2, dy


def check_all(outs, g, L, pre, x, w13, w2, dy, tokens=None, experts=None, mxw=None, tag=""):
    st = gpu_state(L, L.ws_b, B.MOK_WS_BACKWARD, pre)
    gg = dict(g, **outs[0])
    tokens = np.arange(L.T) if tokens is None else tokens
    check_tokens(gg, st, x, w13, w2, dy, True, tokens, mxw=mxw, tag=" mx" + tag)
    for e in (range(L.E) if experts is None else experts):
        check_expert(gg, st, x, w13, w2, dy, True, int(e), mxw=mxw, tag=" mx" + tag)


def test_tiny_config():
    cfg = CONFIGS["tiny"]
    d = inputs(cfg)
    r = np.random.default_rng(78)
    dy = f32_to_bf16_bits(r.standard_normal((cfg.T, cfg.H)).astype(np.float32))
    dims = (cfg.T, cfg.H, cfg.I, cfg.E, cfg.K)
    outs, g, L, pre = gpu_backward_mx(dims, d["x"], d["logits"], d["w13"], d["w2"], dy,
                                      cfg.minibatch, reps=2)
    check_all(outs, g, L, pre, d["x"], d["w13"], d["w2"], dy)
    for k in outs[0]:  # bitwise run to run
        assert same_bits(outs[0][k], outs[1][k]), k


@pytest.mark.parametrize("dims,skew", [((600, 256, 256, 16, 4), 0.0),
                                       ((333, 384, 128, 24, 3), 3.0)])
def test_ragged_and_empty_experts(dims, skew):
    x, lg, w13, w2, dy = small_case(*dims, seed=dims[0] + 1, skew=skew)
    outs, g, L, pre = gpu_backward_mx(dims, x, lg, w13, w2, dy, 100)
    if skew:
        assert len(np.unique(g["idx"])) < dims[3]  # some experts get no rows
    check_all(outs, g, L, pre, x, w13, w2, dy)


@pytest.mark.parametrize("dims", [(600, 256, 256, 16, 4), (2048, 256, 128, 4, 2)])
def test_weight_gradients_on_sm_pairs(dims):
    """The MXFP8 backward's weight gradients (bf16 operands) on SM pairs equal those on one
    SM bit for bit; the second shape (1024 rows per expert) takes the pairs by default."""
    x, lg, w13, w2, dy = small_case(*dims, seed=dims[0] + 3)
    a = gpu_backward_mx(dims, x, lg, w13, w2, dy, 100, flags=B.MOK_FLAG_SM_PAIR_GEMMS)[0]
    b = gpu_backward_mx(dims, x, lg, w13, w2, dy, 100, flags=B.MOK_FLAG_ONE_SM_GEMMS)[0]
    for k in a[0]:
        assert same_bits(a[0][k], b[0][k]), k


def test_full_size_sampled():
    """128 sampled tokens and 4 sampled experts, the hottest among them; the oracle's
    three MXFP8 quantizations of the weights are computed once, by the oracle."""
    cfg = CONFIGS["bwd_bf16"]
    d = inputs(cfg)
    dims = (cfg.T, cfg.H, cfg.I, cfg.E, cfg.K)
    outs, g, L, pre = gpu_backward_mx(dims, d["x"], d["logits"], d["w13"], d["w2"], d["dy"],
                                      cfg.minibatch)
    mxw = (oracle.mxfp8_quantize_bf16(d["w13"]), oracle.quantize_transposed_bf16(d["w13"]),
           oracle.quantize_transposed_bf16(d["w2"]))
    toks = sample_tokens(cfg.T, 128, seed=cfg.seed + 7)
    counts = np.bincount(g["idx"].reshape(-1), minlength=cfg.E)
    r = np.random.default_rng(9)
    experts = list(r.choice(np.flatnonzero(counts > 0), 3, replace=False)) + \
        [int(np.argmax(counts))]
    check_all(outs, g, L, pre, d["x"], d["w13"], d["w2"], d["dy"], tokens=toks,
              experts=experts, mxw=mxw, tag=" full")


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
