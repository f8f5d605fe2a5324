"""GPU parity of the layer forward against the oracle (BF16 and MXFP8), run-to-run and
across ring settings; full-size configurations on sampled tokens."""
import numpy as np
import pytest

import oracle
from harness import (TOL_BF16, TOL_MXFP8, inputs, oracle_forward_tokens, rel_err,
                     sample_tokens, to_dev)
from mixture_experts_layer_deterministic_gb300 import binding as B
from mixture_experts_layer_deterministic_gb300.buffers import MoELayer, quantize_mxfp8
from workloads import CONFIGS
from workloads.synth import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


def gpu_forward(dims, x, logits, w13, w2, prec, MB, ring, preact=False, reps=1, wq=None):
    import torch
    T, H, I, E, K = dims
    L = MoELayer(T, H, I, E, K, MB, ring, prec)
    xd = to_dev(x)
    if prec == B.MOK_MXFP8:
        if wq is None:
            wq = quantize_mxfp8(to_dev(w13)) + quantize_mxfp8(to_dev(w2))
        a13, s13, a2, s2 = wq
    else:
        a13, s13, a2, s2 = to_dev(w13), None, to_dev(w2), None
    L.route(to_dev(logits))
    L.schedule()
    R = T * K
    pre = torch.empty(max(R, 1), 2 * I, dtype=torch.float32, device="cuda") if preact else None
    ys = []
    for _ in range(reps):
        y = torch.empty(max(T, 1), H, dtype=torch.float32, device="cuda")
        L.forward(xd, a13, a2, y, s13, s2, pre)
        ys.append(y)
    torch.cuda.synchronize()
    st, dev = B.mok_read_device_status()
    assert st == B.MOK_OK and dev == B.MOK_OK
    idx = L.idx[:R].view(T, K).cpu().numpy()
    w = L.w[:R].view(T, K).cpu().numpy().astype(np.float64)
    return dict(y=[t[:T].cpu().numpy() for t in ys], idx=idx, w=w, pre=pre, wq=wq, L=L)


def small_case(T, H, I, E, K, seed, scale=0.05):
    r = np.random.default_rng(seed)
    x = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    lg = r.standard_normal((T, E)).astype(np.float32)
    w13 = f32_to_bf16_bits((r.standard_normal((E, 2 * I, H)) * scale).astype(np.float32))
    w2 = f32_to_bf16_bits((r.standard_normal((E, H, I)) * scale).astype(np.float32))
    return x, lg, w13, w2


def oracle_y(x, idx, w, w13, w2, mx):
    if mx:
        q13, s13 = oracle.mxfp8_quantize_bf16(w13)
        q2, s2 = oracle.mxfp8_quantize_bf16(w2)
        return oracle.forward(oracle.bf16_to_f64(x), idx, w, (q13, s13), (q2, s2),
                              mode=oracle.MXFP8, with_slack=True)
    return oracle.forward(oracle.bf16_to_f64(x), idx, w, w13, w2, mode=oracle.BF16,
                          with_slack=True)


@pytest.mark.parametrize("prec", [B.MOK_BF16, B.MOK_MXFP8])
def test_tiny_config(prec):
    cfg = CONFIGS["tiny"]
    d = inputs(cfg)
    g = gpu_forward((cfg.T, cfg.H, cfg.I, cfg.E, cfg.K), d["x"], d["logits"], d["w13"],
                    d["w2"], prec, cfg.minibatch, cfg.ring_capacity, reps=3)
    mx = prec == B.MOK_MXFP8
    y_o, sl = oracle_y(d["x"], g["idx"], g["w"], d["w13"], d["w2"], mx)
    err = rel_err(g["y"][0], y_o, sl)
    assert err <= (TOL_MXFP8 if mx else TOL_BF16), err
    for y in g["y"][1:]:
        np.testing.assert_array_equal(y, g["y"][0])  # bitwise run to run


@pytest.mark.parametrize("prec", [B.MOK_BF16, B.MOK_MXFP8])
def test_ragged_multi_pass_rings(prec):
    """Several tiles per expert, ragged tails, 1 and 2 ring slots and a full ring: every
    ring setting gives the same bits, and they match the oracle."""
    dims = (1000, 512, 256, 16, 4)
    x, lg, w13, w2 = small_case(*dims, seed=11)
    outs = []
    for MB, ring in ((300, 0), (300, 700), (300, 300), (128, 0), (1000, 1000)):
        g = gpu_forward(dims, x, lg, w13, w2, prec, MB, ring)
        outs.append(g)
    for g in outs[1:]:
        np.testing.assert_array_equal(g["y"][0], outs[0]["y"][0])
    mx = prec == B.MOK_MXFP8
    y_o, sl = oracle_y(x, outs[0]["idx"], outs[0]["w"], w13, w2, mx)
    err = rel_err(outs[0]["y"][0], y_o, sl)
    assert err <= (TOL_MXFP8 if mx else TOL_BF16), err


@pytest.mark.parametrize("dims", [(40, 128, 128, 8, 8), (300, 256, 128, 1, 1),
                                  (129, 384, 256, 64, 1), (5, 128, 128, 32, 3)])
def test_edge_shapes(dims):
    x, lg, w13, w2 = small_case(*dims, seed=sum(dims))
    g = gpu_forward(dims, x, lg, w13, w2, B.MOK_BF16, 37, 0)
    y_o, sl = oracle_y(x, g["idx"], g["w"], w13, w2, False)
    assert rel_err(g["y"][0], y_o, sl) <= TOL_BF16


def test_empty_batch():
    import torch
    L = MoELayer(0, 256, 128, 8, 2, 16, 0, B.MOK_BF16)
    dummy = torch.zeros(16, dtype=torch.float32, device="cuda")
    B.check(B.mok_forward(L.cfg, dummy, L.sched.struct, L.w, dummy, None, dummy, None, dummy,
                          None, L.ws_f, L.ws_f_n, None))


def test_saved_preact_matches_oracle_gate_up():
    dims = (64, 256, 128, 4, 2)
    x, lg, w13, w2 = small_case(*dims, seed=5)
    g = gpu_forward(dims, x, lg, w13, w2, B.MOK_BF16, 32, 0, preact=True)
    T, H, I, E, K = dims
    pre = g["pre"].cpu().numpy().astype(np.float64).reshape(T * K, 2 * I)
    so = oracle.schedule(g["idx"], E, 32)
    # a = W13[e] x for each sorted row, as a dense product of the bf16 inputs
    xf = oracle.bf16_to_f64(x)
    wf = oracle.bf16_to_f64(w13)
    for r in range(T * K):
        f = so["perm"][r]
        e = g["idx"].reshape(-1)[f]
        a = wf[e] @ xf[f // K]
        assert rel_err(pre[r], a) <= 1e-5  # fp32 accumulation only


# ---------------------------------------------------------------- full-size configurations

def full_case(name, n_tokens=256):
    cfg = CONFIGS[name]
    d = inputs(cfg)
    prec = B.MOK_MXFP8 if cfg.prec == "mxfp8" else B.MOK_BF16
    g = gpu_forward((cfg.T, cfg.H, cfg.I, cfg.E, cfg.K), d["x"], d["logits"], d["w13"],
                    d["w2"], prec, cfg.minibatch, cfg.ring_capacity, reps=2)
    np.testing.assert_array_equal(g["y"][0], g["y"][1])
    toks = sample_tokens(cfg.T, n_tokens, seed=cfg.seed)
    mx = prec == B.MOK_MXFP8
    if mx:
        # the device-quantized weights must equal the oracle's quantization bit for bit
        q13, s13 = oracle.mxfp8_quantize_bf16(d["w13"])
        q2, s2 = oracle.mxfp8_quantize_bf16(d["w2"])
        a13, g13, a2, g2 = g["wq"]
        for got, want in ((a13, q13), (g13, s13), (a2, q2), (g2, s2)):
            assert np.array_equal(got.cpu().numpy(), want)
        wo = ((q13, s13), (q2, s2))
    else:
        wo = (d["w13"], d["w2"])
    y_o, sl = oracle_forward_tokens(toks, d["x"], g["idx"], g["w"], wo[0], wo[1],
                                    mode=oracle.MXFP8 if mx else oracle.BF16)
    err = rel_err(g["y"][0][toks], y_o, sl)
    assert err <= (TOL_MXFP8 if mx else TOL_BF16), err
    return g


@pytest.mark.parametrize("name", ["fwd_bf16", "fwd_mxfp8", "imbalanced_bf16",
                                  "imbalanced_mxfp8"])
def test_full_size(name):
    full_case(name)
