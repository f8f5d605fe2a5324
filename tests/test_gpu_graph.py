"""The layer's calls are stream-ordered with no host synchronisation and no allocation,
so a training step captures into a CUDA graph; its replay must reproduce the eager
results bit for bit (rings that hold every row, and smaller rings, whose forward is one
persistent launch that resets its own claim counter and tile counters)."""
import numpy as np
import pytest

from harness import same_bits, to_dev
from mixture_experts_layer_deterministic_gb300 import binding as B
from mixture_experts_layer_deterministic_gb300.buffers import MoELayer, SharedExpert
from workloads.synth import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dims,MB,ring", [((256, 256, 128, 8, 2), 64, 0),
                                          ((600, 256, 256, 16, 4), 256, 512)])
def test_captured_step_replays_eager_results(dims, MB, ring):
    import torch
    T, H, I, E, K = dims
    r = np.random.default_rng(T)
    x = to_dev(f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32)))
    lg = to_dev(r.standard_normal((T, E)).astype(np.float32))
    w13 = to_dev(f32_to_bf16_bits((r.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32)))
    w2 = to_dev(f32_to_bf16_bits((r.standard_normal((E, H, I)) * 0.05).astype(np.float32)))
    w13s = to_dev(f32_to_bf16_bits((r.standard_normal((2 * I, H)) * 0.05).astype(np.float32)))
    w2s = to_dev(f32_to_bf16_bits((r.standard_normal((H, I)) * 0.05).astype(np.float32)))
    dy = to_dev(f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32)))
    L = MoELayer(T, H, I, E, K, MB, ring, B.MOK_BF16, backward=True)
    S = SharedExpert(L)
    R = T * K
    f32 = dict(dtype=torch.float32, device="cuda")
    st = dict(dtype=L.dtype, device="cuda")
    pre = torch.empty(R, 2 * I, **st)
    y, dx = torch.empty(T, H, **st), torch.empty(T, H, **st)
    dw13, dw2 = torch.empty(E, 2 * I, H, **st), torch.empty(E, H, I, **st)
    dtk, dlg = torch.empty(R, **f32), torch.empty(T, E, **f32)
    s = torch.cuda.Stream()

    def step():
        L.route(lg, s)
        L.schedule(stream=s)
        L.forward(x, w13, w2, y, saved_preact=pre, stream=s)
        S.forward(x, w13s, w2s, y, stream=s)
        L.backward(x, pre, w13, w2, dy, dx, dw13, dw2, dtk, dlg, stream=s)

    outs = (y, dx, dw13, dw2, dtk, dlg, pre)
    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for t in outs:
        t.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.replay()
        g.replay()
    torch.cuda.synchronize()
    st, dev = B.mok_read_device_status()
    assert st == B.MOK_OK and dev == B.MOK_OK
    for a, b in zip(outs, eager):
        assert same_bits(a, b)


def test_captured_mxfp8_ring_forward_replays_eager_results():
    """MXFP8 forward through a ring of 512 rows (4.7 laps of the 2400 routed rows, one
    persistent launch): replay equals eager bit for bit, twice in a row."""
    import torch
    from mixture_experts_layer_deterministic_gb300.buffers import quantize_mxfp8
    T, H, I, E, K, MB, ring = 600, 256, 256, 16, 4, 256, 512
    r = np.random.default_rng(17)
    x = to_dev(f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32)))
    lg = to_dev(r.standard_normal((T, E)).astype(np.float32))
    q13, s13 = quantize_mxfp8(to_dev(f32_to_bf16_bits(
        (r.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32))))
    q2, s2 = quantize_mxfp8(to_dev(f32_to_bf16_bits(
        (r.standard_normal((E, H, I)) * 0.05).astype(np.float32))))
    L = MoELayer(T, H, I, E, K, MB, ring, B.MOK_MXFP8)
    st = dict(dtype=L.dtype, device="cuda")
    pre = torch.empty(T * K, 2 * I, **st)
    y = torch.empty(T, H, **st)
    s = torch.cuda.Stream()

    def fwd():
        L.route(lg, s)
        L.schedule(stream=s)
        L.forward(x, q13, q2, y, s13, s2, saved_preact=pre, stream=s)

    with torch.cuda.stream(s):
        fwd()
    torch.cuda.synchronize()
    eager = [y.clone(), pre.clone()]
    # the forward through a ring of every row gives the same y, bit for bit
    L1 = MoELayer(T, H, I, E, K, MB, 0, B.MOK_MXFP8)
    y1 = torch.empty(T, H, **st)
    with torch.cuda.stream(s):
        L1.route(lg, s)
        L1.schedule(stream=s)
        L1.forward(x, q13, q2, y1, s13, s2, stream=s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fwd()
    y.fill_(float("nan"))
    pre.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.replay()
        g.replay()
    torch.cuda.synchronize()
    s_, dev = B.mok_read_device_status()
    assert s_ == B.MOK_OK and dev == B.MOK_OK
    assert same_bits(y, eager[0])
    assert same_bits(pre, eager[1])
    assert same_bits(y1, eager[0])
