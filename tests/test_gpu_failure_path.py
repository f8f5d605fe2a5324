"""The kernels' failure path, exercised without a fault: a wait that nothing completes gives
up after its bounded limit, the device status word reads MOK_ERR_TIMEOUT, and the context
keeps working (a layer forward right after still matches the oracle)."""
import time

import numpy as np
import pytest

import oracle
from harness import TOL_BF16, check_tol, host, inputs, to_dev
from mixture_experts_layer_deterministic_gb300 import binding as B
from mixture_experts_layer_deterministic_gb300.buffers import MoELayer
from workloads import CONFIGS

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    import torch
    torch.cuda.synchronize()
    B.check(B.mok_clear_device_status())
    t0 = time.perf_counter()
    assert B.mok_selftest_bounded_wait(20000) == B.MOK_OK  # 20 ms
    st, dev = B.mok_read_device_status()  # synchronises
    elapsed = time.perf_counter() - t0
    assert st == B.MOK_OK and dev == B.MOK_ERR_TIMEOUT, (st, dev)
    assert 0.015 < elapsed < 1.5, elapsed  # it waited about its limit, not the 2 s default
    B.check(B.mok_clear_device_status())
    st, dev = B.mok_read_device_status()
    assert st == B.MOK_OK and dev == B.MOK_OK
    # out-of-range limits are refused before anything is enqueued
    assert B.mok_selftest_bounded_wait(0) == B.MOK_ERR_INVALID_ARG
    assert B.mok_selftest_bounded_wait(1000001) == B.MOK_ERR_INVALID_ARG


def test_context_is_usable_after_a_timeout():
    import torch
    B.check(B.mok_clear_device_status())
    assert B.mok_selftest_bounded_wait(5000) == B.MOK_OK
    st, dev = B.mok_read_device_status()
    assert dev == B.MOK_ERR_TIMEOUT
    B.check(B.mok_clear_device_status())
    cfg = CONFIGS["tiny"]
    d = inputs(cfg)
    L = MoELayer(cfg.T, cfg.H, cfg.I, cfg.E, cfg.K, cfg.minibatch, 0, B.MOK_BF16)
    L.route(to_dev(d["logits"]))
    L.schedule()
    y = torch.empty(cfg.T, cfg.H, dtype=L.dtype, device="cuda")
    L.forward(to_dev(d["x"]), to_dev(d["w13"]), to_dev(d["w2"]), y)
    torch.cuda.synchronize()
    st, dev = B.mok_read_device_status()
    assert st == B.MOK_OK and dev == B.MOK_OK
    R = cfg.T * cfg.K
    idx = L.idx[:R].view(cfg.T, cfg.K).cpu().numpy()
    w = L.w[:R].view(cfg.T, cfg.K).cpu().numpy().astype(np.float64)
    y_o, sl = oracle.forward(oracle.bf16_to_f64(d["x"]), idx, w, d["w13"], d["w2"],
                             mode=oracle.BF16, with_slack=True, store=oracle.STORE_BF16)
    check_tol("y after a timeout", host(y), y_o, sl, TOL_BF16, max_slack_rms=0.2)


def test_ring_counter_wait_times_out_and_reports():
    """The ring forward's producers wait on per-tile counters through a bounded spin: on a
    counter nothing raises it gives up after its limit with MOK_ERR_TIMEOUT recorded, and it
    gives up at once when the status word already holds a problem (as every producer does
    once another CTA has given up)."""
    import torch
    torch.cuda.synchronize()
    B.check(B.mok_clear_device_status())
    t0 = time.perf_counter()
    assert B.mok_selftest_bounded_count_wait(20000) == B.MOK_OK  # 20 ms
    st, dev = B.mok_read_device_status()
    elapsed = time.perf_counter() - t0
    assert st == B.MOK_OK and dev == B.MOK_ERR_TIMEOUT, (st, dev)
    assert 0.015 < elapsed < 1.5, elapsed
    # a problem already recorded: the wait returns without waiting out its limit
    t0 = time.perf_counter()
    assert B.mok_selftest_bounded_count_wait(1000000) == B.MOK_OK  # 1 s limit
    st, dev = B.mok_read_device_status()
    elapsed = time.perf_counter() - t0
    assert dev == B.MOK_ERR_TIMEOUT and elapsed < 0.5, (dev, elapsed)
    B.check(B.mok_clear_device_status())
    assert B.mok_selftest_bounded_count_wait(0) == B.MOK_ERR_INVALID_ARG
    st, dev = B.mok_read_device_status()
    assert st == B.MOK_OK and dev == B.MOK_OK
