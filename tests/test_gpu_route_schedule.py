"""GPU parity of routing and the schedule: bit-exact against the oracle, run to run."""
import numpy as np
import pytest

import oracle
from harness import inputs, to_dev
from mixture_experts_layer_deterministic_gb300 import binding as B
from mixture_experts_layer_deterministic_gb300.buffers import MoELayer
from workloads import CONFIGS

pytestmark = pytest.mark.gpu


def route_and_schedule(logits, E, K, MB, H=256, I=128):
    T = logits.shape[0]
    L = MoELayer(T, H, I, E, K, MB, 0, B.MOK_BF16)
    L.route(to_dev(logits))
    L.schedule()
    import torch
    torch.cuda.synchronize()
    s = L.sched
    R = T * K
    n = int(s.n_segs.cpu()[0])
    return dict(idx=L.idx[:R].view(T, K).cpu().numpy() if R else np.zeros((T, K), np.int32),
                w=L.w[:R].view(T, K).cpu().numpy() if R else np.zeros((T, K), np.float32),
                counts=s.counts.cpu().numpy(), offsets=s.offsets.cpu().numpy(),
                perm=s.perm[:R].cpu().numpy(), inv=s.inv[:R].cpu().numpy(),
                segs=s.segs[: 3 * n].view(-1, 3).cpu().numpy() if n else np.zeros((0, 3)))


def check_against_oracle(logits, E, K, MB, g):
    idx_o, w_o = oracle.route(logits.astype(np.float64), K)
    np.testing.assert_array_equal(g["idx"], idx_o)
    # fp32 softmax against the fp64 oracle: a few ulp
    np.testing.assert_allclose(g["w"], w_o, rtol=4e-6, atol=1e-7)
    so = oracle.schedule(idx_o, E, MB)
    for k in ("counts", "offsets", "perm", "inv"):
        np.testing.assert_array_equal(g[k], so[k], err_msg=k)
    np.testing.assert_array_equal(g["segs"], so["segs"])


@pytest.mark.parametrize("name", ["tiny", "fwd_bf16", "bwd_bf16", "imbalanced_bf16"])
def test_route_schedule_configs(name):
    cfg = CONFIGS[name]
    lg = inputs(cfg, weights=False)["logits"]
    g = route_and_schedule(lg, cfg.E, cfg.K, cfg.minibatch)
    check_against_oracle(lg, cfg.E, cfg.K, cfg.minibatch, g)
    assert g["counts"].sum() == cfg.R  # no routed row is dropped
    g2 = route_and_schedule(lg, cfg.E, cfg.K, cfg.minibatch)
    for k in g:
        np.testing.assert_array_equal(g[k], g2[k])  # run to run


@pytest.mark.parametrize("T,E,K,MB", [(1000, 16, 4, 300), (77, 512, 10, 2368), (333, 1024, 32, 7),
                                      (64, 5, 5, 1), (1, 3, 1, 1), (513, 100, 7, 64)])
def test_route_schedule_ragged_shapes(T, E, K, MB):
    r = np.random.default_rng(T * 7 + E)
    lg = r.standard_normal((T, E)).astype(np.float32)
    g = route_and_schedule(lg, E, K, MB)
    check_against_oracle(lg, E, K, MB, g)


def test_route_ties_and_signed_zero():
    r = np.random.default_rng(3)
    vals = np.array([-1.0, -0.0, 0.0, 0.5, 0.5, 2.0], np.float32)
    lg = r.choice(vals, size=(500, 64)).astype(np.float32)
    g = route_and_schedule(lg, 64, 8, 100)
    check_against_oracle(lg, 64, 8, 100, g)
    # 512 experts (16 per lane) from three values: every round breaks ties both between
    # lanes and between the experts one lane holds
    lg = r.choice(np.array([-0.0, 0.25, 0.25, 1.0], np.float32), size=(300, 512))
    g = route_and_schedule(lg.astype(np.float32), 512, 10, 2368)
    check_against_oracle(lg.astype(np.float32), 512, 10, 2368, g)


def test_route_one_hot_and_all_experts():
    E = 32
    lg = np.full((E, E), -3.0, np.float32)
    lg[np.arange(E), (np.arange(E) * 7) % E] = 3.0
    g = route_and_schedule(lg, E, 1, 5)
    np.testing.assert_array_equal(g["idx"][:, 0], (np.arange(E) * 7) % E)
    np.testing.assert_array_equal(g["w"], 1.0)
    lg2 = np.random.default_rng(1).standard_normal((40, 8)).astype(np.float32)
    g2 = route_and_schedule(lg2, 8, 8, 16)
    check_against_oracle(lg2, 8, 8, 16, g2)


def test_empty_batch():
    g = route_and_schedule(np.zeros((0, 8), np.float32), 8, 2, 16)
    assert g["counts"].sum() == 0 and np.all(g["offsets"] == 0) and len(g["segs"]) == 0


def test_out_of_range_expert_id_is_reported():
    import torch
    T, E, K = 64, 8, 2
    L = MoELayer(T, 256, 128, E, K, 16, 0, B.MOK_BF16)
    idx = torch.randint(0, E, (T * K,), dtype=torch.int32, device="cuda")
    idx[5] = E + 3  # a bad id made on the host
    B.check(B.mok_clear_device_status())
    B.check(B.mok_build_schedule(L.cfg, idx, L.sched.struct, L.ws_s, L.ws_s_n, None))
    st, dev = B.mok_read_device_status()
    assert st == B.MOK_OK and dev == B.MOK_ERR_DEVICE_INVARIANT
    assert int(L.sched.counts.sum()) == T * K - 1  # the bad id is counted nowhere
    B.check(B.mok_clear_device_status())
    st, dev = B.mok_read_device_status()
    assert dev == B.MOK_OK


def test_host_validation_rejects_bad_arguments():
    import torch
    L = MoELayer(64, 256, 128, 8, 2, 16, 0, B.MOK_BF16)
    lg = torch.zeros(64 * 8 + 1, device="cuda")
    assert B.mok_route_topk(L.cfg, lg[1:], L.idx, L.w) == B.MOK_ERR_INVALID_ARG  # misaligned
    assert B.mok_route_topk(L.cfg, None, L.idx, L.w) == B.MOK_ERR_INVALID_ARG
    assert B.mok_build_schedule(L.cfg, L.idx, L.sched.struct, L.ws_s, 16) == B.MOK_ERR_WORKSPACE
    assert B.mok_build_schedule(L.cfg, L.idx, L.sched.struct, None, 0) == B.MOK_ERR_WORKSPACE
    bad = B.make_config(64, 256, 128, 8, 2, 16, 0, B.MOK_BF16, abi_version=B.MOK_ABI_VERSION + 1)
    assert B.mok_route_topk(bad, lg, L.idx, L.w) == B.MOK_ERR_ABI
