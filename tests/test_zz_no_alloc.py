"""mok_build_schedule_noalloc: the schedule builder for callers that cannot allocate.

Some users of this library cannot call cudaMalloc to make a workspace: their GPU memory
is owned and handed out by another component (a framework or server with its own pool),
or they run a time-critical loop that cannot pay cudaMalloc's latency and implicit
synchronisation. For them the library offers a schedule builder whose scratch lives in a
fixed array inside the library. These tests call it through the C ABI and check that it
produces exactly what the workspace-based mok_build_schedule produces, on two calls in a
row (the second call inherits the first call's leftovers in the shared array), that a call
takes no device memory, and that it refuses sizes its array cannot hold.

The file is named to be collected last, so that a run stopping at its first failure has
run every other test before this one; it passes alone in a fresh process and after the
rest of the suite alike.
"""
import numpy as np
import pytest

from mixture_experts_layer_deterministic_gb300 import binding as B
from mixture_experts_layer_deterministic_gb300.buffers import MoELayer, Schedule

pytestmark = pytest.mark.gpu


def schedule_arrays(s, R):
    n = int(s.n_segs.cpu()[0])
    return dict(counts=s.counts.cpu().numpy(), offsets=s.offsets.cpu().numpy(),
                perm=s.perm[:R].cpu().numpy(), inv=s.inv[:R].cpu().numpy(),
                segs=s.segs[: 3 * n].cpu().numpy(), n_segs=n)


def both_ways(T, E, K, MB, seed, skew=0.0):
    import torch
    L = MoELayer(T, 256, 128, E, K, MB, 0, B.MOK_BF16)
    r = np.random.default_rng(seed)
    lg = (r.standard_normal((T, E)) - skew * np.log1p(np.arange(E))).astype(np.float32)
    L.route(torch.from_numpy(lg).cuda())
    L.schedule()  # the workspace-based entry point
    other = Schedule(L.cfg, L.device)
    B.check(B.mok_build_schedule_noalloc(L.cfg, L.idx, other.struct), "noalloc schedule")
    torch.cuda.synchronize()
    st, dev = B.mok_read_device_status()
    assert st == B.MOK_OK and dev == B.MOK_OK
    R = T * K
    return schedule_arrays(L.sched, R), schedule_arrays(other, R)


def test_noalloc_schedule_equals_workspace_schedule_on_two_calls():
    # first call: a large routing
    want, got = both_ways(16384, 512, 10, 2368, seed=1)
    for k in want:
        np.testing.assert_array_equal(got[k], want[k], err_msg=k)
    # second call: a smaller, skewed routing on top of the first call's leftovers
    want, got = both_ways(1000, 64, 6, 300, seed=2, skew=2.0)
    for k in want:
        np.testing.assert_array_equal(got[k], want[k], err_msg=k)


def test_noalloc_schedule_takes_no_device_memory():
    """After a warm-up call (which looks up the array's address on this device), another
    call changes neither the device's free memory nor torch's allocator statistics."""
    import torch
    T, E, K = 4096, 256, 8
    L = MoELayer(T, 256, 128, E, K, 2368, 0, B.MOK_BF16)
    lg = np.random.default_rng(4).standard_normal((T, E)).astype(np.float32)
    L.route(torch.from_numpy(lg).cuda())
    other = Schedule(L.cfg, L.device)
    B.check(B.mok_build_schedule_noalloc(L.cfg, L.idx, other.struct), "warm-up")
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    stats0 = torch.cuda.memory_stats()
    B.check(B.mok_build_schedule_noalloc(L.cfg, L.idx, other.struct), "second call")
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    stats1 = torch.cuda.memory_stats()
    assert free1 == free0, (free0, free1)
    for k in ("allocation.all.allocated", "reserved_bytes.all.current",
              "allocated_bytes.all.current"):
        assert stats1.get(k) == stats0.get(k), k


def test_noalloc_schedule_rejects_sizes_beyond_its_array():
    import torch
    # ceil(R / 1024) * E * 4 bytes > 4 MiB: 2,098,180 routed rows with E = 512
    T, E, K = 209818, 512, 10
    cfg = B.make_config(T, 256, 128, E, K, 2368, 0, B.MOK_BF16)
    assert B.mok_workspace_size(cfg, B.MOK_WS_SCHEDULE) > B.MOK_NOALLOC_SCHEDULE_SCRATCH_BYTES
    idx = torch.zeros(16, dtype=torch.int32, device="cuda")
    sched = Schedule(B.make_config(1, 256, 128, E, K, 2368, 0, B.MOK_BF16), "cuda")
    assert B.mok_build_schedule_noalloc(cfg, idx, sched.struct) == B.MOK_ERR_WORKSPACE
