"""The C ABI without a GPU: the library loads, exports every entry point include/mok.h
declares, and validates configurations on the host."""
import os
import re

import pytest

from mixture_experts_layer_deterministic_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        import mixture_experts_layer_deterministic_gb300 as pkg
        pkg.build()
    return B.lib()


def declared_entry_points():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(mok_\w+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(lib):
    names = declared_entry_points()
    assert "mok_forward" in names and "mok_backward" in names
    for n in sorted(names):
        assert hasattr(lib, n), "missing export " + n
    assert names <= set(B.EXPORTED)


def test_header_is_plain_c(tmp_path):
    """include/mok.h is a C header: a C11 translation unit that includes it and takes the
    address of every declared entry point compiles cleanly with gcc (no C++ needed)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    if gcc is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA headers are not available")
    names = sorted(declared_entry_points())
    src = tmp_path / "uses_mok.c"
    src.write_text('#include "mok.h"\n' + "".join(
        "void *p_%s(void) { return (void *)&%s; }\n" % (n, n) for n in names))
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                        "-I" + os.path.join(ROOT, "include"), "-I" + cuda_inc, str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_client_builds(lib, tmp_path):
    """tests/c_client/c_forward.c, a client that uses nothing but include/mok.h and the CUDA
    runtime, compiles and links against libmok.so (it runs in the GPU tests)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    if gcc is None or not os.path.exists(os.path.join(cuda, "include", "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA toolkit is not available")
    r = subprocess.run([gcc, "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror",
                        "-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(cuda, "include"),
                        os.path.join(ROOT, "tests", "c_client", "c_forward.c"),
                        "-L" + os.path.dirname(B.LIB_PATH), "-lmok",
                        "-L" + os.path.join(cuda, "lib64"), "-lcudart",
                        "-o", str(tmp_path / "c_forward")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    # its failure paths need no GPU: the library's host validation rejects H = 100 before
    # any CUDA call, and missing inputs are reported; neither crashes
    env = dict(os.environ, LD_LIBRARY_PATH=os.pathsep.join(
        [os.path.dirname(B.LIB_PATH), os.path.join(cuda, "lib64"),
         os.environ.get("LD_LIBRARY_PATH", "")]))
    exe = str(tmp_path / "c_forward")
    bad = subprocess.run([exe, "256", "100", "128", "8", "2", "64", "0", str(tmp_path)],
                         env=env, capture_output=True, text=True, timeout=60)
    assert bad.returncode == 1 and "mok_check_config" in bad.stderr
    assert "invalid argument" in bad.stderr
    missing = subprocess.run([exe, "256", "256", "128", "8", "2", "64", "0",
                              str(tmp_path / "absent")], env=env, capture_output=True,
                             text=True, timeout=60)
    assert missing.returncode == 1 and "missing or short input file" in missing.stderr


def test_abi_version_and_strings(lib):
    assert B.mok_abi_version() == B.MOK_ABI_VERSION
    for s in range(8):
        assert B.status_string(s)
    assert B.status_string(0) == "ok"


def cfg(**kw):
    base = dict(T=256, H=256, I=128, E=8, K=2, minibatch=64, ring_capacity=0, prec=B.MOK_BF16)
    base.update(kw)
    return B.make_config(**base)


@pytest.mark.parametrize("kw,want", [
    (dict(), B.MOK_OK),
    (dict(T=0), B.MOK_OK),
    (dict(K=9), B.MOK_ERR_INVALID_ARG),          # K > E
    (dict(K=0), B.MOK_ERR_INVALID_ARG),
    (dict(E=2000, K=2), B.MOK_ERR_INVALID_ARG),   # E > 1024
    (dict(E=64, K=33), B.MOK_ERR_INVALID_ARG),    # K > 32
    (dict(H=200), B.MOK_ERR_INVALID_ARG),         # H % 128
    (dict(I=64), B.MOK_ERR_INVALID_ARG),          # I < 128
    (dict(minibatch=0), B.MOK_ERR_INVALID_ARG),
    (dict(ring_capacity=32), B.MOK_ERR_INVALID_ARG),  # smaller than a minibatch
    (dict(ring_capacity=100), B.MOK_OK),              # a ring smaller than R
    (dict(ring_capacity=10000), B.MOK_OK),            # >= R: holds every row
    (dict(prec=5), B.MOK_ERR_INVALID_ARG),
    (dict(T=1 << 28, K=8, E=8), B.MOK_ERR_INVALID_ARG),  # R >= 2^31
    (dict(abi_version=99), B.MOK_ERR_ABI),
    (dict(flags=B.MOK_FLAG_FP32_STORAGE), B.MOK_OK),
    (dict(flags=B.MOK_FLAG_ONE_SM_GEMMS), B.MOK_OK),
    (dict(flags=B.MOK_FLAG_SM_PAIR_GEMMS), B.MOK_OK),
    (dict(flags=B.MOK_FLAG_ONE_SM_GEMMS | B.MOK_FLAG_SM_PAIR_GEMMS), B.MOK_ERR_INVALID_ARG),
    (dict(flags=8), B.MOK_ERR_INVALID_ARG),       # unknown flag
])
def test_check_config(lib, kw, want):
    assert B.mok_check_config(cfg(**kw)) == want


def test_workspace_sizes(lib):
    c = cfg()
    for which in (B.MOK_WS_SCHEDULE, B.MOK_WS_FORWARD, B.MOK_WS_BACKWARD):
        assert B.mok_workspace_size(c, which) > 0
    # the recompute backward adds the [R][2I] pre-activations (plus alignment): bf16, or
    # fp32 under fp32 storage
    R, I = c.T * c.K, c.I
    for flags, esz in ((0, 2), (B.MOK_FLAG_FP32_STORAGE, 4)):
        cf = cfg(flags=flags)
        extra = (B.mok_workspace_size(cf, B.MOK_WS_BACKWARD_RECOMPUTE) -
                 B.mok_workspace_size(cf, B.MOK_WS_BACKWARD))
        assert R * 2 * I * esz <= extra < R * 2 * I * esz + 256
    # fp32 storage doubles the (token, k) slots of the forward
    H = c.H
    d = (B.mok_workspace_size(cfg(flags=B.MOK_FLAG_FP32_STORAGE), B.MOK_WS_FORWARD) -
         B.mok_workspace_size(c, B.MOK_WS_FORWARD))
    assert R * H * 2 <= d < R * H * 2 + 256
    assert B.mok_workspace_size(c, 99) == 0
    assert B.mok_workspace_size(cfg(K=9), B.MOK_WS_FORWARD) == 0
    # a smaller ring needs a smaller forward workspace
    big = B.mok_workspace_size(cfg(T=4096), B.MOK_WS_FORWARD)
    small = B.mok_workspace_size(cfg(T=4096, ring_capacity=128), B.MOK_WS_FORWARD)
    assert small < big
    # MXFP8 rings hold one byte per element
    assert B.mok_workspace_size(cfg(prec=B.MOK_MXFP8), B.MOK_WS_FORWARD) < \
        B.mok_workspace_size(c, B.MOK_WS_FORWARD)
    # the shared expert: bf16 h [T][I]; MXFP8 holds x and h quantized with their scales and
    # the scale atoms of the weights ([2I][H/32] + [H][I/32]) instead
    T, H = c.T, c.H
    sb = B.mok_workspace_size(c, B.MOK_WS_SHARED)
    sm = B.mok_workspace_size(cfg(prec=B.MOK_MXFP8), B.MOK_WS_SHARED)
    assert T * I * 2 <= sb
    assert T * H + T * I + 3 * I * H // 32 <= sm


def test_partial_ring_workspace(lib):
    """A ring of C < R rows: the x and h rings grow with C (H and I elements per row, and in
    MXFP8 I/32 scales of h); MXFP8 also holds x quantized once per token; the unit order
    (pairs of int32 per unit) and tile lists grow with the tiles a capacity cuts."""
    T, K, MB, H, I, E = 4096, 2, 1000, 256, 128, 8  # R = 8192 routed rows
    c = lambda prec, C: cfg(T=T, K=K, minibatch=MB, ring_capacity=C, prec=prec)  # noqa: E731
    ws = lambda prec, C: B.mok_workspace_size(c(prec, C), B.MOK_WS_FORWARD)  # noqa: E731
    full_bf16 = B.mok_workspace_size(cfg(T=T, K=K, minibatch=MB), B.MOK_WS_FORWARD)
    assert ws(B.MOK_BF16, 2000) < full_bf16 - (T * K - 2000) * H * 2  # no [R][H] x ring
    # 500 more ring rows, less a lap's worth of tile bookkeeping
    assert ws(B.MOK_BF16, 2500) - ws(B.MOK_BF16, 2000) >= 500 * (H + I) * 2 - 4096
    assert ws(B.MOK_MXFP8, 2500) - ws(B.MOK_MXFP8, 2000) >= 500 * (H + I + I // 32) - 4096
    for prec in (B.MOK_BF16, B.MOK_MXFP8):
        esz = 1 if prec == B.MOK_MXFP8 else 2
        for it, width in ((B.MOK_ITEM_H_RING, I), (B.MOK_ITEM_X_RING, H)):
            st, _, n = B.mok_workspace_item(c(prec, 2000), B.MOK_WS_FORWARD, it)
            assert st == B.MOK_OK and n == 2000 * width * esz
    # MXFP8: the scales of x's token rows (quantized once per token)
    st, _, n = B.mok_workspace_item(c(B.MOK_MXFP8, 2000), B.MOK_WS_FORWARD,
                                    B.MOK_ITEM_X_RING_SCALE)
    assert st == B.MOK_OK and n == T * H // 32
    # tiles: at most ceil(R / chunk) + E + laps of the ring; units per tile (32-byte
    # records): the gather's pieces, I/128 gate/up and H/256 down units
    R = T * K
    # (a ring below two tile heights cuts tiles of half the ring)
    for C, chunk in ((2000, 128), (200, 100), (1000, 128), (17, 8)):
        cc = cfg(T=T, K=K, minibatch=min(MB, C), ring_capacity=C)
        st, _, n = B.mok_workspace_item(cc, B.MOK_WS_FORWARD, B.MOK_ITEM_RING_TILES)
        cap = -(-R // chunk) + E + -(-R // C)
        assert st == B.MOK_OK and n == 16 + 16 * cap, (C, n, cap)
        st, _, n = B.mok_workspace_item(cc, B.MOK_WS_FORWARD, B.MOK_ITEM_RING_ORDER)
        n_g = -(-chunk // (4 * min(32, 49152 // (H * 2))))  # gather pieces of 4 stages
        assert st == B.MOK_OK and n == 32 * cap * (n_g + I // 128 + H // 256)
    # a ring that holds every row has no unit order
    for it in (B.MOK_ITEM_RING_TILES, B.MOK_ITEM_RING_ORDER):
        assert B.mok_workspace_item(cfg(T=T, K=K, minibatch=MB), B.MOK_WS_FORWARD,
                                    it)[0] == B.MOK_ERR_INVALID_ARG


def test_segment_capacity(lib):
    # E + ceil(R / MB) - 1
    assert B.mok_segment_capacity(cfg()) == 8 + (512 + 63) // 64 - 1
    assert B.mok_segment_capacity(cfg(T=0)) == 7


def test_device_calls_fail_cleanly_without_gpu(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = B.lib().mok_route_topk(B.ctypes.byref(cfg()), None, None, None, None)
    assert st in (B.MOK_ERR_CUDA, B.MOK_ERR_UNSUPPORTED)


ITEMS = {
    B.MOK_WS_FORWARD: [B.MOK_ITEM_X_RING, B.MOK_ITEM_H_RING, B.MOK_ITEM_SLOTS],
    B.MOK_WS_BACKWARD: [B.MOK_ITEM_PAD_OFFSETS, B.MOK_ITEM_DA, B.MOK_ITEM_WH, B.MOK_ITEM_SLOTS],
    B.MOK_WS_SHARED: [B.MOK_ITEM_H_RING],
    B.MOK_WS_SHARED_BACKWARD: [B.MOK_ITEM_DA, B.MOK_ITEM_WH],
}
MX_ITEMS = {
    B.MOK_WS_FORWARD: [B.MOK_ITEM_X_RING_SCALE, B.MOK_ITEM_H_RING_SCALE],
    B.MOK_WS_BACKWARD: [B.MOK_ITEM_DA_Q, B.MOK_ITEM_DA_SCALE, B.MOK_ITEM_DY_Q,
                        B.MOK_ITEM_DY_SCALE],
    B.MOK_WS_SHARED: [B.MOK_ITEM_X_RING, B.MOK_ITEM_X_RING_SCALE, B.MOK_ITEM_H_RING_SCALE],
    B.MOK_WS_SHARED_BACKWARD: [B.MOK_ITEM_DA_Q, B.MOK_ITEM_DA_SCALE, B.MOK_ITEM_DY_Q,
                               B.MOK_ITEM_DY_SCALE],
}


@pytest.mark.parametrize("prec", [B.MOK_BF16, B.MOK_MXFP8])
@pytest.mark.parametrize("ring", [0, 100])
def test_workspace_items_lie_inside_their_workspace_and_apart(lib, prec, ring):
    c = cfg(prec=prec, ring_capacity=ring)
    R, H, I, T = c.T * c.K, c.H, c.I, c.T
    for which, items in ITEMS.items():
        items = items + (MX_ITEMS[which] if prec == B.MOK_MXFP8 else [])
        if which == B.MOK_WS_FORWARD and ring:
            # a ring smaller than R: the unit order of its one launch
            items = items + [B.MOK_ITEM_RING_TILES, B.MOK_ITEM_RING_ORDER]
        size = B.mok_workspace_size(c, which)
        spans = []
        for it in items:
            st, off, n = B.mok_workspace_item(c, which, it)
            assert st == B.MOK_OK, (which, it)
            assert off % 256 == 0 and n > 0 and off + n <= size, (which, it, off, n, size)
            spans.append((off, off + n))
        spans.sort()
        for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
            assert a1 <= b0  # no two items overlap
    # sizes follow the documented shapes: the x and h rings hold the ring's rows
    rows = R if ring == 0 else ring
    esz = 1 if prec == B.MOK_MXFP8 else 2
    assert B.mok_workspace_item(c, B.MOK_WS_FORWARD, B.MOK_ITEM_X_RING)[2] == rows * H * esz
    assert B.mok_workspace_item(c, B.MOK_WS_FORWARD, B.MOK_ITEM_H_RING)[2] == rows * I * esz
    assert B.mok_workspace_item(c, B.MOK_WS_FORWARD, B.MOK_ITEM_SLOTS)[2] == R * H * 2
    assert B.mok_workspace_item(c, B.MOK_WS_BACKWARD, B.MOK_ITEM_PAD_OFFSETS)[2] == 4 * (c.E + 1)
    rpad = R + 15 * c.E
    assert B.mok_workspace_item(c, B.MOK_WS_BACKWARD, B.MOK_ITEM_DA)[2] == rpad * 2 * I * 2
    # an item a workspace does not hold, an unknown item, an invalid configuration
    if prec == B.MOK_BF16:
        assert B.mok_workspace_item(c, B.MOK_WS_FORWARD, B.MOK_ITEM_X_RING_SCALE)[0] == \
            B.MOK_ERR_INVALID_ARG
    assert B.mok_workspace_item(c, B.MOK_WS_FORWARD, B.MOK_ITEM_DA)[0] == B.MOK_ERR_INVALID_ARG
    assert B.mok_workspace_item(c, B.MOK_WS_FORWARD, 99)[0] == B.MOK_ERR_INVALID_ARG
    assert B.mok_workspace_item(c, 99, B.MOK_ITEM_SLOTS)[0] == B.MOK_ERR_INVALID_ARG
    assert B.mok_workspace_item(cfg(K=9), B.MOK_WS_FORWARD, B.MOK_ITEM_SLOTS)[0] == \
        B.MOK_ERR_INVALID_ARG
