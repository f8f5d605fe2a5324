"""The C ABI from plain C: tests/c_client/c_forward.c (only include/mok.h and the CUDA
runtime) routes, schedules and runs the BF16 forward. Its top-k indices and y must equal the
Python binding's bit for bit (same kernels, same inputs), and y must match the oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from harness import TOL_BF16, check_tol, to_dev
from mixture_experts_layer_deterministic_gb300 import binding as B
from mixture_experts_layer_deterministic_gb300.buffers import MoELayer
from workloads.synth import f32_to_bf16_bits

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def build_client(tmp_path):
    gcc = shutil.which("gcc")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    if gcc is None:
        pytest.skip("gcc is not available")
    exe = tmp_path / "c_forward"
    subprocess.run([gcc, "-std=c11", "-O2", "-I" + os.path.join(ROOT, "include"),
                    "-I" + os.path.join(cuda, "include"),
                    os.path.join(ROOT, "tests", "c_client", "c_forward.c"),
                    "-L" + os.path.dirname(B.LIB_PATH), "-lmok",
                    "-L" + os.path.join(cuda, "lib64"), "-lcudart", "-o", str(exe)],
                   check=True)
    env = dict(os.environ)
    env["LD_LIBRARY_PATH"] = os.pathsep.join(
        [os.path.dirname(B.LIB_PATH), os.path.join(cuda, "lib64"), env.get("LD_LIBRARY_PATH", "")])
    return exe, env


@pytest.mark.parametrize("dims,MB,ring", [((256, 256, 128, 8, 2), 64, 0),
                                          ((600, 256, 256, 16, 4), 256, 512)])
def test_c_client_forward(tmp_path, dims, MB, ring):
    import torch
    T, H, I, E, K = dims
    r = np.random.default_rng(T + 5)
    x = f32_to_bf16_bits(r.standard_normal((T, H)).astype(np.float32))
    lg = r.standard_normal((T, E)).astype(np.float32)
    w13 = f32_to_bf16_bits((r.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32))
    w2 = f32_to_bf16_bits((r.standard_normal((E, H, I)) * 0.05).astype(np.float32))
    for name, a in (("x", x), ("logits", lg), ("w13", w13), ("w2", w2)):
        np.ascontiguousarray(a).tofile(str(tmp_path / (name + ".bin")))
    exe, env = build_client(tmp_path)
    run = subprocess.run([str(exe), str(T), str(H), str(I), str(E), str(K), str(MB), str(ring),
                          str(tmp_path)], env=env, capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stderr
    y_c = np.fromfile(str(tmp_path / "y.bin"), np.uint16).reshape(T, H)
    idx_c = np.fromfile(str(tmp_path / "idx.bin"), np.int32).reshape(T, K)

    L = MoELayer(T, H, I, E, K, MB, ring, B.MOK_BF16)
    L.route(to_dev(lg))
    L.schedule()
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    L.forward(to_dev(x), to_dev(w13), to_dev(w2), y)
    torch.cuda.synchronize()
    R = T * K
    idx = L.idx[:R].view(T, K).cpu().numpy()
    np.testing.assert_array_equal(idx_c, idx)
    np.testing.assert_array_equal(y_c, y.view(torch.int16).cpu().numpy().view(np.uint16))
    w = L.w[:R].view(T, K).cpu().numpy().astype(np.float64)
    y_o, sl = oracle.forward(oracle.bf16_to_f64(x), idx, w, w13, w2, mode=oracle.BF16,
                             with_slack=True, store=oracle.STORE_BF16)
    check_tol("c client y e2e", oracle.bf16_to_f64(y_c), y_o, sl, TOL_BF16, max_slack_rms=0.2)
