"""GPU MXFP8 quantizer: bytes bit-exact against the oracle quantizer."""
import numpy as np
import pytest

import oracle
from harness import bf16_dev_to_np, to_dev
from mixture_experts_layer_deterministic_gb300.buffers import quantize_mxfp8
from workloads.synth import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


def check(bits):
    q, s = quantize_mxfp8(to_dev(bits))
    qo, so = oracle.mxfp8_quantize_bf16(bits)
    np.testing.assert_array_equal(s.cpu().numpy(), so)
    np.testing.assert_array_equal(q.cpu().numpy(), qo)


def test_random_blocks_over_wide_dynamic_range():
    r = np.random.default_rng(0)
    x = r.standard_normal((257, 512)) * np.exp(r.uniform(-80, 80, size=(257, 1)))
    check(f32_to_bf16_bits(x.astype(np.float32)))


def test_special_values():
    r = np.random.default_rng(1)
    x = r.standard_normal((64, 256)).astype(np.float32)
    x[0, :32] = 0.0                       # zero block -> scale byte 0
    x[1, :32] = -0.0                      # signed zeros keep their sign
    x[2, :32] = 1e-40                     # subnormal bf16 block
    x[3, :32] = 3.0e38                    # near the top of the range
    x[4, :32] = np.float32(448.0)
    x[5, :32] = np.float32(511.0)         # saturates
    x[6, 0] = 1.0
    x[6, 1:32] = 2.0 ** -10               # rounds to even (zero)
    x[7, 0] = 1.0
    x[7, 1:32] = 3 * 2.0 ** -11           # rounds up to the smallest subnormal
    x[8, :32] = -x[8, :32]
    x[9, :] = 1.0 + 2.0 ** -4             # exact ties between E4M3 neighbours
    bits = f32_to_bf16_bits(x)
    # every bf16 bit pattern that is finite, scattered over rows
    allp = np.arange(65536, dtype=np.uint32)
    f = (allp << 16).view(np.float32)
    fin = allp[np.isfinite(f)].astype(np.uint16)
    fin = np.concatenate([fin, np.zeros((-fin.size) % 256, np.uint16)]).reshape(-1, 256)
    check(np.concatenate([bits, fin]))


def test_quantized_weights_roundtrip_device_bf16():
    r = np.random.default_rng(2)
    x = (r.standard_normal((8, 2 * 128, 256)) * 0.02).astype(np.float32)
    bits = f32_to_bf16_bits(x)
    d = to_dev(bits)
    np.testing.assert_array_equal(bf16_dev_to_np(d), bits)
    check(bits)
