"""The layer workloads: shapes, value distributions, seeds and scheduling knobs.

The shapes follow the pages' headline case (alphalab.site "Mixture-of-Kittens" analysis,
section 三: 512 experts, hidden 4,096, intermediate 1,024, top-10) and the minibatch
figure of the arex-research.com article (section "pull 代替 push", about 2,368 tokens).
Routing is synthetic Gaussian logits (alphalab.site section 四), optionally skewed by a
per-expert bias for the imbalanced case.
"""
from dataclasses import dataclass, replace
import math


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int                 # tokens
    H: int                 # hidden size
    I: int                 # expert intermediate size
    E: int                 # experts
    K: int                 # experts per token (top-k)
    x_std: float           # activations ~ N(0, x_std^2), stored bf16
    w_std: float           # W13 and W2 ~ N(0, w_std^2), stored bf16
    dy_std: float          # upstream gradient ~ N(0, dy_std^2), stored bf16
    zipf_bias: bool        # logits += -2*ln(e+1) (expert 0 hottest)
    seed: int
    minibatch: int         # routed rows per minibatch
    ring_capacity: int     # ring rows; 0 means "all R routed rows"
    prec: str              # "bf16" or "mxfp8"
    passes: str            # "fwd" or "bwd"

    @property
    def R(self) -> int:
        return self.T * self.K

    def fwd_flops(self) -> float:
        """Useful forward FLOPs: gate/up GEMM 4*R*H*I plus down GEMM 2*R*H*I."""
        return 6.0 * self.R * self.H * self.I

    def bwd_flops(self) -> float:
        """Useful backward FLOPs: G GEMM 2RHI, dgrad 4RHI, wgrad 6RHI."""
        return 12.0 * self.R * self.H * self.I

    def with_(self, **kw) -> "LayerConfig":
        return replace(self, **kw)


_BIG = dict(H=4096, I=1024, E=512, K=10, x_std=1.0, w_std=1.0 / math.sqrt(4096.0),
            dy_std=1.0, zipf_bias=False, minibatch=2368, ring_capacity=0)

CONFIGS = {
    # small case the oracle finishes in seconds
    "tiny": LayerConfig(name="tiny", T=256, H=256, I=128, E=8, K=2, x_std=0.02, w_std=0.02,
                        dy_std=1.0, zipf_bias=False, seed=0, minibatch=64, ring_capacity=0,
                        prec="bf16", passes="fwd"),
    "fwd_bf16": LayerConfig(name="fwd_bf16", T=16384, seed=0, prec="bf16", passes="fwd", **_BIG),
    "fwd_mxfp8": LayerConfig(name="fwd_mxfp8", T=16384, seed=1, prec="mxfp8", passes="fwd", **_BIG),
    # profiling case: same routed rows per expert (320) as fwd_bf16 with a quarter of the
    # experts, so a full counter capture holds a few GB on the device
    "fwd_bf16_e128": LayerConfig(name="fwd_bf16_e128", T=4096, seed=0, prec="bf16",
                                 passes="fwd", **{**_BIG, "E": 128}),
    # counter-capture case: same 320 routed rows per expert, 32 experts (about 3.5 GB held
    # on the device by the benchmark, still larger than L2)
    "fwd_bf16_e32": LayerConfig(name="fwd_bf16_e32", T=1024, seed=0, prec="bf16",
                                passes="fwd", **{**_BIG, "E": 32}),
    "bwd_bf16": LayerConfig(name="bwd_bf16", T=8192, seed=2, prec="bf16", passes="bwd", **_BIG),
    # counter-capture case of the ring forward: the imbalanced routing and ring with 64
    # experts and 8192 tokens (about 4 GB held on the device)
    "ring_bf16_e64": LayerConfig(name="ring_bf16_e64", T=8192, seed=3, prec="bf16",
                                 passes="fwd", **{**_BIG, "E": 64, "zipf_bias": True,
                                                  "ring_capacity": 2960}),
    "imbalanced_bf16": LayerConfig(name="imbalanced_bf16", T=65536, seed=3, prec="bf16",
                                   passes="fwd", **{**_BIG, "zipf_bias": True,
                                                    "ring_capacity": 2960}),
    "imbalanced_mxfp8": LayerConfig(name="imbalanced_mxfp8", T=65536, seed=3, prec="mxfp8",
                                    passes="fwd", **{**_BIG, "zipf_bias": True,
                                                     "ring_capacity": 2960}),
}


def get_config(name: str) -> LayerConfig:
    return CONFIGS[name]
