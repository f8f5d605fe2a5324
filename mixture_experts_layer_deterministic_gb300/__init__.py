"""Deterministic MoE layer core for one GB300 (sm_103a): a C-ABI library (libmok.so) of
hand-written CUDA kernels and a thin Python binding.

    binding   the C entry points by name (ctypes; marshalling only)
    buffers   torch-allocated schedule arrays and workspaces, and a small MoELayer helper
"""
from . import binding  # noqa: F401
from .binding import (  # noqa: F401
    MOK_BF16, MOK_MXFP8, MOK_OK, MokError, mok_abi_version, mok_backward, mok_build_schedule,
    mok_forward, mok_quantize_mxfp8, mok_read_device_status, mok_route_topk,
)


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)
