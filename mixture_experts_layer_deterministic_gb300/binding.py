"""ctypes binding of libmok.so (include/mok.h): argument marshalling only.

Each `mok_*` function here has the name and arguments of the C entry point. Tensor
arguments may be torch tensors (their device pointers are passed) or plain integers
(addresses); `None` is NULL. Streams are torch streams, raw handles or None (the current
torch stream). Nothing here computes any part of the layer: every step runs in the
library's CUDA kernels, and a missing library is an error, never a fallback.
"""
import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmok.so")

MOK_ABI_VERSION = 2

# mok_config.flags
MOK_FLAG_FP32_STORAGE = 1
MOK_FLAG_ONE_SM_GEMMS = 2
MOK_FLAG_SM_PAIR_GEMMS = 4

# mok_status
MOK_OK = 0
MOK_ERR_INVALID_ARG = 1
MOK_ERR_UNSUPPORTED = 2
MOK_ERR_WORKSPACE = 3
MOK_ERR_CUDA = 4
MOK_ERR_TIMEOUT = 5
MOK_ERR_DEVICE_INVARIANT = 6
MOK_ERR_ABI = 7

# mok_precision
MOK_BF16 = 0
MOK_MXFP8 = 1

# mok_workspace_kind
MOK_WS_SCHEDULE = 0
MOK_WS_FORWARD = 1
MOK_WS_BACKWARD = 2
MOK_WS_BACKWARD_RECOMPUTE = 3
MOK_WS_SHARED = 4
MOK_WS_SHARED_BACKWARD = 5

# mok_ws_item
MOK_ITEM_X_RING = 0
MOK_ITEM_X_RING_SCALE = 1
MOK_ITEM_H_RING = 2
MOK_ITEM_H_RING_SCALE = 3
MOK_ITEM_SLOTS = 4
MOK_ITEM_PAD_OFFSETS = 5
MOK_ITEM_DA = 6
MOK_ITEM_WH = 7
MOK_ITEM_DA_Q = 8
MOK_ITEM_DA_SCALE = 9
MOK_ITEM_DY_Q = 10
MOK_ITEM_DY_SCALE = 11
MOK_ITEM_RING_TILES = 12
MOK_ITEM_RING_ORDER = 13

EXPORTED = [
    "mok_abi_version", "mok_status_string", "mok_check_config", "mok_segment_capacity",
    "mok_workspace_size", "mok_route_topk", "mok_build_schedule", "mok_forward",
    "mok_backward", "mok_quantize_mxfp8", "mok_read_device_status",
    "mok_clear_device_status", "mok_profile_enable", "mok_profile_read",
    "mok_build_schedule_noalloc", "mok_shared_expert_forward",
    "mok_quantize_mxfp8_transposed", "mok_backward_mxfp8", "mok_shared_expert_backward",
    "mok_shared_expert_forward_mxfp8", "mok_shared_expert_backward_mxfp8",
    "mok_selftest_bounded_wait", "mok_selftest_bounded_count_wait", "mok_workspace_item",
]

# bytes of the fixed scratch array behind mok_build_schedule_noalloc
MOK_NOALLOC_SCHEDULE_SCRATCH_BYTES = 4 << 20


class MokConfig(ctypes.Structure):
    _fields_ = [("abi_version", ctypes.c_uint32), ("T", ctypes.c_int32), ("H", ctypes.c_int32),
                ("I", ctypes.c_int32), ("E", ctypes.c_int32), ("K", ctypes.c_int32),
                ("minibatch", ctypes.c_int32), ("ring_capacity", ctypes.c_int32),
                ("prec", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class MokSchedule(ctypes.Structure):
    _fields_ = [("counts", ctypes.c_void_p), ("offsets", ctypes.c_void_p),
                ("perm", ctypes.c_void_p), ("inv", ctypes.c_void_p), ("segs", ctypes.c_void_p),
                ("n_segs", ctypes.c_void_p)]


class MokError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = int(status)
        super().__init__("%s: %s (status %d)" % (what or "mok", status_string(status),
                                                 self.status))


_lib = None


def lib():
    """The loaded library; raises if libmok.so has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libmok.so is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        p, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        cfgp = ctypes.POINTER(MokConfig)
        schp = ctypes.POINTER(MokSchedule)
        sig = {
            "mok_abi_version": ([], ctypes.c_uint32),
            "mok_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "mok_check_config": ([cfgp], ctypes.c_int),
            "mok_segment_capacity": ([cfgp], i64),
            "mok_workspace_size": ([cfgp, ctypes.c_int], sz),
            "mok_workspace_item": ([cfgp, ctypes.c_int, ctypes.c_int, ctypes.POINTER(sz),
                                    ctypes.POINTER(sz)], ctypes.c_int),
            "mok_route_topk": ([cfgp, p, p, p, p], ctypes.c_int),
            "mok_build_schedule": ([cfgp, p, schp, p, sz, p], ctypes.c_int),
            "mok_build_schedule_noalloc": ([cfgp, p, schp, p], ctypes.c_int),
            "mok_forward": ([cfgp, p, schp, p, p, p, p, p, p, p, p, sz, p], ctypes.c_int),
            "mok_backward": ([cfgp, p, schp, p, p, p, p, p, p, p, p, p, p, p, sz, p],
                             ctypes.c_int),
            "mok_shared_expert_forward": ([cfgp, p, p, p, p, p, p, sz, p], ctypes.c_int),
            "mok_shared_expert_forward_mxfp8": ([cfgp, p, p, p, p, p, p, p, p, sz, p],
                                                ctypes.c_int),
            "mok_shared_expert_backward_mxfp8": ([cfgp, p, p, p, p, p, p, p, p, p, p, p, sz, p],
                                                 ctypes.c_int),
            "mok_selftest_bounded_wait": ([ctypes.c_uint32, p], ctypes.c_int),
            "mok_selftest_bounded_count_wait": ([ctypes.c_uint32, p], ctypes.c_int),
            "mok_shared_expert_backward": ([cfgp, p, p, p, p, p, p, p, p, p, sz, p],
                                           ctypes.c_int),
            "mok_backward_mxfp8": ([cfgp, p, schp, p, p, p, p, p, p, p, p, p, p, p, p, p, sz,
                                    p], ctypes.c_int),
            "mok_quantize_mxfp8": ([p, i64, i32, p, p, p], ctypes.c_int),
            "mok_quantize_mxfp8_transposed": ([p, i64, i32, i32, p, p, p], ctypes.c_int),
            "mok_read_device_status": ([ctypes.POINTER(ctypes.c_int)], ctypes.c_int),
            "mok_clear_device_status": ([], ctypes.c_int),
            "mok_profile_enable": ([ctypes.c_int], ctypes.c_int),
            "mok_profile_read": ([i32, ctypes.POINTER(i32), ctypes.POINTER(ctypes.c_char_p),
                                  ctypes.POINTER(i64), ctypes.POINTER(ctypes.c_double)],
                                 ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


# ------------------------------------------------------------------------- marshalling

def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def make_config(T, H, I, E, K, minibatch=2368, ring_capacity=0, prec=MOK_BF16,
                abi_version=MOK_ABI_VERSION, flags=0) -> MokConfig:
    return MokConfig(abi_version, T, H, I, E, K, minibatch, ring_capacity, prec, flags)


def make_schedule(counts, offsets, perm, inv, segs, n_segs) -> MokSchedule:
    return MokSchedule(_ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(segs),
                       _ptr(n_segs))


def status_string(s) -> str:
    return lib().mok_status_string(int(s)).decode()


def check(status, what=""):
    if int(status) != MOK_OK:
        raise MokError(status, what)


# ------------------------------------------------------------------------- entry points

def mok_abi_version() -> int:
    return int(lib().mok_abi_version())


def mok_check_config(cfg) -> int:
    return lib().mok_check_config(ctypes.byref(cfg))


def mok_segment_capacity(cfg) -> int:
    return int(lib().mok_segment_capacity(ctypes.byref(cfg)))


def mok_workspace_size(cfg, which) -> int:
    return int(lib().mok_workspace_size(ctypes.byref(cfg), int(which)))


def mok_workspace_item(cfg, which, item):
    """(status, offset, bytes) of an intermediate inside a workspace (see include/mok.h)."""
    off = ctypes.c_size_t(0)
    n = ctypes.c_size_t(0)
    st = lib().mok_workspace_item(ctypes.byref(cfg), int(which), int(item), ctypes.byref(off),
                                  ctypes.byref(n))
    return st, off.value, n.value


def mok_route_topk(cfg, logits, topk_idx, topk_w, stream=None) -> int:
    return lib().mok_route_topk(ctypes.byref(cfg), _ptr(logits), _ptr(topk_idx), _ptr(topk_w),
                                _stream(stream))


def mok_build_schedule(cfg, topk_idx, sched, ws, ws_bytes, stream=None) -> int:
    return lib().mok_build_schedule(ctypes.byref(cfg), _ptr(topk_idx), ctypes.byref(sched),
                                    _ptr(ws), int(ws_bytes), _stream(stream))


def mok_build_schedule_noalloc(cfg, topk_idx, sched, stream=None) -> int:
    """mok_build_schedule for callers that cannot allocate a workspace (see include/mok.h)."""
    return lib().mok_build_schedule_noalloc(ctypes.byref(cfg), _ptr(topk_idx),
                                            ctypes.byref(sched), _stream(stream))


def mok_forward(cfg, x, sched, topk_w, w13, w13_scale, w2, w2_scale, y, saved_preact, ws,
                ws_bytes, stream=None) -> int:
    return lib().mok_forward(ctypes.byref(cfg), _ptr(x), ctypes.byref(sched), _ptr(topk_w),
                             _ptr(w13), _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), _ptr(y),
                             _ptr(saved_preact), _ptr(ws), int(ws_bytes), _stream(stream))


def mok_backward(cfg, x, sched, topk_w, saved_preact, w13, w2, dy, dx, dw13, dw2, d_topk_w,
                 d_logits, ws, ws_bytes, stream=None) -> int:
    return lib().mok_backward(ctypes.byref(cfg), _ptr(x), ctypes.byref(sched), _ptr(topk_w),
                              _ptr(saved_preact), _ptr(w13), _ptr(w2), _ptr(dy), _ptr(dx),
                              _ptr(dw13), _ptr(dw2), _ptr(d_topk_w), _ptr(d_logits), _ptr(ws),
                              int(ws_bytes), _stream(stream))


def mok_shared_expert_forward(cfg, x, w13_s, w2_s, y, saved_preact_s, ws, ws_bytes,
                              stream=None) -> int:
    return lib().mok_shared_expert_forward(ctypes.byref(cfg), _ptr(x), _ptr(w13_s), _ptr(w2_s),
                                           _ptr(y), _ptr(saved_preact_s), _ptr(ws),
                                           int(ws_bytes), _stream(stream))


def mok_backward_mxfp8(cfg, x, sched, topk_w, saved_preact, w13t_q, w13t_s, w2t_q, w2t_s, dy,
                       dx, dw13, dw2, d_topk_w, d_logits, ws, ws_bytes, stream=None) -> int:
    return lib().mok_backward_mxfp8(ctypes.byref(cfg), _ptr(x), ctypes.byref(sched),
                                    _ptr(topk_w), _ptr(saved_preact), _ptr(w13t_q),
                                    _ptr(w13t_s), _ptr(w2t_q), _ptr(w2t_s), _ptr(dy), _ptr(dx),
                                    _ptr(dw13), _ptr(dw2), _ptr(d_topk_w), _ptr(d_logits),
                                    _ptr(ws), int(ws_bytes), _stream(stream))


def mok_shared_expert_forward_mxfp8(cfg, x, w13s_q, w13s_scale, w2s_q, w2s_scale, y,
                                    saved_preact_s, ws, ws_bytes, stream=None) -> int:
    return lib().mok_shared_expert_forward_mxfp8(ctypes.byref(cfg), _ptr(x), _ptr(w13s_q),
                                                 _ptr(w13s_scale), _ptr(w2s_q),
                                                 _ptr(w2s_scale), _ptr(y), _ptr(saved_preact_s),
                                                 _ptr(ws), int(ws_bytes), _stream(stream))


def mok_selftest_bounded_wait(limit_us, stream=None) -> int:
    return lib().mok_selftest_bounded_wait(int(limit_us), _stream(stream))


def mok_selftest_bounded_count_wait(limit_us, stream=None) -> int:
    return lib().mok_selftest_bounded_count_wait(int(limit_us), _stream(stream))


def mok_shared_expert_backward_mxfp8(cfg, x, w13st_q, w13st_scale, w2st_q, w2st_scale,
                                     saved_preact_s, dy, dx, dw13_s, dw2_s, ws, ws_bytes,
                                     stream=None) -> int:
    return lib().mok_shared_expert_backward_mxfp8(
        ctypes.byref(cfg), _ptr(x), _ptr(w13st_q), _ptr(w13st_scale), _ptr(w2st_q),
        _ptr(w2st_scale), _ptr(saved_preact_s), _ptr(dy), _ptr(dx), _ptr(dw13_s), _ptr(dw2_s),
        _ptr(ws), int(ws_bytes), _stream(stream))


def mok_shared_expert_backward(cfg, x, w13_s, w2_s, saved_preact_s, dy, dx, dw13_s, dw2_s, ws,
                               ws_bytes, stream=None) -> int:
    return lib().mok_shared_expert_backward(ctypes.byref(cfg), _ptr(x), _ptr(w13_s),
                                            _ptr(w2_s), _ptr(saved_preact_s), _ptr(dy),
                                            _ptr(dx), _ptr(dw13_s), _ptr(dw2_s), _ptr(ws),
                                            int(ws_bytes), _stream(stream))


def mok_quantize_mxfp8(src, rows, cols, q, scale, stream=None) -> int:
    return lib().mok_quantize_mxfp8(_ptr(src), int(rows), int(cols), _ptr(q), _ptr(scale),
                                    _stream(stream))


def mok_quantize_mxfp8_transposed(src, batch, rows, cols, q, scale, stream=None) -> int:
    return lib().mok_quantize_mxfp8_transposed(_ptr(src), int(batch), int(rows), int(cols),
                                               _ptr(q), _ptr(scale), _stream(stream))


def mok_read_device_status():
    """(call status, device status)."""
    out = ctypes.c_int(0)
    st = lib().mok_read_device_status(ctypes.byref(out))
    return st, out.value


def mok_clear_device_status() -> int:
    return lib().mok_clear_device_status()


def mok_profile_enable(on) -> int:
    return lib().mok_profile_enable(1 if on else 0)


def mok_profile_read(max_kinds=32):
    """{kernel kind: (launches, total ms)} recorded since mok_profile_enable(1)."""
    n = ctypes.c_int32(0)
    names = (ctypes.c_char_p * max_kinds)()
    launches = (ctypes.c_int64 * max_kinds)()
    ms = (ctypes.c_double * max_kinds)()
    check(lib().mok_profile_read(max_kinds, ctypes.byref(n), names, launches, ms), "profile")
    return {names[i].decode(): (int(launches[i]), float(ms[i]))
            for i in range(min(n.value, max_kinds))}
