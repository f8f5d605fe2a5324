"""Device-memory plumbing for the C ABI: torch allocates, the library computes.

`MoELayer` owns the caller-side buffers of one configuration (schedule arrays and the
three workspaces) and strings the entry points together in the order a user calls them:
mok_route_topk -> mok_build_schedule -> mok_forward (-> mok_backward). Every method only
passes pointers; all arithmetic happens in libmok.so.
"""
import torch

from . import binding as B


def _empty(n, dtype, device):
    return torch.empty(max(int(n), 1), dtype=dtype, device=device)


class Schedule:
    """Device arrays of one schedule table (mok_schedule)."""

    def __init__(self, cfg, device):
        R = cfg.T * cfg.K
        self.cap = B.mok_segment_capacity(cfg)
        i32 = torch.int32
        self.counts = _empty(cfg.E, i32, device)
        self.offsets = _empty(cfg.E + 1, i32, device)
        self.perm = _empty(R, i32, device)
        self.inv = _empty(R, i32, device)
        self.segs = _empty(3 * self.cap, i32, device)
        self.n_segs = _empty(1, i32, device)
        self.struct = B.make_schedule(self.counts, self.offsets, self.perm, self.inv, self.segs,
                                      self.n_segs)
        self.R = R


def workspace(cfg, which, device):
    n = B.mok_workspace_size(cfg, which)
    return _empty(n, torch.uint8, device), n


def workspace_item(ws, cfg, which, item):
    """The bytes of one intermediate inside workspace tensor `ws` (a uint8 view, see
    mok_workspace_item); callers view it with the item's dtype and shape."""
    st, off, n = B.mok_workspace_item(cfg, which, item)
    B.check(st, "workspace item")
    return ws[off: off + n]


def stored_dtype(cfg):
    """torch dtype of the values the layer only stores (outputs, slots, saved A)."""
    return torch.float32 if cfg.flags & B.MOK_FLAG_FP32_STORAGE else torch.bfloat16


class MoELayer:
    """One layer configuration with its buffers on `device` (a CUDA device)."""

    def __init__(self, T, H, I, E, K, minibatch=2368, ring_capacity=0, prec=B.MOK_BF16,
                 device="cuda", backward=False, flags=0):
        self.cfg = B.make_config(T, H, I, E, K, minibatch, ring_capacity, prec, flags=flags)
        self.dtype = stored_dtype(self.cfg)
        B.check(B.mok_check_config(self.cfg), "config")
        self.device = torch.device(device)
        self.T, self.H, self.I, self.E, self.K = T, H, I, E, K
        self.sched = Schedule(self.cfg, self.device)
        self.ws_s, self.ws_s_n = workspace(self.cfg, B.MOK_WS_SCHEDULE, self.device)
        self.ws_f, self.ws_f_n = workspace(self.cfg, B.MOK_WS_FORWARD, self.device)
        self.idx = _empty(T * K, torch.int32, self.device)
        self.w = _empty(T * K, torch.float32, self.device)
        self.ws_b = None
        if backward:
            self.ws_b, self.ws_b_n = workspace(self.cfg, B.MOK_WS_BACKWARD, self.device)

    def route(self, logits, stream=None):
        B.check(B.mok_route_topk(self.cfg, logits, self.idx, self.w, stream), "route")
        return self.idx, self.w

    def schedule(self, idx=None, stream=None):
        B.check(B.mok_build_schedule(self.cfg, self.idx if idx is None else idx,
                                     self.sched.struct, self.ws_s, self.ws_s_n, stream),
                "schedule")
        return self.sched

    def forward(self, x, w13, w2, y, w13_scale=None, w2_scale=None, saved_preact=None,
                topk_w=None, stream=None):
        B.check(B.mok_forward(self.cfg, x, self.sched.struct, self.w if topk_w is None else
                              topk_w, w13, w13_scale, w2, w2_scale, y, saved_preact, self.ws_f,
                              self.ws_f_n, stream), "forward")
        return y

    def backward(self, x, saved_preact, w13, w2, dy, dx, dw13, dw2, d_topk_w, d_logits=None,
                 topk_w=None, stream=None):
        if saved_preact is None:  # recompute the pre-activations: larger workspace
            if getattr(self, "ws_r", None) is None:
                self.ws_r, self.ws_r_n = workspace(self.cfg, B.MOK_WS_BACKWARD_RECOMPUTE,
                                                   self.device)
            ws, ws_n = self.ws_r, self.ws_r_n
        else:
            if self.ws_b is None:
                self.ws_b, self.ws_b_n = workspace(self.cfg, B.MOK_WS_BACKWARD, self.device)
            ws, ws_n = self.ws_b, self.ws_b_n
        B.check(B.mok_backward(self.cfg, x, self.sched.struct, self.w if topk_w is None else
                               topk_w, saved_preact, w13, w2, dy, dx, dw13, dw2, d_topk_w,
                               d_logits, ws, ws_n, stream), "backward")
        return dx


def backward_mxfp8(layer, x, saved_preact, w13t, w2t, dy, dx, dw13, dw2, d_topk_w,
                   d_logits=None, topk_w=None, stream=None):
    """MXFP8 backward of a layer built with prec=MOK_MXFP8 (backward=True); w13t, w2t are
    (q, scale) pairs from quantize_mxfp8_transposed of the bf16 W13 and W2."""
    if layer.ws_b is None:
        layer.ws_b, layer.ws_b_n = workspace(layer.cfg, B.MOK_WS_BACKWARD, layer.device)
    B.check(B.mok_backward_mxfp8(layer.cfg, x, layer.sched.struct,
                                 layer.w if topk_w is None else topk_w, saved_preact, w13t[0],
                                 w13t[1], w2t[0], w2t[1], dy, dx, dw13, dw2, d_topk_w, d_logits,
                                 layer.ws_b, layer.ws_b_n, stream), "backward mxfp8")
    return dx


class SharedExpert:
    """The shared expert of a layer configuration (same H, I as the routed experts)."""

    def __init__(self, layer):
        self.cfg = layer.cfg
        self.ws, self.ws_n = workspace(self.cfg, B.MOK_WS_SHARED, layer.device)

    def forward(self, x, w13_s, w2_s, y, saved_preact=None, stream=None):
        """y += the shared expert's output for every token (after the routed forward).
        MXFP8 layers take w13_s, w2_s as (q, scale) pairs from quantize_mxfp8."""
        if self.cfg.prec == B.MOK_MXFP8:
            B.check(B.mok_shared_expert_forward_mxfp8(self.cfg, x, w13_s[0], w13_s[1],
                                                      w2_s[0], w2_s[1], y, saved_preact,
                                                      self.ws, self.ws_n, stream),
                    "shared forward mxfp8")
            return y
        B.check(B.mok_shared_expert_forward(self.cfg, x, w13_s, w2_s, y, saved_preact,
                                            self.ws, self.ws_n, stream), "shared forward")
        return y

    def backward(self, x, w13_s, w2_s, saved_preact, dy, dx, dw13_s, dw2_s, stream=None):
        """dx += the shared expert's input gradient; dw13_s, dw2_s = its weight gradients.
        MXFP8 layers take w13_s, w2_s as (q, scale) pairs from quantize_mxfp8_transposed
        (of W13s[None] and W2s[None])."""
        if getattr(self, "ws_b", None) is None:
            self.ws_b, self.ws_b_n = workspace(self.cfg, B.MOK_WS_SHARED_BACKWARD,
                                               x.device)
        if self.cfg.prec == B.MOK_MXFP8:
            B.check(B.mok_shared_expert_backward_mxfp8(self.cfg, x, w13_s[0], w13_s[1],
                                                       w2_s[0], w2_s[1], saved_preact, dy, dx,
                                                       dw13_s, dw2_s, self.ws_b, self.ws_b_n,
                                                       stream), "shared backward mxfp8")
            return dx
        B.check(B.mok_shared_expert_backward(self.cfg, x, w13_s, w2_s, saved_preact, dy, dx,
                                             dw13_s, dw2_s, self.ws_b, self.ws_b_n, stream),
                "shared backward")
        return dx


def quantize_mxfp8_transposed(src, stream=None):
    """MXFP8 of a [batch][rows][cols] bf16 tensor along rows, stored as [batch][cols][rows]
    (q) and [batch][cols][rows/32] (scale): the MXFP8 backward's pre-quantized weights."""
    b, r, c = src.shape
    q = torch.empty((b, c, r), dtype=torch.uint8, device=src.device)
    s = torch.empty((b, c, r // 32), dtype=torch.uint8, device=src.device)
    B.check(B.mok_quantize_mxfp8_transposed(src, b, r, c, q, s, stream), "quantize_transposed")
    return q, s


def quantize_mxfp8(src, stream=None):
    """MXFP8 along the last axis of a bf16 tensor: (q uint8, scale uint8)."""
    cols = src.shape[-1]
    rows = src.numel() // cols
    q = torch.empty(src.shape, dtype=torch.uint8, device=src.device)
    s = torch.empty(src.shape[:-1] + (cols // 32,), dtype=torch.uint8, device=src.device)
    B.check(B.mok_quantize_mxfp8(src, rows, cols, q, s, stream), "quantize")
    return q, s
