"""Counter-keyed Gaussian draws, rounded to the layer's storage types.

Every tensor is a flat sequence of standard-normal float32 draws cut into chunks of
2**22 elements. Chunk c of tensor `tag` under `seed` comes from its own Philox-4x64
stream keyed (seed, tag << 32 | c), so any row range of a tensor can be regenerated on
its own (the oracle side regenerates only the tokens and experts it samples) and chunks
can be drawn in parallel. Draws are scaled by the tensor's standard deviation in
float32 and, for bf16 tensors, rounded to nearest-even bf16.
"""
from concurrent.futures import ThreadPoolExecutor
import os

import numpy as np

CHUNK = 1 << 22

TAG_X, TAG_LOGITS, TAG_W13, TAG_W2, TAG_DY = 1, 2, 3, 4, 5

_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))
    return _POOL


def _chunk_draw(seed: int, tag: int, c: int, n: int) -> np.ndarray:
    key = np.array([seed & 0xFFFFFFFFFFFFFFFF, ((tag & 0xFFFFFFFF) << 32) | (c & 0xFFFFFFFF)],
                   dtype=np.uint64)
    g = np.random.Generator(np.random.Philox(key=key))
    return g.standard_normal(n, dtype=np.float32)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); finite inputs only."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


def normal_f32(seed: int, tag: int, n: int, std: float = 1.0, out_bf16: np.ndarray = None,
               start: int = 0) -> np.ndarray:
    """Elements [start, start+n) of tensor `tag`, as float32 (or written as bf16 bits).

    When `out_bf16` is given (a uint16 array of n elements), the bf16-rounded values are
    written there and it is returned; otherwise a float32 array is returned.
    """
    std32 = np.float32(std)
    if out_bf16 is None:
        out = np.empty(n, dtype=np.float32)
    else:
        out = out_bf16
        assert out.dtype == np.uint16 and out.size == n
    c0 = start // CHUNK
    c1 = (start + n + CHUNK - 1) // CHUNK if n > 0 else c0

    def work(c):
        lo = max(start, c * CHUNK)
        hi = min(start + n, (c + 1) * CHUNK)
        if hi <= lo:
            return
        # draws are sequential within a chunk, so a prefix of the chunk's stream is enough
        d = _chunk_draw(seed, tag, c, hi - c * CHUNK)
        seg = d[lo - c * CHUNK: hi - c * CHUNK]
        if std32 != np.float32(1.0):
            seg = seg * std32
        if out_bf16 is None:
            out[lo - start: hi - start] = seg
        else:
            out[lo - start: hi - start] = f32_to_bf16_bits(seg)

    list(_pool().map(work, range(c0, c1)))
    return out


def normal_f32_rows(seed: int, tag: int, row_len: int, row0: int, row1: int,
                    std: float = 1.0, bf16: bool = True) -> np.ndarray:
    """Rows [row0, row1) of a row-major tensor with rows of `row_len` elements."""
    n = (row1 - row0) * row_len
    if bf16:
        buf = np.empty(n, dtype=np.uint16)
        normal_f32(seed, tag, n, std, out_bf16=buf, start=row0 * row_len)
        return buf.reshape(row1 - row0, row_len)
    return normal_f32(seed, tag, n, std, start=row0 * row_len).reshape(row1 - row0, row_len)


# ---------------------------------------------------------------------------------------
# the layer's tensors


def make_x(cfg, out=None, rows=None) -> np.ndarray:
    """Token activations X [T, H] as bf16 bits."""
    r0, r1 = rows if rows is not None else (0, cfg.T)
    if out is not None:
        normal_f32(cfg.seed, TAG_X, (r1 - r0) * cfg.H, cfg.x_std, out_bf16=out.reshape(-1),
                   start=r0 * cfg.H)
        return out
    return normal_f32_rows(cfg.seed, TAG_X, cfg.H, r0, r1, cfg.x_std)


def make_dy(cfg, out=None, rows=None) -> np.ndarray:
    """Upstream gradient dY [T, H] as bf16 bits."""
    r0, r1 = rows if rows is not None else (0, cfg.T)
    if out is not None:
        normal_f32(cfg.seed, TAG_DY, (r1 - r0) * cfg.H, cfg.dy_std, out_bf16=out.reshape(-1),
                   start=r0 * cfg.H)
        return out
    return normal_f32_rows(cfg.seed, TAG_DY, cfg.H, r0, r1, cfg.dy_std)


def zipf_bias(E: int) -> np.ndarray:
    """Per-expert logit bias 2*ln(1/rank) with rank(e) = e + 1, in float32."""
    return (-2.0 * np.log(np.arange(1, E + 1, dtype=np.float64))).astype(np.float32)


def make_logits(cfg, rows=None) -> np.ndarray:
    """Router logits [T, E] float32: N(0,1), plus the Zipf-like bias when configured."""
    r0, r1 = rows if rows is not None else (0, cfg.T)
    z = normal_f32_rows(cfg.seed, TAG_LOGITS, cfg.E, r0, r1, 1.0, bf16=False)
    if cfg.zipf_bias:
        z = z + zipf_bias(cfg.E)[None, :]
    return np.ascontiguousarray(z, dtype=np.float32)


def make_w13(cfg, out=None, experts=None) -> np.ndarray:
    """Gate/up weights W13 [E, 2I, H] as bf16 bits (gate rows 0..I-1, up rows I..2I-1)."""
    per = 2 * cfg.I * cfg.H
    if experts is None:
        if out is None:
            out = np.empty(cfg.E * per, dtype=np.uint16)
        normal_f32(cfg.seed, TAG_W13, cfg.E * per, cfg.w_std, out_bf16=out.reshape(-1))
        return out.reshape(cfg.E, 2 * cfg.I, cfg.H)
    res = np.empty((len(experts), 2 * cfg.I, cfg.H), dtype=np.uint16)
    for j, e in enumerate(experts):
        normal_f32(cfg.seed, TAG_W13, per, cfg.w_std, out_bf16=res[j].reshape(-1), start=e * per)
    return res


def make_w2(cfg, out=None, experts=None) -> np.ndarray:
    """Down weights W2 [E, H, I] as bf16 bits."""
    per = cfg.H * cfg.I
    if experts is None:
        if out is None:
            out = np.empty(cfg.E * per, dtype=np.uint16)
        normal_f32(cfg.seed, TAG_W2, cfg.E * per, cfg.w_std, out_bf16=out.reshape(-1))
        return out.reshape(cfg.E, cfg.H, cfg.I)
    res = np.empty((len(experts), cfg.H, cfg.I), dtype=np.uint16)
    for j, e in enumerate(experts):
        normal_f32(cfg.seed, TAG_W2, per, cfg.w_std, out_bf16=res[j].reshape(-1), start=e * per)
    return res


def logit_margin_ok(logits: np.ndarray, K: int, margin: float) -> bool:
    """True when every row's K-th and (K+1)-th largest logits differ by more than margin."""
    s = -np.sort(-logits.astype(np.float64), axis=1)
    if K >= logits.shape[1]:
        return True
    return bool(np.all(s[:, K - 1] - s[:, K] > margin))


__all__ = ["CHUNK", "normal_f32", "normal_f32_rows", "make_x", "make_dy", "make_logits",
           "make_w13", "make_w2", "f32_to_bf16_bits", "bf16_bits_to_f32", "zipf_bias",
           "logit_margin_ok"]
