"""Test-only helpers: device transfer, tolerance checks, and CPU decoders of
the repacked device layouts (written from the layout description in
include/w4a8.h, independent of both the oracle and the CUDA code)."""
from __future__ import annotations

import numpy as np

# rtol of the fp32 outputs, relative to the magnitude of the summed terms
RTOL_W4 = 1e-5
RTOL_GROUP = 1e-4


def cuda_ok() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t) -> np.ndarray:
    return t.detach().cpu().numpy()


def check_close(y_gpu, y_ref, scale, rtol, what=""):
    """|y_gpu - y_ref| <= rtol * scale elementwise (scale = sum of |terms|)."""
    y_gpu = np.asarray(y_gpu, np.float64)
    err = np.abs(y_gpu - y_ref)
    bound = rtol * scale + 1e-30
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} outside tolerance; worst at {i}: "
                             f"gpu {y_gpu[i]!r} ref {y_ref[i]!r} scale {scale[i]!r}")


def w4_scale(acc, sw, sx, bias):
    """sum of |terms| of y = s_w s_x acc + b, shape [M][N]."""
    b = 0.0 if bias is None else np.abs(bias.astype(np.float64))[None, :]
    return np.abs(sw.astype(np.float64)[None, :] * sx.astype(np.float64)[:, None] * acc.astype(np.float64)) + b


def group_scale(acc_g, d, sx, bias):
    """s_x * sum_g |d_g acc_g| + |b|; acc_g [M][N][G], d [N][G] float64."""
    s = np.abs(sx.astype(np.float64))[:, None] * np.sum(np.abs(d[None, :, :] * acc_g.astype(np.float64)), axis=2)
    return s + (0.0 if bias is None else np.abs(bias.astype(np.float64))[None, :])


def q4_0_scales(blocks):
    bits = blocks[:, :, 0].astype(np.uint16) | (blocks[:, :, 1].astype(np.uint16) << 8)
    return bits.view(np.float16).astype(np.float64)


# ------------------------------------------------- device layout decoders
def _tiles(N):
    return (N + 7) // 8


def decode_w4_units(raw: np.ndarray, N: int, K: int, biased: bool = True) -> np.ndarray:
    """Repacked 4-bit units -> int8 values [N][K].  biased: nibble n = q + 8
    (per-row INT4); else 4-bit two's complement (Q4_0)."""
    C = K // 32
    T = _tiles(N)
    units = raw[: T * C * 8 * 16].reshape(T, C, 8, 4, 4)        # t, c, r, word, byte
    lo = (units & 0xF).astype(np.int16)
    hi = (units >> 4).astype(np.int16)
    if biased:
        lo, hi = lo - 8, hi - 8
    else:
        lo = np.where(lo >= 8, lo - 16, lo)
        hi = np.where(hi >= 8, hi - 16, hi)
    # weight index within the chunk: 8*word + byte (low) and 8*word + 4 + byte (high)
    w = np.concatenate([lo, hi], axis=4)                         # t, c, r, word, 8
    w = w.transpose(0, 2, 1, 3, 4).reshape(T * 8, C * 32)
    return w[:N].astype(np.int8)


def decode_group_plane(raw: np.ndarray, N: int, K: int, unit_bytes: int) -> np.ndarray:
    """fp16 scale plane -> float64 [N][K/32]."""
    C = K // 32
    T = _tiles(N)
    off = T * C * 8 * unit_bytes
    plane = raw[off: off + T * C * 8 * 2].view(np.uint16).reshape(T, C, 8)
    return plane.transpose(0, 2, 1).reshape(T * 8, C)[:N].view(np.float16).astype(np.float64)


def decode_i8_units(raw: np.ndarray, N: int, K: int) -> np.ndarray:
    C = K // 32
    T = _tiles(N)
    units = raw[: T * C * 8 * 32].view(np.int8).reshape(T, C, 8, 32)
    return units.transpose(0, 2, 1, 3).reshape(T * 8, K)[:N]


def decode_q6g32(raw: np.ndarray, N: int, K: int):
    """Q6G32 device layout -> (int8 codes [N][K], float64 scales [N][K/32])."""
    C = K // 32
    T = _tiles(N)
    units = T * C * 8
    lo = raw[: units * 16].reshape(T, C, 8, 4, 4)                       # t, c, r, word, byte
    lo_l = (lo & 0xF).astype(np.int16)
    lo_h = (lo >> 4).astype(np.int16)
    low = np.concatenate([lo_l, lo_h], axis=4).reshape(T, C, 8, 32)    # weight 8w+b, 8w+4+b
    hi = raw[units * 16: units * 24].reshape(T, C, 8, 2, 4)            # t, c, r, word h, byte b
    shifts = np.array([0, 2, 4, 6], np.uint8)
    hv = (hi[..., None, :] >> shifts[:, None]) & 3                     # t, c, r, h, s, b
    high = hv.reshape(T, C, 8, 32).astype(np.int16)                    # weight 16h + 4s + b
    n = low + 16 * high
    q = (n - 32).transpose(0, 2, 1, 3).reshape(T * 8, K)[:N].astype(np.int8)
    plane = raw[units * 24: units * 26].view(np.uint16).reshape(T, C, 8)
    d = plane.transpose(0, 2, 1).reshape(T * 8, C)[:N].view(np.float16).astype(np.float64)
    return q, d
