"""CPU oracle for bit-quantized decode GEMV -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
this package never imports the product: the two share no code.

The arithmetic lives in ``w4a8_oracle.c`` (plain C, fp32 quantization
decisions, exact integer dot products, fp64 dequantization).  This module
compiles it with gcc on first use and wraps each function for numpy arrays.

Sources (the two web pages the method is taken from):
  [Orin-INT4]   "Jetson Orin AGX INT4 推理优化实践：super 分支从 9 tok/s 到 24 tok/s"
  [310B-Gemma4] "在香橙派上跑 Gemma4：vLLM 适配昇腾 310B 的内核开发实录"

Every function is pinned by ``tests/test_oracle_pins.py`` against values the
pages print, closed forms, library routines and brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a8_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ORC_OK = 0
ORC_ERR_ARG = 1
ORC_ERR_INT32_OVERFLOW = 2

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source (gcc, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.orc_half_to_float.argtypes = [ctypes.c_uint16]
            lib.orc_half_to_float.restype = ctypes.c_float
            lib.orc_float_to_half.argtypes = [ctypes.c_float]
            lib.orc_float_to_half.restype = ctypes.c_uint16
            for name, args in {
                "orc_quantize_act_int8": [P, I, I, P, P],
                "orc_quantize_rows_int4": [P, I, I, P, P],
                "orc_pack_int4": [P, I, I, P],
                "orc_unpack_int4": [P, I, I, P],
                "orc_gemv_w4a8_acc": [P, P, I, I, I, P],
                "orc_epilogue_w4a8": [P, P, P, P, I, I, P],
                "orc_quantize_q4_0": [P, I, I, P],
                "orc_dequantize_q4_0": [P, I, I, P],
                "orc_gemv_q4_0": [P, P, P, P, I, I, I, P, P],
                "orc_quantize_i8g32": [P, I, I, P, P],
                "orc_gemv_i8g32": [P, P, P, P, P, I, I, I, P, P],
                "orc_glu": [P, P, I, I, P],
                "orc_quantize_rows_int8": [P, I, I, P, P],
                "orc_gemv_weight_only": [P, P, P, P, I, I, I, P],
            }.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = ctypes.c_int
            lib.orc_rmsnorm_f32.argtypes = [P, P, ctypes.c_float, I, I, P]
            lib.orc_rmsnorm_f32.restype = ctypes.c_int
            lib.orc_dp4a.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int32]
            lib.orc_dp4a.restype = ctypes.c_int32
            lib.orc_q4_0_block_bytes.argtypes = []
            lib.orc_q4_0_block_bytes.restype = ctypes.c_int
            lib.orc_row_weight_bytes.argtypes = [I, I]
            lib.orc_row_weight_bytes.restype = ctypes.c_longlong
            _lib = lib
        return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, name):
    if rc != ORC_OK:
        raise OracleError(rc, name)


class OracleError(RuntimeError):
    def __init__(self, rc, name):
        super().__init__(f"{name} returned {rc}")
        self.rc = rc


# ---------------------------------------------------------------- fp16 helpers
def half_to_float(h: int) -> float:
    return float(_load().orc_half_to_float(int(h)))


def float_to_half(f: float) -> int:
    return int(_load().orc_float_to_half(float(f)))


# -------------------------------------------------------------- activations
def quantize_act_int8(x):
    """[Orin-INT4] per-token INT8 quantization: returns (qx int8 [M][K], sx f32 [M])."""
    x = _c(np.atleast_2d(x), np.float32)
    M, K = x.shape
    qx = np.zeros((M, K), np.int8)
    sx = np.zeros(M, np.float32)
    _check(_load().orc_quantize_act_int8(_ptr(x), M, K, _ptr(qx), _ptr(sx)), "quantize_act_int8")
    return qx, sx


# ---------------------------------------------------------- per-row INT4
def quantize_rows_int4(W):
    """Per-row symmetric INT4: returns (q int8 [N][K] in [-8,7], s_w f32 [N])."""
    W = _c(W, np.float32)
    N, K = W.shape
    q = np.zeros((N, K), np.int8)
    sw = np.zeros(N, np.float32)
    _check(_load().orc_quantize_rows_int4(_ptr(W), N, K, _ptr(q), _ptr(sw)), "quantize_rows_int4")
    return q, sw


def pack_int4(q):
    q = _c(q, np.int8)
    N, K = q.shape
    out = np.zeros((N, K // 8), np.uint32)
    _check(_load().orc_pack_int4(_ptr(q), N, K, _ptr(out)), "pack_int4")
    return out


def unpack_int4(packed, K):
    packed = _c(packed, np.uint32)
    N = packed.shape[0]
    q = np.zeros((N, K), np.int8)
    _check(_load().orc_unpack_int4(_ptr(packed), N, K, _ptr(q)), "unpack_int4")
    return q


def dp4a(a: int, b: int, c: int) -> int:
    return int(_load().orc_dp4a(a & 0xFFFFFFFF, b & 0xFFFFFFFF, int(c)))


def gemv_w4a8_acc(packed, qx):
    """Exact int32 accumulators acc[m][j] = sum_i q_w[j,i] qx[m,i]."""
    packed = _c(packed, np.uint32)
    qx = _c(np.atleast_2d(qx), np.int8)
    N = packed.shape[0]
    M, K = qx.shape
    assert packed.shape[1] * 8 == K
    acc = np.zeros((M, N), np.int32)
    _check(_load().orc_gemv_w4a8_acc(_ptr(packed), _ptr(qx), M, N, K, _ptr(acc)), "gemv_w4a8_acc")
    return acc


def epilogue_w4a8(acc, sw, sx, bias=None):
    """y = s_w[j] * s_x[m] * acc[m][j] + b[j] in fp64."""
    acc = _c(np.atleast_2d(acc), np.int32)
    M, N = acc.shape
    sw = _c(sw, np.float32)
    sx = _c(np.atleast_1d(sx), np.float32)
    b = None if bias is None else _c(bias, np.float32)
    y = np.zeros((M, N), np.float64)
    _check(_load().orc_epilogue_w4a8(_ptr(acc), _ptr(sw), _ptr(sx), _ptr(b), M, N, _ptr(y)),
           "epilogue_w4a8")
    return y


def w4a8_linear(packed, sw, x, bias=None):
    """The whole per-row INT4 decode linear: quantize x, integer GEMV, epilogue.

    Returns (y fp64 [M][N], qx, sx, acc)."""
    qx, sx = quantize_act_int8(x)
    acc = gemv_w4a8_acc(packed, qx)
    return epilogue_w4a8(acc, sw, sx, bias), qx, sx, acc


# ---------------------------------------------------------------- Q4_0
def q4_0_block_bytes() -> int:
    return int(_load().orc_q4_0_block_bytes())


def quantize_q4_0(W):
    """Q4_0 blocks, uint8 [N][K/32][18]."""
    W = _c(W, np.float32)
    N, K = W.shape
    blocks = np.zeros((N, K // 32, 18), np.uint8)
    _check(_load().orc_quantize_q4_0(_ptr(W), N, K, _ptr(blocks)), "quantize_q4_0")
    return blocks


def dequantize_q4_0(blocks, K):
    blocks = _c(blocks, np.uint8)
    N = blocks.shape[0]
    W = np.zeros((N, K), np.float64)
    _check(_load().orc_dequantize_q4_0(_ptr(blocks), N, K, _ptr(W)), "dequantize_q4_0")
    return W


def gemv_q4_0(blocks, qx, sx, bias=None, want_acc=False):
    blocks = _c(blocks, np.uint8)
    qx = _c(np.atleast_2d(qx), np.int8)
    sx = _c(np.atleast_1d(sx), np.float32)
    M, K = qx.shape
    N = blocks.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    y = np.zeros((M, N), np.float64)
    acc = np.zeros((M, N, K // 32), np.int32) if want_acc else None
    _check(_load().orc_gemv_q4_0(_ptr(blocks), _ptr(qx), _ptr(sx), _ptr(b), M, N, K, _ptr(acc), _ptr(y)),
           "gemv_q4_0")
    return (y, acc) if want_acc else y


# --------------------------------------------------------------- i8g32
def quantize_i8g32(W):
    """int8 values in [-32,31] and fp16 scale bits per group of 32."""
    W = _c(W, np.float32)
    N, K = W.shape
    q = np.zeros((N, K), np.int8)
    d = np.zeros((N, K // 32), np.uint16)
    _check(_load().orc_quantize_i8g32(_ptr(W), N, K, _ptr(q), _ptr(d)), "quantize_i8g32")
    return q, d


def gemv_i8g32(q, d, qx, sx, bias=None, want_acc=False):
    q = _c(q, np.int8)
    d = _c(d, np.uint16)
    qx = _c(np.atleast_2d(qx), np.int8)
    sx = _c(np.atleast_1d(sx), np.float32)
    M, K = qx.shape
    N = q.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    y = np.zeros((M, N), np.float64)
    acc = np.zeros((M, N, K // 32), np.int32) if want_acc else None
    _check(_load().orc_gemv_i8g32(_ptr(q), _ptr(d), _ptr(qx), _ptr(sx), _ptr(b), M, N, K, _ptr(acc),
                                  _ptr(y)), "gemv_i8g32")
    return (y, acc) if want_acc else y


def row_weight_bytes(K: int, bits: int) -> int:
    return int(_load().orc_row_weight_bytes(K, bits))


# ---------------------------------------------- operators around the linear
GLU_SILU = 1
GLU_GELU_TANH = 2


def rmsnorm_f32(x, g, eps):
    """RMSNorm per token in fp32 steps: (x * (1 / sqrt(sum x^2 / K + eps))) * g."""
    x = _c(np.atleast_2d(x), np.float32)
    M, K = x.shape
    g = _c(g, np.float32)
    assert g.shape == (K,)
    out = np.zeros((M, K), np.float32)
    _check(_load().orc_rmsnorm_f32(_ptr(x), _ptr(g), float(eps), M, K, _ptr(out)), "rmsnorm_f32")
    return out


def glu(gate, up, kind):
    """act(gate) * up in fp64; kind GLU_SILU (SwiGLU) or GLU_GELU_TANH."""
    gate = _c(gate, np.float64)
    up = _c(up, np.float64)
    assert gate.shape == up.shape
    out = np.zeros(gate.shape, np.float64)
    _check(_load().orc_glu(_ptr(gate), _ptr(up), gate.size, int(kind), _ptr(out)), "glu")
    return out


def rmsnorm_w4a8_linear(packed, sw, x, g, eps, bias=None):
    """RMSNorm, then the per-row INT4 decode linear on the normalized tokens.

    Returns (y fp64 [M][N], qx, sx, acc, xn)."""
    xn = rmsnorm_f32(x, g, eps)
    y, qx, sx, acc = w4a8_linear(packed, sw, xn, bias)
    return y, qx, sx, acc, xn


# -------------------------------------- weight-only paths (float activations)
def quantize_rows_int8(W):
    """Per-row symmetric INT8: returns (q int8 [N][K] in [-127,127], s_w f32 [N])."""
    W = _c(W, np.float32)
    N, K = W.shape
    q = np.zeros((N, K), np.int8)
    sw = np.zeros(N, np.float32)
    _check(_load().orc_quantize_rows_int8(_ptr(W), N, K, _ptr(q), _ptr(sw)), "quantize_rows_int8")
    return q, sw


def gemv_weight_only(q, sw, x, bias=None):
    """y = s_w[j] * sum_i q[j,i] x[m,i] + b[j] in fp64, activations not quantized."""
    q = _c(q, np.int8)
    sw = _c(sw, np.float32)
    x = _c(np.atleast_2d(x), np.float32)
    M, K = x.shape
    N = q.shape[0]
    assert q.shape[1] == K
    b = None if bias is None else _c(bias, np.float32)
    y = np.zeros((M, N), np.float64)
    _check(_load().orc_gemv_weight_only(_ptr(q), _ptr(sw), _ptr(x), _ptr(b), M, N, K, _ptr(y)),
           "gemv_weight_only")
    return y
