"""ctypes binding of ``libw4a8.so`` (C ABI declared in include/w4a8.h).

Argument marshalling only: every function takes torch tensors that already
live on the current CUDA device, checks dtypes and shapes, and passes raw
pointers and the current stream to the C entry point of the same name.  All
arithmetic runs in the library's CUDA kernels; there is no CPU path.  If the
library has not been built, loading fails with an error saying how to build
it.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw4a8.so")

W4_OK = 0
STATUS = {
    0: "W4_OK",
    1: "W4_ERR_INVALID_ARG",
    2: "W4_ERR_UNSUPPORTED_SHAPE",
    3: "W4_ERR_MISALIGNED",
    4: "W4_ERR_CUDA",
    5: "W4_ERR_DEVICE_TIMEOUT",
}
W4_FLAG_PDL = 1
TUNE_KEYS = {"blocks_per_sm": 0, "max_stages": 1, "grid_blocks": 2, "tc_min_m": 3, "chain_prefetch_kb": 4, "k_splits": 5,
             "group_launch_tokens": 6}
W4_MAX_M = 16
W4_MAX_K = 131072
W4_MAX_SHARDS = 8

# exported symbol -> (argtypes, restype)
_P = ctypes.c_void_p
_I = ctypes.c_int
_U = ctypes.c_uint
_SZ = ctypes.c_size_t
_PP = ctypes.POINTER(ctypes.c_void_p)
_PI = ctypes.POINTER(ctypes.c_int)
SIGNATURES = {
    "w4_status_str": ([_I], ctypes.c_char_p),
    "w4_version": ([], _I),
    "w4_set_tuning": ([_I, _I], _I),
    "w4_get_tuning": ([_I], _I),
    "w4_quantize_rows": ([_P, _I, _I, _P, _P, _P], _I),
    "q4_0_quantize": ([_P, _I, _I, _P, _P], _I),
    "i8g32_quantize": ([_P, _I, _I, _P, _P, _P], _I),
    "w4_repacked_bytes": ([_I, _I], _SZ),
    "q4_0_repacked_bytes": ([_I, _I], _SZ),
    "i8g32_repacked_bytes": ([_I, _I], _SZ),
    "q6g32_repacked_bytes": ([_I, _I], _SZ),
    "w4_repack": ([_PP, _PI, _I, _I, _P, _SZ, _P], _I),
    "q4_0_repack": ([_PP, _PI, _I, _I, _P, _SZ, _P], _I),
    "i8g32_repack": ([_PP, _PP, _PI, _I, _I, _P, _SZ, _P], _I),
    "q6g32_repack": ([_PP, _PP, _PI, _I, _I, _P, _SZ, _P], _I),
    "w4_concat_f32": ([_PP, _PI, _I, _P, _P], _I),
    "a8_quantize": ([_P, _I, _I, _P, _P, _P], _I),
    "w4a8_gemv": ([_P, _P, _P, _P, _P, _I, _I, _I, _P, _P], _I),
    "q4_0_gemv": ([_P, _P, _P, _P, _I, _I, _I, _P, _P], _I),
    "i8g32_gemv": ([_P, _P, _P, _P, _I, _I, _I, _P, _P], _I),
    "q6g32_gemv": ([_P, _P, _P, _P, _I, _I, _I, _P, _P], _I),
    "w4a8_linear": ([_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _U, _P], _I),
    "q4_0_linear": ([_P, _P, _P, _I, _I, _I, _P, _P, _P, _U, _P], _I),
    "i8g32_linear": ([_P, _P, _P, _I, _I, _I, _P, _P, _P, _U, _P], _I),
    "q6g32_linear": ([_P, _P, _P, _I, _I, _I, _P, _P, _P, _U, _P], _I),
    "w4_device_error": ([ctypes.POINTER(ctypes.c_uint)], _I),
    "w4_clear_device_error": ([], _I),
}


class Fusion(ctypes.Structure):
    """w4_fusion of include/w4a8.h."""
    _fields_ = [("norm_weight", _P), ("norm_eps", ctypes.c_float), ("glu", _I), ("residual", _P)]


W4_GLU_NONE = 0
W4_GLU_SILU = 1
W4_GLU_GELU_TANH = 2
_F = ctypes.c_float
_LL = ctypes.c_longlong
_PF = ctypes.POINTER(Fusion)
SIGNATURES.update({
    "w4_glu_repacked_bytes": ([_I, _I], _SZ),
    "q4_0_glu_repacked_bytes": ([_I, _I], _SZ),
    "w4_repack_glu": ([_P, _P, _I, _I, _P, _SZ, _P], _I),
    "q4_0_repack_glu": ([_P, _P, _I, _I, _P, _SZ, _P], _I),
    "w4a8_linear_fused": ([_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _PF, _U, _P], _I),
    "q4_0_linear_fused": ([_P, _P, _P, _I, _I, _I, _P, _P, _P, _PF, _U, _P], _I),
    "i8g32_linear_fused": ([_P, _P, _P, _I, _I, _I, _P, _P, _P, _PF, _U, _P], _I),
    "q6g32_linear_fused": ([_P, _P, _P, _I, _I, _I, _P, _P, _P, _PF, _U, _P], _I),
    "rms_a8_quantize": ([_P, _P, _F, _I, _I, _P, _P, _U, _P], _I),
    "w4_rmsnorm": ([_P, _P, _F, _I, _I, _P, _U, _P], _I),
    "w4_glu": ([_P, _I, _I, _I, _P, _U, _P], _I),
    "w4_add": ([_P, _P, _LL, _P, _U, _P], _I),
    "w8_quantize_rows": ([_P, _I, _I, _P, _P, _P], _I),
    "w8_repacked_bytes": ([_I, _I], _SZ),
    "w8_repack": ([_PP, _PI, _I, _I, _P, _SZ, _P], _I),
    "w4a32_gemv": ([_P, _P, _P, _P, _I, _I, _I, _P, _U, _P], _I),
    "w8a32_gemv": ([_P, _P, _P, _P, _I, _I, _I, _P, _U, _P], _I),
})


class LinearDesc(ctypes.Structure):
    """w4_linear_desc of include/w4a8.h."""
    _fields_ = [("w", _P), ("s_w", _P), ("bias", _P), ("x", _P), ("y", _P), ("qx", _P), ("sx", _P),
                ("N", _I), ("K", _I)]


class DeviceDesc(ctypes.Structure):
    """w4_device_desc of include/w4a8.h."""
    _fields_ = [("sms", _I), ("smem_per_sm", _I), ("smem_reserved", _I), ("smem_optin", _I)]


class LaunchPlan(ctypes.Structure):
    """w4_launch_plan of include/w4a8.h."""
    _fields_ = [("path", _I), ("quantize_launches", _I), ("grid", _I), ("threads", _I), ("smem_bytes", _I),
                ("stages", _I), ("k_splits", _I), ("gemv_launches", _I)]


FORMATS = {"w4": 0, "q4_0": 1, "i8g32": 2, "q6g32": 3}
W4_PLAN_LINEAR = 1
W4_PLAN_NORM = 2
W4_PLAN_GLU = 4
PATHS = {0: "none", 1: "fused", 2: "codes_smem", 3: "codes_global", 4: "tensor_cores"}
SIGNATURES["w4_plan"] = ([_I, _I, _I, _I, _U, ctypes.POINTER(DeviceDesc), ctypes.POINTER(LaunchPlan)], _I)
SIGNATURES["w4_describe_device"] = ([ctypes.POINTER(DeviceDesc)], _I)
SIGNATURES["w4_chain_workspace_bytes"] = ([], _SZ)
SIGNATURES["w4_chain_noalloc_scratch_bytes"] = ([], _SZ)
SIGNATURES["w4a8_linear_chain_noalloc"] = ([ctypes.POINTER(LinearDesc), _I, _I, _P], _I)
SIGNATURES["w4a8_linear_chain"] = ([ctypes.POINTER(LinearDesc), _I, _I, _P, _SZ, _P], _I)
SIGNATURES["w4_workspace_bytes"] = ([_I, _I, _I], _SZ)
SIGNATURES["w4_quantize_rows_host"] = ([_P, _I, _I, _P, _P], _I)
SIGNATURES["q4_0_quantize_host"] = ([_P, _I, _I, _P], _I)
SIGNATURES["i8g32_quantize_host"] = ([_P, _I, _I, _P, _P], _I)
SIGNATURES["w4_last_device_error"] = ([ctypes.POINTER(ctypes.c_uint)], _I)
SIGNATURES["w4_hbm_read"] = ([_P, _SZ, _P, _P], _I)
SIGNATURES["w4_selftest_wait_timeout"] = ([_I, ctypes.c_uint, _P], _I)
W4_MAX_CHAIN = 128

_lib = None


class W4Error(RuntimeError):
    def __init__(self, name: str, status: int):
        super().__init__(f"{name}: {STATUS.get(status, status)}")
        self.status = status


def load(path: str = LIB_PATH):
    """Load the library (once).  Raises if it is missing: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m bit_quantized_decode_gb300.build` "
                "(needs nvcc); the decode GEMV has no CPU implementation")
        lib = ctypes.CDLL(path)
        for name, (args, res) in SIGNATURES.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
    return _lib


def _check(name: str, st: int):
    if st != W4_OK:
        raise W4Error(name, st)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("tensor must live on a CUDA device")
            if not t.is_contiguous():
                raise ValueError("tensor must be contiguous")


def _ptr_array(ts):
    arr = (ctypes.c_void_p * len(ts))(*[t.data_ptr() if t is not None else None for t in ts])
    return ctypes.cast(arr, _PP), arr


def _int_array(vals):
    arr = (ctypes.c_int * len(vals))(*vals)
    return ctypes.cast(arr, _PI), arr


# ---------------------------------------------------------------- queries
def status_str(st: int) -> str:
    return load().w4_status_str(st).decode()


def version() -> int:
    return load().w4_version()


def w4_describe_device() -> dict:
    """The current device's description (w4_device_desc) as a dict."""
    d = DeviceDesc()
    _check("w4_describe_device", load().w4_describe_device(ctypes.byref(d)))
    return {f: getattr(d, f) for f, _ in DeviceDesc._fields_}


def w4_plan(fmt: str, M: int, N: int, K: int, device: dict, linear: bool = True, norm: bool = False,
            glu: bool = False) -> dict:
    """The launch plan of a call (w4_plan): host computation only, no GPU
    needed.  device: a dict with the w4_device_desc fields."""
    d = DeviceDesc(**{f: int(device[f]) for f, _ in DeviceDesc._fields_})
    what = (W4_PLAN_LINEAR if linear else 0) | (W4_PLAN_NORM if norm else 0) | (W4_PLAN_GLU if glu else 0)
    p = LaunchPlan()
    _check("w4_plan", load().w4_plan(FORMATS[fmt], M, N, K, what, ctypes.byref(d), ctypes.byref(p)))
    out = {f: getattr(p, f) for f, _ in LaunchPlan._fields_}
    out["path"] = PATHS[out["path"]]
    return out


def set_tuning(key: str, value: int):
    """Launch tuning (see include/w4a8.h): blocks_per_sm, max_stages, grid_blocks; 0 = automatic."""
    _check("w4_set_tuning", load().w4_set_tuning(TUNE_KEYS[key], int(value)))


def get_tuning(key: str) -> int:
    return int(load().w4_get_tuning(TUNE_KEYS[key]))


def w4_repacked_bytes(N: int, K: int) -> int:
    return int(load().w4_repacked_bytes(N, K))


def q4_0_repacked_bytes(N: int, K: int) -> int:
    return int(load().q4_0_repacked_bytes(N, K))


def q6g32_repacked_bytes(N: int, K: int) -> int:
    return int(load().q6g32_repacked_bytes(N, K))


def i8g32_repacked_bytes(N: int, K: int) -> int:
    return int(load().i8g32_repacked_bytes(N, K))


# ------------------------------------------------------------- quantizers
def w4_quantize_rows(W, packed, s_w, stream=None):
    """W float32 [N][K] -> packed int32 [N][K/8] (canonical words), s_w float32 [N]."""
    _dev(W, packed, s_w)
    N, K = W.shape
    _check("w4_quantize_rows", load().w4_quantize_rows(_ptr(W), N, K, _ptr(packed), _ptr(s_w), _stream(stream)))


def q4_0_quantize(W, blocks, stream=None):
    """W float32 [N][K] -> blocks uint8 [N][K/32][18]."""
    _dev(W, blocks)
    N, K = W.shape
    _check("q4_0_quantize", load().q4_0_quantize(_ptr(W), N, K, _ptr(blocks), _stream(stream)))


def i8g32_quantize(W, q, d, stream=None):
    """W float32 [N][K] -> q int8 [N][K], d fp16 bits int16 [N][K/32]."""
    _dev(W, q, d)
    N, K = W.shape
    _check("i8g32_quantize", load().i8g32_quantize(_ptr(W), N, K, _ptr(q), _ptr(d), _stream(stream)))


# ------------------------------------------------- quantizers on the host
def _host_arr(a, dtype):
    """A C-contiguous numpy array of `dtype` (the host entry points take host memory)."""
    import numpy as np
    if not isinstance(a, np.ndarray) or a.dtype != dtype or not a.flags.c_contiguous:
        raise ValueError(f"expected a C-contiguous numpy array of {np.dtype(dtype)}")
    return ctypes.c_void_p(a.ctypes.data)


def w4_quantize_rows_host(W):
    """Host numpy float32 [N][K] -> (packed uint32 [N][K/8], s_w float32 [N]), by the library's host code."""
    import numpy as np
    N, K = W.shape
    packed = np.zeros((N, K // 8), np.uint32)
    sw = np.zeros(N, np.float32)
    _check("w4_quantize_rows_host", load().w4_quantize_rows_host(_host_arr(W, np.float32), N, K,
                                                                 _host_arr(packed, np.uint32), _host_arr(sw, np.float32)))
    return packed, sw


def q4_0_quantize_host(W):
    """Host numpy float32 [N][K] -> Q4_0 blocks uint8 [N][K/32][18], by the library's host code."""
    import numpy as np
    N, K = W.shape
    blocks = np.zeros((N, K // 32, 18), np.uint8)
    _check("q4_0_quantize_host", load().q4_0_quantize_host(_host_arr(W, np.float32), N, K,
                                                           _host_arr(blocks, np.uint8)))
    return blocks


def i8g32_quantize_host(W):
    """Host numpy float32 [N][K] -> (q int8 [N][K], d fp16 bits uint16 [N][K/32]), by the library's host code."""
    import numpy as np
    N, K = W.shape
    q = np.zeros((N, K), np.int8)
    d = np.zeros((N, K // 32), np.uint16)
    _check("i8g32_quantize_host", load().i8g32_quantize_host(_host_arr(W, np.float32), N, K, _host_arr(q, np.int8),
                                                             _host_arr(d, np.uint16)))
    return q, d


def workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().w4_workspace_bytes(M, N, K))


# ---------------------------------------------------------------- repack
def w4_repack(shards, K, out, stream=None):
    """shards: list of canonical packed tensors [rows_s][K/8]; out: uint8 buffer."""
    _dev(out, *shards)
    pp, keep = _ptr_array(shards)
    rows, keep2 = _int_array([s.shape[0] for s in shards])
    _check("w4_repack", load().w4_repack(pp, rows, len(shards), K, _ptr(out), out.numel() * out.element_size(),
                                         _stream(stream)))


def q4_0_repack(shards, K, out, stream=None):
    _dev(out, *shards)
    pp, keep = _ptr_array(shards)
    rows, keep2 = _int_array([s.shape[0] for s in shards])
    _check("q4_0_repack", load().q4_0_repack(pp, rows, len(shards), K, _ptr(out), out.numel() * out.element_size(),
                                             _stream(stream)))


def i8g32_repack(q_shards, d_shards, K, out, stream=None):
    _dev(out, *q_shards, *d_shards)
    qp, keep = _ptr_array(q_shards)
    dp, keep2 = _ptr_array(d_shards)
    rows, keep3 = _int_array([s.shape[0] for s in q_shards])
    _check("i8g32_repack", load().i8g32_repack(qp, dp, rows, len(q_shards), K, _ptr(out),
                                               out.numel() * out.element_size(), _stream(stream)))


def q6g32_repack(q_shards, d_shards, K, out, stream=None):
    """Pack I8G32 canonical shards (codes in [-32, 31]) into the 6-bit device layout."""
    _dev(out, *q_shards, *d_shards)
    qp, keep = _ptr_array(q_shards)
    dp, keep2 = _ptr_array(d_shards)
    rows, keep3 = _int_array([s.shape[0] for s in q_shards])
    _check("q6g32_repack", load().q6g32_repack(qp, dp, rows, len(q_shards), K, _ptr(out),
                                               out.numel() * out.element_size(), _stream(stream)))


def w4_concat_f32(parts, out, stream=None):
    _dev(out, *parts)
    pp, keep = _ptr_array(parts)
    lens, keep2 = _int_array([p.numel() for p in parts])
    _check("w4_concat_f32", load().w4_concat_f32(pp, lens, len(parts), _ptr(out), _stream(stream)))


# ------------------------------------------------------------- per token
def a8_quantize(x, qx, sx, stream=None):
    """x float32 [M][K] -> qx int8 [M][K], sx float32 [M]."""
    _dev(x, qx, sx)
    M, K = x.shape
    _check("a8_quantize", load().a8_quantize(_ptr(x), M, K, _ptr(qx), _ptr(sx), _stream(stream)))


def w4a8_gemv(w, s_w, bias, qx, sx, y, stream=None):
    """y[M][N] from repacked per-row INT4 weights and int8 activations."""
    _dev(w, s_w, bias, qx, sx, y)
    M, K = qx.shape
    N = y.shape[1]
    _check("w4a8_gemv", load().w4a8_gemv(_ptr(w), _ptr(s_w), _ptr(bias), _ptr(qx), _ptr(sx), M, N, K, _ptr(y),
                                         _stream(stream)))


def q4_0_gemv(w, bias, qx, sx, y, stream=None):
    _dev(w, bias, qx, sx, y)
    M, K = qx.shape
    N = y.shape[1]
    _check("q4_0_gemv", load().q4_0_gemv(_ptr(w), _ptr(bias), _ptr(qx), _ptr(sx), M, N, K, _ptr(y),
                                         _stream(stream)))


def i8g32_gemv(w, bias, qx, sx, y, stream=None):
    _dev(w, bias, qx, sx, y)
    M, K = qx.shape
    N = y.shape[1]
    _check("i8g32_gemv", load().i8g32_gemv(_ptr(w), _ptr(bias), _ptr(qx), _ptr(sx), M, N, K, _ptr(y),
                                           _stream(stream)))


def q6g32_gemv(w, bias, qx, sx, y, stream=None):
    _dev(w, bias, qx, sx, y)
    M, K = qx.shape
    N = y.shape[1]
    _check("q6g32_gemv", load().q6g32_gemv(_ptr(w), _ptr(bias), _ptr(qx), _ptr(sx), M, N, K, _ptr(y),
                                           _stream(stream)))


def w4a8_linear(w, s_w, bias, x, y, qx, sx, flags: int = 0, stream=None):
    """Quantize x and run the per-row INT4 GEMV in one launch; y[M][N]."""
    _dev(w, s_w, bias, x, y, qx, sx)
    M, K = x.shape
    N = y.shape[1]
    _check("w4a8_linear", load().w4a8_linear(_ptr(w), _ptr(s_w), _ptr(bias), _ptr(x), M, N, K, _ptr(y), _ptr(qx),
                                             _ptr(sx), flags, _stream(stream)))


def q4_0_linear(w, bias, x, y, qx, sx, flags: int = 0, stream=None):
    _dev(w, bias, x, y, qx, sx)
    M, K = x.shape
    N = y.shape[1]
    _check("q4_0_linear", load().q4_0_linear(_ptr(w), _ptr(bias), _ptr(x), M, N, K, _ptr(y), _ptr(qx), _ptr(sx),
                                             flags, _stream(stream)))


def i8g32_linear(w, bias, x, y, qx, sx, flags: int = 0, stream=None):
    _dev(w, bias, x, y, qx, sx)
    M, K = x.shape
    N = y.shape[1]
    _check("i8g32_linear", load().i8g32_linear(_ptr(w), _ptr(bias), _ptr(x), M, N, K, _ptr(y), _ptr(qx), _ptr(sx),
                                               flags, _stream(stream)))


def q6g32_linear(w, bias, x, y, qx, sx, flags: int = 0, stream=None):
    _dev(w, bias, x, y, qx, sx)
    M, K = x.shape
    N = y.shape[1]
    _check("q6g32_linear", load().q6g32_linear(_ptr(w), _ptr(bias), _ptr(x), M, N, K, _ptr(y), _ptr(qx), _ptr(sx),
                                               flags, _stream(stream)))


# ------------------------------------------------ fusions around the linear
def w4_glu_repacked_bytes(I: int, K: int) -> int:
    return int(load().w4_glu_repacked_bytes(I, K))


def q4_0_glu_repacked_bytes(I: int, K: int) -> int:
    return int(load().q4_0_glu_repacked_bytes(I, K))


def w4_repack_glu(gate, up, K, out, stream=None):
    """Canonical packed gate and up [I][K/8] -> the paired device layout."""
    _dev(gate, up, out)
    assert gate.shape == up.shape
    _check("w4_repack_glu", load().w4_repack_glu(_ptr(gate), _ptr(up), gate.shape[0], K, _ptr(out),
                                                 out.numel() * out.element_size(), _stream(stream)))


def q4_0_repack_glu(gate, up, K, out, stream=None):
    """Q4_0 blocks of gate and up [I][K/32][18] -> the paired device layout."""
    _dev(gate, up, out)
    assert gate.shape == up.shape
    _check("q4_0_repack_glu", load().q4_0_repack_glu(_ptr(gate), _ptr(up), gate.shape[0], K, _ptr(out),
                                                     out.numel() * out.element_size(), _stream(stream)))


def fusion(norm_weight=None, eps: float = 0.0, glu: int = W4_GLU_NONE, residual=None):
    """A w4_fusion descriptor.  It holds references to its tensors, so their
    memory stays allocated while the descriptor is alive."""
    _dev(norm_weight, residual)
    fz = Fusion(None if norm_weight is None else norm_weight.data_ptr(), float(eps), int(glu),
                None if residual is None else residual.data_ptr())
    fz._tensors = (norm_weight, residual)
    return fz


def _fused_args(fz):
    return None if fz is None else ctypes.byref(fz)


def w4a8_linear_fused(w, s_w, bias, x, y, qx, sx, fz=None, flags: int = 0, stream=None):
    """w4a8_linear with RMSNorm / GLU / residual fused (fz from fusion()); y[M][N]."""
    _dev(w, s_w, bias, x, y, qx, sx)
    M, K = x.shape
    N = y.shape[1]
    _check("w4a8_linear_fused", load().w4a8_linear_fused(_ptr(w), _ptr(s_w), _ptr(bias), _ptr(x), M, N, K, _ptr(y),
                                                         _ptr(qx), _ptr(sx), _fused_args(fz), flags,
                                                         _stream(stream)))


def _grouped_fused(name, w, bias, x, y, qx, sx, fz, flags, stream):
    _dev(w, bias, x, y, qx, sx)
    M, K = x.shape
    N = y.shape[1]
    _check(name, getattr(load(), name)(_ptr(w), _ptr(bias), _ptr(x), M, N, K, _ptr(y), _ptr(qx), _ptr(sx),
                                       _fused_args(fz), flags, _stream(stream)))


def q4_0_linear_fused(w, bias, x, y, qx, sx, fz=None, flags: int = 0, stream=None):
    _grouped_fused("q4_0_linear_fused", w, bias, x, y, qx, sx, fz, flags, stream)


def i8g32_linear_fused(w, bias, x, y, qx, sx, fz=None, flags: int = 0, stream=None):
    _grouped_fused("i8g32_linear_fused", w, bias, x, y, qx, sx, fz, flags, stream)


def q6g32_linear_fused(w, bias, x, y, qx, sx, fz=None, flags: int = 0, stream=None):
    _grouped_fused("q6g32_linear_fused", w, bias, x, y, qx, sx, fz, flags, stream)


def rms_a8_quantize(x, norm_weight, eps, qx, sx, flags: int = 0, stream=None):
    """RMSNorm(x) then the activation quantizer: qx int8 [M][K], sx float32 [M]."""
    _dev(x, norm_weight, qx, sx)
    M, K = x.shape
    _check("rms_a8_quantize", load().rms_a8_quantize(_ptr(x), _ptr(norm_weight), float(eps), M, K, _ptr(qx),
                                                     _ptr(sx), flags, _stream(stream)))


def w4_rmsnorm(x, norm_weight, eps, out, flags: int = 0, stream=None):
    _dev(x, norm_weight, out)
    M, K = x.shape
    _check("w4_rmsnorm", load().w4_rmsnorm(_ptr(x), _ptr(norm_weight), float(eps), M, K, _ptr(out), flags,
                                           _stream(stream)))


def w4_glu(gu, kind, out, flags: int = 0, stream=None):
    """out[M][I] = act(gu[:, :I]) * gu[:, I:] for a gate|up output gu [M][2I]."""
    _dev(gu, out)
    M, I = out.shape
    assert gu.shape == (M, 2 * I)
    _check("w4_glu", load().w4_glu(_ptr(gu), int(kind), M, I, _ptr(out), flags, _stream(stream)))


def w4_add(a, b, out, flags: int = 0, stream=None):
    _dev(a, b, out)
    assert a.numel() == b.numel() == out.numel()
    _check("w4_add", load().w4_add(_ptr(a), _ptr(b), a.numel(), _ptr(out), flags, _stream(stream)))


# ------------------------------------- weight-only paths on float activations
def w8_quantize_rows(W, q, s_w, stream=None):
    """W float32 [N][K] -> q int8 [N][K] (per-row INT8), s_w float32 [N]."""
    _dev(W, q, s_w)
    N, K = W.shape
    _check("w8_quantize_rows", load().w8_quantize_rows(_ptr(W), N, K, _ptr(q), _ptr(s_w), _stream(stream)))


def w8_repacked_bytes(N: int, K: int) -> int:
    return int(load().w8_repacked_bytes(N, K))


def w8_repack(shards, K, out, stream=None):
    """shards: int8 [rows_s][K] per-row INT8 codes; out: uint8 buffer of w8_repacked_bytes."""
    _dev(out, *shards)
    pp, keep = _ptr_array(shards)
    rows, keep2 = _int_array([s.shape[0] for s in shards])
    _check("w8_repack", load().w8_repack(pp, rows, len(shards), K, _ptr(out), out.numel() * out.element_size(),
                                         _stream(stream)))


def w4a32_gemv(w, s_w, bias, x, y, flags: int = 0, stream=None):
    """Weight-only per-row INT4 (w4_repack layout) on float x [M][K], M <= 4; y[M][N]."""
    _dev(w, s_w, bias, x, y)
    M, K = x.shape
    N = y.shape[1]
    _check("w4a32_gemv", load().w4a32_gemv(_ptr(w), _ptr(s_w), _ptr(bias), _ptr(x), M, N, K, _ptr(y), flags,
                                           _stream(stream)))


def w8a32_gemv(w, s_w, bias, x, y, flags: int = 0, stream=None):
    """Weight-only per-row INT8 (w8_repack layout) on float x [M][K], M <= 4; y[M][N]."""
    _dev(w, s_w, bias, x, y)
    M, K = x.shape
    N = y.shape[1]
    _check("w8a32_gemv", load().w8a32_gemv(_ptr(w), _ptr(s_w), _ptr(bias), _ptr(x), M, N, K, _ptr(y), flags,
                                           _stream(stream)))


# ---------------------------------------------------------------- chains
def chain_workspace_bytes() -> int:
    return int(load().w4_chain_workspace_bytes())


def make_chain_descs(items):
    """items: sequence of (w, s_w, bias, x, y, qx, sx) tensors (bias, qx, sx may be None)."""
    arr = (LinearDesc * len(items))()
    for i, (w, s_w, bias, x, y, qx, sx) in enumerate(items):
        _dev(w, s_w, bias, x, y, qx, sx)
        arr[i] = LinearDesc(w.data_ptr(), s_w.data_ptr(), None if bias is None else bias.data_ptr(), x.data_ptr(),
                            y.data_ptr(), None if qx is None else qx.data_ptr(),
                            None if sx is None else sx.data_ptr(), y.shape[1], x.shape[1])
    return arr


def w4a8_linear_chain(descs, M: int, workspace, stream=None):
    """Run a chain of per-row INT4 linears (descs from make_chain_descs) in one launch."""
    _dev(workspace)
    _check("w4a8_linear_chain", load().w4a8_linear_chain(descs, len(descs), M, _ptr(workspace),
                                                         workspace.numel() * workspace.element_size(),
                                                         _stream(stream)))


def w4a8_linear_chain_noalloc(descs, M: int, stream=None):
    """w4a8_linear_chain with the library's own fixed barrier scratch: for
    callers that cannot allocate device memory.  Calls sharing the scratch
    must not overlap on the GPU."""
    _check("w4a8_linear_chain_noalloc", load().w4a8_linear_chain_noalloc(descs, len(descs), M, _stream(stream)))


# ---------------------------------------------------------- device errors
def device_error() -> int:
    code = ctypes.c_uint(0)
    st = load().w4_device_error(ctypes.byref(code))
    if st not in (W4_OK, 5):
        raise W4Error("w4_device_error", st)
    return int(code.value)


def last_device_error() -> int:
    """w4_last_device_error: the same word as device_error()."""
    code = ctypes.c_uint(0)
    st = load().w4_last_device_error(ctypes.byref(code))
    if st not in (W4_OK, 5):
        raise W4Error("w4_last_device_error", st)
    return int(code.value)


def hbm_read(buf, sink, stream=None):
    """Stream every byte of the device tensor `buf` once (w4_hbm_read); sink:
    a device int32 [1] that receives the XOR of all 32-bit words."""
    _dev(buf, sink)
    _check("w4_hbm_read", load().w4_hbm_read(_ptr(buf), buf.numel() * buf.element_size(), _ptr(sink),
                                             _stream(stream)))


def selftest_wait_timeout(cluster: bool, timeout_us: int, stream=None):
    """A kernel whose bounded wait nothing completes: it gives up after
    timeout_us and sets the device error word to the wait-timeout code."""
    _check("w4_selftest_wait_timeout", load().w4_selftest_wait_timeout(1 if cluster else 0, int(timeout_us),
                                                                        _stream(stream)))


WAIT_TIMEOUT_CODE = 0x57414954


def clear_device_error():
    _check("w4_clear_device_error", load().w4_clear_device_error())
