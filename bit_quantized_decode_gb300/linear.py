"""Load-time preparation of one decode linear and its per-token call.

`QuantLinear.from_float` quantizes float weight shards on the GPU with the
library's kernels, fuses the shards (q/k/v, gate/up) into one repacked
matrix, and keeps it resident; `QuantLinear.__call__` runs the fused
quantize + GEMV launch, optionally with RMSNorm in front, the gated MLP
activation (gate/up weights paired per tile, `glu_pairs=True`) or the
residual add behind it.  Buffers are torch tensors (device memory only).
"""
from __future__ import annotations

import torch

from . import _lib

# "w4a32" and "w8a32" are the weight-only paths on float activations (per-row
# INT4 unpacked to float, per-row INT8); their calls ignore qx and sx.
FORMATS = ("w4", "q4_0", "i8g32", "q6g32", "w4a32", "w8a32")


class QuantLinear:
    def __init__(self, fmt: str, N: int, K: int, w: torch.Tensor, s_w=None, bias=None, canonical=None,
                 glu_pairs: bool = False):
        if fmt not in FORMATS:
            raise ValueError(fmt)
        self.fmt, self.N, self.K = fmt, N, K   # N: outputs per token (a paired gate/up linear: I)
        self.glu_pairs = glu_pairs
        self.w = w                  # repacked device layout, uint8
        self.s_w = s_w              # float32 [N] (w4 only)
        self.bias = bias            # float32 [N] or None
        self.canonical = canonical  # per-shard canonical tensors, if kept

    # ------------------------------------------------------------- building
    @classmethod
    def from_float(cls, fmt: str, shards, biases=None, keep_canonical: bool = False,
                   glu_pairs: bool = False) -> "QuantLinear":
        """shards: float32 CUDA tensors [rows_s][K] concatenated by rows; biases: matching [rows_s] or None.
        glu_pairs: shards are [gate, up] of a gated MLP (W4 or Q4_0), repacked paired per tile for the
        GLU epilogue; the linear then has I = rows outputs and must be called with glu=..."""
        shards = [s.contiguous() for s in shards]
        if glu_pairs and (fmt not in ("w4", "q4_0") or len(shards) != 2 or shards[0].shape != shards[1].shape):
            raise ValueError("glu_pairs needs W4 or Q4_0 gate and up shards of equal shape")
        K = shards[0].shape[1]
        dev = shards[0].device
        N = sum(s.shape[0] for s in shards)
        canon, scales = [], []
        for W in shards:
            n = W.shape[0]
            if fmt == "w8a32":
                q = torch.empty((n, K), dtype=torch.int8, device=dev)
                sw = torch.empty(n, dtype=torch.float32, device=dev)
                _lib.w8_quantize_rows(W, q, sw)
                canon.append(q)
                scales.append(sw)
            elif fmt in ("w4", "w4a32"):
                p = torch.empty((n, K // 8), dtype=torch.int32, device=dev)
                sw = torch.empty(n, dtype=torch.float32, device=dev)
                _lib.w4_quantize_rows(W, p, sw)
                canon.append(p)
                scales.append(sw)
            elif fmt == "q4_0":
                b = torch.empty((n, K // 32, 18), dtype=torch.uint8, device=dev)
                _lib.q4_0_quantize(W, b)
                canon.append(b)
            else:   # i8g32 and q6g32 share the canonical codes (6-bit values in int8)
                q = torch.empty((n, K), dtype=torch.int8, device=dev)
                d = torch.empty((n, K // 32), dtype=torch.int16, device=dev)
                _lib.i8g32_quantize(W, q, d)
                canon.append((q, d))
        w, s_w = cls._repack(fmt, canon, scales, N, K, dev, glu_pairs)
        bias = None
        if biases is not None:
            bias = torch.empty(N, dtype=torch.float32, device=dev)
            _lib.w4_concat_f32([b.contiguous() for b in biases], bias)
        return cls(fmt, N // 2 if glu_pairs else N, K, w, s_w, bias, canon if keep_canonical else None, glu_pairs)

    @classmethod
    def from_canonical(cls, fmt: str, canon, K: int, scales=None, biases=None) -> "QuantLinear":
        """Repack already-quantized canonical shards (device tensors)."""
        grouped = fmt in ("i8g32", "q6g32")
        dev = (canon[0][0] if grouped else canon[0]).device
        N = sum((c[0] if grouped else c).shape[0] for c in canon)
        w, s_w = cls._repack(fmt, canon, scales or [], N, K, dev)
        bias = None
        if biases is not None:
            bias = torch.empty(N, dtype=torch.float32, device=dev)
            _lib.w4_concat_f32([b.contiguous() for b in biases], bias)
        return cls(fmt, N, K, w, s_w, bias, canon)

    @staticmethod
    def _repack(fmt, canon, scales, N, K, dev, glu_pairs=False):
        s_w = None
        if glu_pairs:
            I = N // 2
            if fmt == "w4":
                w = torch.empty(_lib.w4_glu_repacked_bytes(I, K), dtype=torch.uint8, device=dev)
                _lib.w4_repack_glu(canon[0], canon[1], K, w)
                s_w = torch.empty(N, dtype=torch.float32, device=dev)
                _lib.w4_concat_f32(scales, s_w)
            else:
                w = torch.empty(_lib.q4_0_glu_repacked_bytes(I, K), dtype=torch.uint8, device=dev)
                _lib.q4_0_repack_glu(canon[0], canon[1], K, w)
            return w, s_w
        if fmt in ("w4", "w4a32"):
            w = torch.empty(_lib.w4_repacked_bytes(N, K), dtype=torch.uint8, device=dev)
            _lib.w4_repack(canon, K, w)
            s_w = torch.empty(N, dtype=torch.float32, device=dev)
            _lib.w4_concat_f32(scales, s_w)
        elif fmt == "w8a32":
            w = torch.empty(_lib.w8_repacked_bytes(N, K), dtype=torch.uint8, device=dev)
            _lib.w8_repack(canon, K, w)
            s_w = torch.empty(N, dtype=torch.float32, device=dev)
            _lib.w4_concat_f32(scales, s_w)
        elif fmt == "q4_0":
            w = torch.empty(_lib.q4_0_repacked_bytes(N, K), dtype=torch.uint8, device=dev)
            _lib.q4_0_repack(canon, K, w)
        elif fmt == "i8g32":
            w = torch.empty(_lib.i8g32_repacked_bytes(N, K), dtype=torch.uint8, device=dev)
            _lib.i8g32_repack([c[0] for c in canon], [c[1] for c in canon], K, w)
        else:
            w = torch.empty(_lib.q6g32_repacked_bytes(N, K), dtype=torch.uint8, device=dev)
            _lib.q6g32_repack([c[0] for c in canon], [c[1] for c in canon], K, w)
        return w, s_w

    # ------------------------------------------------------------ per token
    def buffers(self, M: int):
        dev = self.w.device
        return (torch.empty((M, self.N), dtype=torch.float32, device=dev),
                torch.empty((M, self.K), dtype=torch.int8, device=dev),
                torch.empty(M, dtype=torch.float32, device=dev))

    def __call__(self, x, y=None, qx=None, sx=None, flags: int = 0, stream=None, norm=None, eps: float = 1e-6,
                 glu: int = _lib.W4_GLU_NONE, residual=None):
        """Quantize x [M][K] and compute y [M][N] (one fused launch when it fits).
        norm: RMSNorm weight [K] applied to x first (with eps); glu: W4_GLU_SILU or W4_GLU_GELU_TANH
        (paired gate/up weights only); residual [M][N]: added to y last (may be y itself)."""
        M = x.shape[0]
        if y is None or qx is None or sx is None:
            y2, q2, s2 = self.buffers(M)
            y = y if y is not None else y2
            qx = qx if qx is not None else q2
            sx = sx if sx is not None else s2
        if self.glu_pairs != (glu != _lib.W4_GLU_NONE):
            raise ValueError("glu is taken exactly by linears built with glu_pairs=True")
        if self.fmt in ("w4a32", "w8a32"):
            if norm is not None or glu != _lib.W4_GLU_NONE or residual is not None:
                raise ValueError("the weight-only paths take no fused operators")
            fn = _lib.w4a32_gemv if self.fmt == "w4a32" else _lib.w8a32_gemv
            fn(self.w, self.s_w, self.bias, x, y, flags, stream)
            return y
        if norm is not None or glu != _lib.W4_GLU_NONE or residual is not None:
            fz = _lib.fusion(norm, eps, glu, residual)
            if self.fmt == "w4":
                _lib.w4a8_linear_fused(self.w, self.s_w, self.bias, x, y, qx, sx, fz, flags, stream)
            else:
                getattr(_lib, f"{self.fmt}_linear_fused")(self.w, self.bias, x, y, qx, sx, fz, flags, stream)
            return y
        if self.fmt == "w4":
            _lib.w4a8_linear(self.w, self.s_w, self.bias, x, y, qx, sx, flags, stream)
        elif self.fmt == "q4_0":
            _lib.q4_0_linear(self.w, self.bias, x, y, qx, sx, flags, stream)
        elif self.fmt == "i8g32":
            _lib.i8g32_linear(self.w, self.bias, x, y, qx, sx, flags, stream)
        else:
            _lib.q6g32_linear(self.w, self.bias, x, y, qx, sx, flags, stream)
        return y

    def gemv(self, qx, sx, y, stream=None):
        """GEMV on already-quantized activations."""
        if self.fmt == "w4":
            _lib.w4a8_gemv(self.w, self.s_w, self.bias, qx, sx, y, stream)
        elif self.fmt == "q4_0":
            _lib.q4_0_gemv(self.w, self.bias, qx, sx, y, stream)
        elif self.fmt == "i8g32":
            _lib.i8g32_gemv(self.w, self.bias, qx, sx, y, stream)
        else:
            _lib.q6g32_gemv(self.w, self.bias, qx, sx, y, stream)
        return y

    @property
    def weight_bytes(self) -> int:
        """Bytes the GEMV streams: repacked weights (+ group scales) and per-row scales."""
        return self.w.numel() + (self.s_w.numel() * 4 if self.s_w is not None else 0)


class LinearChain:
    """A fixed sequence of per-row INT4 linears launched as one chain
    (w4a8_linear_chain).  Linear i+1 may read (part of) linear i's output:
    the chain orders every input read after the previous linear completes.

    items: sequence of (QuantLinear, x, y, qx, sx) with x [M][K] and y [M][N]."""

    def __init__(self, items, M: int):
        if not items:
            raise ValueError("empty chain")
        if len(items) > _lib.W4_MAX_CHAIN:
            raise ValueError(f"at most {_lib.W4_MAX_CHAIN} linears per chain")
        dev = items[0][0].w.device
        self.M = M
        self.items = list(items)
        self.descs = _lib.make_chain_descs([(ql.w, ql.s_w, ql.bias, x, y, qx, sx) for ql, x, y, qx, sx in items])
        self.workspace = torch.zeros(_lib.chain_workspace_bytes(), dtype=torch.uint8, device=dev)

    def __call__(self, stream=None):
        _lib.w4a8_linear_chain(self.descs, self.M, self.workspace, stream)
