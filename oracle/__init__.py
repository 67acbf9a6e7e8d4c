"""CPU oracle for the fused rank-sum + residual add + RMSNorm operator.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg call this package; the product path (the CUDA
library ``libfarn.so`` and ``rank_sum_residual_gb300``) never imports it.

The arithmetic lives in ``oracle.c`` (plain single-threaded C, fp32 with
contraction off); this module only compiles it with gcc and marshals numpy
arrays of bf16 bit patterns (``uint16``) into it.

Method: FlagTree pull request "[TLERaw] Add NVSHMEM allreduce RMSNorm
tutorial", Summary (the three-line contract) and Implementation section 3
(residual + RMSNorm epilogue with FP32 accumulation).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
           "-fPIC", "-shared"]
_lock = threading.Lock()
_lib = None


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``src`` into the shared library ``out`` with gcc."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source if it is missing or stale."""
    with _lock:
        if (force or not os.path.exists(_LIB_PATH)
                or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
            compile_oracle()
    return _LIB_PATH


def _declare(lib):
    u16p = ctypes.POINTER(ctypes.c_uint16)
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_f32_bits_to_bf16.argtypes = [ctypes.c_uint32]
    lib.oracle_f32_bits_to_bf16.restype = ctypes.c_uint16
    lib.oracle_rank_sum.argtypes = [ctypes.POINTER(u16p), ctypes.c_int,
                                    ctypes.c_int64, u16p]
    lib.oracle_rank_sum.restype = None
    lib.oracle_residual_add.argtypes = [u16p, u16p, ctypes.c_int64, u16p]
    lib.oracle_residual_add.restype = None
    lib.oracle_rmsnorm_row.argtypes = [u16p, u16p, ctypes.c_float,
                                       ctypes.c_int64, u16p]
    lib.oracle_rmsnorm_row.restype = ctypes.c_float
    lib.oracle_forward.argtypes = [ctypes.POINTER(u16p), ctypes.c_int, u16p,
                                   u16p, ctypes.c_float, ctypes.c_int64,
                                   ctypes.c_int64, u16p, u16p, u16p]
    lib.oracle_forward.restype = ctypes.c_int
    f32p = ctypes.POINTER(ctypes.c_float)
    lib.oracle_rank_sum_f32.argtypes = [ctypes.POINTER(f32p), ctypes.c_int,
                                        ctypes.c_int64, u16p]
    lib.oracle_rank_sum_f32.restype = None
    lib.oracle_forward_f32.argtypes = [ctypes.POINTER(f32p), ctypes.c_int, u16p,
                                       u16p, ctypes.c_float, ctypes.c_int64,
                                       ctypes.c_int64, u16p, u16p, u16p]
    lib.oracle_forward_f32.restype = ctypes.c_int
    u8p = ctypes.POINTER(ctypes.c_uint8)
    lib.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_e4m3_sat.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_e4m3_sat.restype = ctypes.c_uint8
    lib.oracle_quant_e4m3_row.argtypes = [u16p, ctypes.c_int64, u8p]
    lib.oracle_quant_e4m3_row.restype = ctypes.c_float
    lib.oracle_e2m1_to_f32.argtypes = [ctypes.c_uint8]
    lib.oracle_e2m1_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_e2m1_sat.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_e2m1_sat.restype = ctypes.c_uint8
    lib.oracle_quant_nvfp4_row.argtypes = [u16p, ctypes.c_int64, ctypes.c_float, u8p, u8p]
    lib.oracle_quant_nvfp4_row.restype = None
    lib.oracle_moe_combine.argtypes = [u16p, ctypes.c_int64, ctypes.POINTER(ctypes.c_int32),
                                       ctypes.POINTER(ctypes.c_float), ctypes.c_int, u16p,
                                       u16p, ctypes.c_float, ctypes.c_int64, ctypes.c_int64,
                                       u16p, u16p, u16p]
    lib.oracle_moe_combine.restype = ctypes.c_int
    lib.oracle_moe_combine_acc.argtypes = [u16p, ctypes.c_int64, ctypes.POINTER(ctypes.c_int32),
                                           ctypes.POINTER(ctypes.c_float), ctypes.c_int,
                                           ctypes.c_int64, ctypes.c_int64]
    lib.oracle_moe_combine_acc.restype = ctypes.c_float
    return lib


def load_library(path: str):
    """Load an oracle shared library (the real one, or a test build)."""
    return _declare(ctypes.CDLL(path))


def lib():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns as uint16, got {a.dtype}")
    return a


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def _pf(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


class Oracle:
    """numpy front end over one loaded oracle library."""

    def __init__(self, library=None):
        self.lib = library if library is not None else lib()

    def bf16_to_f32(self, b: int) -> float:
        return float(self.lib.oracle_bf16_to_f32(int(b)))

    def f32_to_bf16(self, f: float) -> int:
        return int(self.lib.oracle_f32_to_bf16(float(np.float32(f))))

    def f32_bits_to_bf16(self, u: int) -> int:
        return int(self.lib.oracle_f32_bits_to_bf16(int(u) & 0xFFFFFFFF))

    def rank_sum(self, xs) -> np.ndarray:
        if np.asarray(xs[0]).dtype == np.float32:
            xs = [np.ascontiguousarray(x, dtype=np.float32) for x in xs]
            out = np.empty(xs[0].shape, np.uint16)
            arr = (ctypes.POINTER(ctypes.c_float) * len(xs))(*[_pf(x) for x in xs])
            self.lib.oracle_rank_sum_f32(arr, len(xs), xs[0].size, _p(out))
            return out
        xs = [_u16(x) for x in xs]
        n = xs[0].size
        out = np.empty(xs[0].shape, np.uint16)
        arr = (ctypes.POINTER(ctypes.c_uint16) * len(xs))(*[_p(x) for x in xs])
        self.lib.oracle_rank_sum(arr, len(xs), n, _p(out))
        return out

    def residual_add(self, reduced, residual) -> np.ndarray:
        reduced, residual = _u16(reduced), _u16(residual)
        out = np.empty(reduced.shape, np.uint16)
        self.lib.oracle_residual_add(_p(reduced), _p(residual), reduced.size,
                                     _p(out))
        return out

    def rmsnorm_row(self, ro, weight, eps: float):
        ro, weight = _u16(ro), _u16(weight)
        out = np.empty(ro.shape, np.uint16)
        rstd = self.lib.oracle_rmsnorm_row(_p(ro), _p(weight), eps, ro.size,
                                           _p(out))
        return out, float(rstd)

    def forward(self, xs, residual, weight, eps: float):
        """All three outputs for W partials [T,H], residual [T,H], weight [H].

        Partials are bf16 patterns (uint16) or fp32 (float32) arrays."""
        f32 = np.asarray(xs[0]).dtype == np.float32
        xs = [np.ascontiguousarray(x, dtype=np.float32) for x in xs] if f32 \
            else [_u16(x) for x in xs]
        residual, weight = _u16(residual), _u16(weight)
        if residual.ndim != 2:
            raise ValueError("residual must be [T, H]")
        T, H = residual.shape
        for x in xs:
            if x.shape != (T, H):
                raise ValueError("every partial must be [T, H] like residual")
        if weight.shape != (H,):
            raise ValueError("weight must be [H]")
        reduced = np.empty((T, H), np.uint16)
        ro = np.empty((T, H), np.uint16)
        norm = np.empty((T, H), np.uint16)
        if f32:
            arr = (ctypes.POINTER(ctypes.c_float) * len(xs))(*[_pf(x) for x in xs])
            rc = self.lib.oracle_forward_f32(arr, len(xs), _p(residual), _p(weight),
                                             eps, T, H, _p(reduced), _p(ro), _p(norm))
        else:
            arr = (ctypes.POINTER(ctypes.c_uint16) * len(xs))(*[_p(x) for x in xs])
            rc = self.lib.oracle_forward(arr, len(xs), _p(residual), _p(weight),
                                         eps, T, H, _p(reduced), _p(ro), _p(norm))
        if rc != 0:
            raise ValueError(f"oracle_forward rejected its arguments (rc={rc})")
        return reduced, ro, norm


def _Oracle_quant(self, norm):
    """E4M3 quantisation of bf16 norm_out rows [T,H]: (q uint8 [T,H],
    scale float32 [T])."""
    norm = _u16(norm)
    if norm.ndim == 1:
        norm = norm[None, :]
    T, H = norm.shape
    q = np.empty((T, H), np.uint8)
    scale = np.empty(T, np.float32)
    for t in range(T):
        row = np.ascontiguousarray(norm[t])
        scale[t] = self.lib.oracle_quant_e4m3_row(
            _p(row), H, q[t].ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)))
    return q, scale


def _Oracle_e4m3(self, f: float) -> int:
    return int(self.lib.oracle_f32_to_e4m3_sat(float(np.float32(f))))


def _Oracle_e4m3_to_f32(self, b: int) -> float:
    return float(self.lib.oracle_e4m3_to_f32(int(b)))


def _Oracle_quant_nvfp4(self, norm, g: float):
    """NVFP4 quantisation of bf16 norm_out rows [T,H] (H % 16 == 0) under
    the tensor scale g: (q uint8 [T,H/2], two E2M1 codes per byte, even
    element in the low nibble; s uint8 [T,H/16], E4M3 block scales)."""
    norm = _u16(norm)
    if norm.ndim == 1:
        norm = norm[None, :]
    T, H = norm.shape
    if H % 16:
        raise ValueError("NVFP4 needs H % 16 == 0")
    q = np.empty((T, H // 2), np.uint8)
    s = np.empty((T, H // 16), np.uint8)
    u8 = ctypes.POINTER(ctypes.c_uint8)
    for t in range(T):
        row = np.ascontiguousarray(norm[t])
        self.lib.oracle_quant_nvfp4_row(_p(row), H, float(np.float32(g)),
                                        q[t].ctypes.data_as(u8), s[t].ctypes.data_as(u8))
    return q, s


def _Oracle_e2m1(self, f: float) -> int:
    return int(self.lib.oracle_f32_to_e2m1_sat(float(np.float32(f))))


def _Oracle_e2m1_to_f32(self, c: int) -> float:
    return float(self.lib.oracle_e2m1_to_f32(int(c)))


def _Oracle_moe_combine(self, expert_out, index, gates, residual, weight, eps: float):
    """MoE combine + residual + RMSNorm: expert_out uint16 [S,H], index
    int32 [T,K], gates float32 [T,K], residual uint16 [T,H], weight [H]."""
    expert_out = _u16(expert_out)
    index = np.ascontiguousarray(index, dtype=np.int32)
    gates = np.ascontiguousarray(gates, dtype=np.float32)
    residual, weight = _u16(residual), _u16(weight)
    T, H = residual.shape
    S = expert_out.shape[0] if expert_out.size else 0
    K = index.shape[1]
    outs = [np.empty((T, H), np.uint16) for _ in range(3)]
    rc = self.lib.oracle_moe_combine(
        _p(expert_out), S, index.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
        _pf(gates), K, _p(residual), _p(weight), eps, T, H, *[_p(o) for o in outs])
    if rc != 0:
        raise ValueError(f"oracle_moe_combine rejected its arguments (rc={rc})")
    return tuple(outs)


def _Oracle_moe_combine_acc(self, expert_out, index_row, gates_row, h: int) -> float:
    """The fp32 accumulator of one element before its bf16 rounding."""
    expert_out = _u16(expert_out)
    index_row = np.ascontiguousarray(index_row, dtype=np.int32)
    gates_row = np.ascontiguousarray(gates_row, dtype=np.float32)
    S, H = expert_out.shape
    return float(self.lib.oracle_moe_combine_acc(
        _p(expert_out), S, index_row.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
        _pf(gates_row), index_row.size, H, h))


Oracle.moe_combine = _Oracle_moe_combine
Oracle.moe_combine_acc = _Oracle_moe_combine_acc
Oracle.quant_e4m3 = _Oracle_quant
Oracle.f32_to_e4m3 = _Oracle_e4m3
Oracle.e4m3_to_f32 = _Oracle_e4m3_to_f32
Oracle.quant_nvfp4 = _Oracle_quant_nvfp4
Oracle.f32_to_e2m1 = _Oracle_e2m1
Oracle.e2m1_to_f32 = _Oracle_e2m1_to_f32


def forward(xs, residual, weight, eps: float):
    """Module-level shorthand for ``Oracle().forward``."""
    return Oracle().forward(xs, residual, weight, eps)
