"""Seeded synthetic inputs for the fused rank-sum + residual + RMSNorm operator.

A module of its own: it makes input bytes and nothing else.  Both the CUDA
path (device fill through ``libfarn_synth.so``) and the CPU oracle's tests
(the numpy twin below) draw their inputs here; it contains none of the
operator's arithmetic.

Recipe (the same on device and host): a SplitMix64 counter stream per
(seed, stream_id), Box-Muller normals or uniforms evaluated in fp64, an
optional outlier multiplier, fp64 -> fp32 round-to-nearest, then bf16 by
truncating the fp32 pattern to its upper 16 bits (fp32 partials keep the
fp32 value).  ``gen.cu`` states the
constants.  The host twin uses numpy's log/cos, the device CUDA's, so the two
can differ in a rare last bit; parity never depends on that, because every
GPU parity test feeds the oracle the bytes the device generated.

Workloads follow the operator page's setting (bf16 partials of W tensor-
parallel ranks, hidden sizes of LLM layers) at the sizes of the five
benchmark shapes below.  "N(m, v)" is read as mean m and VARIANCE v.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.cu")
_LIB_PATH = os.path.join(_HERE, "libfarn_synth.so")
_lock = threading.Lock()
_lib = None

GAMMA = np.uint64(0x9E3779B97F4A7C15)
NORMAL, UNIFORM = 0, 1
STREAM_RESIDUAL, STREAM_WEIGHT = 1000, 1001


# --------------------------------------------------------------------- recipes
@dataclass(frozen=True)
class Dist:
    kind: int            # NORMAL or UNIFORM
    p0: float            # mean, or lower bound
    p1: float            # variance, or upper bound
    outlier_p: float = 0.0
    outlier_scale: float = 1.0

    def describe(self) -> str:
        if self.kind == NORMAL:
            s = f"N(mean={self.p0}, var={self.p1:g}, sigma={self.p1 ** 0.5:.4f})"
        else:
            s = f"U({self.p0}, {self.p1})"
        if self.outlier_p > 0:
            s += f" with {self.outlier_p:g} of entries x{self.outlier_scale:g}"
        return s


@dataclass(frozen=True)
class Problem:
    """One operator call: W partials [T,H], residual [T,H], weight [H]."""
    name: str
    W: int
    T: int
    H: int
    eps: float
    seed: int
    x: Dist
    residual: Dist = Dist(NORMAL, 0.0, 1.0)
    weight: Dist = Dist(NORMAL, 1.0, 0.1)
    partial_dtype: str = "bf16"      # or "f32"
    fp8_out: bool = False            # also write norm_out as E4M3 + row scales
    nvfp4_out: bool = False          # also write norm_out as NVFP4 + block scales
    tensor_scale: float = 1.0        # the NVFP4 tensor scale
    norm_out: bool = True            # write the bf16 norm_out
    kind: str = "rank_sum"           # or "moe_combine" (W = experts per token)

    @property
    def partial_bytes(self) -> int:
        return 4 if self.partial_dtype == "f32" else 2

    def read_bytes(self) -> int:
        """W*T*H*pb partials + T*H*2 residual + H*2 weight (pb = 2 for bf16
        partials, 4 for fp32); for the MoE combine the W gathered expert
        rows of each token (bf16) plus its W int32 indices and fp32 gates."""
        if self.kind == "moe_combine":
            return (self.W * self.T * self.H * 2 + self.T * self.W * 8
                    + self.T * self.H * 2 + self.H * 2)
        return self.W * self.T * self.H * self.partial_bytes + self.T * self.H * 2 + self.H * 2

    def write_bytes(self) -> int:
        """reduced and residual_out (T*H*2 each), norm_out (T*H*2) if
        written, with the FP8 output T*H bytes plus T*4 of scales, with the
        NVFP4 output T*H/2 bytes of codes plus T*H/16 of block scales."""
        n = self.T * self.H
        return 2 * n * 2 + (n * 2 if self.norm_out else 0) + \
            ((n + 4 * self.T) if self.fp8_out else 0) + \
            ((n // 2 + n // 16) if self.nvfp4_out else 0)

    def algorithmic_bytes(self) -> int:
        return self.read_bytes() + self.write_bytes()

    def _replace(self, **kw) -> "Problem":
        d = dict(self.__dict__)
        d.update(kw)
        return Problem(**d)

    def with_seed(self, seed: int) -> "Problem":
        return self._replace(seed=seed)

    def with_T(self, T: int) -> "Problem":
        return self._replace(name=f"{self.name.split('@')[0]}@T{T}", T=T)


N01 = Dist(NORMAL, 0.0, 1.0)
DECODE_TS = (1, 2, 4, 8, 16, 32, 64, 128)


def _decode(T: int) -> Problem:
    return Problem(f"decode@T{T}", 8, T, 4096, 1e-5, T, N01)


WORKLOADS = {
    "c1": [Problem("c1", 4, 16, 2048, 1e-6, 0, N01)],
    "decode": [_decode(T) for T in DECODE_TS],
    "prefill": [Problem("prefill", 8, 8192, 8192, 1e-6, 0,
                        Dist(NORMAL, 0.0, 0.5, 0.001, 50.0),
                        N01, Dist(UNIFORM, 0.5, 1.5))],
    "nonpow2": [Problem("nonpow2", 4, 32768, 5120, 1e-6, 0, N01)],
    "wide": [Problem("wide", 16, 4096, 7168, 1e-6, 0, Dist(NORMAL, 0.0, 1.0 / 16))],
    # residual add + RMSNorm alone (one partial: no rank sum), prefill-sized
    "rmsnorm": [Problem("rmsnorm", 1, 8192, 8192, 1e-6, 0, N01)],
    # MoE combine of 8 experts per token at a 7168 hidden size, 4096 tokens
    "moe_combine": [Problem("moe_combine", 8, 4096, 7168, 1e-6, 0, N01, kind="moe_combine")],
    # the prefill shape writing norm_out as E4M3 + row scales instead of bf16
    "prefill_fp8": [Problem("prefill_fp8", 8, 8192, 8192, 1e-6, 0,
                            Dist(NORMAL, 0.0, 0.5, 0.001, 50.0),
                            N01, Dist(UNIFORM, 0.5, 1.5), fp8_out=True, norm_out=False)],
    # the prefill shape writing norm_out as NVFP4 (E2M1 codes, E4M3 scales
    # per 16 elements) instead of bf16; the tensor scale maps an amax of 16
    # to the top of the E4M3 x E2M1 range (448 * 6 / 16)
    "prefill_nvfp4": [Problem("prefill_nvfp4", 8, 8192, 8192, 1e-6, 0,
                              Dist(NORMAL, 0.0, 0.5, 0.001, 50.0),
                              N01, Dist(UNIFORM, 0.5, 1.5), nvfp4_out=True, norm_out=False,
                              tensor_scale=168.0)],
    # the prefill shape with fp32 partials (e.g. straight from GEMM epilogues)
    "prefill_f32": [Problem("prefill_f32", 8, 8192, 8192, 1e-6, 0,
                            Dist(NORMAL, 0.0, 0.5, 0.001, 50.0),
                            N01, Dist(UNIFORM, 0.5, 1.5), "f32")],
}


def workload(name: str) -> list[Problem]:
    if name not in WORKLOADS:
        raise KeyError(f"unknown workload {name!r}; have {sorted(WORKLOADS)}")
    return WORKLOADS[name]


# ------------------------------------------------------------------ host twin
def _mix64(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * np.uint64(0xBF58476D1CE4E5B9)
    z = z ^ (z >> np.uint64(27))
    z = z * np.uint64(0x94D049BB133111EB)
    z = z ^ (z >> np.uint64(31))
    return z


def _base(seed: int, stream_id: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([stream_id], np.uint64) + GAMMA
        return _mix64(np.array([seed], np.uint64) ^ _mix64(s))[0]


def _unit(z: np.ndarray) -> np.ndarray:
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * 2.0 ** -53


def host_bf16(n: int, seed: int, stream_id: int, dist: Dist) -> np.ndarray:
    """The recipe evaluated with numpy; returns n bf16 patterns (uint16)."""
    with np.errstate(over="ignore"):
        base = _base(seed, stream_id)
        j = np.arange(n, dtype=np.uint64) * np.uint64(3)
        u1 = _unit(_mix64(base + (j + np.uint64(1)) * GAMMA))
        u2 = _unit(_mix64(base + (j + np.uint64(2)) * GAMMA))
        if dist.kind == NORMAL:
            v = dist.p0 + np.sqrt(dist.p1) * (np.sqrt(-2.0 * np.log(u1))
                                              * np.cos(2.0 * np.pi * u2))
        else:
            v = dist.p0 + (dist.p1 - dist.p0) * u1
        if dist.outlier_p > 0:
            u3 = _unit(_mix64(base + (j + np.uint64(3)) * GAMMA))
            v = np.where(u3 < dist.outlier_p, v * dist.outlier_scale, v)
    f = v.astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def host_f32(n: int, seed: int, stream_id: int, dist: Dist) -> np.ndarray:
    """The recipe kept in fp32 (fp32 partials)."""
    with np.errstate(over="ignore"):
        base = _base(seed, stream_id)
        j = np.arange(n, dtype=np.uint64) * np.uint64(3)
        u1 = _unit(_mix64(base + (j + np.uint64(1)) * GAMMA))
        u2 = _unit(_mix64(base + (j + np.uint64(2)) * GAMMA))
        if dist.kind == NORMAL:
            v = dist.p0 + np.sqrt(dist.p1) * (np.sqrt(-2.0 * np.log(u1))
                                              * np.cos(2.0 * np.pi * u2))
        else:
            v = dist.p0 + (dist.p1 - dist.p0) * u1
        if dist.outlier_p > 0:
            u3 = _unit(_mix64(base + (j + np.uint64(3)) * GAMMA))
            v = np.where(u3 < dist.outlier_p, v * dist.outlier_scale, v)
    return v.astype(np.float32)


def moe_routing(p: Problem):
    """index int32 [T,K]: a seeded permutation of the T*K expert-output
    rows (each used once); gates float32 [T,K]: a softmax of N(0,1) logits
    per token."""
    rng = np.random.default_rng(p.seed + 12345)
    index = rng.permutation(p.T * p.W).astype(np.int32).reshape(p.T, p.W)
    logits = rng.normal(size=(p.T, p.W))
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    gates = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    return index, gates


def host_inputs(p: Problem):
    """(partials list of [T,H], residual [T,H], weight [H]); partials are
    uint16 bf16 patterns or float32, residual and weight uint16.  For the
    MoE combine the first item is (expert_out [T*K,H], index, gates)."""
    n = p.T * p.H
    if p.kind == "moe_combine":
        ex = host_bf16(n * p.W, p.seed, 0, p.x).reshape(p.T * p.W, p.H)
        index, gates = moe_routing(p)
        res = host_bf16(n, p.seed, STREAM_RESIDUAL, p.residual).reshape(p.T, p.H)
        w = host_bf16(p.H, p.seed, STREAM_WEIGHT, p.weight)
        return (ex, index, gates), res, w
    if p.partial_dtype == "f32":
        xs = [host_f32(n, p.seed, r, p.x).reshape(p.T, p.H) for r in range(p.W)]
    else:
        xs = [host_bf16(n, p.seed, r, p.x).reshape(p.T, p.H) for r in range(p.W)]
    res = host_bf16(n, p.seed, STREAM_RESIDUAL, p.residual).reshape(p.T, p.H)
    w = host_bf16(p.H, p.seed, STREAM_WEIGHT, p.weight)
    return xs, res, w


# ---------------------------------------------------------------- device fill
def build(force: bool = False) -> str:
    """Compile libfarn_synth.so for sm_103a next to its source."""
    with _lock:
        if (force or not os.path.exists(_LIB_PATH)
                or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.run(
                ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                 "-lineinfo", "-Xcompiler", "-fPIC", "-shared", "-o", tmp, _SRC],
                check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is not built; call synth.build()")
        lib = ctypes.CDLL(_LIB_PATH)
        lib.farn_synth_fill_bf16.argtypes = [
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64,
            ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_double,
            ctypes.c_double, ctypes.c_void_p]
        lib.farn_synth_fill_bf16.restype = ctypes.c_int
        lib.farn_synth_fill_f32.argtypes = lib.farn_synth_fill_bf16.argtypes
        lib.farn_synth_fill_f32.restype = ctypes.c_int
        _lib = lib
    return _lib


def fill_device(t, seed: int, stream_id: int, dist: Dist, stream=None) -> None:
    """Fill a contiguous torch bf16 CUDA tensor in place with the recipe."""
    import torch
    if t.dtype not in (torch.bfloat16, torch.float32) or not t.is_cuda \
            or not t.is_contiguous():
        raise TypeError("fill_device wants a contiguous bf16 or fp32 CUDA tensor")
    s = stream if stream is not None else torch.cuda.current_stream(t.device)
    fn = _load().farn_synth_fill_bf16 if t.dtype == torch.bfloat16 \
        else _load().farn_synth_fill_f32
    rc = fn(t.data_ptr(), t.numel(), seed, stream_id, dist.kind, dist.p0, dist.p1,
            dist.outlier_p, dist.outlier_scale, s.cuda_stream)
    if rc != 0:
        raise RuntimeError(f"farn_synth_fill_bf16 failed (rc={rc})")


def device_inputs(p: Problem, device="cuda", seed: int | None = None):
    """Allocate and fill (partials, residual, weight) on the device."""
    import torch
    sd = p.seed if seed is None else seed
    if p.kind == "moe_combine":
        ex = torch.empty((p.T * p.W, p.H), dtype=torch.bfloat16, device=device)
        fill_device(ex, sd, 0, p.x)
        index, gates = moe_routing(p.with_seed(sd))
        res = torch.empty((p.T, p.H), dtype=torch.bfloat16, device=device)
        fill_device(res, sd, STREAM_RESIDUAL, p.residual)
        w = torch.empty((p.H,), dtype=torch.bfloat16, device=device)
        fill_device(w, sd, STREAM_WEIGHT, p.weight)
        return ((ex, torch.from_numpy(index).to(device), torch.from_numpy(gates).to(device)),
                res, w)
    xs = []
    xdt = torch.float32 if p.partial_dtype == "f32" else torch.bfloat16
    for r in range(p.W):
        t = torch.empty((p.T, p.H), dtype=xdt, device=device)
        fill_device(t, sd, r, p.x)
        xs.append(t)
    res = torch.empty((p.T, p.H), dtype=torch.bfloat16, device=device)
    fill_device(res, sd, STREAM_RESIDUAL, p.residual)
    w = torch.empty((p.H,), dtype=torch.bfloat16, device=device)
    fill_device(w, sd, STREAM_WEIGHT, p.weight)
    return xs, res, w
