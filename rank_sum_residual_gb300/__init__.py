"""Fused rank-sum + residual add + RMSNorm for one GB300 (sm_103a).

    reduced      = sum over ranks r of x[r]            (bf16 [T,H] each)
    residual_out = reduced + residual
    norm_out     = RMSNorm(residual_out, weight, eps)

The operator of FlagTree pull request "[TLERaw] Add NVSHMEM allreduce
RMSNorm tutorial" (Summary; Implementation sections 2-3), computed by the
hand-written CUDA kernels of ``libfarn.so``.  This module is the Python
binding of that library's C ABI (``include/farn.h``): the ``farn_*``
functions have the C names and arguments and only marshal them through
ctypes; ``forward`` is the same call for torch tensors.  Every arithmetic
step runs in the CUDA kernels.  There is no CPU fallback: if the library
is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB_PATH, build_library

__all__ = [
    "FARN_MAX_W", "FarnError", "Context", "build_library", "library_path",
    "farn_create", "farn_destroy", "farn_forward", "farn_check_args",
    "farn_plan", "farn_status_string", "farn_device_status", "farn_forward_noalloc",
    "farn_forward_typed", "farn_plan_typed", "farn_forward_quant", "forward_quant",
    "farn_moe_combine", "moe_combine",
    "FARN_BF16", "FARN_F32",
    "forward", "VARIANTS",
]

FARN_MAX_W = 32
FARN_OK = 0
FARN_ERR_INVALID_ARG = -1
FARN_ERR_UNSUPPORTED = -2
FARN_ERR_ALIAS = -3
FARN_ERR_CUDA = -4
FARN_ERR_NOMEM = -5
VARIANTS = {0: "row", 1: "cluster", 2: "generic", 3: "bulk", 4: "stage", 5: "combine"}
FARN_BF16, FARN_F32 = 0, 1

_lib = None


def library_path() -> str:
    return LIB_PATH


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built (the operator has no CPU fallback); "
                "run rank_sum_residual_gb300.build_library() on a machine with nvcc")
        lib = ctypes.CDLL(LIB_PATH)
        vp, cvp = ctypes.c_void_p, ctypes.c_void_p
        pvp = ctypes.POINTER(ctypes.c_void_p)
        i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
        lib.farn_create.argtypes = [ctypes.POINTER(ctypes.c_void_p), i32]
        lib.farn_create.restype = i32
        lib.farn_destroy.argtypes = [vp]
        lib.farn_destroy.restype = i32
        lib.farn_forward.argtypes = [vp, pvp, i32, cvp, cvp, f32, i64, i64,
                                     vp, vp, vp, vp]
        lib.farn_forward.restype = i32
        lib.farn_forward_typed.argtypes = [vp, pvp, i32, i32, cvp, cvp, f32, i64, i64,
                                           vp, vp, vp, vp]
        lib.farn_forward_typed.restype = i32
        lib.farn_forward_quant.argtypes = [vp, pvp, i32, i32, cvp, cvp, f32, i64, i64,
                                           vp, vp, vp, vp, vp, vp]
        lib.farn_forward_quant.restype = i32
        lib.farn_forward_nvfp4.argtypes = [vp, pvp, i32, i32, cvp, cvp, f32, i64, i64, f32,
                                           vp, vp, vp, vp, vp, vp]
        lib.farn_forward_nvfp4.restype = i32
        lib.farn_moe_combine.argtypes = [vp, cvp, i64, cvp, cvp, i32, cvp, cvp, f32, i64, i64,
                                         vp, vp, vp, vp]
        lib.farn_moe_combine.restype = i32
        lib.farn_check_args.argtypes = [pvp, i32, cvp, cvp, f32, i64, i64,
                                        cvp, cvp, cvp]
        lib.farn_check_args.restype = i32
        lib.farn_plan.argtypes = [vp, i32, i64, i64, pvp, cvp, cvp, cvp, cvp,
                                  cvp, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                  ctypes.POINTER(i32)]
        lib.farn_plan.restype = i32
        lib.farn_plan_typed.argtypes = [vp, i32, i32, i32, i64, i64, pvp, cvp, cvp, cvp,
                                        cvp, cvp, ctypes.POINTER(i32), ctypes.POINTER(i32),
                                        ctypes.POINTER(i32)]
        lib.farn_plan_typed.restype = i32
        lib.farn_plan_moe_combine.argtypes = [vp, i32, i64, i64, cvp, cvp, cvp, cvp, cvp, cvp,
                                              ctypes.POINTER(i32), ctypes.POINTER(i32)]
        lib.farn_plan_moe_combine.restype = i32
        lib.farn_forward_noalloc.argtypes = [i32, pvp, i32, cvp, cvp, f32, i64, i64,
                                             vp, vp, vp, vp, ctypes.POINTER(i32)]
        lib.farn_forward_noalloc.restype = i32
        lib.farn_device_status.argtypes = [vp, ctypes.POINTER(i32)]
        lib.farn_device_status.restype = i32
        lib.farn_status_string.argtypes = [i32]
        lib.farn_status_string.restype = ctypes.c_char_p
        _lib = lib
    return _lib


class FarnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {farn_status_string(status)} (status {status})")


def farn_status_string(status: int) -> str:
    return _load().farn_status_string(int(status)).decode()


def _ptr_array(ptrs):
    return (ctypes.c_void_p * max(1, len(ptrs)))(*[ctypes.c_void_p(int(p)) for p in ptrs])


def farn_create(device: int = 0) -> int:
    """C ``farn_create``: returns the opaque context handle (an int)."""
    h = ctypes.c_void_p()
    st = _load().farn_create(ctypes.byref(h), int(device))
    if st != FARN_OK:
        raise FarnError(st, "farn_create")
    return h.value


def farn_destroy(ctx: int) -> None:
    _load().farn_destroy(ctypes.c_void_p(ctx) if ctx else None)


def farn_forward(ctx, partials, W, residual, weight, eps, T, H,
                 reduced_out, residual_out, norm_out, stream=0) -> int:
    """C ``farn_forward`` on raw device addresses (ints); returns the status."""
    return _load().farn_forward(
        ctypes.c_void_p(ctx) if ctx else None, _ptr_array(partials), int(W),
        ctypes.c_void_p(int(residual)), ctypes.c_void_p(int(weight)), float(eps),
        int(T), int(H), ctypes.c_void_p(int(reduced_out)),
        ctypes.c_void_p(int(residual_out)), ctypes.c_void_p(int(norm_out)),
        ctypes.c_void_p(int(stream)))


def farn_forward_typed(ctx, partials, partial_dtype, W, residual, weight, eps, T, H,
                       reduced_out, residual_out, norm_out, stream=0) -> int:
    """C ``farn_forward_typed``: partials of dtype FARN_BF16 or FARN_F32."""
    return _load().farn_forward_typed(
        ctypes.c_void_p(ctx) if ctx else None, _ptr_array(partials), int(partial_dtype),
        int(W), ctypes.c_void_p(int(residual)), ctypes.c_void_p(int(weight)), float(eps),
        int(T), int(H), ctypes.c_void_p(int(reduced_out)),
        ctypes.c_void_p(int(residual_out)), ctypes.c_void_p(int(norm_out)),
        ctypes.c_void_p(int(stream)))


def farn_forward_quant(ctx, partials, partial_dtype, W, residual, weight, eps, T, H,
                       reduced_out, residual_out, norm_out, norm_q, row_scale,
                       stream=0) -> int:
    """C ``farn_forward_quant``: also writes norm_out as E4M3 bytes plus a
    per-row fp32 scale (norm_out may be 0 to skip it)."""
    return _load().farn_forward_quant(
        ctypes.c_void_p(ctx) if ctx else None, _ptr_array(partials), int(partial_dtype),
        int(W), ctypes.c_void_p(int(residual)), ctypes.c_void_p(int(weight)), float(eps),
        int(T), int(H), ctypes.c_void_p(int(reduced_out)),
        ctypes.c_void_p(int(residual_out)),
        ctypes.c_void_p(int(norm_out)) if norm_out else None,
        ctypes.c_void_p(int(norm_q)), ctypes.c_void_p(int(row_scale)),
        ctypes.c_void_p(int(stream)))


def farn_forward_nvfp4(ctx, partials, partial_dtype, W, residual, weight, eps, T, H,
                       tensor_scale, reduced_out, residual_out, norm_out, norm_fp4,
                       block_scale, stream=0) -> int:
    """C ``farn_forward_nvfp4``: also writes norm_out as NVFP4 (two E2M1
    codes per byte, one E4M3 scale per 16 elements, under tensor_scale);
    norm_out may be 0 to skip it."""
    v = lambda a: ctypes.c_void_p(int(a)) if a else None  # noqa: E731
    return _load().farn_forward_nvfp4(
        ctypes.c_void_p(ctx) if ctx else None, _ptr_array(partials), int(partial_dtype),
        int(W), v(residual), v(weight), float(eps), int(T), int(H), float(tensor_scale),
        v(reduced_out), v(residual_out), v(norm_out), v(norm_fp4), v(block_scale),
        ctypes.c_void_p(int(stream)))


def farn_moe_combine(ctx, expert_out, n_slots, index, gates, K, residual, weight, eps, T, H,
                     reduced_out, residual_out, norm_out, stream=0) -> int:
    """C ``farn_moe_combine`` on raw device addresses (ints)."""
    v = lambda a: ctypes.c_void_p(int(a)) if a else None  # noqa: E731
    return _load().farn_moe_combine(
        ctypes.c_void_p(ctx) if ctx else None, v(expert_out), int(n_slots), v(index), v(gates),
        int(K), v(residual), v(weight), float(eps), int(T), int(H), v(reduced_out),
        v(residual_out), v(norm_out), ctypes.c_void_p(int(stream)))


def farn_forward_noalloc(device, partials, W, residual, weight, eps, T, H,
                         reduced_out, residual_out, norm_out, stream=0,
                         want_status=False):
    """C ``farn_forward_noalloc`` on raw device addresses (ints), for callers
    that cannot allocate device memory: no context, nothing allocated.
    Returns (status, device status word or None); asking for the word makes
    the call wait for the kernel."""
    word = ctypes.c_int(-1)
    st = _load().farn_forward_noalloc(
        int(device), _ptr_array(partials), int(W), ctypes.c_void_p(int(residual)),
        ctypes.c_void_p(int(weight)), float(eps), int(T), int(H),
        ctypes.c_void_p(int(reduced_out)), ctypes.c_void_p(int(residual_out)),
        ctypes.c_void_p(int(norm_out)), ctypes.c_void_p(int(stream)),
        ctypes.byref(word) if want_status else None)
    return st, (word.value if want_status else None)


def farn_device_status(ctx: int) -> int:
    """C ``farn_device_status``: read and clear the device status word."""
    v = ctypes.c_int()
    st = _load().farn_device_status(ctypes.c_void_p(ctx), ctypes.byref(v))
    if st != FARN_OK:
        raise FarnError(st, "farn_device_status")
    return v.value


def farn_check_args(partials, W, residual, weight, eps, T, H, reduced_out,
                    residual_out, norm_out) -> int:
    """C ``farn_check_args``: host-only checks, addresses are only compared."""
    arr = None if partials is None else _ptr_array(partials)
    v = lambda a: ctypes.c_void_p(int(a)) if a else None  # noqa: E731
    return _load().farn_check_args(arr, int(W), v(residual), v(weight),
                                   float(eps), int(T), int(H), v(reduced_out),
                                   v(residual_out), v(norm_out))


def farn_plan(ctx, W, T, H, partials, residual, weight, reduced_out,
              residual_out, norm_out):
    """C ``farn_plan``: (variant name, CTAs per row, threads per CTA)."""
    variant, cs, thr = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    v = lambda a: ctypes.c_void_p(int(a)) if a else None  # noqa: E731
    st = _load().farn_plan(ctypes.c_void_p(ctx), int(W), int(T), int(H),
                           _ptr_array(partials), v(residual), v(weight),
                           v(reduced_out), v(residual_out), v(norm_out),
                           ctypes.byref(variant), ctypes.byref(cs),
                           ctypes.byref(thr))
    if st != FARN_OK:
        raise FarnError(st, "farn_plan")
    return VARIANTS[variant.value], cs.value, thr.value


FARN_PLAN_FP8_OUT = 1
FARN_PLAN_NVFP4_OUT = 2


def farn_plan_typed(ctx, partial_dtype, W, T, H, partials, residual, weight, reduced_out,
                    residual_out, norm_out, flags=0):
    """C ``farn_plan_typed``: (variant name, CTAs per row, threads per CTA)."""
    variant, cs, thr = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    v = lambda a: ctypes.c_void_p(int(a)) if a else None  # noqa: E731
    st = _load().farn_plan_typed(ctypes.c_void_p(ctx), int(partial_dtype), int(flags),
                                 int(W), int(T),
                                 int(H), _ptr_array(partials), v(residual), v(weight),
                                 v(reduced_out), v(residual_out), v(norm_out),
                                 ctypes.byref(variant), ctypes.byref(cs), ctypes.byref(thr))
    if st != FARN_OK:
        raise FarnError(st, "farn_plan_typed")
    return VARIANTS[variant.value], cs.value, thr.value


def farn_plan_moe_combine(ctx, K, T, H, expert_out, residual, weight, reduced_out,
                          residual_out, norm_out):
    """C ``farn_plan_moe_combine``: (variant name, threads per CTA)."""
    variant, thr = ctypes.c_int(), ctypes.c_int()
    v = lambda a: ctypes.c_void_p(int(a)) if a else None  # noqa: E731
    st = _load().farn_plan_moe_combine(ctypes.c_void_p(ctx), int(K), int(T), int(H),
                                       v(expert_out), v(residual), v(weight), v(reduced_out),
                                       v(residual_out), v(norm_out), ctypes.byref(variant),
                                       ctypes.byref(thr))
    if st != FARN_OK:
        raise FarnError(st, "farn_plan_moe_combine")
    return VARIANTS[variant.value], thr.value


class Context:
    """Owns one ``farn_ctx`` for a device (``farn_create``/``farn_destroy``)."""

    def __init__(self, device: int = 0):
        self.device = int(device)
        self.handle = farn_create(self.device)

    def close(self):
        if self.handle:
            farn_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


_default_ctx: dict[int, Context] = {}


def _context_for(device_index: int) -> Context:
    c = _default_ctx.get(device_index)
    if c is None:
        c = _default_ctx[device_index] = Context(device_index)
    return c


def _check_tensor(t, name, shape, device, dtypes=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    dtypes = dtypes or (torch.bfloat16,)
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must be {' or '.join(str(d) for d in dtypes)}, got {t.dtype}")
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


# ------------------------------------------------------------ torch level
class PreparedCall:
    """One operator call whose tensors were checked and whose C-ABI
    arguments were marshalled once.  Calling it launches the kernel on the
    stream given at preparation (asynchronously) and returns the outputs; a
    caller that reuses its buffers (a serving loop, a benchmark) pays only
    the C call each time.  The tensors must stay alive, in place, while the
    object is used."""

    __slots__ = ("_fn", "_args", "_name", "_keep", "outputs")

    def __init__(self, fn, args, name, outputs, keep):
        self._fn, self._args, self._name = fn, args, name
        self.outputs, self._keep = outputs, keep

    def __call__(self):
        st = self._fn(*self._args)
        if st != FARN_OK:
            raise FarnError(st, self._name)
        return self.outputs


def _vp(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _partials_checked(partials, residual, weight):
    import torch
    partials = list(partials)
    if not partials:
        raise ValueError("partials must hold at least one tensor")
    if residual.dim() != 2:
        raise ValueError("residual must be [T, H]")
    T, H = residual.shape
    dev = residual.device
    pdt = partials[0].dtype
    if pdt not in (torch.bfloat16, torch.float32):
        raise TypeError(f"partials must be bfloat16 or float32, got {pdt}")
    for r, x in enumerate(partials):
        _check_tensor(x, f"partials[{r}]", (T, H), dev, (pdt,))
    _check_tensor(residual, "residual", (T, H), dev)
    _check_tensor(weight, "weight", (H,), dev)
    return partials, T, H, dev, (FARN_F32 if pdt == torch.float32 else FARN_BF16)


def _common_args(ctx, partials, dtype, residual, weight, eps, T, H):
    return (ctypes.c_void_p(ctx.handle), _ptr_array([x.data_ptr() for x in partials]),
            ctypes.c_int(dtype), ctypes.c_int(len(partials)), _vp(residual), _vp(weight),
            ctypes.c_float(eps), ctypes.c_int64(T), ctypes.c_int64(H))


def _ctx_stream(ctx, stream, dev):
    import torch
    c = ctx if ctx is not None else _context_for(dev.index)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    return c, ctypes.c_void_p(int(s.cuda_stream))


def prepare_forward(partials, residual, weight, eps: float, out=None, ctx=None, stream=None):
    """``forward`` checked and marshalled once (see ``PreparedCall``)."""
    import torch
    partials, T, H, dev, dtype = _partials_checked(partials, residual, weight)
    if out is None:
        out = tuple(torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(3))
    for name, t in zip(("reduced", "residual_out", "norm_out"), out):
        _check_tensor(t, name, (T, H), dev)
    c, s = _ctx_stream(ctx, stream, dev)
    args = _common_args(c, partials, dtype, residual, weight, eps, T, H) + \
        (_vp(out[0]), _vp(out[1]), _vp(out[2]), s)
    return PreparedCall(_load().farn_forward_typed, args, "farn_forward", tuple(out),
                        (partials, residual, weight, c))


def forward(partials, residual, weight, eps: float, out=None, ctx=None,
            stream=None):
    """The fused operator on torch CUDA tensors.

    partials: sequence of W tensors [T,H], all bf16 or all fp32 (fp32 partials
    are summed as fp32, see farn_forward_typed); residual [T,H] and weight
    [H] bf16; outputs bf16.
    out: optional (reduced, residual_out, norm_out) tensors to write
    (residual_out may be ``residual`` itself).  Runs asynchronously on
    ``stream`` (default: torch's current stream) and returns the outputs.
    """
    return prepare_forward(partials, residual, weight, eps, out, ctx, stream)()


def _check_quant_out(out, T, H, dev, q_shape, q_dtype, s_shape, s_dtype):
    import torch
    if len(out) != 5:
        raise ValueError("out must be (reduced, residual_out, norm_out or None, codes, scales)")
    for name, t in zip(("reduced", "residual_out"), out[:2]):
        _check_tensor(t, name, (T, H), dev)
    if out[2] is not None:
        _check_tensor(out[2], "norm_out", (T, H), dev)
    _check_tensor(out[3], "codes", q_shape, dev, (q_dtype,))
    _check_tensor(out[4], "scales", s_shape, dev, (s_dtype,))


def prepare_forward_quant(partials, residual, weight, eps: float, write_norm: bool = True,
                          out=None, ctx=None, stream=None):
    """``forward_quant`` checked and marshalled once.  out: optional
    (reduced, residual_out, norm_out or None, norm_q, row_scale)."""
    import torch
    partials, T, H, dev, dtype = _partials_checked(partials, residual, weight)
    if out is None:
        out = (torch.empty((T, H), dtype=torch.bfloat16, device=dev),
               torch.empty((T, H), dtype=torch.bfloat16, device=dev),
               torch.empty((T, H), dtype=torch.bfloat16, device=dev) if write_norm else None,
               torch.empty((T, H), dtype=torch.uint8, device=dev),
               torch.empty((T,), dtype=torch.float32, device=dev))
    _check_quant_out(out, T, H, dev, (T, H), torch.uint8, (T,), torch.float32)
    c, s = _ctx_stream(ctx, stream, dev)
    args = _common_args(c, partials, dtype, residual, weight, eps, T, H) + \
        tuple(_vp(t) for t in out) + (s,)
    return PreparedCall(_load().farn_forward_quant, args, "farn_forward_quant", tuple(out),
                        (partials, residual, weight, c))


def forward_quant(partials, residual, weight, eps: float, write_norm: bool = True,
                  ctx=None, stream=None):
    """``forward`` plus the FP8 (E4M3) copy of norm_out and its per-row
    scales.  Returns (reduced, residual_out, norm_out or None, norm_q as a
    uint8 tensor of E4M3 patterns, row_scale float32 [T])."""
    return prepare_forward_quant(partials, residual, weight, eps, write_norm,
                                 ctx=ctx, stream=stream)()


def prepare_forward_nvfp4(partials, residual, weight, eps: float, tensor_scale: float,
                          write_norm: bool = True, out=None, ctx=None, stream=None):
    """``forward_nvfp4`` checked and marshalled once.  out: optional
    (reduced, residual_out, norm_out or None, norm_fp4, block_scale)."""
    import torch
    partials, T, H, dev, dtype = _partials_checked(partials, residual, weight)
    if H % 16:
        raise ValueError(f"NVFP4 output needs H % 16 == 0, got H = {H}")
    if out is None:
        out = (torch.empty((T, H), dtype=torch.bfloat16, device=dev),
               torch.empty((T, H), dtype=torch.bfloat16, device=dev),
               torch.empty((T, H), dtype=torch.bfloat16, device=dev) if write_norm else None,
               torch.empty((T, H // 2), dtype=torch.uint8, device=dev),
               torch.empty((T, H // 16), dtype=torch.uint8, device=dev))
    _check_quant_out(out, T, H, dev, (T, H // 2), torch.uint8, (T, H // 16), torch.uint8)
    c, s = _ctx_stream(ctx, stream, dev)
    args = _common_args(c, partials, dtype, residual, weight, eps, T, H) + \
        (ctypes.c_float(tensor_scale),) + tuple(_vp(t) for t in out) + (s,)
    return PreparedCall(_load().farn_forward_nvfp4, args, "farn_forward_nvfp4", tuple(out),
                        (partials, residual, weight, c))


def forward_nvfp4(partials, residual, weight, eps: float, tensor_scale: float,
                  write_norm: bool = True, ctx=None, stream=None):
    """``forward`` plus the NVFP4 copy of norm_out.  Returns (reduced,
    residual_out, norm_out or None, norm_fp4 uint8 [T,H/2] (two E2M1 codes
    per byte, the even element in the low nibble), block_scale uint8
    [T,H/16] (E4M3 patterns)).  H must be a multiple of 16."""
    return prepare_forward_nvfp4(partials, residual, weight, eps, tensor_scale, write_norm,
                                 ctx=ctx, stream=stream)()


def prepare_moe_combine(expert_out, index, gates, residual, weight, eps: float, out=None,
                        ctx=None, stream=None):
    """``moe_combine`` checked and marshalled once."""
    import torch
    T, H = residual.shape
    dev = residual.device
    S = expert_out.shape[0]
    _check_tensor(expert_out, "expert_out", (S, H), dev)
    K = index.shape[1] if index.dim() == 2 else -1
    _check_tensor(index, "index", (T, K), dev, (torch.int32,))
    _check_tensor(gates, "gates", (T, K), dev, (torch.float32,))
    _check_tensor(residual, "residual", (T, H), dev)
    _check_tensor(weight, "weight", (H,), dev)
    if out is None:
        out = tuple(torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(3))
    for name, t in zip(("reduced", "residual_out", "norm_out"), out):
        _check_tensor(t, name, (T, H), dev)
    c, s = _ctx_stream(ctx, stream, dev)
    args = (ctypes.c_void_p(c.handle), _vp(expert_out), ctypes.c_int64(S), _vp(index),
            _vp(gates), ctypes.c_int(K), _vp(residual), _vp(weight), ctypes.c_float(eps),
            ctypes.c_int64(T), ctypes.c_int64(H), _vp(out[0]), _vp(out[1]), _vp(out[2]), s)
    return PreparedCall(_load().farn_moe_combine, args, "farn_moe_combine", tuple(out),
                        (expert_out, index, gates, residual, weight, c))


def moe_combine(expert_out, index, gates, residual, weight, eps: float, out=None, ctx=None,
                stream=None):
    """MoE combine + residual + RMSNorm on torch CUDA tensors: expert_out bf16
    [S,H], index int32 [T,K], gates fp32 [T,K], residual bf16 [T,H], weight
    bf16 [H].  Returns (reduced, residual_out, norm_out)."""
    return prepare_moe_combine(expert_out, index, gates, residual, weight, eps, out, ctx,
                               stream)()
