"""Rounding-sensitive inputs for every kernel, bit for bit against the oracle.

With N(0,1) data an fp32 sum of a few bf16 values is usually exact, and a
1-ulp fp32 difference reaches the bf16 output only about once in 2^16
elements, so an addition that rounds wrongly, a different order or a fused
multiply-add could pass the ordinary parity tests.  Here every element is
built so that its sequence of fp32 roundings decides its bf16 result: the
first two partials put the exact sum on a bf16 tie (b + half a bf16 ulp of
b) and the others add quarter, half and three-quarter fp32 ulps that the
rank-order fp32 additions either drop or keep.  (The MoE combine's
separately rounded products are covered by its ordinary parity tests: a
fused multiply-add changes most fp32 sums, which shows in bf16 at a rate
those tests' million-element cases catch.)"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import rank_sum_residual_gb300 as farn  # noqa: E402
import synth  # noqa: E402
from parity import assert_parity, u16  # noqa: E402
from gpu_util import make_ctx, oracle_rows  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    farn.build_library()
    synth.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


@pytest.fixture(scope="module")
def O():
    return oracle.Oracle()


def bf16_bits(v: np.ndarray) -> np.ndarray:
    """Exactly representable float32 values -> bf16 patterns."""
    b = v.astype(np.float32).view(np.uint32)
    assert not np.any(b & 0xFFFF), "value not representable in bf16"
    return (b >> 16).astype(np.uint16)


def tie_partials(W, T, H, seed):
    """W partials [T,H] (bf16 patterns) whose rank-order fp32 sum lands on or
    next to a bf16 tie, decided by sub-ulp terms."""
    rng = np.random.default_rng(seed)
    e = rng.integers(-10, 11, size=(T, H))
    m = rng.integers(0, 128, size=(T, H))
    sign = np.where(rng.random((T, H)) < 0.5, -1.0, 1.0)
    base = sign * (1.0 + m / 128.0) * np.exp2(e)
    xs = [base, sign * np.exp2(e - 8)]                  # exact sum: a bf16 tie
    small = np.array([0.0, 1.0, 2.0, 3.0, 4.0, -1.0, -2.0, -3.0, -4.0])
    for _ in range(2, W):
        pick = small[rng.integers(0, len(small), size=(T, H))]
        xs.append(pick * np.exp2(e - 25))               # quarter fp32 ulps of base
    return [bf16_bits(x) for x in xs]


def _device(a, dev):
    return torch.from_numpy(a.astype(np.uint16).view(np.int16)).to(dev).view(torch.bfloat16)


def _run(O, dev, W, T, H, ctx=None, quant=None, what=""):
    xs_h = tie_partials(W, T, H, seed=T * 31 + H)
    rng = np.random.default_rng(5)
    res_h = bf16_bits((rng.integers(-64, 64, size=(T, H)) * 2.0 ** -12).astype(np.float32))
    w_h = bf16_bits(np.ones(H, np.float32))
    xs = [_device(x, dev) for x in xs_h]
    res, w = _device(res_h, dev), _device(w_h, dev)
    if quant == "fp8":
        out = farn.forward_quant(xs, res, w, 1e-6, ctx=ctx)[:3]
    elif quant == "nvfp4":
        out = farn.forward_nvfp4(xs, res, w, 1e-6, 168.0, ctx=ctx)[:3]
    else:
        out = farn.forward(xs, res, w, 1e-6, ctx=ctx)
    torch.cuda.synchronize()
    want = oracle_rows(O, xs, res, w, 1e-6)
    assert_parity([u16(t) for t in out], want, what)
    # the construction really exercises the rounding: a reversed rank order
    # changes many reduced values
    rev = O.forward([u16(x) for x in reversed(xs)], u16(res), u16(w), 1e-6)
    assert np.count_nonzero(rev[0] != want[0]) > T * H // 50


@pytest.mark.parametrize("env,W,T,H,quant", [
    ({}, 8, 2048, 4096, None),                          # stage kernel (packed adds)
    ({}, 8, 200, 4096, None),                           # row kernel
    ({}, 8, 3, 4096, None),                             # cluster kernel
    (dict(FARN_VARIANT="generic"), 6, 50, 2048, None),
    (dict(FARN_VARIANT="bulk"), 8, 600, 4096, None),
    (dict(FARN_VARIANT="stage", FARN_VPT=2), 5, 400, 8192, None),
    ({}, 8, 2048, 4096, "fp8"),                         # FP8 stage kernel (mixed adds)
    ({}, 8, 2048, 4096, "nvfp4"),                       # NVFP4 stage kernel
    ({}, 16, 100, 7168, "fp8"),
], ids=lambda v: (str(v) if not isinstance(v, dict)
                  else "-".join(f"{k[5:].lower()}{x}" for k, x in v.items()) or "auto"))
def test_rank_sum_rounding_boundaries(O, dev, env, W, T, H, quant):
    ctx = make_ctx(**env) if env else None
    try:
        _run(O, dev, W, T, H, ctx=ctx, quant=quant, what=f"ties {env} W={W} T={T} H={H} {quant}")
    finally:
        if ctx is not None:
            ctx.close()
