"""The C ABI on the host (no GPU needed): the library loads, exports every
function include/farn.h declares, and its argument checks return the
documented status without touching the pointers."""
import ctypes
import os
import re

import pytest

import rank_sum_residual_gb300 as farn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "farn.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    farn.build_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(farn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("farn_create", "farn_forward", "farn_destroy", "farn_check_args",
              "farn_status_string", "farn_plan"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(farn.library_path())
    for name in declared_functions():
        assert hasattr(lib, name), f"libfarn.so does not export {name}"


def test_status_strings():
    assert farn.farn_status_string(0) == "ok"
    for st in (-1, -2, -3, -4, -5):
        assert farn.farn_status_string(st) not in ("", "unknown status")
    assert farn.farn_status_string(12345) == "unknown status"


# Fake, never-dereferenced addresses: 1 MiB apart, 16-byte aligned.
MB = 1 << 20
X = [0x10000000 + i * MB for i in range(40)]
RES, WT, RED, RO, NRM = 0x20000000, 0x21000000, 0x22000000, 0x23000000, 0x24000000


def check(partials=None, W=None, residual=RES, weight=WT, eps=1e-6, T=4, H=64,
          red=RED, ro=RO, nrm=NRM):
    partials = X[:4] if partials is None else partials
    W = len(partials) if W is None else W
    return farn.farn_check_args(partials, W, residual, weight, eps, T, H, red, ro, nrm)


def test_valid_arguments_pass():
    assert check() == 0
    assert check(T=0) == 0
    assert check(partials=X[:32]) == 0
    assert check(partials=X[:1]) == 0
    # residual_out may be exactly the residual buffer (in-place update)
    assert check(ro=RES) == 0
    # partials may repeat (read-only inputs may overlap)
    assert check(partials=[X[0], X[0], X[1]]) == 0


@pytest.mark.parametrize("kw", [
    dict(W=0, partials=X[:1]), dict(partials=X[:33]), dict(T=-1), dict(H=0),
    dict(H=-8), dict(eps=-1e-6), dict(eps=float("nan")), dict(eps=float("inf")),
    dict(residual=0), dict(weight=0), dict(red=0), dict(ro=0), dict(nrm=0),
    dict(partials=[X[0], 0, X[1]]), dict(H=1 << 62, T=4),
])
def test_invalid_arguments(kw):
    assert check(**kw) == farn.FARN_ERR_INVALID_ARG


def test_zero_rows_accept_null_tensors():
    # empty tensors have null data pointers; with T == 0 nothing is touched
    assert farn.farn_check_args([0, 0], 2, 0, 0, 1e-6, 0, 64, 0, 0, 0) == 0


def test_null_partials_array():
    assert farn.farn_check_args(None, 2, RES, WT, 1e-6, 4, 64, RED, RO, NRM) \
        == farn.FARN_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [
    dict(red=RO),                          # two outputs the same
    dict(red=RO + 2 * 4 * 64 - 2),         # outputs overlap by one element
    dict(nrm=X[2] + 16),                   # output inside a partial
    dict(red=WT),                          # output over the weight
    dict(nrm=RES),                         # only residual_out may alias residual
    dict(ro=RES + 16),                     # residual_out partially over residual
])
def test_aliasing_rejected(kw):
    assert check(**kw) == farn.FARN_ERR_ALIAS


def test_adjacent_buffers_are_not_aliases():
    nb = 4 * 64 * 2
    assert check(red=RED, ro=RED + nb, nrm=RED + 2 * nb) == 0


def test_forward_rejects_null_context_before_any_cuda_call():
    st = farn.farn_forward(0, X[:4], 4, RES, WT, 1e-6, 4, 64, RED, RO, NRM, 0)
    assert st == farn.FARN_ERR_INVALID_ARG
    st = farn.farn_forward_typed(0, X[:4], farn.FARN_F32, 4, RES, WT, 1e-6, 4, 64,
                                 RED, RO, NRM, 0)
    assert st == farn.FARN_ERR_INVALID_ARG
    st = farn.farn_forward_quant(0, X[:4], farn.FARN_BF16, 4, RES, WT, 1e-6, 4, 64,
                                 RED, RO, NRM, 0x25000000, 0x26000000, 0)
    assert st == farn.FARN_ERR_INVALID_ARG


def test_create_without_a_gpu_reports_cuda_error():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the GPU tests cover farn_create")
    with pytest.raises(farn.FarnError) as e:
        farn.farn_create(0)
    assert e.value.status in (farn.FARN_ERR_CUDA, farn.FARN_ERR_INVALID_ARG)
    with pytest.raises(farn.FarnError) as e:
        farn.farn_create(-1)
    assert e.value.status == farn.FARN_ERR_INVALID_ARG


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    import importlib
    import rank_sum_residual_gb300 as pkg
    monkeypatch.setattr(pkg, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(pkg, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        pkg.farn_status_string(0)
    importlib.reload(pkg)


def test_synth_twin_recipe_statistics():
    import numpy as np
    import synth
    p = synth.workload("wide")[0]
    xs, res, w = synth.host_inputs(p.with_T(64))
    x = (xs[0].astype(np.uint32) << 16).view(np.float32)
    assert abs(x.var() - 1.0 / 16) < 0.005          # N(0, 1/16): variance
    r = (res.astype(np.uint32) << 16).view(np.float32)
    assert abs(r.mean()) < 0.02 and abs(r.var() - 1.0) < 0.05
    # different streams differ, same stream repeats
    assert not np.array_equal(xs[0], xs[1])
    assert np.array_equal(synth.host_bf16(1000, 0, 3, p.x), synth.host_bf16(1000, 0, 3, p.x))


def test_synth_splitmix64_published_vectors():
    """The generator's mixing function is SplitMix64's: with the state
    advanced by the golden gamma from 0 it gives the published first outputs
    0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F."""
    import numpy as np
    import synth
    with np.errstate(over="ignore"):
        got = [int(synth._mix64(np.uint64(k) * synth.GAMMA)) for k in (1, 2, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_synth_moe_routing():
    """Every expert-output row is gathered exactly once, gates are a softmax
    (positive, summing to 1 per token), and the routing is seeded."""
    import numpy as np
    import synth
    p = synth.workload("moe_combine")[0].with_T(300)
    index, gates = synth.moe_routing(p)
    assert index.shape == (300, p.W) and index.dtype == np.int32
    assert np.array_equal(np.sort(index.ravel()), np.arange(300 * p.W))
    assert (gates > 0).all() and np.allclose(gates.sum(axis=1), 1.0, atol=1e-6)
    i2, g2 = synth.moe_routing(p)
    assert np.array_equal(index, i2) and np.array_equal(gates, g2)
    i3, _ = synth.moe_routing(p.with_seed(p.seed + 1))
    assert not np.array_equal(index, i3)


def test_noalloc_host_side_checks():
    """farn_forward_noalloc's argument checks and the empty call need no
    GPU: T = 0 returns FARN_OK with a zero status word and launches nothing
    (null data pointers allowed, as for empty tensors); bad arguments and a
    negative device are refused before any CUDA call."""
    a = 1 << 40
    st, word = farn.farn_forward_noalloc(0, [0, 0], 2, 0, 0, 1e-6, 0, 4096, 0, 0, 0,
                                         want_status=True)
    assert st == farn.FARN_OK and word == 0
    st, _ = farn.farn_forward_noalloc(0, [a], 0, a, a, 1e-6, 4, 4096, a, a, a)
    assert st == farn.FARN_ERR_INVALID_ARG                      # W = 0
    st, _ = farn.farn_forward_noalloc(0, [a] * 33, 33, a, a, 1e-6, 4, 4096, a, a, a)
    assert st == farn.FARN_ERR_INVALID_ARG                      # W > FARN_MAX_W
    st, _ = farn.farn_forward_noalloc(0, [a], 1, a, a, float("nan"), 4, 4096, a, a, a)
    assert st == farn.FARN_ERR_INVALID_ARG                      # eps not finite
    st, _ = farn.farn_forward_noalloc(-1, [a], 1, a, a, 1e-6, 4, 4096, a, a, a)
    assert st == farn.FARN_ERR_INVALID_ARG                      # no such device
    g = 1 << 32
    st, _ = farn.farn_forward_noalloc(0, [a], 1, a + g, a + 2 * g, 1e-6, 4, 4096,
                                      a, a + 3 * g, a + 4 * g)
    assert st == farn.FARN_ERR_ALIAS                            # reduced_out over x[0]
