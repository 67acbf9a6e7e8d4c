"""farn_forward_noalloc, the entry point for callers that cannot allocate
device memory (code inside another framework's plugin or allocator
interface, where every device allocation must go through that framework).

It is called through the C ABI and checked against the ordinary entry point
farn_forward on the same inputs, on two calls in a row (the second call
finds the shared status word as the first one left it), and against the
oracle: reduced and residual_out bit for bit, norm_out within one bf16 ulp.
The row-length limit it documents (H <= 16384, any W <= 32) is tested on
both sides.  This file is collected last so that a run stopping at the
first failure has run everything else; it also passes on its own in a
fresh process.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import rank_sum_residual_gb300 as farn  # noqa: E402
import synth  # noqa: E402
from gpu_util import oracle_rows  # noqa: E402
from parity import assert_parity, sample_rows, u16  # noqa: E402

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


def _noalloc(dev, xs, res, w, eps, outs, stream, want_status=True, device=None):
    T, H = res.shape
    return farn.farn_forward_noalloc(
        dev.index if device is None else device, [x.data_ptr() for x in xs], len(xs),
        res.data_ptr(), w.data_ptr(), eps, T, H, outs[0].data_ptr(), outs[1].data_ptr(),
        outs[2].data_ptr(), stream.cuda_stream, want_status=want_status)


def _check_against_oracle(O, xs, res, w, eps, outs, what, n_rows=None):
    T = res.shape[0]
    rows = None if n_rows is None else sample_rows(T, n_rows, seed=T)
    got = [u16(t) if rows is None else u16(t[torch.as_tensor(rows, device=t.device)])
           for t in outs]
    assert_parity(got, oracle_rows(O, xs, res, w, eps, rows), what)


@pytest.mark.parametrize("name,T", [("decode", 300), ("prefill", 257), ("wide", 160)])
def test_noalloc_matches_farn_forward_twice(O, dev, name, T):
    p = synth.workload(name)[0].with_T(T)
    xs, res, w = synth.device_inputs(p, dev)
    stream = torch.cuda.current_stream(dev)
    ref = farn.forward(xs, res, w, p.eps)          # existing entry point
    torch.cuda.synchronize(dev)
    want = [u16(t) for t in ref]
    for call in range(2):
        outs = [torch.full_like(res, float("nan")) for _ in range(3)]
        st, word = _noalloc(dev, xs, res, w, p.eps, outs, stream)
        assert st == farn.FARN_OK, farn.farn_status_string(st)
        assert word == 0, f"call {call}: status word {word}"
        torch.cuda.synchronize(dev)
        got = [u16(t) for t in outs]
        assert_parity(got, want, f"no-alloc call {call} vs farn_forward ({name}, T={T})")
        assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1])
        _check_against_oracle(O, xs, res, w, p.eps, outs,
                              f"no-alloc call {call} vs oracle ({name}, T={T})")


@pytest.mark.parametrize("W,H", [(32, 16384), (4, 16384), (32, 8192), (1, 16376)])
def test_noalloc_longest_rows_accepted(O, dev, W, H):
    """At the documented limit (H = 16384) and just below it, with up to
    FARN_MAX_W partials: accepted, and equal to the oracle."""
    p = synth.Problem("edge", W, 19, H, 1e-6, 4, synth.N01)
    xs, res, w = synth.device_inputs(p, dev)
    stream = torch.cuda.current_stream(dev)
    outs = [torch.empty_like(res) for _ in range(3)]
    st, word = _noalloc(dev, xs, res, w, p.eps, outs, stream)
    assert st == farn.FARN_OK and word == 0, (farn.farn_status_string(st), word)
    torch.cuda.synchronize(dev)
    _check_against_oracle(O, xs, res, w, p.eps, outs, f"no-alloc W={W} H={H}")
    ref = farn.forward(xs, res, w, p.eps)
    torch.cuda.synchronize(dev)
    assert_parity([u16(t) for t in outs], [u16(t) for t in ref], f"vs farn_forward W={W} H={H}")


@pytest.mark.parametrize("H", [16392, 32768])
def test_noalloc_rows_beyond_the_limit_refused(dev, H):
    """Rows longer than 16384 elements: FARN_ERR_UNSUPPORTED, nothing written."""
    p = synth.Problem("long", 2, 2, H, 1e-6, 1, synth.N01)
    xs, res, w = synth.device_inputs(p, dev)
    stream = torch.cuda.current_stream(dev)
    outs = [torch.full_like(res, 3.0) for _ in range(3)]
    st, _ = _noalloc(dev, xs, res, w, 1e-6, outs, stream)
    assert st == farn.FARN_ERR_UNSUPPORTED
    torch.cuda.synchronize(dev)
    assert all(bool((o == 3.0).all()) for o in outs)


def test_noalloc_asynchronous_call_and_errors(O, dev):
    p = synth.workload("decode")[0].with_T(200)
    xs, res, w = synth.device_inputs(p, dev)
    stream = torch.cuda.current_stream(dev)
    outs = [torch.empty_like(res) for _ in range(3)]
    st, word = _noalloc(dev, xs, res, w, p.eps, outs, stream, want_status=False)
    assert st == farn.FARN_OK and word is None
    torch.cuda.synchronize(dev)
    ref = farn.forward(xs, res, w, p.eps)
    torch.cuda.synchronize(dev)
    assert_parity([u16(t) for t in outs], [u16(t) for t in ref], "asynchronous no-alloc call")
    _check_against_oracle(O, xs, res, w, p.eps, outs, "asynchronous no-alloc call vs oracle")
    # an output over an input: refused before anything runs
    st, _ = _noalloc(dev, xs, res, w, p.eps, (xs[0], outs[1], outs[2]), stream)
    assert st == farn.FARN_ERR_ALIAS
    # a device this process does not have: an invalid argument
    st, _ = _noalloc(dev, xs, res, w, p.eps, outs, stream, device=torch.cuda.device_count())
    assert st == farn.FARN_ERR_INVALID_ARG
    st, _ = _noalloc(dev, xs, res, w, p.eps, outs, stream, device=-1)
    assert st == farn.FARN_ERR_INVALID_ARG
    # and the device itself still works afterwards
    st, word = _noalloc(dev, xs, res, w, p.eps, outs, stream)
    assert st == farn.FARN_OK and word == 0
