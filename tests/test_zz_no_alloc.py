"""farn_forward_noalloc, the entry point for callers that cannot allocate
device memory (code inside another framework's plugin or allocator
interface, where every device allocation must go through that framework).

It is called through the C ABI and checked against the ordinary entry point
farn_forward on the same inputs: reduced and residual_out bit for bit,
norm_out within one bf16 ulp, on two calls in a row (the second call finds
the shared status word as the first one left it).  This file is collected
last so that a run stopping at the first failure has run everything else;
it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import rank_sum_residual_gb300 as farn  # noqa: E402
import synth  # noqa: E402
from parity import assert_parity, u16  # noqa: E402

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


def _noalloc(dev, xs, res, w, eps, outs, stream, want_status=True):
    T, H = res.shape
    return farn.farn_forward_noalloc(
        dev.index, [x.data_ptr() for x in xs], len(xs), res.data_ptr(), w.data_ptr(),
        eps, T, H, outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(),
        stream.cuda_stream, want_status=want_status)


@pytest.mark.parametrize("name,T", [("decode", 300), ("prefill", 257), ("wide", 160)])
def test_noalloc_matches_farn_forward_twice(dev, name, T):
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


def test_noalloc_asynchronous_call_and_errors(dev):
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
    # an output over an input: refused before anything runs
    st, _ = _noalloc(dev, xs, res, w, p.eps, (xs[0], outs[1], outs[2]), stream)
    assert st == farn.FARN_ERR_ALIAS
    # a row too long for the staged kernel: refused, not mis-run
    big = synth.Problem("long", 2, 2, 32768, 1e-6, 1, synth.N01)
    bx, bres, bw = synth.device_inputs(big, dev)
    bouts = [torch.empty_like(bres) for _ in range(3)]
    st, _ = _noalloc(dev, bx, bres, bw, 1e-6, bouts, stream)
    assert st == farn.FARN_ERR_UNSUPPORTED
