"""The NVFP4 copy of norm_out (farn_forward_nvfp4) on the GPU, through the C
ABI, against the oracle: reduced and residual_out bit for bit, norm_out
within one bf16 ulp; given the GPU's own bf16 norm_out, the E2M1 codes and
the E4M3 block scales are unique, so they must match the oracle's
quantisation of that norm_out byte for byte (the decision is taken on the
same bf16 values on both sides)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import rank_sum_residual_gb300 as farn  # noqa: E402
import synth  # noqa: E402
from parity import assert_parity, sample_rows, u16  # noqa: E402
from gpu_util import make_ctx, oracle_rows  # noqa: E402

pytestmark = pytest.mark.gpu

G = 168.0          # the workload's tensor scale: an amax of 16 maps to 448 * 6


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


def _check_codes(O, nrm_u16, q, sc, g, what):
    want_q, want_s = O.quant_nvfp4(nrm_u16, g)
    got_q, got_s = q.cpu().numpy(), sc.cpu().numpy()
    if not np.array_equal(got_s, want_s):
        bad = np.argwhere(got_s != want_s)[:5].tolist()
        raise AssertionError(f"{what}: block scales differ at {bad}: "
                             f"{[(hex(got_s[tuple(b)]), hex(want_s[tuple(b)])) for b in bad]}")
    if not np.array_equal(got_q, want_q):
        bad = np.argwhere(got_q != want_q)[:5].tolist()
        raise AssertionError(f"{what}: codes differ at {bad}: "
                             f"{[(hex(got_q[tuple(b)]), hex(want_q[tuple(b)])) for b in bad]}")


def _check(O, xs, res, w, eps, g, out, what):
    red, ro, nrm, q, sc = out
    assert_parity([u16(red), u16(ro), u16(nrm)], oracle_rows(O, xs, res, w, eps), what)
    _check_codes(O, u16(nrm), q, sc, g, what)


@pytest.mark.parametrize("name,T", [("decode", 1), ("decode", 5), ("decode", 64), ("c1", 16),
                                    ("prefill", 300), ("prefill", 2200), ("wide", 100),
                                    ("nonpow2", 77), ("prefill_f32", 9), ("nonpow2", 2100)])
def test_nvfp4_output(O, dev, name, T):
    p = synth.workload(name)[0].with_T(T)
    xs, res, w = synth.device_inputs(p, dev)
    out = farn.forward_nvfp4(xs, res, w, p.eps, G)
    torch.cuda.synchronize()
    _check(O, xs, res, w, p.eps, G, out, f"nvfp4 {name} T={T}")


@pytest.mark.parametrize("g", [1.0, 0.03125, 3000.0])
def test_nvfp4_tensor_scales(O, dev, g):
    """Scales from underflowing to saturating E4M3 block scales."""
    p = synth.workload("prefill")[0].with_T(40)
    xs, res, w = synth.device_inputs(p, dev)
    out = farn.forward_nvfp4(xs, res, w, p.eps, g)
    torch.cuda.synchronize()
    _check(O, xs, res, w, p.eps, g, out, f"nvfp4 g={g}")


@pytest.mark.parametrize("env", [dict(FARN_VARIANT="generic"), dict(FARN_CLUSTER=2),
                                 dict(FARN_CLUSTER=16), dict(FARN_VARIANT="row", FARN_VPT=4),
                                 dict(FARN_VARIANT="row", FARN_VPT=1),
                                 dict(FARN_VARIANT="stage"), dict(FARN_VARIANT="stage", FARN_VPT=2),
                                 dict(FARN_VARIANT="stage", FARN_STAGE_CTAS=1)],
                         ids=lambda e: "-".join(f"{k[5:].lower()}{v}" for k, v in e.items()))
def test_nvfp4_output_forced_variants(O, dev, env):
    p = synth.Problem("q", 6, 7, 4096, 1e-6, 13, synth.N01)
    xs, res, w = synth.device_inputs(p, dev)
    ctx = make_ctx(**env)
    try:
        out = farn.forward_nvfp4(xs, res, w, p.eps, G, ctx=ctx)
        torch.cuda.synchronize()
        _check(O, xs, res, w, p.eps, G, out, f"nvfp4 {env}")
    finally:
        ctx.close()


@pytest.mark.parametrize("variant", ["auto", "generic"])
def test_nvfp4_specials_and_without_norm_out(O, dev, variant):
    """Rows with a NaN, an overflow (a NaN row), all zeros and tiny values;
    the codes and scales are the same with and without the bf16 norm_out."""
    W, T, H = 4, 6, 1024
    p = synth.Problem("q", W, T, H, 1e-6, 21, synth.N01)
    xs, res, w = synth.device_inputs(p, dev)
    xs[1][0, 5] = float("nan")
    for x in xs:
        x[1, 7] = 3.0e38                 # reduced -> inf, the row's norm -> NaN
        x[2].zero_()
    res[2].zero_()
    for x in xs:
        x[3].view(torch.int16)[:] = 1    # 2^-133 everywhere
    res[3].zero_()
    ctx = make_ctx(FARN_VARIANT=variant) if variant != "auto" else None
    try:
        a = farn.forward_nvfp4(xs, res, w, p.eps, G, ctx=ctx)
        b = farn.forward_nvfp4(xs, res, w, p.eps, G, write_norm=False, ctx=ctx)
        torch.cuda.synchronize()
    finally:
        if ctx is not None:
            ctx.close()
    assert b[2] is None
    _check(O, xs, res, w, p.eps, G, a, f"nvfp4 specials {variant}")
    assert torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])
    assert not a[4][2].any() and not a[3][2].any()          # zero row: scales and codes 0


def test_nvfp4_odd_vector_count_and_alignment(O, dev):
    """H = 4112 (257 blocks): the cluster split keeps whole blocks per CTA or
    is refused; a code buffer that is not 4-byte aligned takes the generic
    kernel."""
    p = synth.Problem("q", 3, 2, 4112, 1e-6, 5, synth.N01)
    xs, res, w = synth.device_inputs(p, dev)
    out = farn.forward_nvfp4(xs, res, w, p.eps, G)
    torch.cuda.synchronize()
    _check(O, xs, res, w, p.eps, G, out, "nvfp4 H=4112")
    ctx = make_ctx(FARN_CLUSTER=2)
    try:
        with pytest.raises(farn.FarnError) as e:
            farn.forward_nvfp4(xs, res, w, p.eps, G, ctx=ctx)
        assert e.value.status == farn.FARN_ERR_UNSUPPORTED
    finally:
        ctx.close()
    T, H = 2, 4112
    red, ro, nrm = (torch.empty_like(res) for _ in range(3))
    qbuf = torch.empty(T * H // 2 + 16, dtype=torch.uint8, device=dev)
    q = qbuf[2:2 + T * H // 2]
    sc = torch.empty((T, H // 16), dtype=torch.uint8, device=dev)
    st = farn.farn_forward_nvfp4(farn._context_for(0).handle, [x.data_ptr() for x in xs],
                                 farn.FARN_BF16, 3, res.data_ptr(), w.data_ptr(), p.eps, T, H, G,
                                 red.data_ptr(), ro.data_ptr(), nrm.data_ptr(), q.data_ptr(),
                                 sc.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == farn.FARN_OK
    torch.cuda.synchronize()
    _check(O, xs, res, w, p.eps, G, (red, ro, nrm, q.view(T, H // 2), sc), "nvfp4 misaligned")


def test_nvfp4_argument_errors(dev):
    p = synth.Problem("q", 2, 4, 2048, 1e-6, 1, synth.N01)
    xs, res, w = synth.device_inputs(p, dev)
    red, ro, nrm = (torch.empty_like(res) for _ in range(3))
    q = torch.empty((4, 1024), dtype=torch.uint8, device=dev)
    sc = torch.empty((4, 128), dtype=torch.uint8, device=dev)
    c = farn._context_for(0)

    def call(H=2048, g=G, qp=None, sp=None):
        return farn.farn_forward_nvfp4(
            c.handle, [x.data_ptr() for x in xs], farn.FARN_BF16, 2, res.data_ptr(),
            w.data_ptr(), p.eps, 4, H, g, red.data_ptr(), ro.data_ptr(), nrm.data_ptr(),
            q.data_ptr() if qp is None else qp, sc.data_ptr() if sp is None else sp)
    for g in (0.0, -1.0, float("nan"), float("inf")):
        assert call(g=g) == farn.FARN_ERR_INVALID_ARG, g
    assert call(H=2040) == farn.FARN_ERR_INVALID_ARG          # H % 16 != 0
    assert call(sp=0) == farn.FARN_ERR_INVALID_ARG            # no block scales
    assert call(qp=red.data_ptr()) == farn.FARN_ERR_ALIAS    # codes over reduced
    assert call(sp=q.data_ptr() + 100) == farn.FARN_ERR_ALIAS  # scales inside the codes
    assert call() == farn.FARN_OK
    ctx = make_ctx(FARN_VARIANT="bulk")
    try:
        with pytest.raises(farn.FarnError) as e:
            farn.forward_nvfp4(xs, res, w, p.eps, G, ctx=ctx)
        assert e.value.status == farn.FARN_ERR_UNSUPPORTED
    finally:
        ctx.close()
    torch.cuda.synchronize()


def test_nvfp4_plan(dev):
    c = farn._context_for(0)
    for T, want in ((8192, "stage"), (100, "row"), (1, "cluster")):
        p = synth.workload("prefill")[0].with_T(T)
        xs, res, w = synth.device_inputs(p, dev)
        red, ro = torch.empty_like(res), torch.empty_like(res)
        v, _, _ = farn.farn_plan_typed(c.handle, farn.FARN_BF16, p.W, T, p.H,
                                       [x.data_ptr() for x in xs], res.data_ptr(), w.data_ptr(),
                                       red.data_ptr(), ro.data_ptr(), 0,
                                       flags=farn.FARN_PLAN_NVFP4_OUT)
        assert v == want, (T, v)
        del xs, res, w, red, ro
    torch.cuda.empty_cache()


def test_nvfp4_full_size_sampled(O, dev):
    """The bench's configuration (8192 x 8192, W = 8, no bf16 norm_out):
    the codes and scales of sampled rows equal those of the call that also
    writes norm_out, which are checked against the oracle."""
    p = synth.workload("prefill_nvfp4")[0]
    xs, res, w = synth.device_inputs(p, dev)
    a = farn.forward_nvfp4(xs, res, w, p.eps, p.tensor_scale)
    b = farn.forward_nvfp4(xs, res, w, p.eps, p.tensor_scale, write_norm=False)
    torch.cuda.synchronize()
    assert torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    rows = sample_rows(p.T, 48, seed=31)
    idx = torch.as_tensor(rows, device=dev)
    want = oracle_rows(O, xs, res, w, p.eps, rows)
    got = [u16(t.index_select(0, idx)) for t in a[:3]]
    assert_parity(got, want, "nvfp4 full size")
    _check_codes(O, got[2], a[3].index_select(0, idx), a[4].index_select(0, idx),
                 p.tensor_scale, "nvfp4 full size")
    del xs, res, w, a, b
    torch.cuda.empty_cache()
