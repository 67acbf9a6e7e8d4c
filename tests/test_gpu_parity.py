"""GPU parity: the CUDA path, called through the C ABI, against the CPU
oracle on the same seeded device-generated inputs.

reduced and residual_out must match bit for bit, norm_out within one bf16
ulp (tests/parity.py).  Covers the five benchmark shapes (full size on
sampled rows, and mid-size shapes spanning many CTAs with a ragged row
count in full), every kernel variant, and the edge cases: empty and
one-row inputs, odd H, misaligned pointers, W = 1 and W = 32, zero rows,
NaN and overflow, in-place residual, guard regions around the outputs,
argument errors and injected launch faults.
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import rank_sum_residual_gb300 as farn  # noqa: E402
import synth  # noqa: E402
from parity import assert_parity, compare, sample_rows, u16  # noqa: E402
from gpu_util import host, make_ctx, oracle_rows  # noqa: E402,F401

pytestmark = pytest.mark.gpu

SENTINEL = 0x7BAD          # a finite bf16 pattern no output of these tests has


@pytest.fixture(scope="session")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    farn.build_library()
    synth.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


@pytest.fixture(scope="session")
def O():
    return oracle.Oracle()


def run_and_check(O, p, dev, ctx=None, rows=None, what=""):
    xs, res, w = synth.device_inputs(p, dev)
    out = farn.forward(xs, res, w, p.eps, ctx=ctx)
    torch.cuda.synchronize()
    want = oracle_rows(O, xs, res, w, p.eps, rows)
    if rows is None:
        got = [u16(t) for t in out]
    else:
        idx = torch.as_tensor(rows, device=dev)
        got = [u16(t.index_select(0, idx)) for t in out]
    return assert_parity(got, want, what or p.name)


# ------------------------------------------------------------ the workloads
def test_c1_full(O, dev):
    run_and_check(O, synth.workload("c1")[0], dev)


@pytest.mark.parametrize("T", synth.DECODE_TS)
def test_decode_sweep_full(O, dev, T):
    p = [q for q in synth.workload("decode") if q.T == T][0]
    run_and_check(O, p, dev)


@pytest.mark.parametrize("name,T", [("prefill", 333), ("nonpow2", 517), ("wide", 257),
                                    ("prefill", 1), ("wide", 9)])
def test_mid_size_full(O, dev, name, T):
    """The large shapes' H, W and value recipes at a row count the oracle
    finishes in seconds, ragged against every grid size."""
    run_and_check(O, synth.workload(name)[0].with_T(T), dev)


@pytest.mark.parametrize("name", ["prefill", "nonpow2", "wide", "rmsnorm"])
def test_full_size_sampled_rows(O, dev, name):
    """Full benchmark size, default launch plan (as the benchmark times it);
    the oracle recomputes 160 sampled rows (first, middle, last, random)."""
    p = synth.workload(name)[0]
    rows = sample_rows(p.T, 160, seed=p.W)
    run_and_check(O, p, dev, rows=rows)
    torch.cuda.empty_cache()


# ------------------------------------------------------------- variants
def _variant_outputs(dev, p, ctx):
    xs, res, w = synth.device_inputs(p, dev)
    out = farn.forward(xs, res, w, p.eps, ctx=ctx)
    torch.cuda.synchronize()
    return xs, res, w, [u16(t) for t in out]


@pytest.mark.parametrize("env", [
    dict(FARN_VARIANT="row"), dict(FARN_VARIANT="generic"),
    dict(FARN_VARIANT="cluster", FARN_CLUSTER=2), dict(FARN_VARIANT="cluster", FARN_CLUSTER=4),
    dict(FARN_VARIANT="cluster", FARN_CLUSTER=8), dict(FARN_VARIANT="cluster", FARN_CLUSTER=16),
    dict(FARN_VARIANT="row", FARN_VPT=1), dict(FARN_VARIANT="row", FARN_VPT=2),
    dict(FARN_VARIANT="row", FARN_VPT=4), dict(FARN_VARIANT="bulk"),
    dict(FARN_VARIANT="stage"), dict(FARN_VARIANT="stage", FARN_STAGE_R=8),
], ids=lambda e: "-".join(f"{k[5:].lower()}{v}" for k, v in e.items()))
@pytest.mark.parametrize("shape", [(8, 5, 4096), (4, 37, 5120), (16, 3, 7168)],
                         ids=lambda s: f"W{s[0]}T{s[1]}H{s[2]}")
def test_forced_variants_match_oracle_and_each_other(O, dev, env, shape):
    W, T, H = shape
    p = synth.Problem("variant", W, T, H, 1e-6, 17, synth.N01)
    ctx = make_ctx(**env)
    try:
        xs, res, w, got = _variant_outputs(dev, p, ctx)
        want = oracle_rows(O, xs, res, w, p.eps)
        assert_parity(got, want, f"{env} {shape}")
        # the default plan on the same input: reduced/residual_out identical
        _, _, _, ref = _variant_outputs(dev, p, None)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
        assert compare(got, ref)["norm_out"]["max_ulp"] <= 1
        assert farn.farn_device_status(ctx.handle) == 0
    finally:
        ctx.close()


@pytest.mark.parametrize("W,T,H,plan", [
    (32, 5, 4096, ("cluster", 4, 128)),   # four batches of partials, cluster split
    (9, 40, 4096, ("row", 1, 512)),       # one full batch and one partial
    (32, 100, 2048, ("row", 1, 256)),
    (12, 1, 8192, ("cluster", 8, 128)),
    (1, 7, 4096, ("cluster", 4, 128)),    # one partial: residual add + RMSNorm
    (3, 151, 4096, ("row", 1, 512)),      # the last latency-bound row count
], ids=lambda v: str(v).replace(" ", ""))
def test_one_row_decode_builds(O, dev, W, T, H, plan):
    """The one-row builds that serve latency-bound calls (first batch of
    partial pointers by constant rank index, later batches at run time;
    one-row clusters store reduced/residual_out after the DSMEM exchange)
    against the oracle, in full."""
    p = synth.Problem("onerow", W, T, H, 1e-5, 21 + W, synth.N01)
    xs, res, w = synth.device_inputs(p, dev)
    outs = [torch.empty_like(res) for _ in range(3)]
    c = farn._context_for(0)
    got_plan = farn.farn_plan(c.handle, W, T, H, [x.data_ptr() for x in xs], res.data_ptr(),
                              w.data_ptr(), *[o.data_ptr() for o in outs])
    assert got_plan == plan
    farn.forward(xs, res, w, p.eps, out=outs)
    torch.cuda.synchronize()
    assert_parity([u16(o) for o in outs], oracle_rows(O, xs, res, w, p.eps),
                  f"one-row build W={W} T={T} H={H}")


@pytest.mark.parametrize("name,T", [("prefill", 1000), ("nonpow2", 613), ("wide", 300),
                                    ("decode", 4096), ("c1", 777), ("small_h", 999),
                                    ("ragged", 401), ("w32_h16384", 40), ("w4_h16384", 333),
                                    ("tiny_h", 157)])
def test_bulk_variant(O, dev, name, T):
    """The TMA-staged persistent kernel on the five shapes' H, W and value
    recipes; T larger than the resident grid, so CTAs loop over rows and
    the shared-memory ring wraps many times.  Also: a row whose last
    segment is shorter than the others (H = 5128: 641 vectors in segments
    of 224), the longest row at the most partials (W = 32, H = 16384: 16
    segments, a 3-stage ring), the longest row at few partials, and rows
    shorter than one warp of vectors."""
    ctx = make_ctx(FARN_VARIANT="bulk")
    try:
        shapes = {"small_h": (5, 1024), "ragged": (6, 5128), "w32_h16384": (32, 16384),
                  "w4_h16384": (4, 16384), "tiny_h": (3, 48)}
        if name in shapes:
            W, H = shapes[name]
            p = synth.Problem(name, W, T, H, 1e-6, 9, synth.N01)
        else:
            p = synth.workload(name)[0].with_T(T)
        xs, res, w = synth.device_inputs(p, dev)
        outs = [torch.empty_like(res) for _ in range(3)]
        plan = farn.farn_plan(ctx.handle, p.W, p.T, p.H, [x.data_ptr() for x in xs],
                              res.data_ptr(), w.data_ptr(), *[o.data_ptr() for o in outs])
        assert plan[0] == "bulk"
        farn.forward(xs, res, w, p.eps, out=outs, ctx=ctx)
        torch.cuda.synchronize()
        assert_parity([u16(o) for o in outs], oracle_rows(O, xs, res, w, p.eps),
                      f"bulk {name} T={T}")
        assert farn.farn_device_status(ctx.handle) == 0
    finally:
        ctx.close()


@pytest.mark.parametrize("W,H,T,threads", [
    (8, 4096, 333, 32 + 512),     # one segment of 512 consumers, 3 stages
    (8, 8192, 419, 32 + 512),     # two segments of 512
    (16, 5120, 257, 32 + 320),    # two segments of 320, a 2-stage ring
    (16, 7168, 301, 32 + 224),    # two segments leave 1 stage: four of 224
    (12, 6144, 190, 32 + 384),    # two segments of 384
    (4, 5120, 211, 32 + 224),     # W < 8: at most 256 consumers, >= 4 stages
    (4, 4096, 150, 32 + 256)])
def test_bulk_consumer_split(O, dev, W, H, T, threads):
    """The TMA-staged kernel's row split: with W >= 8 inputs a row takes one
    or two segments of up to 512 consumer threads (the fewest segments whose
    ring holds 2 stages), with fewer inputs at most 256 consumers and a ring
    of at least 4 stages; every split equal to the oracle."""
    ctx = make_ctx(FARN_VARIANT="bulk")
    try:
        p = synth.Problem("split", W, T, H, 1e-6, W + T, synth.N01)
        xs, res, w = synth.device_inputs(p, dev)
        outs = [torch.empty_like(res) for _ in range(3)]
        plan = farn.farn_plan(ctx.handle, W, T, H, [x.data_ptr() for x in xs], res.data_ptr(),
                              w.data_ptr(), *[o.data_ptr() for o in outs])
        assert plan[0] == "bulk" and plan[2] == threads, plan
        farn.forward(xs, res, w, p.eps, out=outs, ctx=ctx)
        torch.cuda.synchronize()
        assert_parity([u16(o) for o in outs], oracle_rows(O, xs, res, w, p.eps),
                      f"bulk split W={W} H={H}")
        assert farn.farn_device_status(ctx.handle) == 0
    finally:
        ctx.close()


def test_bulk_bounded_wait_expires_and_reports(O, dev):
    """The TMA-staged kernel's waits are bounded.  With FARN_FAULT_INJECT=stall
    (read at create) CTA 0's consumers wait on a barrier that nothing
    completes: they give up after the 2 s limit, the kernel returns (no GPU
    fault, nothing hangs), and the status word says which wait gave up.
    CTA 0's rows are left unwritten, every other row equals the oracle, the
    status read clears it, and the context's next status is clean."""
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    T, W, H = 600, 8, 4096
    p = synth.Problem("stall", W, T, H, 1e-6, 3, synth.N01)
    xs, res, w = synth.device_inputs(p, dev)
    sentinel = 0x7FC1                                    # a NaN no output can be
    outs = [torch.full_like(res, 0).view(torch.int16).fill_(sentinel).view(torch.bfloat16)
            for _ in range(3)]
    ctx = make_ctx(FARN_VARIANT="bulk", FARN_FAULT_INJECT="stall")
    try:
        assert farn.farn_plan(ctx.handle, W, T, H, [x.data_ptr() for x in xs], res.data_ptr(),
                              w.data_ptr(), *[o.data_ptr() for o in outs])[0] == "bulk"
        farn.forward(xs, res, w, p.eps, out=outs, ctx=ctx)
        torch.cuda.synchronize()
        st = farn.farn_device_status(ctx.handle)
        # a consumer gave up (1), or the producer's own limit came first (2)
        assert st != 0 and st & ~3 == 0, st
        assert farn.farn_device_status(ctx.handle) == 0   # the read cleared it
        got = [u16(o) for o in outs]
        cta0 = np.arange(0, T, min(T, nsm))               # rows of CTA 0 (one CTA per SM)
        for g in got:
            assert (g[cta0] == sentinel).all()
        rest = np.setdiff1d(np.arange(T), cta0)
        want = oracle_rows(O, xs, res, w, p.eps)
        assert_parity([g[rest] for g in got], [x[rest] for x in want], "bulk stall, other CTAs")
    finally:
        ctx.close()
    # the same call on a context without the injection: complete and clean
    ctx = make_ctx(FARN_VARIANT="bulk")
    try:
        out = farn.forward(xs, res, w, p.eps, ctx=ctx)
        torch.cuda.synchronize()
        assert farn.farn_device_status(ctx.handle) == 0
        assert_parity([u16(o) for o in out], want, "bulk after stall")
    finally:
        ctx.close()


def test_bulk_moe_bounded_wait_expires_and_reports(O, dev):
    """The same bounded-wait expiry through the MoE combine's TMA-staged
    kernel (its default for long calls): CTA 0's rows unwritten, the status
    word set and cleared by its read, every other row equal to the oracle."""
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    p = _moe(500, 8, 4096, seed=21)
    (ex, index, gates), res, w = synth.device_inputs(p, dev)
    sentinel = 0x7FC1
    outs = tuple(torch.empty_like(res).view(torch.int16).fill_(sentinel).view(torch.bfloat16)
                 for _ in range(3))
    ctx = make_ctx(FARN_VARIANT="bulk", FARN_FAULT_INJECT="stall")
    try:
        farn.moe_combine(ex, index, gates, res, w, p.eps, out=outs, ctx=ctx)
        torch.cuda.synchronize()
        st = farn.farn_device_status(ctx.handle)
        assert st != 0 and st & ~3 == 0, st
        assert farn.farn_device_status(ctx.handle) == 0
    finally:
        ctx.close()
    got = [u16(o) for o in outs]
    cta0 = np.arange(0, p.T, min(p.T, nsm))
    for g in got:
        assert (g[cta0] == sentinel).all()
    rest = np.setdiff1d(np.arange(p.T), cta0)
    want = O.moe_combine(u16(ex), index.cpu().numpy(), gates.cpu().numpy(), u16(res), u16(w),
                         p.eps)
    assert_parity([g[rest] for g in got], [x[rest] for x in want], "moe bulk stall, other CTAs")


@pytest.mark.parametrize("ctas", [1, 2])
def test_bulk_variant_ctas_per_sm(O, dev, ctas):
    """One or two resident TMA-staged CTAs per SM (FARN_BULK_CTAS)."""
    ctx = make_ctx(FARN_VARIANT="bulk", FARN_BULK_CTAS=ctas)
    try:
        for name, T in (("prefill", 700), ("wide", 500), ("nonpow2", 900)):
            p = synth.workload(name)[0].with_T(T)
            xs, res, w = synth.device_inputs(p, dev)
            out = farn.forward(xs, res, w, p.eps, ctx=ctx)
            torch.cuda.synchronize()
            assert_parity([u16(o) for o in out], oracle_rows(O, xs, res, w, p.eps),
                          f"bulk x{ctas} {name}")
            assert farn.farn_device_status(ctx.handle) == 0
    finally:
        ctx.close()


@pytest.mark.parametrize("env", [dict(), dict(FARN_STAGE_R=8), dict(FARN_STAGE_CTAS=2),
                                 dict(FARN_VPT=2)],
                         ids=lambda e: "-".join(f"{k[5:].lower()}{v}" for k, v in e.items()) or "auto")
@pytest.mark.parametrize("name,T", [("prefill", 1000), ("nonpow2", 613), ("wide", 300),
                                    ("decode", 4096), ("c1", 777)])
def test_stage_variant(O, dev, name, T, env):
    """The cp.async-staged persistent kernel: CTAs loop over many rows and
    each thread's slot ring wraps across row boundaries."""
    ctx = make_ctx(FARN_VARIANT="stage", **env)
    try:
        p = synth.workload(name)[0].with_T(T)
        xs, res, w = synth.device_inputs(p, dev)
        outs = [torch.empty_like(res) for _ in range(3)]
        args = (ctx.handle, p.W, p.T, p.H, [x.data_ptr() for x in xs], res.data_ptr(),
                w.data_ptr(), *[o.data_ptr() for o in outs])
        t4 = (p.H // 8 // 4 + 31) // 32 * 32          # threads at 4 and 2 vectors
        t2 = (p.H // 8 // 2 + 31) // 32 * 32
        budget = 232448 // 2 - 1024
        if env.get("FARN_STAGE_CTAS") == 2 and 8 * 4 * t4 * 16 > budget \
                and 8 * 2 * t2 * 16 > budget:
            # even 8 chunks in flight do not fit two CTAs per SM: refused
            with pytest.raises(farn.FarnError) as e:
                farn.farn_plan(*args)
            assert e.value.status == farn.FARN_ERR_UNSUPPORTED
            return
        assert farn.farn_plan(*args)[0] == "stage"
        farn.forward(xs, res, w, p.eps, out=outs, ctx=ctx)
        torch.cuda.synchronize()
        assert_parity([u16(o) for o in outs], oracle_rows(O, xs, res, w, p.eps),
                      f"stage {name} T={T} {env}")
    finally:
        ctx.close()


def test_stage_in_place_and_few_rows(O, dev):
    """Fewer rows than CTAs (T < grid) and an in-place residual update."""
    ctx = make_ctx(FARN_VARIANT="stage")
    try:
        for T in (1, 3, 151):
            xs, res, w = _inputs(dev, 8, T, 8192, seed=T)
            want = oracle_rows(O, xs, res, w, 1e-6)
            red, nrm = torch.empty_like(res), torch.empty_like(res)
            farn.forward(xs, res, w, 1e-6, out=(red, res, nrm), ctx=ctx)
            torch.cuda.synchronize()
            assert_parity([u16(red), u16(res), u16(nrm)], want, f"stage in place T={T}")
    finally:
        ctx.close()


@pytest.mark.parametrize("variant", ["bulk", "stage"])
def test_persistent_variants_full_size_sampled(O, dev, variant):
    ctx = make_ctx(FARN_VARIANT=variant)
    try:
        for name in ("prefill", "wide"):
            p = synth.workload(name)[0]
            run_and_check(O, p, dev, ctx=ctx, rows=sample_rows(p.T, 96, seed=5))
            assert farn.farn_device_status(ctx.handle) == 0
            torch.cuda.empty_cache()
    finally:
        ctx.close()


def test_plan_choices(dev):
    c = farn.Context(0)
    try:
        def plan(W, T, H, off=0):
            # fake, never-dereferenced addresses 4 GiB apart
            a = (1 << 40) + off
            g = 1 << 32
            return farn.farn_plan(c.handle, W, T, H, [a] * W, a + g, a + 2 * g,
                                  a + 3 * g, a + 4 * g, a + 5 * g)
        assert plan(8, 8192, 8192) == ("stage", 1, 512)  # 2 vectors/thread, 1 CTA/SM
        # fewer than 8 partials and a bf16 norm_out: one CTA per row, 4 vectors
        assert plan(4, 32768, 5120) == ("row", 1, 160)
        assert plan(1, 8192, 8192) == ("row", 1, 256)
        assert plan(7, 4096, 4096) == ("row", 1, 128)
        # W >= 12 long calls: the TMA-staged kernel (producer warp + consumers)
        assert plan(16, 4096, 7168) == ("bulk", 1, 32 + 224)   # 4 segments of 224
        assert plan(12, 2048, 4096) == ("bulk", 1, 32 + 512)   # 1 segment of 512
        assert plan(32, 2048, 8192) == ("bulk", 1, 32 + 192)   # 6 segments of 192, 2 stages
        # 8..11 partials: the row length decides
        assert plan(11, 4096, 7168)[0] == "bulk"
        assert plan(8, 4096, 6144)[0] == "bulk"
        assert plan(8, 4096, 5120)[0] == "row"
        assert plan(10, 4096, 4096)[0] == "row"
        assert plan(8, 4096, 12288)[0] == "stage"
        assert plan(16, 1000, 7168)[0] == "bulk"         # W >= 12: from 256 rows on
        assert plan(16, 255, 7168)[0] == "row"
        assert plan(11, 1000, 7168)[0] == "row"          # 8..11: long calls only
        # half the row threshold when the call reads >= 128 MiB
        assert plan(8, 1024, 8192)[0] == "stage"        # 151 MB
        assert plan(8, 1023, 8192)[0] == "row"
        assert plan(4, 1024, 5120)[0] == "row"          # 52 MB
        assert plan(8, 1, 4096) == ("cluster", 4, 128)  # few rows: 128 vectors per CTA
        assert plan(8, 8, 4096) == ("cluster", 4, 128)
        assert plan(8, 1, 8192) == ("cluster", 8, 128)  # longer rows: wider split
        assert plan(8, 1, 1024) == ("row", 1, 128)      # short rows stay in one CTA
        assert plan(8, 16, 4096) == ("row", 1, 512)     # from 16 rows: one CTA per row
        assert plan(8, 64, 4096) == ("row", 1, 512)     # decode: all ranks at once
        assert plan(4, 16, 13)[0] == "generic"          # H % 8 != 0
        assert plan(4, 16, 2048, off=2)[0] == "generic"  # misaligned
        assert plan(4, 4096, 32768)[0] == "generic"     # longer than one CTA
    finally:
        c.close()


@pytest.mark.parametrize("W,H,T,want", [(10, 4096, 2100, "row"), (9, 6144, 2050, "bulk"),
                                         (11, 8192, 2049, "stage"), (12, 3072, 2111, "bulk"),
                                         (5, 7168, 2222, "row")])
def test_long_call_default_plans(O, dev, W, H, T, want):
    """Long calls through the default plan, one per kernel the row length
    and the partial count pick (row / TMA-staged / cp.async-staged), a
    ragged row count each, sampled rows against the oracle."""
    c = farn._context_for(0)
    p = synth.Problem("long", W, T, H, 1e-6, W * T, synth.N01)
    xs, res, w = synth.device_inputs(p, dev)
    outs = [torch.empty_like(res) for _ in range(3)]
    plan = farn.farn_plan(c.handle, W, T, H, [x.data_ptr() for x in xs], res.data_ptr(),
                          w.data_ptr(), *[o.data_ptr() for o in outs])
    assert plan[0] == want, plan
    farn.forward(xs, res, w, p.eps, out=outs)
    torch.cuda.synchronize()
    rows = sample_rows(T, 64, seed=W)
    idx = torch.as_tensor(rows, device=dev)
    got = [u16(o.index_select(0, idx)) for o in outs]
    assert_parity(got, oracle_rows(O, xs, res, w, p.eps, rows=rows), f"default plan W={W} H={H}")
    del xs, res, w, outs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("H,want", [(5120, "row"), (5128, "bulk"), (8184, "bulk"), (8192, "stage")])
def test_mid_w_row_length_boundaries(O, dev, H, want):
    """8 partials on each side of the row-length limits of the default plan
    (5120 for the row kernel, 8192 for the staged one), ragged row count,
    sampled rows against the oracle."""
    c = farn._context_for(0)
    T = 2051
    p = synth.Problem("edge", 8, T, H, 1e-6, H, synth.N01)
    xs, res, w = synth.device_inputs(p, dev)
    outs = [torch.empty_like(res) for _ in range(3)]
    plan = farn.farn_plan(c.handle, 8, T, H, [x.data_ptr() for x in xs], res.data_ptr(),
                          w.data_ptr(), *[o.data_ptr() for o in outs])
    assert plan[0] == want, plan
    farn.forward(xs, res, w, p.eps, out=outs)
    torch.cuda.synchronize()
    rows = sample_rows(T, 48, seed=H)
    idx = torch.as_tensor(rows, device=dev)
    assert_parity([u16(o.index_select(0, idx)) for o in outs],
                  oracle_rows(O, xs, res, w, p.eps, rows=rows), f"boundary H={H}")
    del xs, res, w, outs
    torch.cuda.empty_cache()


def test_deterministic(dev):
    p = synth.workload("decode")[-1]
    a = _variant_outputs(dev, p, None)[3]
    b = _variant_outputs(dev, p, None)[3]
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


# ------------------------------------------------------------ edge cases
@pytest.mark.parametrize("W", [1, 2, 3, 16, 32])
@pytest.mark.parametrize("T,H", [(1, 8), (3, 4), (3, 13), (2, 2048), (3, 5120),
                                 (5, 8192), (2, 16384), (2, 16392), (1, 24576)])
def test_edge_shapes(O, dev, W, T, H):
    p = synth.Problem("edge", W, T, H, 1e-6, 5, synth.N01)
    run_and_check(O, p, dev, what=f"W={W} T={T} H={H}")


def test_empty_rows(dev):
    xs = [torch.empty((0, 64), dtype=torch.bfloat16, device=dev) for _ in range(3)]
    res = torch.empty((0, 64), dtype=torch.bfloat16, device=dev)
    w = torch.ones(64, dtype=torch.bfloat16, device=dev)
    out = farn.forward(xs, res, w, 1e-6)
    torch.cuda.synchronize()
    assert all(t.shape == (0, 64) for t in out)


def _inputs(dev, W, T, H, seed=3):
    p = synth.Problem("x", W, T, H, 1e-6, seed, synth.N01)
    return synth.device_inputs(p, dev)


def test_misaligned_pointers_take_generic_path(O, dev):
    W, T, H = 3, 7, 2048
    xs0, res0, w0 = _inputs(dev, W, T, H)
    def shifted(t):                      # same values, 2-byte-offset storage
        buf = torch.empty(t.numel() + 1, dtype=torch.bfloat16, device=dev)
        v = buf[1:].view(t.shape)
        v.copy_(t)
        return v
    xs = [shifted(x) for x in xs0]
    res, w = shifted(res0), shifted(w0)
    assert xs[0].data_ptr() % 16 == 2
    outs = [shifted(torch.zeros((T, H), dtype=torch.bfloat16, device=dev)) for _ in range(3)]
    c = farn._context_for(0)
    assert farn.farn_plan(c.handle, W, T, H, [x.data_ptr() for x in xs], res.data_ptr(),
                          w.data_ptr(), *[o.data_ptr() for o in outs])[0] == "generic"
    farn.forward(xs, res, w, 1e-6, out=outs)
    torch.cuda.synchronize()
    assert_parity([u16(o) for o in outs], oracle_rows(O, xs0, res0, w0, 1e-6), "misaligned")


def test_special_values(O, dev):
    """A zero row, a NaN in one partial, an overflowing sum, subnormals."""
    W, T, H = 4, 6, 4096
    xs, res, w = _inputs(dev, W, T, H)
    for x in xs:
        x[0].zero_()
    res[0].zero_()
    xs[2][1, 77] = float("nan")
    big = torch.tensor(3.0e38, dtype=torch.bfloat16)
    for x in xs:
        x[2, 5] = big
    for x in xs:                                      # 2^-133 everywhere
        x[3].view(torch.int16)[:] = 1
    res[3].zero_()
    out = farn.forward(xs, res, w, 1e-6)
    torch.cuda.synchronize()
    got = [u16(t) for t in out]
    want = oracle_rows(O, xs, res, w, 1e-6)
    assert_parity(got, want, "special values")
    # a zero row stays zero (-0 where the weight is negative)
    assert np.all(got[0][0] == 0) and np.all((got[2][0] & 0x7FFF) == 0)
    assert np.isnan(out[2][1].float().cpu().numpy()).all()
    assert got[0][2, 5] == 0x7F80                     # +inf
    assert np.all(got[0][3] == 4)                     # 4 * 2^-133, kept, not flushed


def test_in_place_residual(O, dev):
    W, T, H = 8, 40, 4096
    xs, res, w = _inputs(dev, W, T, H)
    want = oracle_rows(O, xs, res, w, 1e-6)
    red = torch.empty_like(res)
    nrm = torch.empty_like(res)
    farn.forward(xs, res, w, 1e-6, out=(red, res, nrm))
    torch.cuda.synchronize()
    assert_parity([u16(red), u16(res), u16(nrm)], want, "in-place residual")


def test_guard_regions_untouched(O, dev):
    """Outputs carved out of larger buffers: the guard words around them
    must keep their sentinel (stands in for a memory checker)."""
    for (W, T, H) in [(8, 3, 4096), (4, 129, 5120), (3, 5, 13)]:
        xs, res, w = _inputs(dev, W, T, H)
        g = 4096
        bufs = [torch.full((T * H + 2 * g,), 0, dtype=torch.int16, device=dev) for _ in range(3)]
        for b in bufs:
            b.fill_(SENTINEL)
        outs = [b[g:g + T * H].view(torch.bfloat16).view(T, H) for b in bufs]
        farn.forward(xs, res, w, 1e-6, out=outs)
        torch.cuda.synchronize()
        for b in bufs:
            h = b.cpu().numpy().view(np.uint16)
            assert np.all(h[:g] == SENTINEL) and np.all(h[g + T * H:] == SENTINEL)
        assert_parity([u16(o) for o in outs], oracle_rows(O, xs, res, w, 1e-6), "guards")


def test_side_stream(O, dev):
    p = synth.workload("decode")[4]
    xs, res, w = synth.device_inputs(p, dev)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = farn.forward(xs, res, w, p.eps)
    s.synchronize()
    assert_parity([u16(t) for t in out], oracle_rows(O, xs, res, w, p.eps), "side stream")


# ------------------------------------------------------ errors on the GPU
def _sentinel_outputs(dev, T, H):
    outs = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(3)]
    for o in outs:
        o.view(torch.int16).fill_(SENTINEL)
    return outs


def test_alias_error_writes_nothing(dev):
    W, T, H = 4, 8, 2048
    xs, res, w = _inputs(dev, W, T, H)
    outs = _sentinel_outputs(dev, T, H)
    with pytest.raises(farn.FarnError) as e:
        farn.forward(xs, res, w, 1e-6, out=(outs[0], outs[0], outs[2]))
    assert e.value.status == farn.FARN_ERR_ALIAS
    with pytest.raises(farn.FarnError) as e:
        farn.forward(xs, res, w, 1e-6, out=(xs[1], outs[1], outs[2]))
    assert e.value.status == farn.FARN_ERR_ALIAS
    torch.cuda.synchronize()
    for o in outs:
        assert np.all(u16(o) == SENTINEL)


def test_bad_eps_and_shapes_raise(dev):
    W, T, H = 2, 4, 64
    xs, res, w = _inputs(dev, W, T, H)
    with pytest.raises(farn.FarnError):
        farn.forward(xs, res, w, float("nan"))
    with pytest.raises(farn.FarnError):
        farn.forward(xs, res, w, -1.0)
    with pytest.raises(ValueError):
        farn.forward(xs, res[:, :32].contiguous(), w, 1e-6)
    with pytest.raises(TypeError):
        farn.forward([x.half() for x in xs], res, w, 1e-6)


def test_injected_launch_fault_launches_nothing(dev):
    """FARN_FAULT_INJECT=launch is read when the context is created (not on
    every call): each launch of that context then fails on the host before
    anything is enqueued, for the rank-sum path and the MoE combine alike."""
    W, T, H = 4, 8, 2048
    xs, res, w = _inputs(dev, W, T, H)
    outs = _sentinel_outputs(dev, T, H)
    bad = make_ctx(FARN_FAULT_INJECT="launch")
    try:
        with pytest.raises(farn.FarnError) as e:
            farn.forward(xs, res, w, 1e-6, out=outs, ctx=bad)
        assert e.value.status == farn.FARN_ERR_CUDA
        pm = synth.Problem("moe", 2, T, H, 1e-6, 5, synth.N01, kind="moe_combine")
        (ex, index, gates), mres, mw = synth.device_inputs(pm, dev)
        with pytest.raises(farn.FarnError) as e:
            farn.moe_combine(ex, index, gates, mres, mw, 1e-6, out=outs, ctx=bad)
        assert e.value.status == farn.FARN_ERR_CUDA
    finally:
        bad.close()
    torch.cuda.synchronize()
    for o in outs:
        assert np.all(u16(o) == SENTINEL)
    # a context created without the variable is unaffected, even while it
    # is set: the library does not look at it per call
    good = farn.Context(0)
    os.environ["FARN_FAULT_INJECT"] = "launch"
    try:
        farn.forward(xs, res, w, 1e-6, out=outs, ctx=good)
    finally:
        os.environ.pop("FARN_FAULT_INJECT")
        torch.cuda.synchronize()
        good.close()
    assert not np.all(u16(outs[2]) == SENTINEL)


def test_injected_create_fault(dev):
    os.environ["FARN_FAULT_INJECT"] = "create"
    try:
        with pytest.raises(farn.FarnError) as e:
            farn.Context(0)
        assert e.value.status == farn.FARN_ERR_CUDA
    finally:
        os.environ.pop("FARN_FAULT_INJECT")


# ------------------------------------------- back-to-back dependent calls
@pytest.mark.parametrize("pdl", [1, 0])
def test_dependent_chain(O, dev, pdl):
    """Each call reads what the previous call wrote (its reduced becomes the
    next rank-0 partial, its residual_out the next residual) and overwrites
    buffers that the previous call read, with programmatic dependent launch
    on and off: the kernel must wait for its predecessor before any global
    access.  reduced and residual_out are exact, so the whole chain must
    match the oracle's chain bit for bit."""
    W, T, H, n = 4, 3, 4096, 12
    xs, res, w = _inputs(dev, W, T, H, seed=23)
    hx = [u16(x) for x in xs]
    hres, hw = u16(res), u16(w)
    ctx = make_ctx(FARN_PDL=pdl)
    try:
        bufs = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(6)]
        cur_x, cur_res = list(xs), res
        for i in range(n):
            red, ro, nrm = bufs[0:3] if i % 2 == 0 else bufs[3:6]
            farn.forward(cur_x, cur_res, w, 1e-6, out=(red, ro, nrm), ctx=ctx)
            cur_x = [red] + cur_x[1:]
            cur_res = ro
        torch.cuda.synchronize()
        got = [u16(red), u16(ro), u16(nrm)]
    finally:
        ctx.close()
    ox, ores = hx, hres
    for i in range(n):
        want = O.forward(ox, ores, hw, 1e-6)
        ox = [want[0]] + ox[1:]
        ores = want[1]
    assert_parity(got, want, f"chain of {n} dependent calls, pdl={pdl}")


def test_bulk_forced_on_unsupported_shape_is_an_error(dev):
    """Forcing the TMA-staged kernel where it cannot cover the row is
    refused, not mis-run: at most 4 segments per row (FARN_VPT=4) of at
    most 256 vectors cannot hold 12288 elements, and no plan takes rows
    longer than 16384 elements."""
    ctx = make_ctx(FARN_VARIANT="bulk", FARN_VPT=4)
    try:
        xs, res, w = _inputs(dev, 4, 8, 12288)
        with pytest.raises(farn.FarnError) as e:
            farn.forward(xs, res, w, 1e-6, ctx=ctx)
        assert e.value.status == farn.FARN_ERR_UNSUPPORTED
    finally:
        ctx.close()
    ctx = make_ctx(FARN_VARIANT="bulk")
    try:
        xs, res, w = _inputs(dev, 2, 4, 16392)
        with pytest.raises(farn.FarnError) as e:
            farn.forward(xs, res, w, 1e-6, ctx=ctx)
        assert e.value.status == farn.FARN_ERR_UNSUPPORTED
    finally:
        ctx.close()


@pytest.mark.parametrize("name", ["rmsnorm", "prefill"])
def test_full_size_in_place(O, dev, name):
    """residual_out written over the residual at full size, default plan."""
    p = synth.workload(name)[0]
    xs, res, w = synth.device_inputs(p, dev)
    rows = sample_rows(p.T, 96, seed=11)
    idx = torch.as_tensor(rows, device=dev)
    want = O.forward([u16(x.index_select(0, idx)) for x in xs],
                     u16(res.index_select(0, idx)), u16(w), p.eps)
    red, nrm = torch.empty_like(res), torch.empty_like(res)
    farn.forward(xs, res, w, p.eps, out=(red, res, nrm))
    torch.cuda.synchronize()
    got = [u16(t.index_select(0, idx)) for t in (red, res, nrm)]
    assert_parity(got, want, f"{name} in place")
    del xs, res, w, red, nrm
    torch.cuda.empty_cache()


# ---------------------------------------------------------- fp32 partials
def _f32(name, T, W=None, H=None):
    p = synth.workload(name)[0].with_T(T) if name in synth.WORKLOADS else None
    if p is None or W is not None:
        p = synth.Problem(name, W, T, H, 1e-6, 31, synth.N01)
    return synth.Problem(p.name, p.W, p.T, p.H, p.eps, p.seed, p.x, p.residual,
                         p.weight, "f32")


@pytest.mark.parametrize("prob", [
    ("prefill_f32", 333), ("prefill_f32", 2500), ("nonpow2", 517), ("wide", 300),
    ("wide", 2100), ("dec", 1, 8, 4096), ("dec", 5, 8, 4096), ("dec", 64, 8, 4096),
    ("odd", 3, 3, 1000), ("w1", 40, 1, 2048), ("w32", 6, 32, 1024)],
    ids=lambda p: "-".join(str(v) for v in p))
def test_f32_partials(O, dev, prob):
    """fp32 partials (residual, weight, outputs bf16) against the oracle's
    fp32-partial path, on the default launch plan."""
    p = _f32(*prob) if len(prob) == 2 else _f32(prob[0], prob[1], prob[2], prob[3])
    run_and_check(O, p, dev, what=f"f32 partials {prob}")


def test_f32_partials_full_size_sampled(O, dev):
    p = synth.workload("prefill_f32")[0]
    run_and_check(O, p, dev, rows=sample_rows(p.T, 128, seed=2))
    torch.cuda.empty_cache()


@pytest.mark.parametrize("env", [
    dict(FARN_VARIANT="row"), dict(FARN_VARIANT="generic"),
    dict(FARN_VARIANT="cluster", FARN_CLUSTER=2), dict(FARN_VARIANT="cluster", FARN_CLUSTER=8),
    dict(FARN_VARIANT="cluster", FARN_CLUSTER=16), dict(FARN_VARIANT="row", FARN_VPT=4),
    dict(FARN_VARIANT="row", FARN_VPT=1), dict(FARN_VARIANT="row", FARN_VPT=2)],
    ids=lambda e: "-".join(f"{k[5:].lower()}{v}" for k, v in e.items()))
def test_f32_partials_forced_variants(O, dev, env):
    p = _f32("v", 37, 6, 4096)
    ctx = make_ctx(**env)
    try:
        run_and_check(O, p, dev, ctx=ctx, what=f"f32 {env}")
    finally:
        ctx.close()


@pytest.mark.parametrize("variant", ["bulk", "stage"])
def test_f32_partials_staged_kernels_refused(dev, variant):
    """The TMA- and cp.async-staged kernels stage bf16 rows only: forcing
    either with fp32 partials is refused (the row kernel serves them)."""
    p = _f32("v", 4, 2, 2048)
    xs, res, w = synth.device_inputs(p, dev)
    ctx = make_ctx(FARN_VARIANT=variant)
    try:
        with pytest.raises(farn.FarnError) as e:
            farn.forward(xs, res, w, p.eps, ctx=ctx)
        assert e.value.status == farn.FARN_ERR_UNSUPPORTED
    finally:
        ctx.close()


def test_f32_partials_misaligned_and_specials(O, dev):
    W, T, H = 3, 5, 1024
    p = _f32("m", T, W, H)
    xs0, res, w = synth.device_inputs(p, dev)
    xs = []
    for x in xs0:                        # 4-byte offset: not 16-byte aligned
        buf = torch.empty(x.numel() + 1, dtype=torch.float32, device=dev)
        v = buf[1:].view(T, H)
        v.copy_(x)
        xs.append(v)
    xs[0][0, 3] = float("nan")
    xs[1][1, 7] = float("inf")
    xs[2][2, 9] = 3.0e38
    xs[1][2, 9] = 3.0e38                 # overflows the fp32 sum
    xs[0][3].zero_(); xs[1][3].zero_(); xs[2][3].zero_()
    xs[0][4, 0] = 1.0
    xs[1][4, 0] = 2.0 ** -10
    xs[2][4, 0] = -1.0                   # (1 + 2^-10) - 1 = 2^-10 exactly
    assert xs[0].data_ptr() % 16 == 4
    out = farn.forward(xs, res, w, p.eps)
    torch.cuda.synchronize()
    got = [u16(t) for t in out]
    assert_parity(got, oracle_rows(O, xs, res, w, p.eps), "f32 misaligned + specials")
    assert got[0][4, 0] == 0x3A80


def test_f32_partials_alias_uses_four_byte_extent(dev):
    """An output over the second half of an fp32 partial overlaps it (the
    partial spans T*H*4 bytes), so it is refused."""
    T, H = 8, 256
    x = torch.zeros((T, H), dtype=torch.float32, device=dev)
    res = torch.zeros((T, H), dtype=torch.bfloat16, device=dev)
    w = torch.ones(H, dtype=torch.bfloat16, device=dev)
    inside = x.view(torch.bfloat16).view(-1)[T * H: 2 * T * H].view(T, H)
    outs = (inside, torch.empty_like(res), torch.empty_like(res))
    with pytest.raises(farn.FarnError) as e:
        farn.forward([x], res, w, 1e-6, out=outs)
    assert e.value.status == farn.FARN_ERR_ALIAS


def test_f32_partials_plan(dev):
    c = farn.Context(0)
    try:
        a, g = (1 << 40), (1 << 34)
        args = ([a] * 8, a + g, a + 2 * g, a + 3 * g, a + 4 * g, a + 5 * g)
        assert farn.farn_plan_typed(c.handle, farn.FARN_F32, 8, 8192, 8192, *args)[0] == "row"
        assert farn.farn_plan_typed(c.handle, farn.FARN_BF16, 8, 8192, 8192, *args)[0] == "stage"
        assert farn.farn_plan_typed(c.handle, farn.FARN_F32, 8, 2, 4096, *args)[0] == "row"
        assert farn.farn_plan_typed(c.handle, farn.FARN_F32, 8, 2, 8192, *args)[0] == "cluster"
        with pytest.raises(farn.FarnError):
            farn.farn_plan_typed(c.handle, 7, 8, 2, 4096, *args)
        # with the FP8 output (norm_out written or not) the same kernel choice
        assert farn.farn_plan_typed(c.handle, farn.FARN_BF16, 8, 8192, 8192, *args,
                                    flags=farn.FARN_PLAN_FP8_OUT)[0] == "stage"
        noq = args[:5] + (0,)
        assert farn.farn_plan_typed(c.handle, farn.FARN_BF16, 8, 8192, 8192, *noq,
                                    flags=farn.FARN_PLAN_FP8_OUT)[0] == "stage"
        assert farn.farn_plan_typed(c.handle, farn.FARN_F32, 8, 8192, 8192, *noq,
                                    flags=farn.FARN_PLAN_FP8_OUT)[0] == "row"
        # fewer than 8 bf16 partials: the row kernel, but the stage kernel
        # for the quantised outputs
        assert farn.farn_plan_typed(c.handle, farn.FARN_BF16, 4, 8192, 8192, *args)[0] == "row"
        assert farn.farn_plan_typed(c.handle, farn.FARN_BF16, 4, 8192, 8192, *args,
                                    flags=farn.FARN_PLAN_FP8_OUT)[0] == "stage"
        assert farn.farn_plan_typed(c.handle, farn.FARN_BF16, 4, 8192, 8192, *noq,
                                    flags=farn.FARN_PLAN_NVFP4_OUT)[0] == "stage"
        # quantised outputs of one or two partials, or of short rows: the row kernel
        assert farn.farn_plan_typed(c.handle, farn.FARN_BF16, 1, 8192, 8192, *noq,
                                    flags=farn.FARN_PLAN_FP8_OUT)[0] == "row"
        assert farn.farn_plan_typed(c.handle, farn.FARN_BF16, 2, 8192, 8192, *noq,
                                    flags=farn.FARN_PLAN_NVFP4_OUT)[0] == "row"
        # many rows of one or two partials and 256..511 vectors: 4 per thread
        assert farn.farn_plan_typed(c.handle, farn.FARN_BF16, 1, 8192, 2048, *args) == \
            ("row", 1, 64)
        assert farn.farn_plan_typed(c.handle, farn.FARN_BF16, 4, 8192, 2048, *args) == \
            ("row", 1, 128)
        assert farn.farn_plan_typed(c.handle, farn.FARN_BF16, 4, 8192, 4096, *noq,
                                    flags=farn.FARN_PLAN_NVFP4_OUT)[0] == "row"
        assert farn.farn_plan_typed(c.handle, farn.FARN_BF16, 8, 8192, 4096, *noq,
                                    flags=farn.FARN_PLAN_FP8_OUT)[0] == "stage"
    finally:
        c.close()


# --------------------------------------------------- graphs and streams
@pytest.mark.parametrize("name,T", [("decode", 1), ("decode", 64), ("prefill", 2300),
                                    ("wide", 300), ("prefill_f32", 40)])
def test_cuda_graph_capture_and_replay(O, dev, name, T):
    """Calls captured in a CUDA graph (as the benchmark runs them, with
    programmatic dependent launch) give the oracle's results on replay,
    including after the inputs change in place between replays."""
    p = synth.workload(name)[0].with_T(T)
    xs, res, w = synth.device_inputs(p, dev)
    outs = tuple(torch.empty_like(res) for _ in range(3))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        farn.forward(xs, res, w, p.eps, out=outs)          # warm-up / module load
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        farn.forward(xs, res, w, p.eps, out=outs, stream=s)
        farn.forward(xs, res, w, p.eps, out=outs, stream=s)  # two dependent launches
    for k in range(2):
        if k:
            synth.fill_device(xs[0], 99, 0, p.x)            # new values, same buffers
            torch.cuda.synchronize()
        for o in outs:
            o.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert_parity([u16(t) for t in outs], oracle_rows(O, xs, res, w, p.eps),
                      f"graph replay {k} {name} T={T}")


def test_cuda_graph_quantised_and_moe(O, dev):
    """The NVFP4 and FP8 outputs and the staged MoE combine captured in one
    CUDA graph, replayed twice: the same bytes as eager calls."""
    p = synth.workload("prefill")[0].with_T(2100)
    xs, res, w = synth.device_inputs(p, dev)
    pm = _moe(2100, 8, 2048, seed=21)
    (ex, index, gates), mres, mw = synth.device_inputs(pm, dev)
    eager = [farn.forward_nvfp4(xs, res, w, p.eps, 168.0), farn.forward_quant(xs, res, w, p.eps),
             farn.moe_combine(ex, index, gates, mres, mw, pm.eps)]
    torch.cuda.synchronize()
    outs4 = tuple(torch.empty_like(t) for t in eager[0])
    outs8 = tuple(torch.empty_like(t) for t in eager[1])
    outsm = tuple(torch.empty_like(t) for t in eager[2])
    c = farn._context_for(0)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    ptrs = [x.data_ptr() for x in xs]
    with torch.cuda.graph(g, stream=s):
        assert farn.farn_forward_nvfp4(c.handle, ptrs, farn.FARN_BF16, p.W, res.data_ptr(),
                                       w.data_ptr(), p.eps, p.T, p.H, 168.0,
                                       *[t.data_ptr() for t in outs4], s.cuda_stream) == 0
        assert farn.farn_forward_quant(c.handle, ptrs, farn.FARN_BF16, p.W, res.data_ptr(),
                                       w.data_ptr(), p.eps, p.T, p.H,
                                       *[t.data_ptr() for t in outs8], s.cuda_stream) == 0
        farn.moe_combine(ex, index, gates, mres, mw, pm.eps, out=outsm, stream=s)
    for k in range(2):
        for t in outs4 + outs8 + outsm:
            t.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        for got, want in zip((outs4, outs8, outsm), eager):
            for a, b in zip(got, want):
                assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"replay {k}"


@pytest.mark.parametrize("variant", ["auto", "stage", "row", "bulk"])
def test_moe_combine_32_experts(O, dev, variant):
    """K = 32 (every lane of the routing registers in use), many rows per
    persistent CTA."""
    ctx = make_ctx(FARN_VARIANT=variant) if variant != "auto" else None
    try:
        _run_moe(O, dev, _moe(700, 32, 1024, seed=17), ctx=ctx, what=f"moe K=32 {variant}")
    finally:
        if ctx is not None:
            ctx.close()


def test_two_streams_concurrently(O, dev):
    """Independent calls on two streams at once (one long, one decode-sized)."""
    pa = synth.workload("prefill")[0].with_T(4096)
    pb = synth.workload("decode")[-1]
    a = synth.device_inputs(pa, dev)
    b = synth.device_inputs(pb, dev)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs_a, outs_b = [], []
    for _ in range(3):
        with torch.cuda.stream(s1):
            outs_a.append(farn.forward(*a, pa.eps))
        with torch.cuda.stream(s2):
            outs_b.append(farn.forward(*b, pb.eps))
    torch.cuda.synchronize()
    rows = sample_rows(pa.T, 64, seed=4)
    idx = torch.as_tensor(rows, device=dev)
    want_a = oracle_rows(O, *a, pa.eps, rows)
    want_b = oracle_rows(O, *b, pb.eps)
    for oa, ob in zip(outs_a, outs_b):
        assert_parity([u16(t.index_select(0, idx)) for t in oa], want_a, "stream 1")
        assert_parity([u16(t) for t in ob], want_b, "stream 2")


# ------------------------------------------------------ FP8 norm output
def _check_quant(O, xs, res, w, eps, red, ro, nrm, q, scale, what):
    """norm_out within 1 ulp of the oracle; given the GPU's norm_out, the
    E4M3 bytes and the row scales are unique: bit-exact against the
    oracle's quantisation of that norm_out (NaN by pattern class)."""
    assert_parity([u16(red), u16(ro), u16(nrm)], oracle_rows(O, xs, res, w, eps), what)
    want_q, want_s = O.quant_e4m3(u16(nrm))
    got_q = q.cpu().numpy()
    got_s = scale.cpu().numpy()
    assert np.array_equal(got_s.view(np.uint32), want_s.view(np.uint32)), what
    nan_w = (want_q & 0x7F) == 0x7F
    assert np.array_equal((got_q & 0x7F) == 0x7F, nan_w), what
    assert np.array_equal(np.where(nan_w, 0, got_q), np.where(nan_w, 0, want_q)), what


@pytest.mark.parametrize("name,T", [("decode", 1), ("decode", 5), ("decode", 64),
                                    ("prefill", 300), ("prefill", 2200), ("wide", 100),
                                    ("nonpow2", 77), ("prefill_f32", 9)])
def test_fp8_output(O, dev, name, T):
    p = synth.workload(name)[0].with_T(T)
    xs, res, w = synth.device_inputs(p, dev)
    red, ro, nrm, q, scale = farn.forward_quant(xs, res, w, p.eps)
    torch.cuda.synchronize()
    _check_quant(O, xs, res, w, p.eps, red, ro, nrm, q, scale, f"fp8 {name} T={T}")


@pytest.mark.parametrize("env", [dict(FARN_VARIANT="generic"), dict(FARN_CLUSTER=2),
                                 dict(FARN_CLUSTER=16), dict(FARN_VARIANT="row", FARN_VPT=4),
                                 dict(FARN_VARIANT="stage"), dict(FARN_VARIANT="stage", FARN_VPT=2),
                                 dict(FARN_VARIANT="stage", FARN_STAGE_CTAS=1)],
                         ids=lambda e: "-".join(f"{k[5:].lower()}{v}" for k, v in e.items()))
def test_fp8_output_forced_variants(O, dev, env):
    p = synth.Problem("q", 6, 7, 4096, 1e-6, 13, synth.N01)
    xs, res, w = synth.device_inputs(p, dev)
    ctx = make_ctx(**env)
    try:
        red, ro, nrm, q, scale = farn.forward_quant(xs, res, w, p.eps, ctx=ctx)
        torch.cuda.synchronize()
        _check_quant(O, xs, res, w, p.eps, red, ro, nrm, q, scale, f"fp8 {env}")
    finally:
        ctx.close()


def test_fp8_output_without_norm_out_and_specials(O, dev):
    """norm_out not written: the same E4M3 bytes and scales as with it;
    rows with a NaN, an overflow, all zeros and tiny values."""
    W, T, H = 4, 6, 1000                 # H % 8 != 0: generic kernel
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
    red, ro, nrm, q, scale = farn.forward_quant(xs, res, w, p.eps)
    red2, ro2, nrm2, q2, scale2 = farn.forward_quant(xs, res, w, p.eps, write_norm=False)
    torch.cuda.synchronize()
    assert nrm2 is None
    _check_quant(O, xs, res, w, p.eps, red, ro, nrm, q, scale, "fp8 specials")
    assert torch.equal(q, q2) and torch.equal(scale.view(torch.int32), scale2.view(torch.int32))
    assert scale[2].item() == 1.0 and not q[2].any()      # zero row


def test_fp8_output_vector_path_without_norm_out(O, dev):
    p = synth.workload("prefill")[0].with_T(500)
    xs, res, w = synth.device_inputs(p, dev)
    a = farn.forward_quant(xs, res, w, p.eps)
    b = farn.forward_quant(xs, res, w, p.eps, write_norm=False)
    torch.cuda.synchronize()
    _check_quant(O, xs, res, w, p.eps, *a, "fp8 with norm")
    assert torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])


@pytest.mark.parametrize("variant", ["bulk"])
def test_fp8_output_refused_by_staged_kernels(dev, variant):
    p = synth.Problem("q", 2, 4, 2048, 1e-6, 1, synth.N01)
    xs, res, w = synth.device_inputs(p, dev)
    ctx = make_ctx(FARN_VARIANT=variant)
    try:
        with pytest.raises(farn.FarnError) as e:
            farn.forward_quant(xs, res, w, p.eps, ctx=ctx)
        assert e.value.status == farn.FARN_ERR_UNSUPPORTED
    finally:
        ctx.close()


def test_fp8_output_aliasing(dev):
    p = synth.Problem("q", 2, 4, 2048, 1e-6, 1, synth.N01)
    xs, res, w = synth.device_inputs(p, dev)
    red, ro, nrm = (torch.empty_like(res) for _ in range(3))
    scale = torch.empty(4, dtype=torch.float32, device=dev)
    c = farn._context_for(0)
    # the E4M3 output over the reduced output: refused
    st = farn.farn_forward_quant(c.handle, [x.data_ptr() for x in xs], farn.FARN_BF16, 2,
                                 res.data_ptr(), w.data_ptr(), p.eps, 4, 2048, red.data_ptr(),
                                 ro.data_ptr(), nrm.data_ptr(), red.data_ptr(), scale.data_ptr())
    assert st == farn.FARN_ERR_ALIAS
    # a missing scale output: invalid
    q = torch.empty((4, 2048), dtype=torch.uint8, device=dev)
    st = farn.farn_forward_quant(c.handle, [x.data_ptr() for x in xs], farn.FARN_BF16, 2,
                                 res.data_ptr(), w.data_ptr(), p.eps, 4, 2048, red.data_ptr(),
                                 ro.data_ptr(), nrm.data_ptr(), q.data_ptr(), 0)
    assert st == farn.FARN_ERR_INVALID_ARG


# ---------------------------------------------------------- MoE combine
def _moe(T, K, H, seed=3):
    return synth.Problem("moe", K, T, H, 1e-6, seed, synth.N01, kind="moe_combine")


def _run_moe(O, dev, p, ins=None, rows=None, ctx=None, what=""):
    (ex, index, gates), res, w = ins if ins is not None else synth.device_inputs(p, dev)
    out = farn.moe_combine(ex, index, gates, res, w, p.eps, ctx=ctx)
    torch.cuda.synchronize()
    if rows is None:
        want = O.moe_combine(u16(ex), index.cpu().numpy(), gates.cpu().numpy(), u16(res),
                             u16(w), p.eps)
        got = [u16(t) for t in out]
    else:
        idx = torch.as_tensor(rows, device=dev)
        want = O.moe_combine(u16(ex), index.index_select(0, idx).cpu().numpy(),
                             gates.index_select(0, idx).cpu().numpy(),
                             u16(res.index_select(0, idx)), u16(w), p.eps)
        got = [u16(t.index_select(0, idx)) for t in out]
    return assert_parity(got, want, what or f"moe T={p.T} K={p.W} H={p.H}")


@pytest.mark.parametrize("T,K,H", [(1, 8, 7168), (5, 8, 4096), (64, 8, 7168), (300, 8, 7168),
                                   (200, 1, 2048), (40, 32, 1024), (9, 3, 1000), (3, 6, 13)])
def test_moe_combine(O, dev, T, K, H):
    _run_moe(O, dev, _moe(T, K, H))


def test_moe_combine_full_size_sampled(O, dev):
    p = synth.workload("moe_combine")[0]
    _run_moe(O, dev, p, rows=sample_rows(p.T, 96, seed=8))
    torch.cuda.empty_cache()


@pytest.mark.parametrize("env", [dict(FARN_VARIANT="generic"), dict(FARN_VPT=1),
                                 dict(FARN_VPT=2), dict(FARN_VPT=4), dict(FARN_VARIANT="stage"),
                                 dict(FARN_VARIANT="stage", FARN_VPT=2),
                                 dict(FARN_VARIANT="stage", FARN_VPT=4),
                                 dict(FARN_VARIANT="stage", FARN_STAGE_CTAS=1),
                                 dict(FARN_VARIANT="bulk"), dict(FARN_VARIANT="bulk", FARN_BULK_CTAS=1),
                                 dict(FARN_VARIANT="bulk", FARN_BULK_CTAS=2)],
                         ids=lambda e: "-".join(f"{k[5:].lower()}{v}" for k, v in e.items()))
def test_moe_combine_variants(O, dev, env):
    ctx = make_ctx(**env)
    try:
        _run_moe(O, dev, _moe(33, 8, 4096, seed=9), ctx=ctx, what=f"moe {env}")
    finally:
        ctx.close()


@pytest.mark.parametrize("T,K,H", [(40, 8, 4096), (37, 8, 7168), (19, 8, 8192), (23, 8, 12288),
                                   (9, 16, 7168), (5, 32, 16384), (11, 1, 2048)])
def test_moe_combine_bulk_segments(O, dev, T, K, H):
    """The TMA-staged combine over one segment of up to 512 consumer threads
    (H <= 4096), two of up to 512 (H = 7168, 8192), and more of at most 256
    (longer rows, or rows whose K + 1 inputs leave room for fewer stages)."""
    ctx = make_ctx(FARN_VARIANT="bulk")
    try:
        _run_moe(O, dev, _moe(T, K, H, seed=T + K), ctx=ctx, what=f"moe bulk T={T} K={K} H={H}")
    finally:
        ctx.close()


@pytest.mark.parametrize("variant", ["row", "stage", "bulk"])
def test_moe_combine_skipped_and_bad_slots(O, dev, variant):
    """-1 and out-of-range slots are skipped (never read); a token with no
    valid slot gets reduced = -0."""
    p = _moe(12, 6, 2048, seed=4)
    (ex, index, gates), res, w = synth.device_inputs(p, dev)
    index[0, 1] = -1
    index[1, :] = -1
    index[2, 3] = ex.shape[0]            # one past the end
    index[3, 0] = 2 ** 31 - 1
    index[4, 5] = -7
    ctx = make_ctx(FARN_VARIANT=variant)
    try:
        _run_moe(O, dev, p, ins=((ex, index, gates), res, w), ctx=ctx,
                 what=f"moe bad slots {variant}")
    finally:
        ctx.close()


@pytest.mark.parametrize("variant", ["auto", "stage", "stage-vpt4", "bulk"])
def test_moe_combine_mid_size(O, dev, variant):
    """Many rows per persistent CTA for the staged gather kernel (its
    two-vector build, which reads the weight per row, and its four-vector
    build, which holds it in registers)."""
    env = dict(FARN_VARIANT="stage", FARN_VPT=4) if variant == "stage-vpt4" else \
        dict(FARN_VARIANT=variant)
    ctx = make_ctx(**env)
    try:
        _run_moe(O, dev, _moe(2100, 8, 7168, seed=14), ctx=ctx, what=f"moe {variant}")
    finally:
        ctx.close()


def test_moe_combine_plan(dev):
    """Long inputs take the TMA-staged kernel while a row fits two segments
    of at most 512 consumer threads, else the staged gather kernel; shorter
    ones one CTA per row, odd alignments the generic kernel; FARN_VARIANT
    forces each."""
    c = farn._context_for(0)
    # long from 2048 rows, or from 1024 rows reading >= 128 MiB
    for T, K, H, want in ((4096, 8, 7168, "bulk"), (2047, 8, 7168, "bulk"),
                          (1100, 8, 7168, "bulk"), (1000, 8, 7168, "combine"),
                          (1, 8, 7168, "combine"), (2048, 8, 4096, "bulk"),
                          (2048, 8, 12288, "bulk"),      # 6 segments of the full 256
                          (2048, 16, 7168, "stage"),     # 4 segments of only 224
                          (2048, 4, 4096, "combine"),    # short rows, few experts
                          (2048, 8, 3072, "combine")):   # short rows
        p = _moe(T, K, H)
        (ex, index, gates), res, w = synth.device_inputs(p, dev)
        outs = [torch.empty_like(res) for _ in range(3)]
        v, thr = farn.farn_plan_moe_combine(c.handle, K, T, p.H, ex.data_ptr(), res.data_ptr(),
                                            w.data_ptr(), *[o.data_ptr() for o in outs])
        assert v == want, (T, K, H, v)
        assert 32 <= thr <= 544
        if want == "bulk":
            # one producer warp and 896 / 2 (H = 7168), 512 (H = 4096) or the
            # full 256 (H = 12288) consumers
            assert thr == 32 + {7168: 448, 4096: 512, 12288: 256}[H], (T, H, thr)
        if want == "stage":
            # two vectors per thread where that fits 512 threads, else four
            nt2 = 32 * ((H // 16 + 31) // 32)
            assert thr == (nt2 if nt2 <= 512 else 32 * ((H // 32 + 31) // 32)), (T, H, thr)
        if T == 4096:
            v, _ = farn.farn_plan_moe_combine(c.handle, 8, T, p.H, ex.data_ptr() + 2,
                                              res.data_ptr(), w.data_ptr(),
                                              *[o.data_ptr() for o in outs])
            assert v == "generic"
            for env, want_v in ((dict(FARN_VARIANT="row"), "combine"),
                                (dict(FARN_VARIANT="generic"), "generic"),
                                (dict(FARN_VARIANT="stage"), "stage"),
                                (dict(FARN_STAGE=0), "combine"),
                                (dict(FARN_VARIANT="bulk"), "bulk"),
                                (dict(FARN_BULK=1), "bulk")):
                ctx = make_ctx(**env)
                try:
                    v, _ = farn.farn_plan_moe_combine(ctx.handle, 8, T, p.H, ex.data_ptr(),
                                                      res.data_ptr(), w.data_ptr(),
                                                      *[o.data_ptr() for o in outs])
                    assert v == want_v, (env, v)
                finally:
                    ctx.close()
        del ex, index, gates, res, w, outs
    torch.cuda.empty_cache()


def test_moe_combine_unit_gates_match_forward(O, dev):
    """Gates of 1 and the slot layout of stacked partials: the combine and
    the rank-sum kernel give the same bits."""
    T, K, H = 50, 4, 4096
    p = synth.Problem("x", K, T, H, 1e-6, 6, synth.N01)
    xs, res, w = synth.device_inputs(p, dev)
    ex = torch.cat(xs, dim=0).contiguous()
    index = torch.tensor([[k * T + t for k in range(K)] for t in range(T)], dtype=torch.int32,
                         device=dev)
    gates = torch.ones((T, K), dtype=torch.float32, device=dev)
    a = farn.moe_combine(ex, index, gates, res, w, 1e-6)
    b = farn.forward(xs, res, w, 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert compare([u16(t) for t in a], [u16(t) for t in b])["norm_out"]["max_ulp"] <= 1


def test_moe_combine_in_place_and_aliasing(O, dev):
    p = _moe(20, 4, 2048, seed=12)
    (ex, index, gates), res, w = synth.device_inputs(p, dev)
    want = O.moe_combine(u16(ex), index.cpu().numpy(), gates.cpu().numpy(), u16(res), u16(w),
                         p.eps)
    red, nrm = torch.empty_like(res), torch.empty_like(res)
    farn.moe_combine(ex, index, gates, res, w, p.eps, out=(red, res, nrm))
    torch.cuda.synchronize()
    assert_parity([u16(red), u16(res), u16(nrm)], want, "moe in place")
    with pytest.raises(farn.FarnError) as e:       # output over an expert row
        farn.moe_combine(ex, index, gates, res, w, p.eps, out=(ex[:20], red, nrm))
    assert e.value.status == farn.FARN_ERR_ALIAS


@pytest.mark.parametrize("name", ["prefill", "wide", "prefill_f32"])
def test_synth_device_fill_matches_host_twin(dev, name):
    """The device generator and its numpy twin follow one recipe: the same
    bytes, up to a rare last-bit difference of the fp64 transcendental
    functions surviving the rounding to fp32 (and bf16)."""
    p = synth.workload(name)[0].with_T(128)
    xs_d, res_d, w_d = synth.device_inputs(p, dev)
    xs_h, res_h, w_h = synth.host_inputs(p)
    pairs = [(host(x), xh) for x, xh in zip(xs_d, xs_h)] + [(u16(res_d), res_h), (u16(w_d), w_h)]
    n = bad = 0
    for a, b in pairs:
        a, b = np.asarray(a).ravel(), np.asarray(b).ravel()
        assert a.shape == b.shape
        n += a.size
        bad += int(np.count_nonzero(a.view(np.uint16 if a.dtype == np.uint16 else np.uint32)
                                    != b.view(np.uint16 if b.dtype == np.uint16 else np.uint32)))
    assert bad <= max(2, n // 100000), f"{bad} of {n} generated values differ"


def test_prepared_calls_reuse_their_buffers(O, dev):
    """A prepared call, launched again after its inputs change in place,
    gives the oracle's results each time; the prepared FP8, NVFP4 and MoE
    calls give the same bytes as the immediate functions."""
    p = synth.workload("prefill")[0].with_T(300)
    xs, res, w = synth.device_inputs(p, dev)
    call = farn.prepare_forward(xs, res, w, p.eps)
    for k in range(2):
        if k:
            synth.fill_device(xs[1], 77, 1, p.x)
        out = call()
        torch.cuda.synchronize()
        assert_parity([u16(t) for t in out], oracle_rows(O, xs, res, w, p.eps), f"prepared {k}")
    q8 = farn.prepare_forward_quant(xs, res, w, p.eps)()
    q4 = farn.prepare_forward_nvfp4(xs, res, w, p.eps, 168.0, write_norm=False)()
    a8 = farn.forward_quant(xs, res, w, p.eps)
    a4 = farn.forward_nvfp4(xs, res, w, p.eps, 168.0, write_norm=False)
    pm = _moe(200, 8, 2048, seed=5)
    (ex, index, gates), mres, mw = synth.device_inputs(pm, dev)
    m1 = farn.prepare_moe_combine(ex, index, gates, mres, mw, pm.eps)()
    m2 = farn.moe_combine(ex, index, gates, mres, mw, pm.eps)
    torch.cuda.synchronize()
    for got, want in ((q8, a8), (q4, a4), (m1, m2)):
        for a, b in zip(got, want):
            assert (a is None and b is None) or torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    with pytest.raises(ValueError):
        bad = (q8[0], q8[1], q8[2], q8[3][:, :10], q8[4])   # codes of the wrong shape
        farn.prepare_forward_quant(xs, res, w, p.eps, out=bad)
