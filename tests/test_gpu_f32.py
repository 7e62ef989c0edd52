"""The q6_K GEMV against an f32 activation row (the dequantize-and-FMA
family of the D3 page, §2.3 and §3.3), through the C ABI, against the oracle.

Bar, derived from the kernel's f32 arithmetic: every product (q - 32) * x
and every partial sum rounds once; per row the longest chain is a 16-term
sub-block FMA chain, two FMAs per chunk a warp streams, the lane butterfly
and the split combine.  So

    |y_gpu - y_oracle| <= (2 * nchunks + 64) * 2^-24 * sum_e |w_e x_e|

which stays below the 1e-4 * sum |terms| bar of the q8 GEMV at every
shape the kernel accepts.
"""
import os

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
U = 2.0 ** -24


@pytest.fixture(scope="module")
def mq():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quant_quantized_gemv_gb300 import build
    build.build()
    import quant_quantized_gemv_gb300 as m
    m.lib()
    yield m
    m.mq_set_pdl(False)


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    import torch
    torch.cuda.synchronize()
    return t.cpu().numpy()


def threads():
    return len(os.sched_getaffinity(0))


def bound(cols, absum):
    nchunks = -(-(cols // 256) // 4)
    return (2 * nchunks + 64) * U * absum + 1e-30


def check(y, ref, absum, cols):
    err = np.abs(y.astype(np.float64) - ref)
    b = bound(cols, absum)
    assert np.all(err <= b), float(np.max(err / b))


def setup(mq, rows, cols, tag, xs=1.0):
    g = synth.rng("f32", tag, rows, cols)
    W = synth.q6k_blocks(g, rows, cols)
    x = (synth.normal(g, cols) * np.float32(xs)).astype(np.float32)
    return W, x, dev(mq.mq_repack_q6k(W, rows, cols)), dev(x)


SHAPES = [(512, 2048), (1024, 5120), (2048, 4864), (37, 1280), (1, 256), (8, 2304), (3584, 18944),
          (13, 56576), (152064, 5120)]


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_default_plan_against_oracle(mq, orc, rows, cols):
    W, x, Wp, xd = setup(mq, rows, cols, "default")
    y = host(mq.mq_gemv_q6k_f32(Wp, xd, rows, cols))
    ref, absum = orc.gemv_q6k_f32(W, x, rows, cols, threads=threads())
    check(y, ref, absum, cols)


def test_outlier_magnitudes(mq, orc):
    """Activations spanning ~2^40 (a few huge, many tiny), as the D3a page's
    tolerance check uses outlier-magnitude data."""
    rows, cols = 96, 4096
    W, x, _, _ = setup(mq, rows, cols, "outlier")
    g = synth.rng("f32-outlier")
    big = g.integers(0, cols, 16)
    x = (x * np.float32(1e-6)).astype(np.float32)
    x[big] = np.float32(1e6)
    Wp, xd = dev(mq.mq_repack_q6k(W, rows, cols)), dev(x)
    y = host(mq.mq_gemv_q6k_f32(Wp, xd, rows, cols))
    ref, absum = orc.gemv_q6k_f32(W, x, rows, cols)
    check(y, ref, absum, cols)


def test_every_plan(mq, orc):
    rows, cols = 40, 256 * 11            # 5 tiles, 3 chunks (the last of 3 super-blocks)
    W, x, Wp, xd = setup(mq, rows, cols, "plans")
    ref, absum = orc.gemv_q6k_f32(W, x, rows, cols)
    whole = None
    for tpi in range(1, 6):
        y = host(mq.mq_gemv_q6k_f32(Wp, xd, rows, cols, plan=(1, 3, tpi)))
        check(y, ref, absum, cols)
        if whole is None:
            whole = y
        assert np.array_equal(y, whole), tpi  # same order of additions per row
    for splits, cps in ((2, 2), (3, 1)):
        y = host(mq.mq_gemv_q6k_f32(Wp, xd, rows, cols, plan=(splits, cps, 1)))
        check(y, ref, absum, cols)


def test_twelve_splits_and_default_cap(mq, orc):
    rows, cols = 16, 256 * 4 * 48         # 2 tiles of 48 chunks
    W, x, Wp, xd = setup(mq, rows, cols, "cap")
    ref, absum = orc.gemv_q6k_f32(W, x, rows, cols)
    s, c, t = mq.mq_gemv_q6k_f32_plan_of(rows, cols)
    assert 1 <= s <= 12 and (s - 1) * c < 48 <= s * c
    check(host(mq.mq_gemv_q6k_f32(Wp, xd, rows, cols)), ref, absum, cols)
    check(host(mq.mq_gemv_q6k_f32(Wp, xd, rows, cols, plan=(12, 4, 1))), ref, absum, cols)


def test_agrees_with_q8_path_on_q8_values(mq, orc):
    """x = f16(d8) * q8 exactly: both GEMVs compute the same real number."""
    rows, cols = 256, 5120
    W, x, Wp, _ = setup(mq, rows, cols, "q8vals")
    d8, q8, _ = orc.quantize_q8(x)
    xh = (np.repeat(np.array([orc.f16_to_f32(h) for h in d8]), 32) * q8).astype(np.float32)
    y32 = host(mq.mq_gemv_q6k_f32(Wp, dev(xh), rows, cols))
    plane = mq.mq_quantize_q8(dev(x))
    y8 = host(mq.mq_gemv_q6k_q8(Wp, plane, rows, cols, ws=mq.mq_gemv_workspace(rows, cols)))
    ref, absum = orc.gemv_q6k_f32(W, xh, rows, cols)
    check(y32, ref, absum, cols)
    assert np.all(np.abs(y8.astype(np.float64) - ref) <= 1e-4 * absum + 1e-30)


def test_bad_calls_are_refused_and_nothing_runs(mq):
    import torch
    rows, cols = 24, 256 * 9
    W, x, Wp, xd = setup(mq, rows, cols, "bad")
    y = torch.full((rows,), 7.0, device="cuda")
    for plan in [(13, 1, 1), (2, 1, 1), (4, 1, 1), (1, 2, 1), (2, 2, 2), (0, 3, 1)]:
        with pytest.raises(mq.MQError) as e:
            mq.mq_gemv_q6k_f32(Wp, xd, rows, cols, y=y, plan=plan)
        assert e.value.status == mq.MQ_ERR_COVERAGE, plan
    big = 256 * 228                        # 233472 bytes of f32: more than one CTA stages
    Wb = dev(mq.mq_repack_q6k(synth.q6k_blocks(synth.rng("f32-big"), 8, big), 8, big))
    with pytest.raises(mq.MQError) as e:
        mq.mq_gemv_q6k_f32(Wb, torch.zeros(big, device="cuda"), 8, big, y=y[:8])
    assert e.value.status == mq.MQ_ERR_SHAPE
    buf = torch.zeros(cols + 4, device="cuda")
    with pytest.raises(mq.MQError) as e:
        mq.mq_gemv_q6k_f32(Wp, buf[1:1 + cols], rows, cols, y=y)
    assert e.value.status == mq.MQ_ERR_ALIGN
    with pytest.raises(mq.MQError) as e:
        mq.mq_gemv_q6k_f32(Wp, xd, rows, 1000, y=y)
    assert e.value.status == mq.MQ_ERR_SHAPE
    assert torch.all(y == 7.0)


@pytest.mark.parametrize("h,rows", [(5120, 1024), (1024, 20000)])   # split CTAs; whole tiles
def test_pdl_chain_with_the_rms_producer(mq, h, rows):
    """rms_norm (its f32 output) -> f32 GEMV, 6 steps, with and without PDL
    and under graph capture: identical outputs."""
    import torch
    s, _, _ = mq.mq_gemv_q6k_f32_plan_of(rows, h)
    assert (s == 1) == (rows == 20000)
    g = synth.rng("f32-chain")
    Wp = dev(mq.mq_repack_q6k(synth.q6k_blocks(g, rows, h), rows, h))
    gain = dev(synth.normal(g, h, 1.0, 0.1))
    xs = [dev(synth.normal(g, h)) for _ in range(6)]
    x = torch.empty(h, device="cuda")
    xn = torch.empty(h, device="cuda")
    qa = torch.empty(mq.mq_q8_bytes(h), dtype=torch.uint8, device="cuda")
    out = torch.empty(rows, device="cuda")

    def step():
        mq.mq_rmsnorm_quant_q8(x, gain, 1e-6, y=xn, q8=qa)
        mq.mq_gemv_q6k_f32(Wp, xn, rows, h, y=out)

    def run(pdl, graph):
        mq.mq_set_pdl(pdl)
        res = []
        st = torch.cuda.Stream()
        with torch.cuda.stream(st):
            if graph:
                x.copy_(xs[0])
                step()
                torch.cuda.synchronize()
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr, stream=st):
                    step()
            for xi in xs:
                x.copy_(xi)
                gr.replay() if graph else step()
                res.append(out.clone())
        torch.cuda.synchronize()
        mq.mq_set_pdl(False)
        return [r.cpu().numpy() for r in res]

    ref = run(False, False)
    for pdl, graph in ((True, False), (False, True), (True, True)):
        for a, b in zip(ref, run(pdl, graph)):
            assert np.array_equal(a, b), (pdl, graph)
