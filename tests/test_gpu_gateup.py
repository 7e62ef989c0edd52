"""Gate||up GEMV with the fused SwiGLU -> q8 epilogue, through the C ABI.

Bar: act and its q8 plane identical, bit for bit, to the three-launch chain
GEMV(gate), GEMV(up) (whole-tile plan) and mq_swiglu_quant_q8; act against
the oracle chain within the bound the GEMV tolerance implies; the q8 plane
equal to the oracle quantizer applied to the act the kernel wrote.
"""
import os

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
TOL = 1e-4


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


def setup(mq, fmt, rows, cols, seed):
    g = synth.rng("gateup", fmt, rows, cols, seed)
    Wg = synth.blocks(fmt, g, rows, cols)
    Wu = synth.blocks(fmt, g, rows, cols)
    x, gain = synth.normal(g, cols), synth.normal(g, cols, 1.0, 0.1)
    _, plane = mq.mq_rmsnorm_quant_q8(dev(x), dev(gain), 1e-6)
    return Wg, Wu, dev(mq.mq_repack(fmt, Wg, rows, cols)), dev(mq.mq_repack(fmt, Wu, rows, cols)), plane


def fields(mq, plane, n):
    """(d, codes, sums) of a q8 plane: the padding between its sections is
    not part of the plane's value."""
    return mq.mq_q8_unpack_host(host(plane), n)


def same_plane(mq, a, b, n):
    return all(np.array_equal(x, y) for x, y in zip(fields(mq, a, n), fields(mq, b, n)))


def unfused(mq, fmt, Wgp, Wup, plane, rows, cols):
    nch = -(-(cols // 256) // 4)
    yg = mq.mq_gemv(fmt, Wgp, plane, rows, cols, plan=(1, nch, 1))
    yu = mq.mq_gemv(fmt, Wup, plane, rows, cols, plan=(1, nch, 1))
    return mq.mq_swiglu_quant_q8(yg, yu)


SHAPES = [("q4k", 13824, 5120), ("q4k", 18944, 3584), ("q6k", 256, 18944), ("q4k", 32, 1280),
          ("q6k", 96, 4608), ("q5k", 13824, 5120), ("q5k", 64, 2304)]


@pytest.mark.parametrize("fmt,rows,cols", SHAPES)
def test_fused_equals_three_launches_bitwise(mq, fmt, rows, cols):
    Wg, Wu, Wgp, Wup, plane = setup(mq, fmt, rows, cols, 0)
    act, q8 = mq.mq_gemv_gateup_swiglu_q8(fmt, Wgp, Wup, plane, rows, cols)
    act2, q82 = unfused(mq, fmt, Wgp, Wup, plane, rows, cols)
    assert np.array_equal(host(act), host(act2))
    assert same_plane(mq, q8, q82, rows)


@pytest.mark.parametrize("fmt", ["q4k", "q6k", "q5k"])
def test_every_plan_gives_the_same_bits(mq, fmt):
    rows, cols = 320, 2304                        # 10 blocks of 32 rows; 9 super-blocks: 3 chunks
    Wg, Wu, Wgp, Wup, plane = setup(mq, fmt, rows, cols, 1)
    ref_act, ref_q8 = unfused(mq, fmt, Wgp, Wup, plane, rows, cols)
    ref_act = host(ref_act)
    for w in range(1, 9):
        for ctas in (1, 3, 7, 10):
            act, q8 = mq.mq_gemv_gateup_swiglu_q8(fmt, Wgp, Wup, plane, rows, cols, plan=(w, ctas))
            assert np.array_equal(host(act), ref_act), (w, ctas)
            assert same_plane(mq, q8, ref_q8, rows), (w, ctas)


@pytest.mark.parametrize("fmt,rows,cols", [("q4k", 13824, 5120), ("q6k", 96, 4608), ("q5k", 320, 2304)])
def test_fused_against_the_oracle_chain(mq, orc, fmt, rows, cols):
    Wg, Wu, Wgp, Wup, plane = setup(mq, fmt, rows, cols, 2)
    act, q8 = mq.mq_gemv_gateup_swiglu_q8(fmt, Wgp, Wup, plane, rows, cols)
    acth = host(act)
    d, q, _ = mq.mq_q8_unpack_host(host(plane), cols)
    th = len(os.sched_getaffinity(0))
    g, ag = orc.gemv(fmt, Wg, d, q, rows, cols, threads=th)
    u, au = orc.gemv(fmt, Wu, d, q, rows, cols, threads=th)
    ref = orc.swiglu(g.astype(np.float32), u.astype(np.float32))
    # |d act| <= |silu'(g)| |u| |dg| + |silu(g)| |du| with |silu'| < 1.1 and
    # |dg| <= 1e-4 sum|terms| (the GEMV bound), plus f32 rounding of act
    silu = g / (1.0 + np.exp(-g))
    bound = 1.1 * np.abs(u) * TOL * ag + np.abs(silu) * TOL * au + 1e-6 * np.abs(ref) + 1e-30
    assert np.all(np.abs(acth - ref) <= bound), float(np.max(np.abs(acth - ref) / bound))
    d0, q0, s0 = orc.quantize_q8(acth)
    d1, q1, s1 = mq.mq_q8_unpack_host(host(q8), rows)
    assert np.array_equal(d0, d1) and np.array_equal(q0, q1) and np.array_equal(s0, s1)


def test_bad_calls_are_refused_and_nothing_runs(mq):
    import torch
    fmt, rows, cols = "q4k", 64, 1024
    Wg, Wu, Wgp, Wup, plane = setup(mq, fmt, rows, cols, 3)
    act = torch.full((rows,), 5.0, device="cuda")
    for plan in [(0, 1), (9, 1), (4, 0), (4, 3)]:          # rows / 32 = 2 blocks
        with pytest.raises(mq.MQError) as e:
            mq.mq_gemv_gateup_swiglu_q8(fmt, Wgp, Wup, plane, rows, cols, act=act, plan=plan)
        assert e.value.status == mq.MQ_ERR_COVERAGE, plan
    with pytest.raises(mq.MQError) as e:
        mq.mq_gemv_gateup_swiglu_q8(fmt, Wgp[: Wgp.numel() // 2], Wup, plane, 48, cols, act=act[:48],
                                    q8_out=torch.empty(128, dtype=torch.uint8, device="cuda"))
                                                        # 48 rows: not whole q8 blocks
    assert e.value.status == mq.MQ_ERR_SHAPE
    assert torch.all(act == 5.0)


def test_pdl_chain_with_the_fused_kernel(mq):
    """rms -> fused gate||up -> down, 8 steps, with and without PDL and
    under graph capture: identical outputs."""
    import torch
    h, i = 2048, 5376
    g = synth.rng("gateup-chain")
    Wg = dev(mq.mq_repack_q4k(synth.q4k_blocks(g, i, h), i, h))
    Wu = dev(mq.mq_repack_q4k(synth.q4k_blocks(g, i, h), i, h))
    Wd = dev(mq.mq_repack_q6k(synth.q6k_blocks(g, h, i), h, i))
    gain = dev(synth.normal(g, h, 1.0, 0.1))
    xs = [dev(synth.normal(g, h)) for _ in range(8)]
    x = torch.empty(h, device="cuda")
    xn = torch.empty(h, device="cuda")
    qa = torch.empty(mq.mq_q8_bytes(h), dtype=torch.uint8, device="cuda")
    act = torch.empty(i, device="cuda")
    qb = torch.empty(mq.mq_q8_bytes(i), dtype=torch.uint8, device="cuda")
    out = torch.empty(h, device="cuda")
    wsd = mq.mq_gemv_workspace(h, i)

    def step():
        mq.mq_rmsnorm_quant_q8(x, gain, 1e-6, y=xn, q8=qa)
        mq.mq_gemv_gateup_swiglu_q8("q4k", Wg, Wu, qa, i, h, act=act, q8_out=qb)
        mq.mq_gemv_q6k_q8(Wd, qb, h, i, y=out, ws=wsd)

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
        got = run(pdl, graph)
        for a, b in zip(ref, got):
            assert np.array_equal(a, b), (pdl, graph)
