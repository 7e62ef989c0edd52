"""The single-token GEMV's weight ring (mq_set_gemv_ring): every depth, with
every number of stages requested before the grid-dependency wait, gives the
bits of the register-only path (stages 0) under the same explicit plan --
whole tiles, CTA splits and workspace splits, every format, ragged rows and
chunks, groups of mixed formats -- and each default plan stays within the
parity bar of the oracle (|dy| <= 1e-4 * sum |terms| per row)."""
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
    m.mq_set_gemv_ring(-1, -1)
    m.mq_set_pdl(False)


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


RINGS = [(1, 0), (1, 1), (2, 0), (2, 1), (2, 2), (3, 1), (3, 3)]
SHAPES = [  # fmt, rows, cols, explicit plans (splits, chunks_per_split, tiles_per_item)
    ("q6k", 61, 4864, [(1, 5, 1), (1, 5, 3), (3, 2, 1), (5, 1, 1)]),
    ("q4k", 100, 3328, [(1, 4, 2), (2, 2, 1), (4, 1, 1)]),
    ("q5k", 37, 5120, [(1, 5, 1), (3, 2, 1), (5, 1, 1)]),
    ("q6k", 24, 18944, [(1, 19, 1), (10, 2, 1), (19, 1, 1)]),   # 19 splits meet in the workspace
    ("q4k", 16, 16384, [(16, 1, 1), (8, 2, 1), (1, 16, 2)]),
]


@pytest.mark.parametrize("fmt,rows,cols,plans", SHAPES)
def test_ring_bits_equal_register_path(mq, orc, fmt, rows, cols, plans):
    g = synth.rng("ring", fmt, rows, cols)
    W = synth.blocks(fmt, g, rows, cols)
    Wp = dev(mq.mq_repack(fmt, W, rows, cols))
    x = synth.normal(g, cols)
    plane = mq.mq_quantize_q8(dev(x))
    d, q, _ = orc.quantize_q8(x)
    yref, absum = orc.gemv(fmt, W, d, q, rows, cols, threads=8)
    for plan in plans:
        ws = mq.mq_gemv_workspace(rows, cols, plan=plan)
        mq.mq_set_gemv_ring(0, 0)
        base = mq.mq_gemv(fmt, Wp, plane, rows, cols, ws=ws, plan=plan).cpu().numpy()
        assert np.all(np.abs(base.astype(np.float64) - yref) <= TOL * absum), plan
        for st, pre in RINGS:
            mq.mq_set_gemv_ring(st, pre)
            y = mq.mq_gemv(fmt, Wp, plane, rows, cols, ws=ws, plan=plan).cpu().numpy()
            assert np.array_equal(y, base), (plan, st, pre)
    mq.mq_set_gemv_ring(-1, -1)


@pytest.mark.parametrize("st,pre", [(0, 0), (1, 1), (2, 1), (3, 3), (-1, -1)])
@pytest.mark.parametrize("fmt,rows,cols", [("q6k", 3584, 18944), ("q4k", 5120, 5120),
                                           ("q4k", 13824, 5120), ("q6k", 1024, 5120)])
def test_default_plans_at_every_depth(mq, orc, st, pre, fmt, rows, cols):
    """The default plan a depth leads to (its shared memory changes the
    occupancy) is checked on every row against the oracle."""
    import os
    mq.mq_set_gemv_ring(st, pre)
    try:
        g = synth.rng("ring-default", fmt, rows, cols)
        W = synth.blocks(fmt, g, rows, cols)
        Wp = dev(mq.mq_repack(fmt, W, rows, cols))
        x = synth.normal(g, cols)
        plane = mq.mq_quantize_q8(dev(x))
        ws = mq.mq_gemv_workspace(rows, cols)
        y1 = mq.mq_gemv(fmt, Wp, plane, rows, cols, ws=ws).cpu().numpy()
        y2 = mq.mq_gemv(fmt, Wp, plane, rows, cols, ws=ws).cpu().numpy()
        assert np.array_equal(y1, y2)
        d, q, _ = orc.quantize_q8(x)
        yref, absum = orc.gemv(fmt, W, d, q, rows, cols, threads=len(os.sched_getaffinity(0)))
        assert np.all(np.abs(y1.astype(np.float64) - yref) <= TOL * absum)
    finally:
        mq.mq_set_gemv_ring(-1, -1)


def test_grouped_mixed_formats_with_ring(mq, orc):
    """q, k, v of a layer in one launch (q4_K, q4_K, q6_K: slots sized for
    q6_K) under every ring depth: the bits of the register-only path."""
    import torch
    g = synth.rng("ring-group")
    cols = 2560
    spec = [("q4k", 136), ("q4k", 40), ("q6k", 40)]
    Ws = [synth.blocks(f, g, r, cols) for f, r in spec]
    Wps = [dev(mq.mq_repack(f, W, r, cols)) for (f, r), W in zip(spec, Ws)]
    x = synth.normal(g, cols)
    plane = mq.mq_quantize_q8(dev(x))
    parts = [(f, Wp, r) for (f, r), Wp in zip(spec, Wps)]

    def run():
        ys = [torch.empty(r, device="cuda") for _, r in spec]
        ws = mq.mq_gemv_group_workspace(parts, cols, plan=(3, 1, 1))
        mq.mq_gemv_group_q8(parts, plane, cols, ys=ys, ws=ws, plan=(3, 1, 1))
        return [y.cpu().numpy() for y in ys]

    mq.mq_set_gemv_ring(0, 0)
    base = run()
    d, q, _ = orc.quantize_q8(x)
    for (f, r), W, y in zip(spec, Ws, base):
        yref, absum = orc.gemv(f, W, d, q, r, cols)
        assert np.all(np.abs(y.astype(np.float64) - yref) <= TOL * absum)
    for st, pre in RINGS:
        mq.mq_set_gemv_ring(st, pre)
        for a, b in zip(run(), base):
            assert np.array_equal(a, b), (st, pre)
    mq.mq_set_gemv_ring(-1, -1)


def test_ring_under_pdl_graph(mq, orc):
    """quantize -> GEMV steps captured in one graph with PDL, every ring
    depth: each step's output equals the eager no-PDL register-path run."""
    import torch
    rows, cols = 2048, 4864
    g = synth.rng("ring-pdl")
    W = synth.q6k_blocks(g, rows, cols)
    Wp = dev(mq.mq_repack_q6k(W, rows, cols))
    xs = [dev(synth.normal(g, cols)) for _ in range(6)]
    x = torch.empty(cols, device="cuda")
    plane = torch.empty(mq.mq_q8_bytes(cols), dtype=torch.uint8, device="cuda")
    y = torch.empty(rows, device="cuda")
    ws = mq.mq_gemv_workspace(rows, cols)

    def step():
        mq.mq_quantize_q8(x, q8=plane)
        mq.mq_gemv_q6k_q8(Wp, plane, rows, cols, y=y, ws=ws)

    def run(pdl, graph):
        mq.mq_set_pdl(pdl)
        outs = []
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
                outs.append(y.clone())
        torch.cuda.synchronize()
        mq.mq_set_pdl(False)
        return [o.cpu().numpy() for o in outs]

    mq.mq_set_gemv_ring(0, 0)
    ref = run(False, False)
    for st, pre in ((1, 1), (2, 2), (2, 0), (3, 3)):
        mq.mq_set_gemv_ring(st, pre)
        # the same plan at every depth?  compare against the oracle when not
        splits = mq.mq_gemv_plan(rows, cols, "q6k")
        got = run(True, True)
        mq.mq_set_gemv_ring(0, 0)
        same_plan = mq.mq_gemv_plan(rows, cols, "q6k") == splits
        for i, (a, b) in enumerate(zip(ref, got)):
            if same_plan:
                assert np.array_equal(a, b), (st, pre, i)
            d, q, _ = orc.quantize_q8(xs[i].cpu().numpy())
            yref, absum = orc.gemv("q6k", W, d, q, rows, cols, threads=8)
            assert np.all(np.abs(b.astype(np.float64) - yref) <= TOL * absum), (st, pre, i)
    mq.mq_set_gemv_ring(-1, -1)
