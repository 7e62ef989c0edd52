"""Device-side coverage: the GEMV's own work decomposition, run by the kernel,
touches every (tile, chunk) unit exactly once, for every kind of plan (whole
tiles with several tiles per warp, CTA splits, workspace splits), for groups
of parts with mixed formats, and at the benchmark shapes' default plans.
Its outputs equal the plain GEMV's bit for bit (the count is a side effect)."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mq():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quant_quantized_gemv_gb300 import build
    build.build()
    import quant_quantized_gemv_gb300 as m
    m.lib()
    return m


def setup(mq, specs, cols, seed):
    import torch
    g = synth.rng("cover", cols, seed, len(specs))
    parts = []
    for fmt, rows in specs:
        W = synth.blocks(fmt, g, rows, cols)
        parts.append((fmt, torch.from_numpy(mq.mq_repack(fmt, W, rows, cols)).cuda(), rows))
    plane = mq.mq_quantize_q8(torch.from_numpy(synth.normal(g, cols)).cuda())
    return parts, plane


def check(mq, parts, plane, cols, plan):
    import torch
    spec = [(f, W, r) for f, W, r in parts]
    ws = mq.mq_gemv_group_workspace(spec, cols, plan=plan)
    ys, counts = mq.mq_gemv_group_q8_coverage(spec, plane, cols, ws=ws, plan=plan)
    ref = mq.mq_gemv_group_q8(spec, plane, cols, ws=ws, plan=plan)
    torch.cuda.synchronize()
    c = counts.cpu().numpy()
    assert np.all(c == 1), (plan, int(c.min()), int(c.max()), int((c != 1).sum()))
    for a, b in zip(ys, ref):
        assert torch.equal(a, b)


@pytest.mark.parametrize("cols", [256, 2304, 4864, 18944])
def test_every_plan_of_one_matrix(mq, cols):
    rows = 41                                    # 6 tiles, the last ragged
    parts, plane = setup(mq, [("q6k", rows)], cols, 0)
    nch = -(-(cols // 256) // 4)
    plans = [None] + [(1, nch, t) for t in (1, 2, 4, 6)]
    for s in range(2, nch + 1):
        cps = -(-nch // s)
        if (s - 1) * cps < nch:
            plans.append((s, cps, 1))            # CTA splits (<= 12) and workspace splits (> 12)
    for plan in plans:
        check(mq, parts, plane, cols, plan)


def test_groups_of_mixed_formats(mq):
    cols = 5120
    parts, plane = setup(mq, [("q4k", 5120), ("q4k", 1024), ("q6k", 1024), ("q5k", 24)], cols, 1)
    for plan in [None, (1, 5, 1), (1, 5, 3), (2, 3, 1), (5, 1, 1)]:
        check(mq, parts, plane, cols, plan)


@pytest.mark.parametrize("fmt,rows,cols", [("q6k", 3584, 18944), ("q6k", 5120, 13824), ("q4k", 13824, 5120),
                                           ("q6k", 152064, 5120), ("q6k", 512, 18944)])
def test_default_plans_of_the_benchmark_shapes(mq, fmt, rows, cols):
    parts, plane = setup(mq, [(fmt, rows)], cols, 2)
    check(mq, parts, plane, cols, None)
