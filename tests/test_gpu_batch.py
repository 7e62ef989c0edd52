"""Small-batch path (nt tokens against one pass over the weights) through the
C ABI, against the oracle applied token by token.

Bar: q8 planes bit-exact per row; f32 GEMV outputs within 1e-4 * sum|terms|
per row and token; every plan deterministic run to run; a batched producer's
row identical to the single-row producer on that row.
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


def planes_fields(mq, planes, n, nt):
    """Split nt back-to-back planes (host bytes) into per-token (d, q, sum)."""
    pb = mq.mq_q8_bytes(n)
    raw = host(planes)
    assert raw.size == nt * pb
    return [mq.mq_q8_unpack_host(np.ascontiguousarray(raw[t * pb:(t + 1) * pb]), n) for t in range(nt)]


def oracle_rows(orc, fmt, W, rows, cols, fields):
    ys, sums = [], []
    for d, q, _ in fields:
        y, a = orc.gemv(fmt, W, d, q, rows, cols, threads=len(os.sched_getaffinity(0)))
        ys.append(y)
        sums.append(a)
    return np.stack(ys), np.stack(sums)


def assert_close(y, yref, absum):
    err = np.abs(y.astype(np.float64) - yref)
    bad = err > TOL * absum
    assert not bad.any(), f"{bad.sum()} outputs out of tolerance; worst {np.max(err / np.maximum(absum, 1e-300))}"


def make(mq, fmt, rows, cols, nt, seed):
    g = synth.rng("batch", fmt, rows, cols, nt, seed)
    W = synth.blocks(fmt, g, rows, cols)
    Wp = dev(mq.mq_repack(fmt, W, rows, cols))
    x = np.stack([synth.normal(g, cols) for _ in range(nt)]).astype(np.float32)
    return W, Wp, x


def batch_fn(mq, fmt):
    return getattr(mq, f"mq_gemv_{fmt}_q8_batch")


# ------------------------------------------------------------------ producers
@pytest.mark.parametrize("nt", [1, 3, 8])
@pytest.mark.parametrize("n", [96, 5120, 18944])
def test_quantize_batch_rows_bit_exact(mq, orc, nt, n):
    g = synth.rng("qbatch", nt, n)
    x = np.stack([synth.normal(g, n) for _ in range(nt)]).astype(np.float32)
    x[0, :32] = 0.0                                  # an all-zero block
    planes = mq.mq_quantize_q8_batch(dev(x))
    for t, (d, q, s) in enumerate(planes_fields(mq, planes, n, nt)):
        d0, q0, s0 = orc.quantize_q8(x[t])
        assert np.array_equal(d, d0) and np.array_equal(q, q0) and np.array_equal(s, s0), t


@pytest.mark.parametrize("nt", [1, 2, 5, 8])
@pytest.mark.parametrize("n", [32, 5120, 13824, 131168])
def test_rmsnorm_batch_each_row_its_own_scale(mq, orc, nt, n):
    g = synth.rng("rbatch", nt, n)
    x = np.stack([synth.normal(g, n, 0.0, 1.0 + t) for t in range(nt)]).astype(np.float32)
    gain = synth.normal(g, n, 1.0, 0.1)
    y, planes = mq.mq_rmsnorm_quant_q8_batch(dev(x), dev(gain), 1e-6)
    yh = host(y)
    fields = planes_fields(mq, planes, n, nt)
    for t in range(nt):
        yref = orc.rmsnorm(x[t], gain, 1e-6)
        assert np.all(np.abs(yh[t] - yref) <= TOL * np.abs(yref) + 1e-30), t
        d0, q0, s0 = orc.quantize_q8(yh[t])
        d, q, s = fields[t]
        assert np.array_equal(d, d0) and np.array_equal(q, q0) and np.array_equal(s, s0), t


@pytest.mark.parametrize("nt", [1, 4, 8])
@pytest.mark.parametrize("n", [64, 13824, 18944])
def test_swiglu_batch(mq, orc, nt, n):
    g = synth.rng("sbatch", nt, n)
    gv = np.stack([synth.normal(g, n) for _ in range(nt)]).astype(np.float32)
    uv = np.stack([synth.normal(g, n) for _ in range(nt)]).astype(np.float32)
    y, planes = mq.mq_swiglu_quant_q8_batch(dev(gv), dev(uv))
    yh = host(y)
    fields = planes_fields(mq, planes, n, nt)
    for t in range(nt):
        yref = orc.swiglu(gv[t], uv[t])
        assert np.all(np.abs(yh[t] - yref) <= TOL * np.abs(yref) + 1e-30), t
        d0, q0, s0 = orc.quantize_q8(yh[t])
        d, q, s = fields[t]
        assert np.array_equal(d, d0) and np.array_equal(q, q0) and np.array_equal(s, s0), t


def test_batch_producer_row_equals_single_row_call(mq):
    """A row of the batched producer is the single-row producer on that row, bit for bit."""
    n, nt = 4608, 5
    g = synth.rng("rowsame")
    x = np.stack([synth.normal(g, n) for _ in range(nt)]).astype(np.float32)
    gain = synth.normal(g, n, 1.0, 0.1)
    yb, pb = mq.mq_rmsnorm_quant_q8_batch(dev(x), dev(gain), 1e-6)
    pbh = host(pb)
    size = mq.mq_q8_bytes(n)
    for t in range(nt):
        y1, p1 = mq.mq_rmsnorm_quant_q8(dev(x[t]), dev(gain), 1e-6)
        assert np.array_equal(host(y1), host(yb)[t])
        assert np.array_equal(host(p1), pbh[t * size:(t + 1) * size])


# ------------------------------------------------------------------ GEMV
SHAPES = [(37, 4608), (64, 18944), (9, 1280), (8, 256), (200, 5120)]


@pytest.mark.parametrize("fmt", ["q6k", "q4k", "q5k"])
@pytest.mark.parametrize("nt", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_batch_gemv_matches_oracle_per_token(mq, orc, fmt, nt, rows, cols):
    W, Wp, x = make(mq, fmt, rows, cols, nt, 0)
    planes = mq.mq_quantize_q8_batch(dev(x))
    y = host(batch_fn(mq, fmt)(Wp, planes, nt, rows, cols))
    assert y.shape == (nt, rows)
    yref, absum = oracle_rows(orc, fmt, W, rows, cols, planes_fields(mq, planes, cols, nt))
    assert_close(y, yref, absum)


def valid_plans(nchunks, ntiles):
    out = []
    for S in range(1, 13):
        cps = -(-nchunks // S)
        if (S - 1) * cps >= nchunks:
            continue
        G = 12 // S
        groups = -(-ntiles // G)
        for tpi in sorted({1, 2, 3, groups}):
            out.append((S, cps, tpi))
        if (S - 1) * (cps + 1) < nchunks:         # a longer range than needed, last split short
            out.append((S, cps + 1, 1))
    return out


@pytest.mark.parametrize("fmt", ["q6k", "q4k", "q5k"])
@pytest.mark.parametrize("nt", [1, 2, 6])
def test_batch_every_plan_agrees_and_is_deterministic(mq, orc, fmt, nt):
    rows, cols = 61, 7936                         # 8 tiles (ragged), 8 chunks (last: 3 blocks)
    W, Wp, x = make(mq, fmt, rows, cols, nt, 1)
    planes = mq.mq_quantize_q8_batch(dev(x))
    yref, absum = oracle_rows(orc, fmt, W, rows, cols, planes_fields(mq, planes, cols, nt))
    nchunks, ntiles = -(-cols // 1024), -(-rows // 8)
    plans = valid_plans(nchunks, ntiles)
    assert len(plans) > 10
    fn = batch_fn(mq, fmt)
    for plan in plans:
        y1 = host(fn(Wp, planes, nt, rows, cols, plan=plan))
        y2 = host(fn(Wp, planes, nt, rows, cols, plan=plan))
        assert np.array_equal(y1, y2), plan
        assert_close(y1, yref, absum)


@pytest.mark.parametrize("fmt", ["q6k", "q4k", "q5k"])
@pytest.mark.parametrize("nt", [3, 8])
def test_batch_zero_token_gives_exact_zeros(mq, orc, fmt, nt):
    """A degenerate token (an all-zero activation row: every q8 block d = 0,
    q = 0, sum = 0) among ordinary ones: its outputs are 0.0 exactly, the
    other tokens' are within the bar of the oracle."""
    rows, cols = 37, 4608
    W, Wp, x = make(mq, fmt, rows, cols, nt, 7)
    z = nt // 2
    x[z] = 0.0
    planes = mq.mq_quantize_q8_batch(dev(x))
    y = host(batch_fn(mq, fmt)(Wp, planes, nt, rows, cols))
    assert np.array_equal(y[z], np.zeros(rows, np.float32))
    yref, absum = oracle_rows(orc, fmt, W, rows, cols, planes_fields(mq, planes, cols, nt))
    keep = [t for t in range(nt) if t != z]
    assert_close(y[keep], yref[keep], absum[keep])


def test_batch_bad_plans_refused(mq):
    import torch
    rows, cols, nt = 16, 4096, 2                  # 4 chunks
    W, Wp, x = make(mq, "q6k", rows, cols, nt, 2)
    planes = mq.mq_quantize_q8_batch(dev(x))
    y = torch.full((nt, rows), 7.0, device="cuda")
    for plan in [(3, 1, 1), (2, 1, 1), (9, 1, 1), (13, 1, 1), (0, 4, 1), (2, 2, 0), (4, 2, 1)]:
        with pytest.raises(mq.MQError) as e:
            mq.mq_gemv_q6k_q8_batch(Wp, planes, nt, rows, cols, y=y, plan=plan)
        assert e.value.status == mq.MQ_ERR_COVERAGE, plan
    for bad_nt in (0, 9):
        with pytest.raises(mq.MQError) as e:
            mq.mq_gemv_q6k_q8_batch(Wp, planes, bad_nt, rows, cols, y=y)
        assert e.value.status == mq.MQ_ERR_SHAPE
    assert torch.all(y == 7.0)                    # nothing ran


@pytest.mark.parametrize("fmt", ["q6k", "q4k", "q5k"])
def test_batch_of_one_needs_no_workspace(mq, orc, fmt):
    """One token through the batch entry point: long rows and few tiles (the
    single-token GEMV would take a workspace plan here), no workspace given."""
    rows, cols = 40, 18944
    W, Wp, x = make(mq, fmt, rows, cols, 1, 3)
    plane = mq.mq_quantize_q8(dev(x[0]))
    assert mq.mq_gemv_workspace_bytes(rows, cols) > 0
    yb = host(batch_fn(mq, fmt)(Wp, plane, 1, rows, cols))
    yref, absum = oracle_rows(orc, fmt, W, rows, cols, planes_fields(mq, plane, cols, 1))
    assert_close(yb, yref, absum)


@pytest.mark.parametrize("fmt", ["q6k", "q4k", "q5k"])
@pytest.mark.parametrize("rows,cols", [(3584, 18944), (1000, 5120), (13824, 5120)])
def test_batch_of_one_is_the_single_token_gemv(mq, orc, fmt, rows, cols):
    """One token whose single-token default plan needs no workspace runs the
    single-token GEMV through the batch entry point: the same bits as
    mq_gemv_*_q8, and the oracle's values within tolerance."""
    W, Wp, x = make(mq, fmt, rows, cols, 1, 4)
    plane = mq.mq_quantize_q8(dev(x[0]))
    assert mq.mq_gemv_workspace_bytes(rows, cols) == 0
    yb = host(batch_fn(mq, fmt)(Wp, plane, 1, rows, cols))
    ys = host(getattr(mq, f"mq_gemv_{fmt}_q8")(Wp, plane, rows, cols))
    assert np.array_equal(yb.reshape(-1), ys)
    yref, absum = oracle_rows(orc, fmt, W, rows, cols, planes_fields(mq, plane, cols, 1))
    assert_close(yb, yref, absum)


def test_planes_too_large_for_shared_memory(mq):
    rows, cols, nt = 8, 65536, 8                 # 8 planes of 69.6 KB
    W, Wp, x = make(mq, "q4k", rows, cols, nt, 4)
    planes = mq.mq_quantize_q8_batch(dev(x))
    with pytest.raises(mq.MQError) as e:
        mq.mq_gemv_q4k_q8_batch(Wp, planes, nt, rows, cols)
    assert e.value.status == mq.MQ_ERR_SHAPE


@pytest.mark.parametrize("fmt,nt", [("q6k", 8), ("q4k", 2), ("q5k", 5)])
def test_widest_row_the_staged_planes_allow(mq, orc, fmt, nt):
    """Maximum size: the widest row whose nt q8 planes every CTA still stages,
    in the opt-in shared memory less 8 KiB (23552 values at 8 tokens on
    GB300).  Every row of every token against the oracle; one super-block
    wider is refused before anything runs (y untouched)."""
    import torch
    optin = getattr(torch.cuda.get_device_properties(0), "shared_memory_per_block_optin", 0)
    if not optin:
        pytest.skip("the device's opt-in shared memory per block is not reported")
    limit = (optin - 8192) & ~15
    cols = 256
    while nt * mq.mq_q8_bytes(cols + 256) <= limit:
        cols += 256
    rows = 19                                            # 3 tiles, the last ragged
    W, Wp, x = make(mq, fmt, rows, cols, nt, 6)
    planes = mq.mq_quantize_q8_batch(dev(x))
    fn = batch_fn(mq, fmt)
    y = host(fn(Wp, planes, nt, rows, cols))
    yref, absum = oracle_rows(orc, fmt, W, rows, cols, planes_fields(mq, planes, cols, nt))
    assert_close(y, yref, absum)
    yw = torch.full((nt, rows), 7.0, device="cuda")
    with pytest.raises(mq.MQError) as e:
        fn(Wp, planes, nt, rows, cols + 256, y=yw)
    assert e.value.status == mq.MQ_ERR_SHAPE
    assert bool((yw == 7.0).all())


FULL = [("ffn_down_7b", "q6k", 3584, 18944, "swiglu", 4),
        ("ffn_down_7b", "q6k", 3584, 18944, "swiglu", 7),
        ("ffn_down_7b", "q6k", 3584, 18944, "swiglu", 8),
        ("ffn_down_14b_q5k", "q5k", 5120, 13824, "swiglu", 6),
        ("attn_v_14b", "q6k", 1024, 5120, "rms", 8),
        ("ffn_gate_14b", "q4k", 13824, 5120, "rms", 8),
        ("lm_head_14b", "q6k", 152064, 5120, "rms", 2),
        ("ffn_down_14b_q5k", "q5k", 5120, 13824, "swiglu", 4)]


@pytest.mark.parametrize("name,fmt,rows,cols,producer,nt", FULL)
def test_batch_full_size_every_row(mq, orc, name, fmt, rows, cols, producer, nt):
    """Full-size matrices in the default batch plan, fed by the batched
    producers: every row of every token against the oracle; two runs equal."""
    g = synth.rng("batch-full", name, nt)
    W = synth.blocks(fmt, g, rows, cols)
    Wp = dev(mq.mq_repack(fmt, W, rows, cols))
    if producer == "swiglu":
        gv = np.stack([synth.normal(g, cols) for _ in range(nt)]).astype(np.float32)
        uv = np.stack([synth.normal(g, cols) for _ in range(nt)]).astype(np.float32)
        _, planes = mq.mq_swiglu_quant_q8_batch(dev(gv), dev(uv))
    else:
        x = np.stack([synth.normal(g, cols) for _ in range(nt)]).astype(np.float32)
        gain = synth.normal(g, cols, 1.0, 0.1)
        _, planes = mq.mq_rmsnorm_quant_q8_batch(dev(x), dev(gain), 1e-6)
    fn = batch_fn(mq, fmt)
    y1 = host(fn(Wp, planes, nt, rows, cols))
    y2 = host(fn(Wp, planes, nt, rows, cols))
    assert np.array_equal(y1, y2)
    yref, absum = oracle_rows(orc, fmt, W, rows, cols, planes_fields(mq, planes, cols, nt))
    assert_close(y1, yref, absum)
