"""Parity of the CUDA path (through the C ABI) against the oracle.

Bar (written here, from the arithmetic of the method):
  * q8 planes, integer sub-block dots: bit-exact.
  * f32 GEMV outputs: |y_gpu - y_oracle| <= 1e-4 * sum_terms |term| per row.
  * f32 producer outputs: |y_gpu - y_oracle| <= 1e-4 * |y_oracle| per element
    (+1e-30 absolute for exact zeros).
A fused producer's q8 must equal the oracle quantizer applied to the f32
output the producer wrote (the q8 bytes are a per-element function of it).
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
    return m


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    import torch
    torch.cuda.synchronize()
    return t.cpu().numpy()


def repack_dev(mq, fmt, W, rows, cols):
    return dev(mq.mq_repack(fmt, W, rows, cols))


def q8_fields(mq, plane, n):
    return mq.mq_q8_unpack_host(host(plane), n)


def gemv(mq, fmt, Wp, q8, rows, cols, plan=None, ws=None):
    if ws is None:
        ws = mq.mq_gemv_workspace(rows, cols, plan=plan)
    return mq.mq_gemv(fmt, Wp, q8, rows, cols, ws=ws, plan=plan)


def assert_gemv_close(y, yref, absum):
    err = np.abs(y.astype(np.float64) - yref)
    bad = err > TOL * absum
    assert not bad.any(), f"{bad.sum()} rows out of tolerance; worst {np.max(err / np.maximum(absum, 1e-300))}"


def special_activation(n, seed):
    """N(0,1) with hand-placed blocks: zeros, exact ties, one-hots, tiny and
    huge scales (subnormal and large fp16 d)."""
    g = synth.rng("act", seed, n)
    x = synth.normal(g, n)
    nb = n // 32
    if nb >= 6:
        x[0:32] = 0.0
        x[32:64] = 0.0
        x[32:42] = [127, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5, 126.5, -3.5, 5.5]
        x[64:96] = 0.0
        x[64 + 7] = -1.0
        x[96:128] *= np.float32(1e-4)
        x[128:160] *= np.float32(3e3)
    return x


# ------------------------------------------------------------------ producers
@pytest.mark.parametrize("n", [32, 96, 2048, 4128, 18944])
def test_quantize_q8_bit_exact(mq, orc, n):
    x = special_activation(n, "quant")
    plane = mq.mq_quantize_q8(dev(x))
    d, q, s = q8_fields(mq, plane, n)
    d0, q0, s0 = orc.quantize_q8(x)
    assert np.array_equal(d, d0) and np.array_equal(q, q0) and np.array_equal(s, s0)


@pytest.mark.parametrize("n", [64, 5120, 13824, 18944])
def test_swiglu_quant_q8(mq, orc, n):
    g = synth.rng("swiglu", n)
    gv = synth.normal(g, n)
    uv = synth.normal(g, n)
    y, plane = mq.mq_swiglu_quant_q8(dev(gv), dev(uv))
    yh = host(y)
    yref = orc.swiglu(gv, uv)
    assert np.all(np.abs(yh - yref) <= TOL * np.abs(yref) + 1e-30)
    d, q, s = q8_fields(mq, plane, n)
    d0, q0, s0 = orc.quantize_q8(yh)          # the plane is the quantization of y as written
    assert np.array_equal(d, d0) and np.array_equal(q, q0) and np.array_equal(s, s0)


def test_swiglu_in_place(mq, orc):
    n = 4096
    g = synth.rng("swiglu-inplace")
    gv, uv = synth.normal(g, n), synth.normal(g, n)
    gd = dev(gv)
    y, plane = mq.mq_swiglu_quant_q8(gd, dev(uv), y=gd)
    assert np.all(np.abs(host(gd) - orc.swiglu(gv, uv)) <= TOL * np.abs(orc.swiglu(gv, uv)) + 1e-30)


@pytest.mark.parametrize("n", [32, 4128, 5120, 13824, 40960, 131168])
def test_rmsnorm_quant_q8(mq, orc, n):
    g = synth.rng("rms", n)
    x = synth.normal(g, n)
    gain = synth.normal(g, n, 1.0, 0.1)
    y, plane = mq.mq_rmsnorm_quant_q8(dev(x), dev(gain), 1e-6)
    yh = host(y)
    yref = orc.rmsnorm(x, gain, 1e-6)
    assert np.all(np.abs(yh - yref) <= TOL * np.abs(yref) + 1e-30)
    d, q, s = q8_fields(mq, plane, n)
    d0, q0, s0 = orc.quantize_q8(yh)
    assert np.array_equal(d, d0) and np.array_equal(q, q0) and np.array_equal(s, s0)


def test_rmsnorm_one_scale_for_the_whole_row(mq, orc):
    """A constant row with unit gain: every y must be the same f32 value, so
    every CTA of the producer applied the same scale (the row spans many
    CTAs and more than one slice per CTA)."""
    n = 131168
    x = np.full(n, 0.37, np.float32)
    gain = np.ones(n, np.float32)
    y, plane = mq.mq_rmsnorm_quant_q8(dev(x), dev(gain), 1e-6)
    yh = host(y)
    assert np.all(yh == yh[0])
    yref = orc.rmsnorm(x, gain, 1e-6)
    assert np.all(np.abs(yh - yref) <= TOL * np.abs(yref))


# ------------------------------------------------------------------ integer path
@pytest.mark.parametrize("fmt", ["q6k", "q4k", "q5k"])
@pytest.mark.parametrize("rows,cols", [(16, 2048), (13, 1280), (9, 18944), (1, 256)])
def test_subdots_bit_exact(mq, orc, fmt, rows, cols):
    g = synth.rng("subdots", fmt, rows, cols)
    W = synth.blocks(fmt, g, rows, cols)
    x = special_activation(cols, "subdots")
    Wp = repack_dev(mq, fmt, W, rows, cols)
    plane = mq.mq_quantize_q8(dev(x))
    fn = getattr(mq, f"mq_gemv_{fmt}_q8_subdots")
    got = host(fn(Wp, plane, rows, cols))
    _, q0, _ = orc.quantize_q8(x)
    want = orc.subdots(fmt, W, q0, rows, cols)
    assert np.array_equal(got, want)


# ------------------------------------------------------------------ GEMV
SHAPES = [(512, 2048), (13, 1280), (1, 256), (37, 4608), (64, 18944), (8, 32768), (200, 5120)]


@pytest.mark.parametrize("fmt", ["q6k", "q4k", "q5k"])
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_gemv_matches_oracle(mq, orc, fmt, rows, cols):
    g = synth.rng("gemv", fmt, rows, cols)
    W = synth.blocks(fmt, g, rows, cols)
    x = special_activation(cols, "gemv")
    Wp = repack_dev(mq, fmt, W, rows, cols)
    plane = mq.mq_quantize_q8(dev(x))
    y = host(gemv(mq, fmt, Wp, plane, rows, cols))
    d0, q0, _ = orc.quantize_q8(x)
    yref, absum = orc.gemv(fmt, W, d0, q0, rows, cols, threads=8)
    assert_gemv_close(y, yref, absum)


def widest_cols(reserve, staged_bytes):
    """The widest row (a multiple of 256 values) whose staged shared memory,
    staged_bytes(cols), fits one CTA's opt-in shared memory less `reserve`
    bytes (rounded down to 16, as the library rounds it)."""
    import torch
    optin = getattr(torch.cuda.get_device_properties(0), "shared_memory_per_block_optin", 0)
    if not optin:
        pytest.skip("the device's opt-in shared memory per block is not reported")
    limit = (optin - reserve) & ~15
    cols = 256
    while staged_bytes(cols + 256) <= limit:
        cols += 256
    return cols


@pytest.mark.parametrize("fmt", ["q6k", "q4k"])
def test_widest_row_the_staged_plane_allows(mq, orc, fmt):
    """Maximum size: the widest row whose q8 plane (rounded up to 128 bytes)
    a whole-tile CTA still stages, in the opt-in shared memory less 1 KiB
    (194816 values on GB300).  The default plan (workspace splits for 2
    tiles) and an explicit whole-tile plan, every row against the oracle;
    one super-block wider is refused before anything runs (y untouched)."""
    import torch
    cols = widest_cols(1024, lambda c: (mq.mq_q8_bytes(c) + 127) & ~127)
    rows = 11                                            # 2 tiles, the second ragged
    g = synth.rng("widest", fmt, cols)
    W = synth.blocks(fmt, g, rows, cols)
    x = special_activation(cols, "widest")
    Wp = repack_dev(mq, fmt, W, rows, cols)
    plane = mq.mq_quantize_q8(dev(x))
    d0, q0, _ = orc.quantize_q8(x)
    yref, absum = orc.gemv(fmt, W, d0, q0, rows, cols, threads=8)
    nch = -(-(cols // 256) // 4)
    for plan in (None, (1, nch, 1)):
        assert_gemv_close(host(gemv(mq, fmt, Wp, plane, rows, cols, plan=plan)), yref, absum)
    y = torch.full((rows,), 7.0, device="cuda")
    for plan in (None, (1, -(-((cols + 256) // 256) // 4), 1)):
        with pytest.raises(mq.MQError) as e:
            mq.mq_gemv(fmt, Wp, plane, rows, cols + 256, y=y, plan=plan)
        assert e.value.status == mq.MQ_ERR_SHAPE
    assert bool((y == 7.0).all())


@pytest.mark.parametrize("fmt", ["q6k", "q4k", "q5k"])
def test_zero_activation_or_zero_scales_give_exact_zeros(mq, fmt):
    """Degenerate cases with an exact answer: an all-zero activation row
    (every q8 block d = 0, q = 0, sum = 0) and weights whose fp16 scales d
    (and dmin) are all zero give y == 0.0 exactly, under the default plan, a
    CTA-split plan and a workspace-split plan."""
    import torch
    rows, cols = 37, 18944                                   # 5 tiles (ragged) x 19 chunks
    g = synth.rng("zeros", fmt)
    W = synth.blocks(fmt, g, rows, cols)
    x = synth.normal(g, cols)
    bb = {"q6k": 210, "q4k": 144, "q5k": 176}[fmt]
    Wz = W.copy().reshape(rows, cols // 256, bb)
    if fmt == "q6k":
        Wz[:, :, 208:210] = 0                                # d (fp16) is the last field
    else:
        Wz[:, :, 0:4] = 0                                    # d and dmin lead the block
    cases = [(repack_dev(mq, fmt, W, rows, cols), mq.mq_quantize_q8(dev(np.zeros(cols, np.float32)))),
             (repack_dev(mq, fmt, Wz.reshape(W.shape), rows, cols), mq.mq_quantize_q8(dev(x)))]
    for Wp, plane in cases:
        for plan in (None, (4, 5, 1), (19, 1, 1)):
            y = host(gemv(mq, fmt, Wp, plane, rows, cols, plan=plan))
            assert np.array_equal(y, np.zeros(rows, np.float32)), plan


def all_plans(ntiles, nch):
    plans = []
    for s in range(2, nch + 1):
        cps = -(-nch // s)
        if (s - 1) * cps < nch:
            plans.append((s, cps, 1))
    plans += [(1, nch, tpi) for tpi in range(1, ntiles + 1)]
    return plans


@pytest.mark.parametrize("fmt", ["q6k", "q4k", "q5k"])
def test_every_plan_agrees_and_is_deterministic(mq, orc, fmt):
    """Every valid plan of a 5-tile x 19-chunk matrix (every split count,
    every tiles-per-item) against the oracle, twice, bitwise repeatable."""
    import torch
    rows, cols = 37, 18944                                  # 5 tiles (ragged) x 19 chunks
    g = synth.rng("splits", fmt)
    W = synth.blocks(fmt, g, rows, cols)
    x = synth.normal(g, cols)
    Wp = repack_dev(mq, fmt, W, rows, cols)
    plane = mq.mq_quantize_q8(dev(x))
    d0, q0, _ = orc.quantize_q8(x)
    yref, absum = orc.gemv(fmt, W, d0, q0, rows, cols)
    for plan in all_plans(5, 19):
        ws = mq.mq_gemv_workspace(rows, cols, plan=plan)
        y1 = host(gemv(mq, fmt, Wp, plane, rows, cols, plan=plan, ws=ws))
        y2 = host(gemv(mq, fmt, Wp, plane, rows, cols, plan=plan, ws=ws))
        assert_gemv_close(y1, yref, absum)
        assert np.array_equal(y1, y2), plan                 # fixed combine order
        if ws is not None:                                  # counters back to zero
            assert torch.count_nonzero(ws[:4 * 5]).item() == 0


def test_bad_plan_is_refused_and_nothing_runs(mq):
    import torch
    rows, cols = 16, 18944                                  # 2 tiles x 19 chunks
    g = synth.rng("badplan")
    W = synth.q6k_blocks(g, rows, cols)
    Wp = repack_dev(mq, "q6k", W, rows, cols)
    plane = mq.mq_quantize_q8(dev(synth.normal(g, cols)))
    y = torch.full((rows,), float("nan"), device="cuda")
    ws = mq.mq_gemv_workspace(rows, cols, plan=(19, 1, 1))
    # 15 of 19 chunks; an empty split; a one-split plan short of the row;
    # splits together with multi-tile items
    for bad in ((5, 3, 1), (10, 2, 2), (1, 18, 1), (4, 5, 2)):
        with pytest.raises(mq.MQError) as e:
            mq.mq_gemv_q6k_q8(Wp, plane, rows, cols, y=y, ws=ws, plan=bad)
        assert e.value.status == mq.MQ_ERR_COVERAGE, bad
    torch.cuda.synchronize()
    assert torch.isnan(y).all().item()


# ------------------------------------------------------------------ chains
def test_swiglu_to_gemv_chain(mq, orc):
    """The 7B ffn_down chain at reduced rows: swiglu -> q8 -> q6_K split-K GEMV,
    against the oracle chain computed from the same f32 inputs only."""
    rows, cols = 256, 18944
    g = synth.rng("chain-swiglu")
    W = synth.q6k_blocks(g, rows, cols)
    gv, uv = synth.normal(g, cols), synth.normal(g, cols)
    Wp = repack_dev(mq, "q6k", W, rows, cols)
    _, plane = mq.mq_swiglu_quant_q8(dev(gv), dev(uv))
    y = host(gemv(mq, "q6k", Wp, plane, rows, cols))
    d0, q0, _ = orc.quantize_q8(orc.swiglu(gv, uv).astype(np.float32))
    yref, absum = orc.gemv("q6k", W, d0, q0, rows, cols, threads=8)
    assert_gemv_close(y, yref, absum)


def test_rms_to_gemv_chain(mq, orc):
    rows, cols = 320, 5120
    g = synth.rng("chain-rms")
    W = synth.q4k_blocks(g, rows, cols)
    x, gain = synth.normal(g, cols), synth.normal(g, cols, 1.0, 0.1)
    Wp = repack_dev(mq, "q4k", W, rows, cols)
    _, plane = mq.mq_rmsnorm_quant_q8(dev(x), dev(gain), 1e-6)
    y = host(gemv(mq, "q4k", Wp, plane, rows, cols))
    d0, q0, _ = orc.quantize_q8(orc.rmsnorm(x, gain, 1e-6).astype(np.float32))
    yref, absum = orc.gemv("q4k", W, d0, q0, rows, cols, threads=8)
    assert_gemv_close(y, yref, absum)


# ------------------------------------------------------------------ full sizes
FULL = [("ffn_down_7b", "q6k", 3584, 18944, "swiglu"),
        ("attn_v_14b", "q6k", 1024, 5120, "rms"),
        ("ffn_down_14b", "q6k", 5120, 13824, "rms"),
        ("attn_q_14b", "q4k", 5120, 5120, "rms"),
        ("attn_k_14b", "q4k", 1024, 5120, "rms"),
        ("ffn_gate_14b", "q4k", 13824, 5120, "rms"),
        ("lm_head_14b", "q6k", 152064, 5120, "rms"),
        # q5_K at the 14B ffn_down and gate shapes (the class of q5_K_M files)
        ("ffn_down_14b_q5k", "q5k", 5120, 13824, "swiglu"),
        ("ffn_gate_14b_q5k", "q5k", 13824, 5120, "rms")]


@pytest.mark.parametrize("name,fmt,rows,cols,producer", FULL)
def test_full_size_every_row(mq, orc, name, fmt, rows, cols, producer):
    """Full-size matrices in the launch configuration the benchmark times:
    every row against the oracle (dropped work hides from row samples), and
    every output identical across two runs."""
    g = synth.rng("full", name)
    W = synth.blocks(fmt, g, rows, cols)
    Wp = repack_dev(mq, fmt, W, rows, cols)
    if producer == "swiglu":
        gv, uv = synth.normal(g, cols), synth.normal(g, cols)
        yprod, plane = mq.mq_swiglu_quant_q8(dev(gv), dev(uv))
    else:
        x, gain = synth.normal(g, cols), synth.normal(g, cols, 1.0, 0.1)
        yprod, plane = mq.mq_rmsnorm_quant_q8(dev(x), dev(gain), 1e-6)
    ws = mq.mq_gemv_workspace(rows, cols)
    y1 = host(gemv(mq, fmt, Wp, plane, rows, cols, ws=ws))
    y2 = host(gemv(mq, fmt, Wp, plane, rows, cols, ws=ws))
    assert np.all(np.isfinite(y1)) and np.array_equal(y1, y2)
    # every row against the oracle, fed the oracle's own quantization of the
    # producer output (checked bit-exact against the plane above)
    d, q, _ = orc.quantize_q8(host(yprod))
    dg, qg, _ = q8_fields(mq, plane, cols)
    assert np.array_equal(d, dg) and np.array_equal(q, qg)
    yref, absum = orc.gemv(fmt, W, d, q, rows, cols, threads=len(os.sched_getaffinity(0)))
    assert_gemv_close(y1, yref, absum)


# ------------------------------------------------------------------ groups
GROUPS = [
    # q, k, v of a layer (q4_K, q4_K, q6_K), ragged rows, ragged last chunk
    (4608, [("q4k", 40), ("q4k", 13), ("q6k", 24)]),
    # a gate/up pair and a third part with long rows (19 chunks: > 12 splits possible)
    (18944, [("q4k", 16), ("q4k", 16), ("q6k", 9)]),
    # all three formats in one launch
    (5120, [("q5k", 24), ("q6k", 8), ("q4k", 17), ("q5k", 3)]),
]


@pytest.mark.parametrize("cols,spec", GROUPS)
def test_group_matches_oracle_under_every_plan(mq, orc, cols, spec):
    import torch
    g = synth.rng("group", cols)
    Ws = [synth.blocks(fmt, g, rows, cols) for fmt, rows in spec]
    Wps = [repack_dev(mq, fmt, W, rows, cols) for (fmt, rows), W in zip(spec, Ws)]
    x = special_activation(cols, "group")
    plane = mq.mq_quantize_q8(dev(x))
    d0, q0, _ = orc.quantize_q8(x)
    refs = [orc.gemv(fmt, W, d0, q0, rows, cols) for (fmt, rows), W in zip(spec, Ws)]
    parts = [(fmt, Wp, rows) for (fmt, rows), Wp in zip(spec, Wps)]
    ntiles = sum(-(-rows // 8) for _, rows in spec)
    nch = -(-(cols // 256) // 4)
    plans = [None] + all_plans(ntiles, nch)
    for plan in plans:
        ws = mq.mq_gemv_group_workspace(parts, cols, plan=plan)
        ys1 = mq.mq_gemv_group_q8(parts, plane, cols, ws=ws, plan=plan)
        ys2 = mq.mq_gemv_group_q8(parts, plane, cols, ws=ws, plan=plan)
        for y1, y2, (yref, absum) in zip(ys1, ys2, refs):
            assert_gemv_close(host(y1), yref, absum)
            assert np.array_equal(host(y1), host(y2)), plan
        if ws is not None:
            assert torch.count_nonzero(ws[:4 * ntiles]).item() == 0


def test_group_of_one_is_the_single_gemv(mq):
    rows, cols = 3584, 18944
    g = synth.rng("group-one")
    W = synth.q6k_blocks(g, rows, cols)
    Wp = repack_dev(mq, "q6k", W, rows, cols)
    plane = mq.mq_quantize_q8(dev(synth.normal(g, cols)))
    y1 = host(gemv(mq, "q6k", Wp, plane, rows, cols))
    (y2,) = mq.mq_gemv_group_q8([("q6k", Wp, rows)], plane, cols,
                                ws=mq.mq_gemv_group_workspace([("q6k", Wp, rows)], cols))
    assert np.array_equal(y1, host(y2))


def test_read_floor_runs(mq):
    """The measurement aid reads a buffer without error (bench.py times it)."""
    import torch
    buf = torch.ones(1 << 20, dtype=torch.uint8, device="cuda")
    mq.mq_read_floor(buf)
    mq.mq_read_floor(buf, 4096)
    torch.cuda.synchronize()
    with pytest.raises(mq.MQError):
        mq.mq_read_floor(buf, 4095)


def test_group_instance_matches_the_standard_instance(mq, orc):
    """A default-plan grouped launch of q6_K/q4_K parts runs the kernel's
    grouped-launch instance (fewer registers, its own occupancy); explicit
    plans run the standard instance.  Both compute the same sub-dots in the
    same order, so the default launch must equal, bit for bit, the explicit
    launch of whichever plan it chose -- here on the 14B q, k, v shapes."""
    import torch
    g = synth.rng("group-instance")
    cols = 5120
    spec = [("q4k", 5120), ("q4k", 1024), ("q6k", 1024)]
    Ws = [synth.blocks(f, g, r, cols) for f, r in spec]
    parts = [(f, repack_dev(mq, f, W, r, cols), r) for (f, r), W in zip(spec, Ws)]
    x = synth.normal(g, cols)
    plane = mq.mq_quantize_q8(dev(x))
    ys = mq.mq_gemv_group_q8(parts, plane, cols, ws=mq.mq_gemv_group_workspace(parts, cols))
    got = [host(y) for y in ys]
    nch = cols // 256 // 4
    plans = [(s, -(-nch // s), 1) for s in range(2, nch + 1)
             if (s - 1) * -(-nch // s) < nch]  # no empty split
    plans += [(1, nch, t) for t in (1, 2, 3, 4)]
    matches = []
    for plan in plans:
        ws = mq.mq_gemv_group_workspace(parts, cols, plan=plan)
        ref = [host(y) for y in mq.mq_gemv_group_q8(parts, plane, cols, ws=ws, plan=plan)]
        if all(np.array_equal(a, b) for a, b in zip(got, ref)):
            matches.append(plan)
    assert matches, "the default grouped launch matches no explicit plan bit for bit"
    d, q, _ = orc.quantize_q8(x)
    for (f, r), W, y in zip(spec, Ws, got):
        yref, absum = orc.gemv(f, W, d, q, r, cols, threads=len(os.sched_getaffinity(0)))
        assert_gemv_close(y, yref, absum)
