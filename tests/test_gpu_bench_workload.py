"""The benchmark's own workload, in the launch configuration bench.py times,
against the oracle: a two-layer Qwen2.5-14B decode sweep (every shape of the
48-layer sweep: the grouped q/k/v launch, attn_output, the fused gate||up
launch with its SwiGLU -> q8 epilogue, ffn_down, and the 152064 x 5120 head,
with their rms_norm and quantize producers), built by bench.DeviceWorkload
with the same grouping, fusion, plans and workspaces, and run as one step in
a CUDA graph with programmatic dependent launch.  After the step:

  * every producer's q8 plane is bit for bit the oracle's quantization of
    the producer's f32 output, and rms_norm's output is within 1e-4 of the
    oracle's;
  * sampled 16-row windows of every GEMV output (first, middle, last rows of
    each part) are within 1e-4 * sum|terms| of the oracle fed the plane the
    GEMV read;
  * gate||up's act rows in sampled 32-row blocks are within the bound the
    GEMV tolerance implies through SwiGLU, and its q8 plane is bit for bit the
    oracle's quantization of act.
"""
import os

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(scope="module")
def step():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quant_quantized_gemv_gb300 import build
    build.build()
    import quant_quantized_gemv_gb300 as mq
    import bench
    name = "sweep_14b_2_layers"
    synth.WORKLOADS[name] = synth.Workload(name, synth._sweep_14b(2))
    dev = torch.device("cuda", 0)
    l2 = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    wl = bench.DeviceWorkload(name, dev, l2)
    stream = torch.cuda.Stream(device=dev)
    prev = mq.mq_set_pdl(True)
    try:
        sg = bench.StepGraphs(wl.run, wl.n_copies, 1, stream)
        sg.prepare(0, 1)
        with torch.cuda.stream(stream):
            sg.enqueue(0, 1)
        torch.cuda.synchronize()
    finally:
        mq.mq_set_pdl(bool(prev))
    yield mq, wl
    del synth.WORKLOADS[name]


def host(t):
    return t.detach().cpu().numpy()


def threads():
    return len(os.sched_getaffinity(0))


def windows(rows, g, width=16):
    mid = int(g.integers(1, max(2, rows // width - 1))) * width
    return sorted({(0, min(width, rows)), (min(mid, rows - width), min(mid, rows - width) + width),
                   (rows - width, rows)})


def test_the_step_is_the_sweep_pattern(step):
    mq, wl = step
    kinds = [o[0] for o in wl.ops]
    # per layer: rms, q/k/v group, quantize, attn_output, rms, gate||up, ffn_down; then rms, head
    assert kinds == ["rms", "gemv", "quant", "gemv", "rms", "gateup", "gemv"] * 2 + ["rms", "gemv"]
    assert [len(o[3]) for o in wl.ops if o[0] == "gemv"] == [3, 1, 1] * 2 + [1]


def test_producers_against_the_oracle(step, orc):
    mq, wl = step
    for o in wl.ops:
        if o[0] == "rms":
            _, x, gain, y, plane, n = o
            yh = host(y)
            yref = orc.rmsnorm(host(x), host(gain), 1e-6)
            assert np.all(np.abs(yh - yref) <= TOL * np.abs(yref) + 1e-30)
            src = yh
        elif o[0] == "quant":
            _, x, plane, n = o
            src = host(x)
        else:
            continue
        d0, q0, s0 = orc.quantize_q8(src)
        d1, q1, s1 = mq.mq_q8_unpack_host(host(plane), n)
        assert np.array_equal(d0, d1) and np.array_equal(q0, q1) and np.array_equal(s0, s1)


def test_gemv_rows_against_the_oracle(step, orc):
    mq, wl = step
    g = synth.rng("bench-workload-rows")
    for o in wl.ops:
        if o[0] != "gemv":
            continue
        _, plane, cols, parts, _ = o
        d, q, _ = mq.mq_q8_unpack_host(host(plane), cols)
        for fmt, _, rows, y, gname in parts:
            W = wl.host_w[(fmt, rows, cols)]
            yh = host(y)
            assert np.all(np.isfinite(yh)), gname
            for r0, r1 in windows(rows, g):
                yref, absum = orc.gemv(fmt, W, d, q, rows, cols, row_range=(r0, r1), threads=threads())
                err = np.abs(yh[r0:r1].astype(np.float64) - yref)
                assert np.all(err <= TOL * absum), (gname, r0, float(np.max(err / (TOL * absum))))


def test_gateup_against_the_oracle_chain(step, orc):
    mq, wl = step
    g = synth.rng("bench-workload-gateup")
    for o in wl.ops:
        if o[0] != "gateup":
            continue
        _, plane, cols, parts, act, plane_out = o
        (fmt, _, rows, _, gname), (fmt_u, _, rows_u, _, _) = parts
        Wg, Wu = wl.host_w[(fmt, rows, cols)], wl.host_w[(fmt_u, rows_u, cols)]
        d, q, _ = mq.mq_q8_unpack_host(host(plane), cols)
        acth = host(act)
        for r0, r1 in windows(rows, g, 32):
            gv, ag = orc.gemv(fmt, Wg, d, q, rows, cols, row_range=(r0, r1), threads=threads())
            uv, au = orc.gemv(fmt_u, Wu, d, q, rows, cols, row_range=(r0, r1), threads=threads())
            ref = orc.swiglu(gv.astype(np.float32), uv.astype(np.float32))
            silu = gv / (1.0 + np.exp(-gv))
            bound = 1.1 * np.abs(uv) * TOL * ag + np.abs(silu) * TOL * au + 1e-6 * np.abs(ref) + 1e-30
            assert np.all(np.abs(acth[r0:r1] - ref) <= bound), (gname, r0)
        d0, q0, s0 = orc.quantize_q8(acth)
        d1, q1, s1 = mq.mq_q8_unpack_host(host(plane_out), rows)
        assert np.array_equal(d0, d1) and np.array_equal(q0, q1) and np.array_equal(s0, s1)
