"""Host-resident activations: the producers read their inputs, and the GEMVs
write their outputs, in pinned host memory directly (over NVLink-C2C on
GB300), so that a decode step needs no copy in or out.  The kernels are the
same as for device memory, so every result must equal the device-memory run
bit for bit; one case per producer is also checked against the oracle."""
import ctypes

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
    yield m
    m.mq_set_pdl(False)


def pinned(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def test_device_address(mq):
    import torch
    d = torch.zeros(64, device="cuda")
    assert mq.mq_device_address(d.data_ptr()) == d.data_ptr()
    h = torch.zeros(64).pin_memory()
    assert mq.mq_device_address(h.data_ptr()) != 0
    with pytest.raises(mq.MQError) as e:
        mq.mq_device_address(torch.zeros(64).data_ptr())      # pageable
    assert e.value.status == mq.MQ_ERR_ACCESS
    out = ctypes.c_void_p(0)
    assert mq.lib().mq_device_address(None, ctypes.byref(out)) == mq.MQ_ERR_NULL


def test_pageable_activation_refused(mq):
    import torch
    with pytest.raises(TypeError):
        mq.mq_quantize_q8(torch.zeros(256))
    Wp = torch.zeros(mq.mq_repacked_bytes_q6k(8, 256), dtype=torch.uint8, device="cuda")
    q8 = torch.zeros(mq.mq_q8_bytes(256), dtype=torch.uint8, device="cuda")
    with pytest.raises(TypeError):
        mq.mq_gemv_q6k_q8(Wp, q8, 8, 256, y=torch.zeros(8))


@pytest.mark.parametrize("n", [256, 5120, 13824, 18944])
def test_producers_read_pinned_input(mq, orc, n):
    import torch
    g = synth.rng("host-producers", n)
    x, gate, up = (synth.normal(g, n) for _ in range(3))
    gain = torch.from_numpy(synth.normal(g, n, 1.0, 0.1)).cuda()
    for name, args_h, args_d in [
        ("quant", (pinned(x),), (torch.from_numpy(x).cuda(),)),
        ("swiglu", (pinned(gate), pinned(up)), (torch.from_numpy(gate).cuda(), torch.from_numpy(up).cuda())),
        ("rms", (pinned(x),), (torch.from_numpy(x).cuda(),)),
    ]:
        if name == "quant":
            qh, qd = mq.mq_quantize_q8(*args_h), mq.mq_quantize_q8(*args_d)
        elif name == "swiglu":
            qh, qd = mq.mq_swiglu_quant_q8(*args_h)[1], mq.mq_swiglu_quant_q8(*args_d)[1]
        else:
            qh = mq.mq_rmsnorm_quant_q8(*args_h, gain, 1e-6)[1]
            qd = mq.mq_rmsnorm_quant_q8(*args_d, gain, 1e-6)[1]
        torch.cuda.synchronize()
        assert qh.is_cuda and torch.equal(qh, qd), name
    # the quantizer against the oracle: codes, scales and sums bit for bit
    d, qs, s = mq.mq_q8_unpack_host(mq.mq_quantize_q8(pinned(x)).cpu().numpy(), n)
    od, oq, os_ = orc.quantize_q8(x)
    assert np.array_equal(d, od) and np.array_equal(qs, oq) and np.array_equal(s, os_)


def test_batch_producers_read_pinned_input(mq):
    import torch
    nt, n = 3, 5120
    g = synth.rng("host-batch-producers")
    x = np.stack([synth.normal(g, n) for _ in range(nt)])
    u = np.stack([synth.normal(g, n) for _ in range(nt)])
    gain = torch.from_numpy(synth.normal(g, n, 1.0, 0.1)).cuda()
    xd, ud = torch.from_numpy(x).cuda(), torch.from_numpy(u).cuda()
    pairs = [
        (mq.mq_quantize_q8_batch(pinned(x)), mq.mq_quantize_q8_batch(xd)),
        (mq.mq_swiglu_quant_q8_batch(pinned(x), pinned(u))[1], mq.mq_swiglu_quant_q8_batch(xd, ud)[1]),
        (mq.mq_rmsnorm_quant_q8_batch(pinned(x), gain, 1e-6)[1], mq.mq_rmsnorm_quant_q8_batch(xd, gain, 1e-6)[1]),
    ]
    torch.cuda.synchronize()
    for a, b in pairs:
        assert torch.equal(a, b)


def _plane(mq, n, seed):
    import torch
    x = torch.from_numpy(synth.normal(synth.rng("host-plane", seed), n)).cuda()
    return mq.mq_quantize_q8(x)


# whole tiles, CTA splits and a workspace split (the 7B ffn_down shape)
@pytest.mark.parametrize("fmt,rows,cols", [("q6k", 1024, 5120), ("q4k", 13824, 5120), ("q5k", 520, 4096),
                                           ("q6k", 3584, 18944), ("q4k", 8, 256)])
def test_gemv_writes_pinned_output(mq, fmt, rows, cols):
    import torch
    g = synth.rng("host-gemv", fmt, rows, cols)
    Wp = torch.from_numpy(mq.mq_repack(fmt, synth.blocks(fmt, g, rows, cols), rows, cols)).cuda()
    q8 = _plane(mq, cols, rows)
    fn = getattr(mq, f"mq_gemv_{fmt}_q8")
    ws = mq.mq_gemv_workspace(rows, cols)
    yd = fn(Wp, q8, rows, cols, ws=ws)
    yh = torch.full((rows,), np.nan, dtype=torch.float32).pin_memory()
    fn(Wp, q8, rows, cols, y=yh, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(yh, yd.cpu())


def test_batch_group_f32_noalloc_write_pinned_output(mq):
    import torch
    rows, cols, nt = 1000, 5120, 3
    g = synth.rng("host-gemv-kinds")
    W6 = torch.from_numpy(mq.mq_repack("q6k", synth.blocks("q6k", g, rows, cols), rows, cols)).cuda()
    W4 = torch.from_numpy(mq.mq_repack("q4k", synth.blocks("q4k", g, 512, cols), 512, cols)).cuda()
    x = torch.from_numpy(np.stack([synth.normal(g, cols) for _ in range(nt)])).cuda()
    planes = mq.mq_quantize_q8_batch(x)
    q8 = planes[:mq.mq_q8_bytes(cols)]
    # batch
    yd = mq.mq_gemv_q6k_q8_batch(W6, planes, nt, rows, cols)
    yh = torch.full((nt, rows), np.nan).pin_memory()
    mq.mq_gemv_q6k_q8_batch(W6, planes, nt, rows, cols, y=yh)
    # group of two formats on one plane
    parts = [("q6k", W6, rows), ("q4k", W4, 512)]
    gd = mq.mq_gemv_group_q8(parts, q8, cols, ws=mq.mq_gemv_group_workspace(parts, cols))
    gh = [torch.full((rows,), np.nan).pin_memory(), torch.full((512,), np.nan).pin_memory()]
    mq.mq_gemv_group_q8(parts, q8, cols, ys=gh, ws=mq.mq_gemv_group_workspace(parts, cols))
    # f32 activations
    fd = mq.mq_gemv_q6k_f32(W6, x[0], rows, cols)
    fh = torch.full((rows,), np.nan).pin_memory()
    mq.mq_gemv_q6k_f32(W6, x[0], rows, cols, y=fh)
    # no caller workspace
    nd = mq.mq_gemv_q6k_q8_noalloc(W6, q8, rows, cols)
    nh = torch.full((rows,), np.nan).pin_memory()
    mq.mq_gemv_q6k_q8_noalloc(W6, q8, rows, cols, y=nh)
    torch.cuda.synchronize()
    assert torch.equal(yh, yd.cpu())
    assert torch.equal(gh[0], gd[0].cpu()) and torch.equal(gh[1], gd[1].cpu())
    assert torch.equal(fh, fd.cpu())
    assert torch.equal(nh, nd.cpu())


def test_decode_steps_in_a_graph_with_pdl(mq):
    """pinned g, u -> SwiGLU -> q8 -> q6_K GEMV -> pinned y: 6 steps, each with
    its own host input and output buffers, captured in one CUDA graph with
    PDL; every step's output equals the same step run on device copies."""
    import torch
    inter, rows = 18944, 3584
    g = synth.rng("host-chain")
    Wp = torch.from_numpy(mq.mq_repack_q6k(synth.q6k_blocks(g, rows, inter), rows, inter)).cuda()
    ins = [(pinned(synth.normal(g, inter)), pinned(synth.normal(g, inter))) for _ in range(6)]
    outs = [torch.full((rows,), np.nan).pin_memory() for _ in range(6)]
    act = torch.empty(inter, device="cuda")
    q8 = torch.empty(mq.mq_q8_bytes(inter), dtype=torch.uint8, device="cuda")
    ws = mq.mq_gemv_workspace(rows, inter)
    expect = []
    for gh, uh in ins:
        _, qd = mq.mq_swiglu_quant_q8(gh.cuda(), uh.cuda())
        expect.append(mq.mq_gemv_q6k_q8(Wp, qd, rows, inter, ws=ws).cpu())
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    prev = mq.mq_set_pdl(True)
    try:
        def steps():
            for (gh, uh), yo in zip(ins, outs):
                mq.mq_swiglu_quant_q8(gh, uh, y=act, q8=q8)
                mq.mq_gemv_q6k_q8(Wp, q8, rows, inter, y=yo, ws=ws)
        with torch.cuda.stream(stream):
            steps()                                   # eager, outside capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            steps()
        for o in outs:
            o.fill_(np.nan)
        graph.replay()
        torch.cuda.synchronize()
    finally:
        mq.mq_set_pdl(bool(prev))
    for o, e in zip(outs, expect):
        assert torch.equal(o, e)


def test_rewritten_host_buffers_in_a_replayed_graph(mq):
    """One pinned input buffer and one pinned output buffer, captured once
    (SwiGLU -> q8 -> q6_K GEMV, PDL), the host writing a new input between
    replays: every replay sees the new input and returns its own result."""
    import torch
    inter, rows = 13824, 1024
    g = synth.rng("host-rewrite")
    Wp = torch.from_numpy(mq.mq_repack_q6k(synth.q6k_blocks(g, rows, inter), rows, inter)).cuda()
    gh = torch.empty(inter).pin_memory()
    uh = torch.empty(inter).pin_memory()
    yo = torch.empty(rows).pin_memory()
    act = torch.empty(inter, device="cuda")
    q8 = torch.empty(mq.mq_q8_bytes(inter), dtype=torch.uint8, device="cuda")
    ws = mq.mq_gemv_workspace(rows, inter)
    stream = torch.cuda.Stream()
    prev = mq.mq_set_pdl(True)
    try:
        def step():
            mq.mq_swiglu_quant_q8(gh, uh, y=act, q8=q8)
            mq.mq_gemv_q6k_q8(Wp, q8, rows, inter, y=yo, ws=ws)
        gh.copy_(torch.from_numpy(synth.normal(g, inter)))
        uh.copy_(torch.from_numpy(synth.normal(g, inter)))
        with torch.cuda.stream(stream):
            step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        seen = []
        for _ in range(4):
            a, b = synth.normal(g, inter), synth.normal(g, inter)
            gh.copy_(torch.from_numpy(a))
            uh.copy_(torch.from_numpy(b))
            graph.replay()
            torch.cuda.synchronize()
            got = yo.clone()
            _, qd = mq.mq_swiglu_quant_q8(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda())
            want = mq.mq_gemv_q6k_q8(Wp, qd, rows, inter, ws=mq.mq_gemv_workspace(rows, inter)).cpu()
            assert torch.equal(got, want)
            seen.append(got)
    finally:
        mq.mq_set_pdl(bool(prev))
    assert not torch.equal(seen[0], seen[1])
