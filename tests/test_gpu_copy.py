"""mq_copy: the kernel copy between device memory and pinned host memory that
carries a decode step's input in and its result out.  Bit-exact: it moves
bytes."""
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


@pytest.mark.parametrize("n", [4, 1024, 37888, 1 << 20])
def test_host_to_device_to_host(mq, n):
    import torch
    g = synth.rng("copy", n)
    src = torch.from_numpy(synth.normal(g, n)).pin_memory()
    mid = torch.full((n,), -1.0, device="cuda")
    out = torch.full((n,), -2.0).pin_memory()
    mq.mq_copy(mid, src)
    mq.mq_copy(out, mid)
    torch.cuda.synchronize()
    assert torch.equal(mid.cpu(), src) and torch.equal(out, src)


def test_device_to_device_and_partial(mq):
    import torch
    a = torch.arange(4096, dtype=torch.float32, device="cuda")
    b = torch.zeros(4096, device="cuda")
    mq.mq_copy(b, a, nbytes=1024 * 4)
    torch.cuda.synchronize()
    assert torch.equal(b[:1024], a[:1024]) and torch.all(b[1024:] == 0)


def test_refusals(mq):
    import torch
    d = torch.zeros(64, device="cuda")
    pageable = torch.ones(64)
    L = mq.lib()
    import ctypes
    st = L.mq_copy(ctypes.c_void_p(d.data_ptr()), ctypes.c_void_p(pageable.data_ptr()), 256, None)
    assert st == mq.MQ_ERR_ACCESS
    assert L.mq_copy(ctypes.c_void_p(d.data_ptr()), ctypes.c_void_p(d.data_ptr() + 4), 128, None) == \
        mq.MQ_ERR_ALIGN
    assert L.mq_copy(ctypes.c_void_p(d.data_ptr()), ctypes.c_void_p(d.data_ptr()), 100, None) == \
        mq.MQ_ERR_SHAPE
    torch.cuda.synchronize()
    assert torch.all(d == 0)


def test_decode_step_in_a_graph_with_pdl(mq):
    """pinned x -> (copy) -> rms_norm -> q8 -> q6_K GEMV -> (copy) -> pinned y,
    6 steps captured in one CUDA graph with PDL: each step's y equals the
    same step run eagerly with torch copies."""
    import torch
    h, rows = 5120, 1024
    g = synth.rng("copy-chain")
    Wp = torch.from_numpy(mq.mq_repack_q6k(synth.q6k_blocks(g, rows, h), rows, h)).cuda()
    gain = torch.from_numpy(synth.normal(g, h, 1.0, 0.1)).cuda()
    xs = [torch.from_numpy(synth.normal(g, h)).pin_memory() for _ in range(6)]
    x = torch.empty(h, device="cuda")
    xn = torch.empty(h, device="cuda")
    qa = torch.empty(mq.mq_q8_bytes(h), dtype=torch.uint8, device="cuda")
    y = torch.empty(rows, device="cuda")
    ws = mq.mq_gemv_workspace(rows, h)
    outs = [torch.empty(rows).pin_memory() for _ in range(6)]

    def step(i, kernel_copies):
        if kernel_copies:
            mq.mq_copy(x, xs[i])
        else:
            x.copy_(xs[i], non_blocking=True)
        mq.mq_rmsnorm_quant_q8(x, gain, 1e-6, y=xn, q8=qa)
        mq.mq_gemv_q6k_q8(Wp, qa, rows, h, y=y, ws=ws)
        if kernel_copies:
            mq.mq_copy(outs[i], y)
        else:
            outs[i].copy_(y, non_blocking=True)

    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for i in range(6):
            step(i, False)
    torch.cuda.synchronize()
    ref = [o.clone() for o in outs]
    for o in outs:
        o.fill_(0.0)
    mq.mq_set_pdl(True)
    with torch.cuda.stream(st):
        step(0, True)
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=st):
        for i in range(6):
            step(i, True)
    for o in outs:
        o.fill_(0.0)
    with torch.cuda.stream(st):
        gr.replay()
    torch.cuda.synchronize()
    mq.mq_set_pdl(False)
    for a, b in zip(ref, outs):
        assert torch.equal(a, b)
