"""The allocation-free q6_K GEMV entry point (mq_gemv_q6k_q8_noalloc).

It serves callers that are handed only input and output pointers and may
not allocate device memory, so they cannot pass the split-K workspace the
regular entry point needs.  This file runs last so that a failure here comes
after every other test has run; it also passes on its own in a fresh
process.  It calls the entry point through the C ABI twice in a row and
checks each result against mq_gemv_q6k_q8 with a caller workspace (the
same kernel and default plan, so the same bits) and against the oracle
(the parity tests' bar: |dy| <= 1e-4 * sum |terms| per row)."""
import ctypes

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


@pytest.mark.parametrize("rows,cols", [(512, 18944), (1024, 5120), (968, 18944)])
def test_noalloc_matches_regular_entry_point(mq, orc, rows, cols):
    import torch
    g = synth.rng("noalloc", rows, cols)
    W = synth.q6k_blocks(g, rows, cols)
    x = synth.normal(g, cols)
    Wp = torch.from_numpy(mq.mq_repack_q6k(W, rows, cols)).cuda()
    plane = mq.mq_quantize_q8(torch.from_numpy(x).cuda())
    splits, _, _ = mq.mq_gemv_plan(rows, cols, "q6k")
    assert splits > 1
    need = mq.mq_gemv_workspace_bytes(rows, cols)
    if rows == 512:                                      # few tiles, long rows: the scratch path
        assert need > 0
    if rows == 968:
        # 121 tiles x 19 splits on a 152-SM GB300: more than 64 KiB of scratch.
        # The plan depends on the device; say so rather than pass vacuously.
        if need == 0:
            pytest.skip(f"default plan {mq.mq_gemv_plan(rows, cols, 'q6k')} needs no scratch on "
                        f"this device ({mq.mq_device_sms()} SMs): the large-scratch case is not covered")
        assert 64 * 1024 < need <= 128 * 1024, need
    ws = mq.mq_gemv_workspace(rows, cols)
    y_ref = mq.mq_gemv_q6k_q8(Wp, plane, rows, cols, ws=ws).cpu().numpy()
    d0, q0, _ = orc.quantize_q8(x)
    y_or, absum = orc.gemv("q6k", W, d0, q0, rows, cols, threads=8)
    assert np.all(np.abs(y_ref.astype(np.float64) - y_or) <= TOL * absum)
    L = mq.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):                                   # two calls in a row share the array
        y = torch.full((rows,), float("nan"), device="cuda")
        st = L.mq_gemv_q6k_q8_noalloc(ctypes.c_void_p(Wp.data_ptr()), ctypes.c_void_p(plane.data_ptr()),
                                      ctypes.c_void_p(y.data_ptr()), rows, cols, stream)
        assert st == mq.MQ_OK, mq.lib().mq_strerror(st)
        torch.cuda.synchronize()
        yn = y.cpu().numpy()
        # the same kernel with the same default plan: the same bits
        assert np.array_equal(yn, y_ref)
        assert np.all(np.abs(yn.astype(np.float64) - y_or) <= TOL * absum)


def test_noalloc_rejects_bad_arguments_before_launch(mq):
    L = mq.lib()
    null = ctypes.c_void_p(0)
    assert L.mq_gemv_q6k_q8_noalloc(null, null, null, 8, 1024, null) == mq.MQ_ERR_NULL


def test_noalloc_in_a_pdl_graph_chain(mq, orc):
    """quantize -> no-alloc GEMV steps with programmatic dependent launch,
    captured in one CUDA graph and replayed: every step's output equals the
    regular entry point's (same plan, caller workspace) bit for bit.  The
    first call on the device comes before the capture (it looks up the
    array's device address)."""
    import torch
    rows, cols = 512, 18944                              # a plan with scratch
    g = synth.rng("noalloc-pdl")
    W = synth.q6k_blocks(g, rows, cols)
    Wp = torch.from_numpy(mq.mq_repack_q6k(W, rows, cols)).cuda()
    xs = [torch.from_numpy(synth.normal(g, cols)).cuda() for _ in range(4)]
    x = torch.empty(cols, device="cuda")
    plane = torch.empty(mq.mq_q8_bytes(cols), dtype=torch.uint8, device="cuda")
    y = torch.empty(rows, device="cuda")
    L = mq.lib()

    def noalloc_step(stream):
        mq.mq_quantize_q8(x, q8=plane)
        st = L.mq_gemv_q6k_q8_noalloc(ctypes.c_void_p(Wp.data_ptr()), ctypes.c_void_p(plane.data_ptr()),
                                      ctypes.c_void_p(y.data_ptr()), rows, cols, ctypes.c_void_p(stream))
        assert st == mq.MQ_OK, mq.lib().mq_strerror(st)

    ws = mq.mq_gemv_workspace(rows, cols)
    refs = []
    for xi in xs:                                        # regular entry point, no PDL
        refs.append(mq.mq_gemv_q6k_q8(Wp, mq.mq_quantize_q8(xi), rows, cols, ws=ws).cpu().numpy())
    prev = mq.mq_set_pdl(True)
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            x.copy_(xs[0])
            noalloc_step(s.cuda_stream)                  # first call outside capture
            torch.cuda.synchronize()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=s):
                noalloc_step(s.cuda_stream)
            outs = []
            for xi in xs:
                x.copy_(xi)
                gr.replay()
                outs.append(y.clone())
        torch.cuda.synchronize()
    finally:
        mq.mq_set_pdl(prev)
    for a, b in zip(outs, refs):
        assert np.array_equal(a.cpu().numpy(), b)
