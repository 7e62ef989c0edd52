"""mq_repack_device: the repack as a kernel, for GGUF rows already in device
memory.  Bar: the bytes equal the host repack's, bit for bit (padding rows
included), for every format and for ragged tiles and chunks."""
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


SHAPES = [(1, 256), (8, 1024), (37, 1280), (61, 2304), (64, 4864), (3584, 18944)]


@pytest.mark.parametrize("fmt", ["q6k", "q4k", "q5k"])
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_device_repack_equals_host_repack(mq, fmt, rows, cols):
    import torch
    g = synth.rng("repack-dev", fmt, rows, cols)
    W = synth.blocks(fmt, g, rows, cols)
    host = mq.mq_repack(fmt, W, rows, cols)
    dev = mq.mq_repack_device(fmt, torch.from_numpy(np.ascontiguousarray(W)).cuda(), rows, cols)
    torch.cuda.synchronize()
    assert np.array_equal(dev.cpu().numpy(), host)


def test_device_repack_overwrites_a_dirty_buffer(mq):
    import torch
    rows, cols = 13, 1280                      # 2 tiles, the second with 3 padding rows
    W = synth.q6k_blocks(synth.rng("repack-dirty"), rows, cols)
    out = torch.full((mq.mq_repacked_bytes_q6k(rows, cols),), 0xAB, dtype=torch.uint8, device="cuda")
    mq.mq_repack_device("q6k", torch.from_numpy(W).cuda(), rows, cols, out=out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), mq.mq_repack("q6k", W, rows, cols))


def test_device_repack_refusals(mq):
    import ctypes
    import torch
    L = mq.lib()
    src = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    dst = torch.full((8192,), 7, dtype=torch.uint8, device="cuda")
    P = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + off)
    assert L.mq_repack_device(7, P(src), P(dst), 8, 256, None) == mq.MQ_ERR_SHAPE
    assert L.mq_repack_device(6, P(src), P(dst), 8, 1000, None) == mq.MQ_ERR_SHAPE
    assert L.mq_repack_device(6, P(src), P(dst, 8), 8, 256, None) == mq.MQ_ERR_ALIGN
    assert L.mq_repack_device(6, P(src, 1), P(dst), 8, 256, None) == mq.MQ_ERR_ALIGN
    assert L.mq_repack_device(6, ctypes.c_void_p(0), P(dst), 8, 256, None) == mq.MQ_ERR_NULL
    torch.cuda.synchronize()
    assert torch.all(dst == 7)
