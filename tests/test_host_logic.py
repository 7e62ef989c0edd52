"""Host-side logic of the C-ABI library, no GPU needed: the library loads and
exports every symbol include/mq.h declares; the repack is a lossless,
content-dense permutation; the dispatch plan always covers every chunk
exactly once; argument validation rejects bad calls before any launch."""
import ctypes
import os
import re

import numpy as np
import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mq():
    from quant_quantized_gemv_gb300 import build
    build.build()
    import quant_quantized_gemv_gb300 as m
    m.lib()
    return m


def header_functions():
    src = open(os.path.join(ROOT, "include", "mq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mq_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(mq):
    names = header_functions()
    assert len(names) >= 20
    L = ctypes.CDLL(mq.library_path())
    for n in names:
        assert hasattr(L, n), n
    assert sorted(mq.EXPORTS) == names


@pytest.mark.parametrize("fmt", ["q6k", "q4k", "q5k"])
@pytest.mark.parametrize("rows,cols", [(1, 256), (7, 512), (8, 1024), (13, 1280), (24, 4608), (9, 18944)])
def test_repack_round_trip_and_size(mq, fmt, rows, cols):
    g = synth.rng("host", "repack", fmt, rows, cols)
    W = synth.blocks(fmt, g, rows, cols)
    bb = {"q6k": 210, "q4k": 144, "q5k": 176}[fmt]
    unrep = getattr(mq, f"mq_unrepack_{fmt}")
    P = mq.mq_repack(fmt, W, rows, cols)
    nb = cols // 256
    tiles = -(-rows // 8)
    assert P.size == tiles * 8 * nb * bb                  # zero padding beyond whole tiles
    assert np.array_equal(unrep(P, rows, cols), W)         # lossless
    # a permutation of bits: the same number of set bits
    assert np.unpackbits(P).sum() == np.unpackbits(W.reshape(-1)).sum()
    if rows % 8 == 0:
        assert P.size == W.size                            # exactly the content bytes


@pytest.mark.parametrize("fmt,bb", [("q6k", 210), ("q4k", 144), ("q5k", 176)])
def test_repack_differs_only_by_bit_permutation(mq, fmt, bb):
    """Flipping one source bit flips exactly one repacked bit, and distinct
    source bits map to distinct repacked bits (an injective bit map)."""
    rows, cols = 8, 1024
    W = np.zeros((rows, cols // 256 * bb), np.uint8)
    seen = set()
    rng = synth.rng("host", "bits", fmt)
    for pos in rng.choice(W.size * 8, 400, replace=False):
        Wb = W.copy().reshape(-1)
        Wb[pos // 8] = 1 << (pos % 8)
        P = mq.mq_repack(fmt, Wb.reshape(rows, -1), rows, cols)
        on = np.flatnonzero(np.unpackbits(P))
        assert on.size == 1
        assert on[0] not in seen
        seen.add(int(on[0]))


def test_q8_plane_size_and_unpack(mq):
    assert mq.mq_q8_bytes(33) == 0 and mq.mq_q8_bytes(0) == 0
    n = 2048
    nb = mq.mq_q8_bytes(n)
    assert nb >= n + n // 32 * 6 and nb % 16 == 0
    plane = np.arange(nb, dtype=np.uint32).astype(np.uint8)
    d, qs, s = mq.mq_q8_unpack_host(plane, n)
    assert np.array_equal(qs.view(np.uint8), plane[:n])


def test_coverage_check_rejects_the_pages_dropped_work(mq, facts):
    """The pipelined kernel of the D4-2 page covered 2 units x 256 threads =
    512 units; npair 592 lost 80 units (13.5%).  The same plan must be refused."""
    npair, covered = facts["npair_q6k_18944"], facts["pf_units_covered"]
    assert npair == 18944 // facts["q6k_weights_per_unit"]
    assert npair - covered == facts["dropped_units_18944"]
    assert round(100 * (npair - covered) / npair, 1) == facts["dropped_percent_18944"]
    assert mq.mq_check_coverage(npair, 256, 2) == mq.MQ_ERR_COVERAGE
    assert mq.mq_check_coverage(npair, 296, 2) == mq.MQ_OK
    assert mq.mq_check_coverage(19, 5, 4) == mq.MQ_OK
    assert mq.mq_check_coverage(19, 5, 3) == mq.MQ_ERR_COVERAGE     # 15 < 19: dropped chunks
    assert mq.mq_check_coverage(19, 11, 2) == mq.MQ_ERR_COVERAGE    # split 10 would be empty
    assert mq.mq_check_coverage(19, 0, 19) == mq.MQ_ERR_COVERAGE
    assert mq.mq_check_coverage(1, 1, 1) == mq.MQ_OK


def test_unit_counts_match_pages(facts):
    assert 5120 // facts["q6k_weights_per_unit"] == facts["npair_q6k_5120"]
    assert 13824 // facts["q6k_weights_per_unit"] == facts["npair_q6k_13824"]
    assert 5120 // facts["q4k_weights_per_unit"] == facts["npair_q4k_5120"]
    assert 13824 // facts["q4k_weights_per_unit"] == facts["npair_q4k_13824"]
    # the padded layout the repack removes, and the page's dense-row example
    assert facts["dpl_nbe_example"] * facts["q6k_block_bytes"] == facts["dpl_row_content"]
    assert (facts["dpl_row_content"] + 15) & ~15 == facts["dpl_row_stride"]
    assert 1024 * (5120 // 256) * facts["q6k_padded_stride"] == facts["attn_v_padded_bytes"]


def model_ctas(w, regs=168):
    return min(65536 // (w * 32 * regs), 2048 // (32 * w), 32)


@pytest.mark.parametrize("sms,regs", [(1, 168), (8, 168), (76, 128), (148, 200), (152, 168), (160, 96)])
def test_plan_always_covers(mq, sms, regs):
    shapes = [(r, c) for r in (1, 5, 8, 64, 512, 1024, 3584, 5120, 13824, 152064)
              for c in (256, 1024, 1280, 2048, 5120, 13824, 18944, 32768)]
    for rows, cols in shapes:
        s, cps, tpi = mq.mq_gemv_plan_for(rows, cols, sms, regs)
        ntiles, nch = -(-rows // 8), -(-(cols // 256) // 4)
        assert mq.mq_check_coverage(nch, s, cps) == mq.MQ_OK, (rows, cols, sms, s, cps)
        assert s * cps >= nch and (s - 1) * cps < nch
        assert s == 1 or tpi == 1
        wave = sms * model_ctas(4, regs) * 4
        if s == 1:
            assert -(-ntiles // tpi) <= wave                     # one resident wave
        elif s <= 12:
            assert ntiles <= sms * model_ctas(s, regs)           # one CTA per tile, one wave
        else:
            assert ntiles * s <= wave and nch > 12               # workspace splits
        ws = mq.mq_gemv_workspace_bytes_for(rows, cols, (s, cps, tpi))
        assert (ws > 0) == (s > 12)


def test_plans_of_the_benchmark_shapes(mq):
    """GB300: 152 SMs, 128 registers -> 4 four-warp CTAs (16 warps) per SM."""
    assert mq.mq_gemv_plan_for(3584, 18944, 152, 128) == (5, 4, 1)     # 448 tiles x 5 splits
    assert mq.mq_gemv_plan_for(152064, 5120, 152, 128) == (1, 5, 8)    # 8 whole tiles per warp
    assert mq.mq_gemv_plan_for(5120, 13824, 152, 128) == (3, 5, 1)
    assert mq.mq_gemv_plan_for(5120, 5120, 152, 128) == (3, 2, 1)
    assert mq.mq_gemv_plan_for(1024, 5120, 152, 128) == (5, 1, 1)
    assert mq.mq_gemv_plan_for(13824, 5120, 152, 128) == (1, 5, 1)
    assert mq.mq_gemv_plan_for(512, 18944, 152, 128) == (19, 1, 1)     # few tiles: workspace splits
    # the same shapes at 168 registers (12 warps per SM)
    assert mq.mq_gemv_plan_for(3584, 18944, 152, 168) == (4, 5, 1)
    assert mq.mq_gemv_plan_for(152064, 5120, 152, 168) == (1, 5, 11)
    assert mq.mq_gemv_plan_for(5120, 13824, 152, 168) == (2, 7, 1)


def test_workspace_sizes(mq):
    # 100 rows -> 13 tiles; 16384 cols -> 16 chunks
    assert mq.mq_gemv_workspace_bytes_for(100, 16384, (1, 16, 1)) == 0
    assert mq.mq_gemv_workspace_bytes_for(100, 16384, (1, 16, 5)) == 0
    assert mq.mq_gemv_workspace_bytes_for(100, 16384, (4, 4, 1)) == 0           # CTA splits
    assert mq.mq_gemv_workspace_bytes_for(100, 16384, (12, 2, 1)) == 0          # (8 would do; valid)
    assert mq.mq_gemv_workspace_bytes_for(100, 16384, (16, 1, 1)) == 64 + 13 * 16 * 8 * 4
    assert mq.mq_gemv_workspace_bytes_for(100, 16384, (2, 7, 1)) == 0           # invalid: drops chunks
    assert mq.mq_gemv_workspace_bytes_for(100, 16384, (16, 1, 3)) == 0          # invalid: splits with tpi


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="fake device pointers are only passed where no GPU exists")
def test_validation_rejects_before_launch(mq):
    L = mq.lib()
    A = ctypes.c_void_p(0x10000)       # aligned, never dereferenced: every call below
    B = ctypes.c_void_p(0x20000)       # must fail validation before any launch
    Y = ctypes.c_void_p(0x30000)
    N = ctypes.c_void_p(0)
    S = ctypes.c_void_p(0)
    assert L.mq_gemv_q6k_q8(N, B, Y, 8, 1024, N, 0, S) == mq.MQ_ERR_NULL
    assert L.mq_gemv_q6k_q8(A, B, Y, 8, 1000, N, 0, S) == mq.MQ_ERR_SHAPE
    assert L.mq_gemv_q6k_q8(A, B, Y, 0, 1024, N, 0, S) == mq.MQ_ERR_SHAPE
    assert L.mq_gemv_q4k_q8(ctypes.c_void_p(0x10008), B, Y, 8, 1024, N, 0, S) == mq.MQ_ERR_ALIGN
    # 64 x 18944: 8 tiles x 19 chunks.  Plans that drop or duplicate work
    # never launch
    assert L.mq_gemv_q6k_q8_plan(A, B, Y, 64, 18944, 5, 3, 1, N, 0, S) == mq.MQ_ERR_COVERAGE
    assert L.mq_gemv_q6k_q8_plan(A, B, Y, 64, 18944, 11, 2, 1, N, 0, S) == mq.MQ_ERR_COVERAGE
    assert L.mq_gemv_q6k_q8_plan(A, B, Y, 64, 18944, 1, 18, 1, N, 0, S) == mq.MQ_ERR_COVERAGE
    assert L.mq_gemv_q6k_q8_plan(A, B, Y, 64, 18944, 4, 5, 2, N, 0, S) == mq.MQ_ERR_COVERAGE
    assert L.mq_gemv_q6k_q8_plan(A, B, Y, 64, 18944, 1, 19, 0, N, 0, S) == mq.MQ_ERR_COVERAGE
    # a workspace plan (> 12 splits) needs (enough) workspace, or it never launches
    assert L.mq_gemv_q6k_q8_plan(A, B, Y, 64, 18944, 19, 1, 1, N, 0, S) == mq.MQ_ERR_NULL
    assert L.mq_gemv_q6k_q8_plan(A, B, Y, 64, 18944, 19, 1, 1, ctypes.c_void_p(0x40000), 16, S) == \
        mq.MQ_ERR_WORKSPACE
    assert L.mq_quantize_q8(A, B, 48, S) == mq.MQ_ERR_SHAPE
    assert L.mq_swiglu_quant_q8(A, B, N, Y, 64, S) == mq.MQ_ERR_NULL
    assert L.mq_rmsnorm_quant_q8(A, ctypes.c_void_p(0x20004), ctypes.c_float(1e-6), Y, B, 64, S) == \
        mq.MQ_ERR_ALIGN
    assert L.mq_repack_q6k(N, A, 8, 1024) == mq.MQ_ERR_NULL
    assert mq.mq_repacked_bytes_q6k(8, 1000) == 0


def test_empty_and_negative_sizes_are_shape_errors(mq):
    """Empty inputs (no rows, no columns, no values, no tokens) and negative
    sizes are refused with MQ_ERR_SHAPE before anything runs; sizes of
    empty buffers are 0."""
    L = mq.lib()
    A, B, Y = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000)
    N = S = ctypes.c_void_p(0)
    E = mq.MQ_ERR_SHAPE
    for rows, cols in ((8, 0), (0, 256), (8, -256), (-8, 256)):
        assert L.mq_gemv_q6k_q8(A, B, Y, rows, cols, N, 0, S) == E
        assert L.mq_gemv_q4k_q8(A, B, Y, rows, cols, N, 0, S) == E
        assert L.mq_gemv_q5k_q8(A, B, Y, rows, cols, N, 0, S) == E
        assert L.mq_gemv_q6k_f32(A, A, Y, rows, cols, S) == E
        assert L.mq_gemv_q6k_q8_batch(A, B, 2, Y, rows, cols, S) == E
        assert L.mq_gemv_gateup_swiglu_q8(4, A, A, B, rows, cols, Y, B, S) == E
    for n in (0, -32):
        assert L.mq_quantize_q8(A, B, n, S) == E
        assert L.mq_rmsnorm_quant_q8(A, A, ctypes.c_float(1e-6), Y, B, n, S) == E
        assert L.mq_swiglu_quant_q8(A, A, Y, B, n, S) == E
        assert L.mq_quantize_q8_batch(A, B, n, 2, S) == E
    for nt in (0, -1, mq.MQ_MAX_TOKENS + 1):
        assert L.mq_gemv_q6k_q8_batch(A, B, nt, Y, 8, 256, S) == E
        assert L.mq_quantize_q8_batch(A, B, 256, nt, S) == E
    assert mq.mq_q8_bytes(0) == 0
    assert mq.mq_repacked_bytes_q6k(0, 256) == 0 and mq.mq_repacked_bytes_q4k(8, 0) == 0


def test_binding_refuses_cpu_tensors(mq):
    import torch
    with pytest.raises(TypeError):
        mq.mq_quantize_q8(torch.zeros(64))
    with pytest.raises(TypeError):                       # pageable: the kernels cannot reach it
        mq.mq_swiglu_quant_q8(torch.zeros(64), torch.zeros(64))


def test_device_address_argument_checks(mq):
    """NULL arguments are refused before any CUDA call."""
    import ctypes
    out = ctypes.c_void_p(0)
    L = mq.lib()
    assert L.mq_device_address(None, ctypes.byref(out)) == mq.MQ_ERR_NULL
    assert L.mq_device_address(ctypes.c_void_p(16), None) == mq.MQ_ERR_NULL
    assert out.value is None


def test_group_workspace_and_validation(mq):
    qkv = [("q4k", None, 5120), ("q4k", None, 1024), ("q6k", None, 1024)]    # 640 + 128 + 128 tiles
    assert mq.mq_gemv_group_workspace_bytes(qkv, 16384, (4, 4, 1)) == 0      # CTA splits
    assert mq.mq_gemv_group_workspace_bytes(qkv, 16384, (16, 1, 1)) == 896 * 4 + 896 * 16 * 8 * 4
    assert mq.mq_gemv_group_workspace_bytes(qkv, 16384, (1, 16, 3)) == 0     # whole tiles
    assert mq.mq_gemv_group_workspace_bytes(qkv, 16384, (2, 7, 1)) == 0      # invalid plan
    with pytest.raises(ValueError):
        mq.mq_gemv_group_workspace_bytes([("q3k", None, 8)], 1024, (1, 1, 1))
    arr = (mq.MQGemvPart * 1)()
    arr[0].fmt, arr[0].rows = 7, 8                  # no such format: no plan, no bytes
    assert mq.lib().mq_gemv_group_workspace_bytes(arr, 1, 1024, 16, 1, 1) == 0
    assert mq.mq_gemv_group_workspace_bytes(qkv * 3, 1024, (1, 1, 1)) == 0   # 9 parts > MQ_MAX_GROUP
    assert mq.MQ_MAX_GROUP == 8


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="fake device pointers are only passed where no GPU exists")
def test_group_validation_rejects_before_launch(mq):
    L = mq.lib()
    arr = (mq.MQGemvPart * 3)()
    for i, (fmt, rows) in enumerate(((4, 5120), (4, 1024), (6, 1024))):
        arr[i].fmt, arr[i].rows, arr[i].Wp, arr[i].y = fmt, rows, 0x10000 * (i + 1), 0x100000 * (i + 1)
    Q = ctypes.c_void_p(0x900000)
    N = ctypes.c_void_p(0)
    assert L.mq_gemv_group_q8(arr, 0, Q, 5120, N, 0, N) == mq.MQ_ERR_SHAPE
    assert L.mq_gemv_group_q8(arr, 9, Q, 5120, N, 0, N) == mq.MQ_ERR_SHAPE
    assert L.mq_gemv_group_q8(arr, 3, N, 5120, N, 0, N) == mq.MQ_ERR_NULL
    assert L.mq_gemv_group_q8_plan(arr, 3, Q, 5120, 3, 1, 1, N, 0, N) == mq.MQ_ERR_COVERAGE
    arr[2].fmt = 7                                   # no such format
    assert L.mq_gemv_group_q8(arr, 3, Q, 5120, N, 0, N) == mq.MQ_ERR_SHAPE
    arr[2].fmt = 6
    arr[1].y = 0x100008
    assert L.mq_gemv_group_q8(arr, 3, Q, 5120, N, 0, N) == mq.MQ_ERR_ALIGN


# ------------------------------------------------------------------ small batch
@pytest.mark.parametrize("nt", [1, 2, 4, 8])
@pytest.mark.parametrize("sms", [1, 20, 152])
def test_batch_plan_always_covers(mq, nt, sms):
    shapes = [(r, c) for r in (1, 8, 61, 512, 1024, 3584, 5120, 13824, 152064)
              for c in (256, 1024, 1280, 5120, 13824, 18944)]
    for rows, cols in shapes:
        s, cps, tpi = mq.mq_gemv_batch_plan_for(rows, cols, nt, sms)
        nch = -(-(cols // 256) // 4)
        assert 1 <= s <= 12 and tpi >= 1
        assert mq.mq_check_coverage(nch, s, cps) == mq.MQ_OK, (rows, cols, nt, s, cps)


def test_batch_plans_of_the_benchmark_shapes(mq):
    """GB300 model: 152 SMs, 168 registers -> one 12-warp CTA per SM.  7B
    ffn_down: 4 splits x 3 tiles per CTA (150 CTAs); lm_head: whole rows, 12
    tiles per group, 11 groups per CTA."""
    for nt in (1, 2, 4, 8):
        assert mq.mq_gemv_batch_plan_for(3584, 18944, nt, 152) == (4, 5, 1)
        assert mq.mq_gemv_batch_plan_for(152064, 5120, nt, 152) == (1, 5, 11)
        assert mq.mq_gemv_batch_plan_for(5120, 13824, nt, 152) == (2, 7, 1)
        assert mq.mq_gemv_batch_plan_for(1024, 5120, nt, 152) == (5, 1, 1)
        assert mq.mq_gemv_batch_plan_for(13824, 5120, nt, 152) == (1, 5, 1)


def test_batch_plans_with_sixteen_warp_ctas(mq):
    """At 128 registers a CTA holds 16 warps: 7B ffn_down takes 5 splits x 3
    tiles (15 warps) per CTA."""
    assert mq.mq_gemv_batch_plan_for(3584, 18944, 2, 152, 128) == (5, 4, 1)
    for nt in (2, 3):
        for rows, cols in [(152064, 5120), (5120, 13824), (1024, 5120), (61, 1280)]:
            s, cps, tpi = mq.mq_gemv_batch_plan_for(rows, cols, nt, 152, 128)
            nch = -(-(cols // 256) // 4)
            assert 1 <= s <= 12 and mq.mq_check_coverage(nch, s, cps) == mq.MQ_OK


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="fake device pointers are only passed where no GPU exists")
def test_batch_validation_rejects_before_launch(mq):
    L = mq.lib()
    A, B, Y = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000)
    N = ctypes.c_void_p(0)
    # 64 x 4096: 8 tiles x 4 chunks
    for nt in (0, 9, -1):
        assert L.mq_gemv_q6k_q8_batch(A, B, nt, Y, 64, 4096, N) == mq.MQ_ERR_SHAPE
        assert L.mq_gemv_q4k_q8_batch_plan(A, B, nt, Y, 64, 4096, 1, 4, 1, N) == mq.MQ_ERR_SHAPE
    assert L.mq_gemv_q6k_q8_batch(N, B, 2, Y, 64, 4096, N) == mq.MQ_ERR_NULL
    assert L.mq_gemv_q6k_q8_batch(A, B, 2, Y, 64, 4000, N) == mq.MQ_ERR_SHAPE
    assert L.mq_gemv_q6k_q8_batch(A, ctypes.c_void_p(0x20008), 2, Y, 64, 4096, N) == mq.MQ_ERR_ALIGN
    for plan in [(3, 1, 1), (4, 2, 1), (9, 1, 1), (13, 1, 1), (0, 4, 1), (2, 2, 0)]:
        assert L.mq_gemv_q6k_q8_batch_plan(A, B, 4, Y, 64, 4096, *plan, N) == mq.MQ_ERR_COVERAGE, plan
    assert L.mq_quantize_q8_batch(A, B, 64, 0, N) == mq.MQ_ERR_SHAPE
    assert L.mq_quantize_q8_batch(A, B, 48, 2, N) == mq.MQ_ERR_SHAPE
    assert L.mq_swiglu_quant_q8_batch(A, B, N, Y, 64, 2, N) == mq.MQ_ERR_NULL
    assert L.mq_rmsnorm_quant_q8_batch(A, B, ctypes.c_float(1e-6), Y, ctypes.c_void_p(0x40004), 64, 9,
                                       N) == mq.MQ_ERR_SHAPE


# ------------------------------------------------------------------ gate||up + SwiGLU -> q8
def test_gateup_plans(mq):
    """GB300 model (152 SMs, 168 registers): the most warps per CTA whose
    one-CTA-per-32-row-block grid fits one wave (12 warps per SM)."""
    assert mq.mq_gemv_gateup_plan_for(13824, 152) == (4, 432)     # 14B: 432 CTAs x 4 warps
    assert mq.mq_gemv_gateup_plan_for(18944, 152) == (3, 592)     # 7B: 592 CTAs x 3 warps
    assert mq.mq_gemv_gateup_plan_for(32, 152) == (8, 1)
    w, c = mq.mq_gemv_gateup_plan_for(152064, 152)                # more blocks than a wave holds
    assert w == 4 and c == 152 * 3
    for rows in (32, 4096, 13824, 18944, 27648, 65536):
        w, c = mq.mq_gemv_gateup_plan_for(rows, 152)
        assert 1 <= w <= 8 and 1 <= c <= rows // 32
        assert c * w <= 152 * model_ctas(w) * w                   # one resident wave


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="fake device pointers are only passed where no GPU exists")
def test_gateup_validation_rejects_before_launch(mq):
    L = mq.lib()
    G, U, Q = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000)
    A, O, N = ctypes.c_void_p(0x40000), ctypes.c_void_p(0x50000), ctypes.c_void_p(0)
    assert L.mq_gemv_gateup_swiglu_q8(4, N, U, Q, 64, 1024, A, O, N) == mq.MQ_ERR_NULL
    assert L.mq_gemv_gateup_swiglu_q8(7, G, U, Q, 64, 1024, A, O, N) == mq.MQ_ERR_SHAPE
    assert L.mq_gemv_gateup_swiglu_q8(4, G, U, Q, 48, 1024, A, O, N) == mq.MQ_ERR_SHAPE
    assert L.mq_gemv_gateup_swiglu_q8(4, G, U, Q, 64, 1000, A, O, N) == mq.MQ_ERR_SHAPE
    assert L.mq_gemv_gateup_swiglu_q8(4, G, U, Q, 64, 1024, ctypes.c_void_p(0x40004), O, N) == \
        mq.MQ_ERR_ALIGN
    for w, c in ((0, 1), (9, 1), (4, 0), (4, 3)):
        assert L.mq_gemv_gateup_swiglu_q8_plan(4, G, U, Q, 64, 1024, A, O, w, c, N) == \
            mq.MQ_ERR_COVERAGE


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="needs a machine without a usable GPU")
def test_cuda_failure_names_its_call(mq):
    """Without a device, a valid call fails in its first device query with
    MQ_ERR_CUDA, and mq_last_error names the query and CUDA's reason."""
    L = mq.lib()
    A, B, Y = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000)
    N = ctypes.c_void_p(0)
    assert L.mq_gemv_q6k_q8(A, B, Y, 8, 1024, N, 0, N) == mq.MQ_ERR_CUDA
    msg = L.mq_last_error().decode()
    assert msg and ":" in msg
    with pytest.raises(mq.MQError) as e:
        mq._check(mq.MQ_ERR_CUDA, "probe")
    assert msg in str(e.value)


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="fake device pointers are only passed where no GPU exists")
def test_read_floor_validation(mq):
    L = mq.lib()
    N = ctypes.c_void_p(0)
    assert L.mq_read_floor(N, 1024, N) == mq.MQ_ERR_NULL
    assert L.mq_read_floor(ctypes.c_void_p(0x10000), 1000, N) == mq.MQ_ERR_SHAPE
    assert L.mq_read_floor(ctypes.c_void_p(0x10000), 0, N) == mq.MQ_ERR_SHAPE
    assert L.mq_read_floor(ctypes.c_void_p(0x10008), 1024, N) == mq.MQ_ERR_ALIGN


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="fake device pointers are only passed where no GPU exists")
def test_f32_gemv_validation_rejects_before_launch(mq):
    L = mq.lib()
    A, X, Y = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000)
    N = ctypes.c_void_p(0)
    assert L.mq_gemv_q6k_f32(N, X, Y, 8, 1024, N) == mq.MQ_ERR_NULL
    assert L.mq_gemv_q6k_f32(A, N, Y, 8, 1024, N) == mq.MQ_ERR_NULL
    assert L.mq_gemv_q6k_f32(A, X, Y, 8, 1000, N) == mq.MQ_ERR_SHAPE
    assert L.mq_gemv_q6k_f32(A, ctypes.c_void_p(0x20004), Y, 8, 1024, N) == mq.MQ_ERR_ALIGN
    # 64 x 18944: 19 chunks.  Dropped, empty, workspace-sized or zero plans never launch
    for plan in [(5, 3, 1), (11, 2, 1), (1, 18, 1), (4, 5, 2), (19, 1, 1), (13, 2, 1), (0, 19, 1)]:
        assert L.mq_gemv_q6k_f32_plan(A, X, Y, 64, 18944, *plan, N) == mq.MQ_ERR_COVERAGE, plan
    s, c, t = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    assert L.mq_gemv_q6k_f32_plan_of(64, 18944, N, ctypes.byref(c), ctypes.byref(t)) == mq.MQ_ERR_NULL
    assert L.mq_gemv_q6k_f32_plan_of(64, 1000, ctypes.byref(s), ctypes.byref(c),
                                     ctypes.byref(t)) == mq.MQ_ERR_SHAPE


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="fake device pointers are only passed where no GPU exists")
def test_copy_validation(mq):
    L = mq.lib()
    N = ctypes.c_void_p(0)
    A, B = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000)
    assert L.mq_copy(N, B, 1024, N) == mq.MQ_ERR_NULL
    assert L.mq_copy(A, N, 1024, N) == mq.MQ_ERR_NULL
    assert L.mq_copy(A, B, 1000, N) == mq.MQ_ERR_SHAPE
    assert L.mq_copy(A, B, 0, N) == mq.MQ_ERR_SHAPE
    assert L.mq_copy(A, ctypes.c_void_p(0x20008), 1024, N) == mq.MQ_ERR_ALIGN
    assert L.mq_copy(A, B, 1024, N) == mq.MQ_ERR_ACCESS      # nothing CUDA knows
    assert b"pageable" in L.mq_strerror(mq.MQ_ERR_ACCESS)


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="fake device pointers are only passed where no GPU exists")
def test_device_repack_validation(mq):
    L = mq.lib()
    N = ctypes.c_void_p(0)
    A, B = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000)
    assert L.mq_repack_device(6, N, B, 8, 256, N) == mq.MQ_ERR_NULL
    assert L.mq_repack_device(6, A, N, 8, 256, N) == mq.MQ_ERR_NULL
    assert L.mq_repack_device(3, A, B, 8, 256, N) == mq.MQ_ERR_SHAPE
    assert L.mq_repack_device(4, A, B, 0, 256, N) == mq.MQ_ERR_SHAPE
    assert L.mq_repack_device(5, A, B, 8, 300, N) == mq.MQ_ERR_SHAPE
    assert L.mq_repack_device(6, A, ctypes.c_void_p(0x20004), 8, 256, N) == mq.MQ_ERR_ALIGN
    assert L.mq_repack_device(6, ctypes.c_void_p(0x10001), B, 8, 256, N) == mq.MQ_ERR_ALIGN


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="fake device pointers are only passed where no GPU exists")
def test_coverage_mode_validation(mq):
    L = mq.lib()
    N = ctypes.c_void_p(0)
    Q, C = ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000)
    arr = (mq.MQGemvPart * 1)(mq.MQGemvPart(6, 64, 0x10000, 0x40000))
    assert L.mq_gemv_group_q8_coverage(arr, 1, Q, 18944, 4, 5, 1, N, 0, N, N) == mq.MQ_ERR_NULL
    assert L.mq_gemv_group_q8_coverage(arr, 1, Q, 18944, 4, 5, 1, N, 0, ctypes.c_void_p(0x30004), N) == \
        mq.MQ_ERR_ALIGN
    assert L.mq_gemv_group_q8_coverage(arr, 1, Q, 18944, 5, 3, 1, N, 0, C, N) == mq.MQ_ERR_COVERAGE
    assert L.mq_gemv_group_q8_coverage(arr, 0, Q, 18944, 4, 5, 1, N, 0, C, N) == mq.MQ_ERR_SHAPE
