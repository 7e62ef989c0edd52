"""Pins for the oracle against things other than itself.

Each test checks one oracle function against what the minfer pages or the
mathematics fix: printed layout facts, closed forms on hand-built blocks, a
second formulation of the same GGUF decode, textbook/library routines (numpy
float16, scipy expit) and brute force (dequantize, then an fp64 matmul).  A
plausible slip in the oracle (a wrong nibble, shift, scale index, sign,
rounding mode or activation index) fails at least one of them.
"""
import numpy as np
import pytest

import synth

F16_ONE = 0x3C00


# ---------------------------------------------------------------- helpers
def q6k_block(ql, qh, sc, d_bits=F16_ONE):
    blk = np.zeros(210, np.uint8)
    blk[0:128] = ql
    blk[128:192] = qh
    blk[192:208] = np.asarray(sc, np.int8).view(np.uint8)
    blk[208] = d_bits & 0xFF
    blk[209] = d_bits >> 8
    return blk


def q6k_dequant_alt(blocks):
    """GGUF q6_K decode written per half-block: for l in 0..31 the weights at
    l, l+32, l+64, l+96 of a 128-weight half take (low ql[l], qh[l] bits 0-1),
    (low ql[l+32], bits 2-3), (high ql[l], bits 4-5), (high ql[l+32], bits 6-7);
    the scale of position p of half h is sc[8h + p//16]."""
    blocks = blocks.reshape(-1, 210).astype(np.int64)
    out = np.zeros((blocks.shape[0], 256))
    d = np.array([np.uint16(b[208] | (b[209] << 8)).view(np.float16) for b in blocks], np.float64)
    sc = blocks[:, 192:208].astype(np.uint8).view(np.int8).astype(np.int64)
    for h in range(2):
        ql = blocks[:, 64 * h:64 * h + 64]
        qh = blocks[:, 128 + 32 * h:128 + 32 * h + 32]
        parts = [(ql[:, :32] & 15) | ((qh & 3) << 4),
                 (ql[:, 32:] & 15) | (((qh >> 2) & 3) << 4),
                 (ql[:, :32] >> 4) | (((qh >> 4) & 3) << 4),
                 (ql[:, 32:] >> 4) | (((qh >> 6) & 3) << 4)]
        for k, qv in enumerate(parts):
            for l in range(32):
                p = 32 * k + l
                out[:, 128 * h + p] = d * sc[:, 8 * h + p // 16] * (qv[:, l] - 32)
    return out.reshape(-1)


def q4k_pack_scales(sc, m):
    """Pack eight 6-bit scales and mins into GGUF q4_K's 12 bytes: bytes 0-3
    hold sc0..3 (bits 0-5) and the top two bits of sc4..7 (bits 6-7), bytes
    4-7 the same for m0..3 / m4..7, bytes 8-11 the low nibbles of sc4..7
    (bits 0-3) and m4..7 (bits 4-7)."""
    s = np.zeros(12, np.uint8)
    for k in range(4):
        s[k] = (sc[k] & 63) | ((sc[k + 4] >> 4) << 6)
        s[k + 4] = (m[k] & 63) | ((m[k + 4] >> 4) << 6)
        s[k + 8] = (sc[k + 4] & 15) | ((m[k + 4] & 15) << 4)
    return s


def q4k_block(d_bits, dmin_bits, sc, m, qs):
    blk = np.zeros(144, np.uint8)
    blk[0], blk[1] = d_bits & 0xFF, d_bits >> 8
    blk[2], blk[3] = dmin_bits & 0xFF, dmin_bits >> 8
    blk[4:16] = q4k_pack_scales(sc, m)
    blk[16:] = qs
    return blk


def q4k_dequant_alt(blocks, orc):
    """GGUF q4_K decode written per 64-weight group j: the first 32 weights are
    the low nibbles of qs[32j:32j+32] with (sc, m) of sub-block 2j, the next 32
    the high nibbles with sub-block 2j+1; w = d*sc*q - dmin*m."""
    blocks = blocks.reshape(-1, 144)
    out = np.zeros((blocks.shape[0], 256))
    for i, b in enumerate(blocks):
        d = float(np.uint16(int(b[0]) | (int(b[1]) << 8)).view(np.float16))
        dmin = float(np.uint16(int(b[2]) | (int(b[3]) << 8)).view(np.float16))
        for j in range(4):
            q = b[16 + 32 * j:16 + 32 * j + 32].astype(np.int64)
            for hsel, qv in ((0, q & 15), (1, q >> 4)):
                sc, m = orc.q4k_scale_min(b, 2 * j + hsel)
                out[i, 64 * j + 32 * hsel:64 * j + 32 * hsel + 32] = d * sc * qv - dmin * m
    return out.reshape(-1)


def q5k_block(d_bits, dmin_bits, sc, m, qh, qs):
    blk = np.zeros(176, np.uint8)
    blk[0], blk[1] = d_bits & 0xFF, d_bits >> 8
    blk[2], blk[3] = dmin_bits & 0xFF, dmin_bits >> 8
    blk[4:16] = q4k_pack_scales(sc, m)
    blk[16:48] = qh
    blk[48:] = qs
    return blk


def q5k_dequant_alt(blocks, orc):
    """GGUF q5_K decode written per 64-weight group j with two moving bit
    masks u1 = 1 << 2j, u2 = 2 << 2j: weight 64j + l (l < 32) is the low
    nibble of qs[32j + l] plus 16 if qh[l] & u1, weight 64j + 32 + l the high
    nibble plus 16 if qh[l] & u2; scales as q4_K."""
    blocks = blocks.reshape(-1, 176)
    out = np.zeros((blocks.shape[0], 256))
    for i, b in enumerate(blocks):
        d = float(np.uint16(int(b[0]) | (int(b[1]) << 8)).view(np.float16))
        dmin = float(np.uint16(int(b[2]) | (int(b[3]) << 8)).view(np.float16))
        qh = b[16:48].astype(np.int64)
        u1, u2 = 1, 2
        for j in range(4):
            q = b[48 + 32 * j:48 + 32 * j + 32].astype(np.int64)
            lo = (q & 15) + np.where(qh & u1, 16, 0)
            hi = (q >> 4) + np.where(qh & u2, 16, 0)
            for hsel, qv in ((0, lo), (1, hi)):
                sc, m = orc.q4k_scale_min(b, 2 * j + hsel)
                out[i, 64 * j + 32 * hsel:64 * j + 32 * hsel + 32] = d * sc * qv - dmin * m
            u1 <<= 2
            u2 <<= 2
    return out.reshape(-1)


def xhat(orc, x):
    d, q, _ = orc.quantize_q8(x)
    dd = np.array([orc.f16_to_f32(h) for h in d])
    return d, q, np.repeat(dd, 32) * q.astype(np.float64)


# ---------------------------------------------------------------- layout facts
def test_q6k_block_offsets_match_pages(orc, facts):
    """Byte offsets of ql/qh/sc/d (D4-2 §3.2 Excerpt C) and the 210 B block."""
    assert facts["q6k_block_bytes"] == 210 == orc.Q6K_BYTES
    assert facts["q6k_off_qh"] - facts["q6k_off_ql"] == 128
    assert facts["q6k_off_sc"] - facts["q6k_off_qh"] == 64
    assert facts["q6k_off_d"] - facts["q6k_off_sc"] == 16
    base = q6k_block(0, 0, np.ones(16, np.int8))
    w0 = orc.dequant_q6k(base)
    assert np.all(w0 == -32.0)                      # q = 0 - 32, sc = 1, d = 1
    # d at offset 208: fp16 2.0 doubles every weight
    b = base.copy(); b[facts["q6k_off_d"] + 1] = 0x40
    assert np.all(orc.dequant_q6k(b) == 2 * w0)
    # a scale byte at 192 + s rescales exactly the 16 weights of sub-block s
    for s in (0, 5, 15):
        b = base.copy(); b[facts["q6k_off_sc"] + s] = 3
        w = orc.dequant_q6k(b)
        changed = np.nonzero(w != w0)[0]
        assert list(changed) == list(range(16 * s, 16 * s + 16))
    # ql byte 0 feeds element 0 (low nibble) and element 64 (high nibble)
    b = base.copy(); b[facts["q6k_off_ql"]] = 0x21
    w = orc.dequant_q6k(b)
    assert list(np.nonzero(w != w0)[0]) == [0, 64] and w[0] == -31 and w[64] == -30
    # qh byte 0 feeds elements 0, 32, 64, 96 through bit pairs 0, 2, 4, 6
    b = base.copy(); b[facts["q6k_off_qh"]] = 0b11100100
    w = orc.dequant_q6k(b)
    assert list(np.nonzero(w != w0)[0]) == [32, 64, 96]
    assert (w[0], w[32], w[64], w[96]) == (-32, 16 - 32, 32 - 32, 48 - 32)


def test_q6k_closed_form_pattern(orc):
    """ql = 0x21 (low 1, high 2), qh = 0xE4 (fields 0,1,2,3), sc_s = s - 8:
    the four 32-weight groups g of each half decode to q = -31, -15, 2, 18."""
    blk = q6k_block(0x21, 0xE4, np.arange(16) - 8)
    w = orc.dequant_q6k(blk)
    per_g = [1 - 32, (1 | 16) - 32, (2 | 32) - 32, (2 | 48) - 32]
    expect = np.array([(e // 16 - 8) * per_g[(e // 32) % 4] for e in range(256)], float)
    assert np.array_equal(w, expect)


def test_q6k_matches_second_formulation(orc):
    g = synth.rng("pin", "q6k-alt")
    W = synth.q6k_blocks(g, 6, 1024)
    assert np.array_equal(orc.dequant_q6k(W), q6k_dequant_alt(W))


def test_q6k_subdots_brute(orc):
    g = synth.rng("pin", "q6k-subdots")
    W = synth.q6k_blocks(g, 3, 768).reshape(-1, 210).copy()
    W[:, 192:208] = 1                                   # sc = 1
    W[:, 208], W[:, 209] = F16_ONE & 0xFF, F16_ONE >> 8  # d = 1  -> dequant = q - 32
    q = orc.dequant_q6k(W).astype(np.int64).reshape(3, 3, 16, 16)
    x8 = g.integers(-128, 128, size=768).astype(np.int8)
    got = orc.subdots("q6k", W, x8, 3, 768)
    want = (q * x8.astype(np.int64).reshape(1, 3, 16, 16)).sum(-1)
    assert np.array_equal(got, want)


# ---------------------------------------------------------------- f16
def test_f16_to_f32_all_patterns(orc):
    for h in range(65536):
        ref = np.uint16(h).view(np.float16).astype(np.float32)
        got = np.float32(orc.f16_to_f32(h))
        assert (np.isnan(ref) and np.isnan(got)) or ref.view(np.uint32) == got.view(np.uint32), h


def test_f32_to_f16_matches_numpy_rne(orc):
    g = synth.rng("pin", "f16")
    mags = np.exp2(g.uniform(-28, 17, 6000)).astype(np.float32)
    vals = np.concatenate([mags, -mags,
                           np.float32([0.0, -0.0, 65504, 65519.99, 65520, 65536, 1e30, -1e30,
                                       2 ** -24, 2 ** -25, 3 * 2 ** -26, 2 ** -14, 2 ** -14 - 2 ** -25,
                                       1 + 2 ** -11, 1 + 3 * 2 ** -11, 2049, 2051, np.inf, -np.inf])])
    # exact halfway cases between neighbouring f16 values
    h = np.arange(0x0400, 0x7bff, 97, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float32)
    hi = (h + 1).view(np.float16).astype(np.float32)
    vals = np.concatenate([vals, (lo + hi) / 2]).astype(np.float32)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    for v, r in zip(vals, ref):
        assert orc.f32_to_f16(v) == int(r), v


# ---------------------------------------------------------------- q8 quantizer
def test_q8_rounds_half_to_even(orc):
    """D3-5 §3.2 quantizes with rintf(x * di): ties go to even.  With
    am = 127, d = 1 and di = 1, so x*di is exact and x.5 are true ties."""
    x = np.zeros(32, np.float32)
    x[:10] = [127, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5, 126.5, -3.5, 5.5]
    d, q, s = orc.quantize_q8(x)
    assert d[0] == F16_ONE
    assert list(q[:10]) == [127, 2, 4, -2, 0, 2, 0, 126, -4, 6]
    assert s[0] == sum(int(v) for v in q)


def test_q8_zero_block_and_one_hot(orc):
    d, q, s = orc.quantize_q8(np.zeros(64, np.float32))
    assert np.all(d == 0) and np.all(q == 0) and np.all(s == 0)
    for v, k in ((1.0, 0), (-3.7, 17), (1e-3, 31), (250.0, 9)):
        x = np.zeros(32, np.float32); x[k] = v
        d, q, s = orc.quantize_q8(x)
        assert q[k] == (127 if v > 0 else -127) and np.count_nonzero(q) == 1 and s[0] == q[k]
        # f16 rounding: half an ulp, relative 2^-11 when normal, absolute 2^-25 when subnormal
        assert abs(orc.f16_to_f32(d[0]) - abs(v) / 127) <= max(abs(v) / 127 * 2 ** -11, 2 ** -25)


def test_q8_invariants_and_error_bound(orc):
    g = synth.rng("pin", "q8")
    x = np.concatenate([synth.normal(g, 4096), synth.normal(g, 4096, std=40.0)])
    d, q, s = orc.quantize_q8(x)
    xb, qb = x.reshape(-1, 32), q.reshape(-1, 32).astype(np.int64)
    assert np.all(np.abs(qb) <= 127)
    am_idx = np.argmax(np.abs(xb), axis=1)
    assert np.all(np.abs(qb[np.arange(len(qb)), am_idx]) == 127)     # d = am / 127
    assert np.array_equal(qb.sum(1), s)
    d2, q2, s2 = orc.quantize_q8(-x)                                  # odd symmetry
    assert np.array_equal(q2, -q) and np.array_equal(d2, d) and np.array_equal(s2, -s)
    dd = np.array([orc.f16_to_f32(h) for h in d])
    dtrue = np.abs(xb).max(1) / 127.0
    err = np.abs(xb - dd[:, None] * qb)
    assert np.all(err <= dtrue[:, None] * (0.5 + 1e-4) + 127 * np.abs(dd - dtrue)[:, None] + 1e-12)


# ---------------------------------------------------------------- q6_K GEMV
def test_gemv_q6k_brute_force(orc):
    g = synth.rng("pin", "gemv-q6k")
    rows, cols = 7, 1024
    W = synth.q6k_blocks(g, rows, cols)
    d8, q8, xh = xhat(orc, synth.normal(g, cols))
    y, a = orc.gemv("q6k", W, d8, q8, rows, cols)
    ref = orc.dequant_q6k(W).reshape(rows, cols) @ xh
    assert np.all(np.abs(y - ref) <= 1e-12 * a)
    # absum is the sum of |terms|, at least |y| and at most sum |w||x_hat|
    assert np.all(a >= np.abs(y)) and np.all(a <= np.abs(orc.dequant_q6k(W).reshape(rows, cols)) @ np.abs(xh) * (1 + 1e-12))


def test_gemv_q6k_one_hot_picks_each_weight(orc):
    g = synth.rng("pin", "gemv-onehot")
    W = synth.q6k_blocks(g, 2, 512)
    w = orc.dequant_q6k(W).reshape(2, 512)
    for k in range(512):
        x = np.zeros(512, np.float32); x[k] = 1.0
        d8, q8, _ = orc.quantize_q8(x)
        y, _ = orc.gemv("q6k", W, d8, q8, 2, 512)
        assert np.array_equal(y, w[:, k] * 127 * orc.f16_to_f32(d8[k // 32]))


def test_gemv_threaded_rows_equal_serial(orc):
    g = synth.rng("pin", "gemv-thr")
    W = synth.q6k_blocks(g, 37, 512)
    d8, q8, _ = xhat(orc, synth.normal(g, 512))
    y1, a1 = orc.gemv("q6k", W, d8, q8, 37, 512)
    y4, a4 = orc.gemv("q6k", W, d8, q8, 37, 512, threads=4)
    assert np.array_equal(y1, y4) and np.array_equal(a1, a4)


# ---------------------------------------------------------------- q6_K x f32 GEMV
def test_gemv_q6k_f32_brute_force(orc):
    """Against the second q6_K decode (q6k_dequant_alt) and an fp64 matmul."""
    g = synth.rng("pin", "gemv-q6k-f32")
    rows, cols = 9, 1280
    W = synth.q6k_blocks(g, rows, cols)
    x = synth.normal(g, cols)
    y, a = orc.gemv_q6k_f32(W, x, rows, cols)
    w = q6k_dequant_alt(W).reshape(rows, cols)
    ref = w @ x.astype(np.float64)
    assert np.all(np.abs(y - ref) <= 1e-12 * a)
    assert np.allclose(a, np.abs(w) @ np.abs(x.astype(np.float64)), rtol=1e-12, atol=0)


def test_gemv_q6k_f32_one_hot_picks_each_weight(orc):
    g = synth.rng("pin", "gemv-f32-onehot")
    W = synth.q6k_blocks(g, 3, 512)
    w = q6k_dequant_alt(W).reshape(3, 512)
    for k in range(0, 512, 7):
        x = np.zeros(512, np.float32)
        x[k] = -2.5
        y, _ = orc.gemv_q6k_f32(W, x, 3, 512)
        assert np.array_equal(y, -2.5 * w[:, k])


def test_gemv_q6k_f32_closed_form(orc):
    """Every code 45 (q = 13), sub-block scales 1..16, d = 2^-3, x = 1 on
    every element: y = 2^-3 * 13 * 16 * (1 + 2 + ... + 16) per block."""
    ql = np.full(128, 0xDD, np.uint8)            # low and high nibbles 13
    qh = np.zeros(64, np.uint8)
    blk = q6k_block(ql, qh, np.arange(1, 17), d_bits=0x3000)   # fp16 0.125
    nb = 3
    W = np.tile(blk, nb)
    y, a = orc.gemv_q6k_f32(W, np.ones(256 * nb, np.float32), 1, 256 * nb)
    assert y[0] == 0.125 * (13 - 32) * 16 * 136 * nb and a[0] == abs(y[0])


def test_gemv_q6k_f32_equals_q8_path_on_q8_values(orc):
    """When x is exactly f16(d8) * q8 (representable in f32), the f32-activation
    GEMV and the q8 GEMV compute the same real number."""
    g = synth.rng("pin", "gemv-f32-q8")
    rows, cols = 6, 2048
    W = synth.q6k_blocks(g, rows, cols)
    d8, q8, xh = xhat(orc, synth.normal(g, cols))
    assert np.array_equal(xh.astype(np.float32).astype(np.float64), xh)
    y1, a1 = orc.gemv_q6k_f32(W, xh.astype(np.float32), rows, cols)
    y2, _ = orc.gemv("q6k", W, d8, q8, rows, cols)
    assert np.all(np.abs(y1 - y2) <= 1e-12 * a1)


def test_gemv_q6k_f32_threaded_rows_equal_serial(orc):
    g = synth.rng("pin", "gemv-f32-thr")
    W = synth.q6k_blocks(g, 29, 512)
    x = synth.normal(g, 512)
    y1, a1 = orc.gemv_q6k_f32(W, x, 29, 512)
    y4, a4 = orc.gemv_q6k_f32(W, x, 29, 512, threads=4)
    assert np.array_equal(y1, y4) and np.array_equal(a1, a4)


# ---------------------------------------------------------------- q4_K
def test_q4k_scale_min_unpack(orc):
    g = synth.rng("pin", "q4k-sm")
    for _ in range(50):
        sc = g.integers(0, 64, 8); m = g.integers(0, 64, 8)
        blk = q4k_block(F16_ONE, F16_ONE, sc, m, np.zeros(128, np.uint8))
        for k in range(8):
            assert orc.q4k_scale_min(blk, k) == (sc[k], m[k])


def test_q4k_closed_forms(orc):
    qs = (np.arange(128) * 37 % 256).astype(np.uint8)
    nib = np.zeros(256)
    for j in range(4):
        nib[64 * j:64 * j + 32] = qs[32 * j:32 * j + 32] & 15
        nib[64 * j + 32:64 * j + 64] = qs[32 * j:32 * j + 32] >> 4
    # d = 1, dmin = 0, sc = 1: the bare nibbles
    w = orc.dequant_q4k(q4k_block(F16_ONE, 0, np.ones(8, int), np.full(8, 63), qs))
    assert np.array_equal(w, nib)
    # d = 0, dmin = 1, m = k + 1: the pure (subtracted) min term
    w = orc.dequant_q4k(q4k_block(0, F16_ONE, np.full(8, 63), np.arange(8) + 1, qs))
    assert np.array_equal(w, -np.repeat(np.arange(8) + 1.0, 32))
    # d = 2, dmin = 0.5, sc = 3, m = 4:  w = 6 q - 2
    w = orc.dequant_q4k(q4k_block(0x4000, 0x3800, np.full(8, 3), np.full(8, 4), qs))
    assert np.array_equal(w, 6 * nib - 2)


def test_q4k_matches_second_formulation(orc):
    g = synth.rng("pin", "q4k-alt")
    W = synth.q4k_blocks(g, 3, 768)
    assert np.array_equal(orc.dequant_q4k(W), q4k_dequant_alt(W, orc))


def test_q4k_subdots_and_gemv_brute(orc):
    g = synth.rng("pin", "gemv-q4k")
    rows, cols = 6, 1280
    W = synth.q4k_blocks(g, rows, cols)
    d8, q8, xh = xhat(orc, synth.normal(g, cols))
    y, a = orc.gemv("q4k", W, d8, q8, rows, cols)
    ref = orc.dequant_q4k(W).reshape(rows, cols) @ xh
    assert np.all(np.abs(y - ref) <= 1e-12 * a)
    # sub-dots against nibbles recovered from a d = 1, dmin = 0, sc = 1 copy
    Wn = W.reshape(-1, 144).copy()
    Wn[:, 0], Wn[:, 1], Wn[:, 2], Wn[:, 3] = F16_ONE & 0xFF, F16_ONE >> 8, 0, 0
    Wn[:, 4:16] = q4k_pack_scales(np.ones(8, int), np.zeros(8, int))
    nib = orc.dequant_q4k(Wn).astype(np.int64).reshape(rows, cols // 256, 8, 32)
    got = orc.subdots("q4k", W, q8, rows, cols)
    want = (nib * q8.astype(np.int64).reshape(1, cols // 256, 8, 32)).sum(-1)
    assert np.array_equal(got, want)


# ---------------------------------------------------------------- q5_K
def test_q5k_without_fifth_bits_is_q4k(orc):
    """A q5_K block whose qh bytes are zero decodes like the q4_K block with
    the same d, dmin, scales and nibbles (whose decode is pinned above)."""
    g = synth.rng("pin", "q5k-q4k")
    W5 = synth.q5k_blocks(g, 2, 1024).reshape(-1, 176).copy()
    W5[:, 16:48] = 0
    W4 = np.concatenate([W5[:, :16], W5[:, 48:]], axis=1)
    assert np.array_equal(orc.dequant_q5k(W5), orc.dequant_q4k(W4))


def test_q5k_closed_forms(orc):
    qs = (np.arange(128) * 59 % 256).astype(np.uint8)
    nib = np.zeros(256)
    for j in range(4):
        nib[64 * j:64 * j + 32] = qs[32 * j:32 * j + 32] & 15
        nib[64 * j + 32:64 * j + 64] = qs[32 * j:32 * j + 32] >> 4
    one, zero = np.ones(8, int), np.zeros(8, int)
    # every fifth bit set: d = 1, dmin = 0, sc = 1 gives nibble + 16
    w = orc.dequant_q5k(q5k_block(F16_ONE, 0, one, zero, np.full(32, 255, np.uint8), qs))
    assert np.array_equal(w, nib + 16)
    # one fifth bit at a time: bit k of qh[l] lifts weight 32k + l alone
    for k in range(8):
        for l in (0, 13, 31):
            qh = np.zeros(32, np.uint8)
            qh[l] = 1 << k
            w = orc.dequant_q5k(q5k_block(F16_ONE, 0, one, zero, qh, qs))
            want = nib.copy()
            want[32 * k + l] += 16
            assert np.array_equal(w, want), (k, l)
    # d = 2, dmin = 0.5, sc = 3, m = 4, all fifth bits: w = 6 (q + 16) - 2
    w = orc.dequant_q5k(q5k_block(0x4000, 0x3800, np.full(8, 3), np.full(8, 4),
                                  np.full(32, 255, np.uint8), qs))
    assert np.array_equal(w, 6 * (nib + 16) - 2)


def test_q5k_matches_second_formulation(orc):
    g = synth.rng("pin", "q5k-alt")
    W = synth.q5k_blocks(g, 3, 768)
    assert np.array_equal(orc.dequant_q5k(W), q5k_dequant_alt(W, orc))


def test_q5k_subdots_and_gemv_brute(orc):
    g = synth.rng("pin", "gemv-q5k")
    rows, cols = 6, 1280
    W = synth.q5k_blocks(g, rows, cols)
    d8, q8, xh = xhat(orc, synth.normal(g, cols))
    y, a = orc.gemv("q5k", W, d8, q8, rows, cols)
    ref = orc.dequant_q5k(W).reshape(rows, cols) @ xh
    assert np.all(np.abs(y - ref) <= 1e-12 * a)
    # sub-dots against codes recovered from a d = 1, dmin = 0, sc = 1 copy
    Wn = W.reshape(-1, 176).copy()
    Wn[:, 0], Wn[:, 1], Wn[:, 2], Wn[:, 3] = F16_ONE & 0xFF, F16_ONE >> 8, 0, 0
    Wn[:, 4:16] = q4k_pack_scales(np.ones(8, int), np.zeros(8, int))
    codes = orc.dequant_q5k(Wn).astype(np.int64).reshape(rows, cols // 256, 8, 32)
    assert codes.min() >= 0 and codes.max() <= 31
    got = orc.subdots("q5k", W, q8, rows, cols)
    want = (codes * q8.astype(np.int64).reshape(1, cols // 256, 8, 32)).sum(-1)
    assert np.array_equal(got, want)


# ---------------------------------------------------------------- producers
def test_rmsnorm_closed_forms(orc):
    g = synth.rng("pin", "rms")
    gain = synth.normal(g, 64, 1.0, 0.1)
    for c in (0.75, -3.0):
        x = np.full(64, c, np.float32)
        assert np.allclose(orc.rmsnorm(x, gain, 0.0), np.sign(c) * gain, rtol=1e-15, atol=0)
        # eps sits inside the root, added to the mean square: eps = c^2 gives 1/sqrt(2)
        y = orc.rmsnorm(x, gain, np.float32(c * c))
        assert np.allclose(y, np.sign(c) * gain / np.sqrt(2.0), rtol=1e-7, atol=0)
    assert np.all(orc.rmsnorm(np.zeros(64, np.float32), gain, 1e-6) == 0)
    x = synth.normal(g, 4096)
    y = orc.rmsnorm(x, np.ones(4096, np.float32), 1e-6)
    ms = float(np.mean(x.astype(np.float64) ** 2))
    assert abs(np.mean(y ** 2) - ms / (ms + 1e-6)) < 1e-12
    # scale invariance with eps = 0
    assert np.allclose(orc.rmsnorm(x * np.float32(8.0), gain[:1].repeat(4096), 0.0),
                       orc.rmsnorm(x, gain[:1].repeat(4096), 0.0), rtol=1e-14, atol=0)


def test_swiglu_identities(orc):
    special = pytest.importorskip("scipy.special")
    g = synth.rng("pin", "swiglu")
    gv = synth.normal(g, 4096, std=4.0)
    uv = synth.normal(g, 4096)
    y = orc.swiglu(gv, uv)
    assert np.allclose(y, gv.astype(np.float64) * special.expit(gv.astype(np.float64)) * uv,
                       rtol=1e-13, atol=1e-300)
    one = np.ones(4096, np.float32)
    # silu(g) - silu(-g) = g pins the sign inside the exponential
    assert np.allclose(orc.swiglu(gv, one) - orc.swiglu(-gv, one), gv, rtol=1e-12, atol=1e-12)
    assert np.all(orc.swiglu(np.zeros(8, np.float32), one[:8]) == 0)
