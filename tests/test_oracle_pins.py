"""Pins for the CPU oracle: each check ties it to something other than itself.

* IEEE binary16 decoding: exhaustive against numpy's float16, plus hand-worked
  values from the binary16 definition (tests/golden/fp16_special_values.txt).
* Q8_0 dequant: hand-built blocks with closed-form values (column mapping,
  sign, extremes -128/127, negative scale).
* Q4_K dequant: hand-worked scale/min byte patterns
  (tests/golden/q4k_scale_fields.txt), a field-wise encoder written from the
  layout description (round trip), one-hot scale/min superblocks that light
  exactly one sub-block, and a nibble-order pattern.
* GEMV: one-hot x extracts a column of a non-square W (catches transposes);
  exact rational (fractions.Fraction) dot products on tiny shapes; linearity.
* SwiGLU / FFN: silu identities and closed forms; one-hot W_up rows; W_down = 0
  gives the residual exactly; identity W_down gives residual + mid.
* Batch GEMM: M = 1 equals the GEMV; permuting X rows permutes Y rows.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from conftest import GOLDEN

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- fp16 decode

def test_fp16_decoder_exhaustive_against_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.fp16_bits_to_f64(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_fp16_decoder_golden_values():
    rows = []
    with open(os.path.join(GOLDEN, "fp16_special_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            b, v = line.split()
            rows.append((int(b, 16), float(v)))
    got = oracle.fp16_bits_to_f64(np.array([b for b, _ in rows], dtype=np.uint16))
    for (b, v), g in zip(rows, got):
        if math.isnan(v):
            assert math.isnan(g), hex(b)
        else:
            assert g == v and math.copysign(1, g) == math.copysign(1, v), (hex(b), g, v)


# ---------------------------------------------------------------- Q8_0

def _q8_block(d_bits: int, q):
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (32,)
    return np.concatenate([[d_bits & 0xFF, d_bits >> 8], (q & 0xFF)]).astype(np.uint8)


def test_q8_0_unit_scale_block():
    # d = 1.0 (0x3c00), q[k] = k - 16  ->  weight k = k - 16
    blk = _q8_block(0x3C00, np.arange(32) - 16)
    w = oracle.q8_0_dequant(blk[None, :], 1, 32)
    assert w.dtype == np.float32
    assert np.array_equal(w[0], np.arange(32, dtype=np.float32) - 16)


def test_q8_0_full_int8_range_power_of_two_scale():
    # d = 2^-10 (0x1400); q runs over all of int8 including -128 -> q * 2^-10 exactly
    qs = np.arange(-128, 128)
    row = np.concatenate([_q8_block(0x1400, qs[32 * b: 32 * b + 32]) for b in range(8)])
    w = oracle.q8_0_dequant(row[None, :], 1, 256)
    assert np.array_equal(w[0], (qs * 2.0 ** -10).astype(np.float32))


def test_q8_0_column_mapping_and_sign():
    # 2 rows x 64 cols; block b of row r has its own scale; element k of block b is column 32b+k
    scales = {(0, 0): (0x3C00, 1.0), (0, 1): (0x4000, 2.0), (1, 0): (0xBC00, -1.0), (1, 1): (0x3800, 0.5)}
    rows = []
    for r in range(2):
        blocks = []
        for b in range(2):
            q = (np.arange(32) + 1) * (1 if b == 0 else -1) + 10 * r
            blocks.append(_q8_block(scales[(r, b)][0], q))
        rows.append(np.concatenate(blocks))
    w = oracle.q8_0_dequant(np.stack(rows), 2, 64)
    for r in range(2):
        for b in range(2):
            q = (np.arange(32) + 1) * (1 if b == 0 else -1) + 10 * r
            assert np.array_equal(w[r, 32 * b: 32 * b + 32], (scales[(r, b)][1] * q).astype(np.float32))


def test_q8_0_extremes_exact():
    # largest |d| and |q|: 65504 * -128 is exact in f32
    blk = _q8_block(0x7BFF, np.array([-128, 127] + [0] * 30))
    w = oracle.q8_0_dequant(blk[None, :], 1, 32)
    assert w[0, 0] == np.float32(-8384512.0) and w[0, 1] == np.float32(65504.0 * 127)


# ---------------------------------------------------------------- Q4_K

def _golden_scale_rows():
    out = []
    with open(os.path.join(GOLDEN, "q4k_scale_fields.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            b, sc, m = [p.strip() for p in line.split("|")]
            out.append((np.array([int(t, 16) for t in b.split()], dtype=np.uint8),
                        [int(t) for t in sc.split()], [int(t) for t in m.split()]))
    return out


@pytest.mark.parametrize("row", range(20))
def test_q4k_scale_fields_golden(row):
    b, sc, m = _golden_scale_rows()[row]
    got_sc, got_m = oracle.q4k_scales_mins(b[None, :])
    assert list(got_sc[0]) == sc and list(got_m[0]) == m


def _encode_scale_fields(sc, m):
    """Field-wise encoder written from the placement description (not by inverting the decoder)."""
    out = [0] * 12
    for j in range(8):
        if j < 4:
            out[j] |= sc[j] & 63
            out[4 + j] |= m[j] & 63
        else:
            lo_sc, hi_sc = sc[j] & 15, sc[j] >> 4
            lo_m, hi_m = m[j] & 15, m[j] >> 4
            out[8 + (j - 4)] |= lo_sc | (lo_m << 4)
            out[j - 4] |= hi_sc << 6
            out[4 + (j - 4)] |= hi_m << 6
    return np.array(out, dtype=np.uint8)


def test_q4k_scale_fields_roundtrip_random():
    rng = np.random.default_rng(1234)
    for _ in range(500):
        sc = rng.integers(0, 64, 8)
        m = rng.integers(0, 64, 8)
        got_sc, got_m = oracle.q4k_scales_mins(_encode_scale_fields(sc, m)[None, :])
        assert np.array_equal(got_sc[0], sc) and np.array_equal(got_m[0], m)


def _q4k_superblock(d_bits, dmin_bits, scales12, qs128):
    return np.concatenate([[d_bits & 0xFF, d_bits >> 8, dmin_bits & 0xFF, dmin_bits >> 8],
                           scales12, qs128]).astype(np.uint8)


def _nibble_pattern():
    # byte i: low nibble = i % 16, high nibble = 15 - i % 16
    i = np.arange(128)
    return ((i % 16) | ((15 - i % 16) << 4)).astype(np.uint8)


def _expected_q_of_pattern():
    q = np.empty(256, dtype=np.int64)
    for c in range(4):
        for l in range(32):
            q[64 * c + l] = (32 * c + l) % 16
            q[64 * c + 32 + l] = 15 - (32 * c + l) % 16
    return q


@pytest.mark.parametrize("j", range(8))
@pytest.mark.parametrize("v", [1, 37, 63])
def test_q4k_one_hot_scale_lights_one_subblock(j, v):
    sc = [0] * 8
    sc[j] = v
    sb = _q4k_superblock(0x3C00, 0x3C00, _encode_scale_fields(sc, [0] * 8), _nibble_pattern())
    w = oracle.q4k_dequant(sb[None, :], 1, 256)[0]
    q = _expected_q_of_pattern()
    expect = np.zeros(256)
    expect[32 * j: 32 * j + 32] = v * q[32 * j: 32 * j + 32]
    assert np.array_equal(w, expect.astype(np.float32))


@pytest.mark.parametrize("j", range(8))
def test_q4k_one_hot_min_lights_one_subblock(j):
    m = [0] * 8
    m[j] = 63
    # d = 1, dmin = 0.5, all scales 0  ->  weight = -0.5 * 63 in sub-block j, 0 elsewhere
    sb = _q4k_superblock(0x3C00, 0x3800, _encode_scale_fields([0] * 8, m), _nibble_pattern())
    w = oracle.q4k_dequant(sb[None, :], 1, 256)[0]
    expect = np.zeros(256)
    expect[32 * j: 32 * j + 32] = -0.5 * 63
    assert np.array_equal(w, expect.astype(np.float32))


def test_q4k_nibble_order_and_formula():
    # all sc = 1, m = 2, d = 2, dmin = 0.25: weight = 2*q - 0.5 with q from the pattern
    sb = _q4k_superblock(0x4000, 0x3400, _encode_scale_fields([1] * 8, [2] * 8), _nibble_pattern())
    w = oracle.q4k_dequant(sb[None, :], 1, 256)[0]
    assert np.array_equal(w, (2.0 * _expected_q_of_pattern() - 0.5).astype(np.float32))


def test_q4k_multi_superblock_rows():
    # 2 rows x 2 superblocks with distinct d: superblock s of row r covers columns 256s..256s+255
    d_bits = [[0x3C00, 0x4000], [0x3800, 0xBC00]]
    d_val = [[1.0, 2.0], [0.5, -1.0]]
    rows = []
    for r in range(2):
        rows.append(np.concatenate([
            _q4k_superblock(d_bits[r][s], 0x0000, _encode_scale_fields([3] * 8, [0] * 8), _nibble_pattern())
            for s in range(2)]))
    w = oracle.q4k_dequant(np.stack(rows), 2, 512)
    q = _expected_q_of_pattern()
    for r in range(2):
        for s in range(2):
            assert np.array_equal(w[r, 256 * s: 256 * s + 256], (d_val[r][s] * 3 * q).astype(np.float32))


def test_q4k_subtraction_rounds_once_in_f32():
    # a = d*sc*q and b = dmin*m chosen so that a - b needs more than 24 bits:
    # d = 2^-14 (0x0400), sc = 63, q = 15 -> a = 945 * 2^-14; dmin = 65504 (0x7bff), m = 63
    sc = [63] * 8
    m = [63] * 8
    qs = np.full(128, 0xFF, dtype=np.uint8)
    sb = _q4k_superblock(0x0400, 0x7BFF, _encode_scale_fields(sc, m), qs)
    w = oracle.q4k_dequant(sb[None, :], 1, 256)[0]
    a = Fraction(945, 2 ** 14)
    b = Fraction(65504 * 63)
    expect = _round_to_f32(a - b)
    assert Fraction(float(expect)) != a - b              # the difference is not representable
    assert np.all(w == expect)


def _round_to_f32(fr: Fraction) -> np.float32:
    """Round an exact rational to the nearest f32 (ties to even), by comparing exact distances."""
    f = np.float32(float(fr))
    best = None
    for c in (np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))):
        dist = abs(Fraction(float(c)) - fr)
        even = (int(np.array(c).view(np.uint32)) & 1) == 0
        key = (dist, not even)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


# ---------------------------------------------------------------- GEMV

def _small_q8(n_out, n_in, seed):
    return oracle.q8_0_dequant(synth.q8_0_blocks(np.random.default_rng(seed), n_out, n_in), n_out, n_in)


def _small_q4k(n_out, n_in, seed):
    return oracle.q4k_dequant(synth.q4k_blocks(np.random.default_rng(seed), n_out, n_in), n_out, n_in)


@pytest.mark.parametrize("fmt", ["q8_0", "q4k"])
def test_gemv_one_hot_extracts_column(fmt):
    n_out, n_in = (5, 96) if fmt == "q8_0" else (3, 512)
    w = _small_q8(n_out, n_in, 7) if fmt == "q8_0" else _small_q4k(n_out, n_in, 7)
    for k in [0, 1, n_in // 2 + 3, n_in - 1]:
        x = np.zeros((1, n_in), np.float32)
        x[0, k] = 1.0
        y, a = oracle.gemv(w, x)
        assert np.array_equal(y[0], w[:, k].astype(np.float64))
        assert np.array_equal(a[0], np.abs(w[:, k]).astype(np.float64))


@pytest.mark.parametrize("fmt", ["q8_0", "q4k"])
def test_gemv_exact_rational_tiny(fmt):
    n_out, n_in = (3, 64) if fmt == "q8_0" else (2, 256)
    w = _small_q8(n_out, n_in, 11) if fmt == "q8_0" else _small_q4k(n_out, n_in, 11)
    x = synth.activations(np.random.default_rng(3), 2, n_in)
    y, a = oracle.gemv(w, x)
    for b in range(2):
        for r in range(n_out):
            exact = sum(Fraction(float(w[r, k])) * Fraction(float(x[b, k])) for k in range(n_in))
            exact_a = sum(abs(Fraction(float(w[r, k])) * Fraction(float(x[b, k]))) for k in range(n_in))
            assert abs(Fraction(y[b, r]) - exact) <= Fraction(exact_a) * Fraction(1, 2 ** 45)
            assert abs(Fraction(a[b, r]) - exact_a) <= Fraction(exact_a) * Fraction(1, 2 ** 45)


def test_gemv_linearity():
    w = _small_q8(17, 160, 5)
    rng = np.random.default_rng(9)
    x1 = synth.activations(rng, 1, 160)
    x2 = synth.activations(rng, 1, 160)
    y1, a1 = oracle.gemv(w, x1)
    y2, a2 = oracle.gemv(w, x2)
    y12, _ = oracle.gemv(w, 2.0 * x1.astype(np.float64) - 0.5 * x2.astype(np.float64))
    assert np.all(np.abs(y12 - (2.0 * y1 - 0.5 * y2)) <= 1e-12 * (2 * a1 + 0.5 * a2))


def test_gemv_batch_rows_are_independent():
    w = _small_q4k(4, 256, 2)
    x = synth.activations(np.random.default_rng(4), 3, 256)
    yb, ab = oracle.gemv(w, x)
    for b in range(3):
        y, a = oracle.gemv(w, x[b:b + 1])
        assert np.array_equal(yb[b], y[0]) and np.array_equal(ab[b], a[0])


# ---------------------------------------------------------------- SwiGLU / FFN

def test_silu_closed_forms():
    z = np.array([0.0, math.log(3.0), -math.log(3.0), 40.0, -800.0, 1.0])
    s = oracle.silu(z)
    assert s[0] == 0.0
    assert abs(s[1] - 0.75 * math.log(3.0)) <= 1e-15          # sigmoid(ln 3) = 3/4
    assert abs(s[2] + 0.25 * math.log(3.0)) <= 1e-15          # sigmoid(-ln 3) = 1/4
    assert abs(s[3] - 40.0) <= 40.0 * 1e-15
    assert s[4] <= 0.0 and abs(s[4]) < 1e-300
    # silu(z) - silu(-z) = z for any z
    zz = np.linspace(-30, 30, 601)
    assert np.all(np.abs(oracle.silu(zz) - oracle.silu(-zz) - zz) <= 1e-13 * (1 + np.abs(zz)))


def test_swiglu_one_hot_up_rows():
    n_ff, n_embd = 8, 256
    wg = _small_q4k(n_ff, n_embd, 21)
    wu = np.zeros((n_ff, n_embd), np.float32)
    cols = [5, 0, 255, 17, 100, 3, 64, 128]
    for i, k in enumerate(cols):
        wu[i, k] = 1.0
    x = synth.activations(np.random.default_rng(22), 1, n_embd)
    s = oracle.swiglu(wg, wu, x)
    g, _ = oracle.gemv(wg, x)
    for i, k in enumerate(cols):
        gi = g[0, i]
        assert s["u"][0, i] == float(x[0, k])
        assert abs(s["mid"][0, i] - gi / (1.0 + math.exp(-gi)) * float(x[0, k])) <= 1e-15 * abs(gi * x[0, k]) + 1e-300


def test_ffn_zero_down_gives_residual_exactly():
    n_embd, n_ff = 256, 512
    wg, wu = _small_q4k(n_ff, n_embd, 31), _small_q4k(n_ff, n_embd, 32)
    wd = np.zeros((n_embd, n_ff), np.float32)
    x, res = (synth.activations(np.random.default_rng(s), 1, n_embd) for s in (33, 34))
    o = oracle.ffn_residual(wg, wu, wd, x, res)
    assert np.array_equal(o["out"], res.astype(np.float64))


def test_ffn_identity_down_gives_residual_plus_mid():
    n = 256
    wg, wu = _small_q4k(n, n, 41), _small_q4k(n, n, 42)
    wd = np.eye(n, dtype=np.float32)
    x, res = (synth.activations(np.random.default_rng(s), 1, n) for s in (43, 44))
    o = oracle.ffn_residual(wg, wu, wd, x, res)
    assert np.array_equal(o["out"], res.astype(np.float64) + o["mid"])


# ---------------------------------------------------------------- fused QKV

def test_qkv_one_hot_extracts_each_matrix_column():
    # distinct matrices and a non-square Q: one-hot x gives column j of each, in its own output
    n_q, n_kv, n_in = 12, 4, 512
    wq, wk, wv = _small_q4k(n_q, n_in, 61), _small_q4k(n_kv, n_in, 62), _small_q4k(n_kv, n_in, 63)
    for j in (0, 255, 256, 511):
        x = np.zeros((1, n_in), np.float32)
        x[0, j] = 1.0
        o = oracle.qkv(wq, wk, wv, x)
        assert o["q"].shape == (1, n_q) and o["k"].shape == (1, n_kv) and o["v"].shape == (1, n_kv)
        assert np.array_equal(o["q"][0], wq[:, j].astype(np.float64))
        assert np.array_equal(o["k"][0], wk[:, j].astype(np.float64))
        assert np.array_equal(o["v"][0], wv[:, j].astype(np.float64))


def test_qkv_closed_form_constant_matrices():
    # W_q = 1, W_k = 2, W_v = -3 everywhere (d = 1, q = 1, 2, -3) and x = 1: q = n_in, k = 2 n_in, v = -3 n_in
    n_q, n_kv, n_in = 8, 2, 64
    def const_q8(rows, val):
        blk = np.zeros((rows, n_in // 32, 34), np.uint8)
        blk[..., 0:2] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
        blk[..., 2:] = np.uint8(val & 0xFF)
        return oracle.q8_0_dequant(blk.reshape(rows, -1), rows, n_in)
    o = oracle.qkv(const_q8(n_q, 1), const_q8(n_kv, 2), const_q8(n_kv, -3), np.ones((1, n_in), np.float32))
    assert np.all(o["q"] == n_in) and np.all(o["k"] == 2 * n_in) and np.all(o["v"] == -3 * n_in)
    assert np.all(o["A_v"] == 3 * n_in)


def test_qkv_rejects_kv_wider_than_q():
    w = _small_q8(4, 64, 1)
    with pytest.raises(ValueError):
        oracle.qkv(w[:2], w, w, np.ones((1, 64), np.float32))
    with pytest.raises(ValueError):
        oracle.qkv(w, w[:2], w[:3], np.ones((1, 64), np.float32))


# ---------------------------------------------------------------- output projection + argmax

def test_logits_argmax_closed_form_and_first_of_ties():
    # one-hot x picks column 5; rows 3 and 7 hold the same largest value there (index 3, the
    # first of the tie); row 9's large weight sits in a column x does not use
    n_vocab, n_in = 12, 64
    w = np.zeros((n_vocab, n_in), np.float32)
    w[:, 5] = np.arange(n_vocab, dtype=np.float32) * 0.25 - 2.0
    w[3, 5] = w[7, 5] = 9.5
    w[9, 6] = 100.0
    x = np.zeros((2, n_in), np.float32)
    x[0, 5] = 1.0
    x[1, 5] = -1.0                      # negated: the smallest entry of column 5 wins
    o = oracle.logits_argmax(w, x)
    assert o["index"][0] == 3 and o["value"][0] == 9.5
    assert o["index"][1] == 0 and o["value"][1] == 2.0


def test_logits_argmax_nan_wins_and_matches_numpy():
    rng = np.random.default_rng(71)
    w = _small_q8(300, 96, 72)
    x = synth.activations(rng, 3, 96)
    o = oracle.logits_argmax(w, x)
    assert np.array_equal(o["index"], np.argmax(o["logits"], axis=1))
    assert np.array_equal(o["value"], o["logits"].max(axis=1))
    x[1, 10] = np.nan
    o = oracle.logits_argmax(w, x)
    assert o["index"][1] == 0 and np.isnan(o["value"][1])
    assert np.array_equal(o["index"], np.argmax(o["logits"], axis=1))


# ---------------------------------------------------------------- batch GEMM

def test_gemm_batch_m1_equals_gemv_and_permutes_rows():
    w = _small_q8(24, 128, 51)
    x = synth.activations(np.random.default_rng(52), 9, 128)
    y, a = oracle.gemm_batch(w, x)
    y1, _ = oracle.gemv(w, x[4:5])
    assert np.array_equal(y[4], y1[0])
    perm = np.random.default_rng(53).permutation(9)
    yp, ap = oracle.gemm_batch(w, x[perm])
    assert np.array_equal(yp, y[perm]) and np.array_equal(ap, a[perm])


# ---------------------------------------------------------------- Q6_K

def _q6k_block(ql=None, qh=None, scales=None, d_bits=0x3C00):
    """One 210-byte Q6_K superblock: ql (128), qh (64), int8 scales (16), fp16 d."""
    b = np.zeros(210, dtype=np.uint8)
    if ql is not None:
        b[0:128] = ql
    if qh is not None:
        b[128:192] = qh
    if scales is not None:
        b[192:208] = np.asarray(scales, dtype=np.int64).astype(np.int8).view(np.uint8)
    b[208], b[209] = d_bits & 0xFF, d_bits >> 8
    return b


def _golden_q6k():
    rows = []
    with open(os.path.join(GOLDEN, "q6k_quants.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("|")
            ql, qh = np.zeros(128, np.uint8), np.zeros(64, np.uint8)
            for tok in lhs.split():
                name, val = tok.split("=")
                plane, idx = name.rstrip("]").split("[")
                (ql if plane == "ql" else qh)[int(idx)] = int(val, 16)
            want = np.zeros(256, np.int64)
            for tok in rhs.split():
                e, q = tok.split("=")
                want[int(e)] = int(q)
            rows.append((ql, qh, want))
    return rows


@pytest.mark.parametrize("row", range(6))
def test_q6k_quants_golden(row):
    ql, qh, want = _golden_q6k()[row]
    assert np.array_equal(oracle.q6k_quants(ql[None], qh[None])[0], want)


def _q6k_encode(q):
    """Field-wise encoder written from the placement text, one weight at a time."""
    ql, qh = np.zeros(128, np.uint8), np.zeros(64, np.uint8)
    for e in range(256):
        h, p = divmod(e, 128)
        t, l = divmod(p, 32)
        i = 64 * h + 32 * (t & 1) + l
        ql[i] |= (int(q[e]) & 0xF) << (4 * (t >> 1))
        qh[32 * h + l] |= (int(q[e]) >> 4) << (2 * t)
    return ql, qh


def test_q6k_quants_roundtrip_random():
    rng = np.random.default_rng(91)
    for _ in range(20):
        q = rng.integers(0, 64, 256)
        ql, qh = _q6k_encode(q)
        assert np.array_equal(oracle.q6k_quants(ql[None], qh[None])[0], q)


@pytest.mark.parametrize("j", range(16))
def test_q6k_one_hot_scale_lights_one_subblock(j):
    # every q = 33 (q - 32 = 1), d = 1, only scale j non-zero: weights 16j..16j+15 equal it
    ql, qh = _q6k_encode(np.full(256, 33))
    sc = np.zeros(16, np.int64)
    sc[j] = -77
    w = oracle.q6k_dequant(_q6k_block(ql, qh, sc), 1, 256)[0]
    want = np.zeros(256, np.float32)
    want[16 * j: 16 * j + 16] = -77.0
    assert np.array_equal(w, want)


def test_q6k_extremes_exact_and_two_rows():
    # q = 0 and 63 against scale -128 and the largest fp16 d: d*sc*(q-32) exact in f32
    q = np.where(np.arange(256) % 2 == 0, 0, 63)
    ql, qh = _q6k_encode(q)
    d_max = 0x7BFF  # 65504
    b0 = _q6k_block(ql, qh, np.full(16, -128), d_max)
    b1 = _q6k_block(ql, qh, np.arange(16) - 8, 0x0001)  # smallest subnormal d = 2^-24
    w = oracle.q6k_dequant(np.stack([np.concatenate([b0, b1]), np.concatenate([b1, b0])]), 2, 512)
    for r, (first, second) in enumerate(((b0, b1), (b1, b0))):
        for half, blk in enumerate((first, second)):
            d = Fraction(65504) if blk is b0 else Fraction(1, 2 ** 24)
            for e in (0, 1, 17, 254, 255):
                sc = -128 if blk is b0 else (e // 16) - 8
                exact = d * sc * (int(q[e]) - 32)
                assert Fraction(float(w[r, 256 * half + e])) == exact


def test_q6k_gemv_one_hot_extracts_column():
    wb = synth.q6k_blocks(np.random.default_rng(92), 7, 512)
    w = oracle.q6k_dequant(wb, 7, 512)
    for k in (0, 15, 16, 255, 256, 511):
        x = np.zeros((1, 512), np.float32)
        x[0, k] = 1.0
        y, a = oracle.gemv(w, x)
        assert np.array_equal(y[0], w[:, k].astype(np.float64))


def test_get_rows_picks_rows_and_nans_bad_ids():
    w = _small_q8(10, 64, 93)
    out = oracle.get_rows(w, [3, 0, 9, 3, 10, -1])
    assert np.array_equal(out[0], w[3]) and np.array_equal(out[1], w[0]) and np.array_equal(out[2], w[9])
    assert np.array_equal(out[3], w[3]) and np.all(np.isnan(out[4])) and np.all(np.isnan(out[5]))


# ---------------------------------------------------------------- top-k

def test_logits_topk_closed_form_with_ties():
    # one-hot rows: logit r = x[col(r)]; rows 1 and 3 tie at 7, rows 0 and 5 tie at 9
    w = np.eye(6, dtype=np.float32)[[3, 1, 4, 1, 0, 3]]
    x = np.array([[5, 7, 2, 9, 1, 0]], np.float32)
    o = oracle.logits_topk(w, x, 6)
    assert list(o["index"][0]) == [0, 5, 1, 3, 4, 2]
    assert list(o["value"][0]) == [9, 9, 7, 7, 5, 1]


def test_logits_topk_matches_lexsort_and_argmax():
    rng = np.random.default_rng(94)
    w = _small_q8(500, 96, 95)
    x = synth.activations(rng, 3, 96)
    for k in (1, 8, 40):
        o = oracle.logits_topk(w, x, k)
        for b in range(3):
            order = np.lexsort((np.arange(500), -o["logits"][b]))   # value desc, then index asc
            assert np.array_equal(o["index"][b], order[:k])
            assert np.array_equal(o["value"][b], o["logits"][b][order[:k]])
        if k == 1:
            assert np.array_equal(o["index"][:, 0], oracle.logits_argmax(w, x)["index"])


def test_logits_topk_nan_first():
    w = _small_q8(50, 64, 96)
    x = synth.activations(np.random.default_rng(97), 2, 64)
    x[1, 3] = np.nan
    o = oracle.logits_topk(w, x, 5)
    assert list(o["index"][1]) == [0, 1, 2, 3, 4] and np.all(np.isnan(o["value"][1]))
    assert np.all(np.isfinite(o["value"][0]))
