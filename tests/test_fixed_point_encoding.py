"""Kernel-claims test (not an oracle pin): the block fixed-point activation
encoding of the batch-1 kernels' opt-in arithmetic (QDQ_OPT_XS_FLOAT_X = 0),
restated in numpy and checked against the claims its stated error bound rests on:

* e = 148 - max(E, 1), E the biased exponent of the block's largest |x|, puts
  every X_j = rint(x_j 2^e) in [-2^22, 2^22];
* |x_j - X_j 2^-e| <= 2^-22 max|x| (so a row's error is at most
  2^-22 sum_b max_b|x| sum_b |w| before f32 rounding);
* X_j = L2 2^16 + L1 2^8 + L0 with L0, L1 unsigned bytes and L2 in [-64, 64],
  so each limb fits the byte lanes of a dp4a;
* q_j int8 or u4 against those limbs: every per-limb dot product over 32 weights
  fits int32, and so does c0 + 256 c1;
* the Q4_K sub-block shift applied to the exact sums, hi = c2 - mu S2 and
  lo = c0 + 256 c1 - mu (S0 + 256 S1) with S_l = sum_j L_l, stays within int32 and
  reassembles sum (q - mu) X exactly.

This is a statement of the arithmetic, not a copy of the kernel: the GPU tests
compare the kernel itself with the oracle.
"""
import numpy as np
import pytest


def encode(xb):
    """One 32-element f32 block -> (X int64[32], e)."""
    xb = np.asarray(xb, dtype=np.float32)
    m = np.abs(xb).max()
    E = int(m.view(np.uint32)) >> 23
    assert E < 255
    e = 148 - max(E, 1)
    X = np.rint(xb.astype(np.float64) * 2.0 ** e).astype(np.int64)  # x 2^e exact in float64
    return X, e


def limbs(X):
    L0 = X & 0xFF
    L1 = (X >> 8) & 0xFF
    L2 = X >> 16
    return L0, L1, L2


def _blocks(rng):
    yield rng.standard_normal(32).astype(np.float32)
    yield (1e4 * rng.standard_normal(32)).astype(np.float32)
    yield np.float32(3e38) * np.sign(rng.standard_normal(32)).astype(np.float32)   # largest finite
    yield np.full(32, np.float32(1.0))                                             # exact powers of two
    yield np.full(32, np.float32(-2.0 ** -126))
    yield (np.float32(1e-40) * rng.standard_normal(32)).astype(np.float32)        # subnormal maximum
    yield np.zeros(32, np.float32)
    b = (1e-3 * rng.standard_normal(32)).astype(np.float32)
    b[7] = 1e4                                                                      # huge in-block range
    yield b
    yield np.nextafter(np.float32(2.0), np.float32(0.0)) * np.ones(32, np.float32)  # just below 2^E+1


def test_exponent_range_and_rounding_bound():
    rng = np.random.default_rng(0)
    for xb in list(_blocks(rng)) + [rng.standard_normal(32).astype(np.float32) * 10.0 ** rng.uniform(-30, 30)
                                    for _ in range(2000)]:
        X, e = encode(xb)
        assert -106 <= e <= 147
        assert np.abs(X).max() <= 2 ** 22
        m = float(np.abs(xb).max())
        err = np.abs(xb.astype(np.float64) - X * 2.0 ** -e)
        if m >= 2.0 ** -126:       # normal maximum: the relative bound
            assert np.all(err <= 2.0 ** -22 * m)
        else:                      # zero or subnormal maximum: absolute 2^-148
            assert np.all(err <= 2.0 ** -148)
        if m >= 2.0 ** -126:       # the largest element keeps 21+ bits
            assert np.abs(X).max() >= 2 ** 21


def test_limb_identity_and_ranges():
    rng = np.random.default_rng(1)
    X = np.concatenate([np.arange(-2 ** 22, -2 ** 22 + 5000), np.arange(-5000, 5000),
                        np.arange(2 ** 22 - 5000, 2 ** 22 + 1), rng.integers(-2 ** 22, 2 ** 22 + 1, 100000)])
    L0, L1, L2 = limbs(X)
    assert np.all((0 <= L0) & (L0 <= 255)) and np.all((0 <= L1) & (L1 <= 255))
    assert np.all((-64 <= L2) & (L2 <= 64))
    assert np.array_equal(L2 * 65536 + L1 * 256 + L0, X)


@pytest.mark.parametrize("q_lo,q_hi", [(-128, 127), (0, 15)])
def test_limb_dot_products_fit_int32(q_lo, q_hi):
    # worst case over 32 weights: every |q| at its largest against the largest limbs
    q = np.full(32, q_lo if abs(q_lo) > abs(q_hi) else q_hi, dtype=np.int64)
    for L in (np.full(32, 255), np.full(32, 0), np.full(32, -64), np.full(32, 64)):
        c = int((q * L).sum())
        assert -2 ** 31 <= c < 2 ** 31
    c0 = int(np.abs(q).sum()) * 255
    c1 = int(np.abs(q).sum()) * 255
    assert c0 + 256 * c1 < 2 ** 31


def test_limb_dot_products_reassemble_the_exact_sum():
    rng = np.random.default_rng(2)
    for _ in range(200):
        xb = (rng.standard_normal(32) * 10.0 ** rng.uniform(-5, 5)).astype(np.float32)
        X, e = encode(xb)
        L0, L1, L2 = limbs(X)
        q = rng.integers(-128, 128, 32)
        c0, c1, c2 = int((q * L0).sum()), int((q * L1).sum()), int((q * L2).sum())
        assert c2 * 65536 + (c0 + 256 * c1) == int((q * X).sum())


@pytest.mark.parametrize("mu", [0, 7, 15])
def test_q4k_shifted_limb_sums_fit_int32_and_reassemble(mu):
    rng = np.random.default_rng(7 + mu)
    for xb in _blocks(rng):
        X, _ = encode(xb)
        L0, L1, L2 = limbs(X)
        for q in (np.full(32, 15), np.zeros(32, np.int64), rng.integers(0, 16, 32)):
            c0, c1, c2 = (int((q * L).sum()) for L in (L0, L1, L2))
            hi = c2 - mu * int(L2.sum())
            lo = c0 + 256 * c1 - mu * int((X & 0xFFFF).sum())
            assert abs(hi) < 2 ** 17 and abs(lo) < 2 ** 26
            assert hi * 65536 + lo == int(((q - mu) * X).sum())
