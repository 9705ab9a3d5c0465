"""The accuracy argument of the chunked backward's products (three TF32 passes), checked on
the CPU from the TF32 format's definition (8 exponent bits and 10 explicit mantissa bits;
conversion from fp32 rounds to nearest, ties away from zero): an fp32 value x splits into
hi = tf32(x) and lo = tf32(x - hi), and hi_a hi_b + hi_a lo_b + lo_a hi_b reproduces a b to
within a few 2^-22 relative, the fp32 level, while one TF32 pass is off by up to ~2^-10."""
import numpy as np


def tf32_rna(x):
    """fp32 -> TF32 (kept in an fp32 container): round to nearest, ties away from zero, at
    the 13th bit below the mantissa's top; finite inputs well inside the fp32 range."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x1000) & 0xFFFFE000
    return b.astype(np.uint32).view(np.float32)


def split(x):
    x = np.asarray(x, np.float32)
    hi = tf32_rna(x)
    lo = tf32_rna(x - hi)  # x - hi is exact in fp32
    return hi, lo


def test_tf32_rounding_keeps_ten_mantissa_bits():
    x = np.float32([1.0, 1.0 + 2.0 ** -10, 1.0 + 2.0 ** -11, 1.0 + 2.0 ** -12, -3.0 - 2.0 ** -10,
                    -3.0 - 2.0 ** -11])
    got = tf32_rna(x)
    assert got[0] == 1.0 and got[1] == 1.0 + 2.0 ** -10  # representable: unchanged
    assert got[2] == 1.0 + 2.0 ** -10  # a tie rounds away from zero
    assert got[3] == 1.0  # below half an ulp rounds down
    assert got[4] == -3.0 - 2.0 ** -9  # ties away from zero for negatives too (ulp 2^-9 at 2..4)
    assert got[5] == -3.0  # below half an ulp there
    assert np.all((got.view(np.uint32) & 0x1FFF) == 0)


def test_split_reconstructs_to_22_bits():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    hi, lo = split(x)
    err = np.abs((hi.astype(np.float64) + lo) - x.astype(np.float64)) / np.abs(x.astype(np.float64))
    assert err.max() <= 2.0 ** -21


def test_three_pass_product_is_fp32_accurate_and_one_pass_is_not():
    rng = np.random.default_rng(1)
    n = 200000
    a = (rng.standard_normal(n) * np.exp(rng.uniform(-10, 10, n))).astype(np.float32)
    b = (rng.standard_normal(n) * np.exp(rng.uniform(-10, 10, n))).astype(np.float32)
    ah, al = split(a)
    bh, bl = split(b)
    exact = a.astype(np.float64) * b.astype(np.float64)
    three = (ah.astype(np.float64) * bh + ah.astype(np.float64) * bl + al.astype(np.float64) * bh)
    one = ah.astype(np.float64) * bh
    rel3 = np.abs(three - exact) / np.abs(exact)
    rel1 = np.abs(one - exact) / np.abs(exact)
    assert rel3.max() <= 2.0 ** -20
    assert rel1.max() >= 2.0 ** -11  # a single TF32 pass is far from fp32


def test_three_pass_dot_products_meet_fp32_level_error():
    """Length-128 dot products (the chain's contraction length) accumulated in fp32 from
    the three products per term stay within a small multiple of fp32 accumulation error."""
    rng = np.random.default_rng(2)
    A = rng.standard_normal((2000, 128)).astype(np.float32)
    B = rng.standard_normal((2000, 128)).astype(np.float32)
    Ah, Al = split(A)
    Bh, Bl = split(B)
    terms = (Ah.astype(np.float64) * Bh + Ah.astype(np.float64) * Bl + Al.astype(np.float64) * Bh)
    acc = np.zeros(2000, np.float32)
    for k in range(128):  # fp32 accumulation, as in the MMA accumulators
        acc = (acc + terms[:, k].astype(np.float32)).astype(np.float32)
    exact = np.sum(A.astype(np.float64) * B, axis=1)
    scale = np.sum(np.abs(A.astype(np.float64) * B), axis=1)
    assert (np.abs(acc - exact) / scale).max() <= 128 * 2.0 ** -23
