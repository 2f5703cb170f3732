"""The GPU verifier sums the fixed-point masses rint(e * 2^40) of a row as two
32-bit partials, from three fp32 FMAs and one subtraction per element (the
top-p reading: masses in 64-bit fixed point, "vLLM PR #65007", Part 2). This
checks, with fp32 arithmetic emulated exactly in fp64, that the split gives
rint(e * 2^40) for every fp32 e in [0, 1] on a stride through the whole
range, densely around the powers of two, and at 0 and 1."""
import numpy as np

MAGIC = 1.5 * 2.0 ** 23
MAGIC_BITS = int(np.float32(MAGIC).view(np.uint32))


def _f32(x):
    return np.asarray(x, np.float64).astype(np.float32)


def split_mass(e32):
    e = e32.astype(np.float64)
    s = _f32(e * 2.0 ** 20 + MAGIC)             # fma(e, 2^20, magic), one rounding
    vh = _f32(s.astype(np.float64) - MAGIC)     # exact
    f64 = e * 2.0 ** 20 - vh.astype(np.float64)
    f = _f32(f64)                               # fma(e, 2^20, -vh)
    assert np.array_equal(f.astype(np.float64), f64), "the fraction must be exact"
    r = _f32(f.astype(np.float64) * 2.0 ** 20 + MAGIC)   # fma(f, 2^20, magic)
    hi = s.view(np.uint32).astype(np.int64) - MAGIC_BITS
    lo = r.view(np.uint32).astype(np.int64) - MAGIC_BITS
    return hi * 2 ** 20 + lo


def test_split_fixed_point_mass_is_rint_e_times_2_40():
    one = 0x3F800000
    strided = np.arange(0, one + 1, 4099, dtype=np.int64)
    dense = [np.arange(c - 3000, c + 3000, dtype=np.int64)
             for c in (one, 0x3F000000, 0x3E800000, 0x35800000, 0x34000000, 0x2B800000, 0x2B000000)]
    bits = np.clip(np.concatenate([strided] + dense + [np.array([0, 1, one])]), 0, one)
    e = bits.astype(np.uint32).view(np.float32)
    want = np.rint(e.astype(np.float64) * 2.0 ** 40).astype(np.int64)  # half to even
    np.testing.assert_array_equal(split_mass(e), want)
