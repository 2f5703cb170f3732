"""The GPU verifier's fixed-point mass of one value, rint(e * 2^40) for an
fp32 e in [0, 1] (the top-p reading: masses in 64-bit fixed point, vLLM PR
#65007, Part 2). The device forms v = e * 2^40 (exact in fp32) and, below
2^23, rounds it to an integer by adding 2^23 in fp32 and reading the
mantissa bits; from 2^23 up v is already an integer, its 24-bit significand
shifted left. This checks that construction, with the fp32 addition done by
numpy (IEEE, nearest even), against rint on a stride through every fp32
value in [0, 1], densely around the powers of two, and at 0 and 1."""
import numpy as np


def device_fixed_mass(e32):
    v = (e32.astype(np.float32) * np.float32(2.0 ** 40)).astype(np.float32)  # exact
    lo = ((v + np.float32(8388608.0)).astype(np.float32).view(np.uint32).astype(np.int64)
          - 0x4B000000)
    bits = v.view(np.uint32).astype(np.int64)
    sh = ((bits >> 23) - 150) & 63
    hi = ((bits & 0x7FFFFF) | 0x800000) << sh
    return np.where(v < np.float32(8388608.0), lo, hi)


def test_fixed_mass_is_rint_e_times_2_40():
    one = 0x3F800000
    strided = np.arange(0, one + 1, 4099, dtype=np.int64)
    dense = [np.arange(c - 3000, c + 3000, dtype=np.int64)
             for c in (one, 0x3F000000, 0x3E800000, 0x35800000, 0x35000000, 0x34000000,
                       0x2B800000, 0x2B000000)]
    bits = np.clip(np.concatenate([strided] + dense + [np.array([0, 1, one])]), 0, one)
    e = bits.astype(np.uint32).view(np.float32)
    want = np.rint(e.astype(np.float64) * 2.0 ** 40).astype(np.int64)  # half to even
    np.testing.assert_array_equal(device_fixed_mass(e), want)
