"""The device noise generator against the oracle's: Philox words and
uniforms bit-exact (pure integer and exact fp32 arithmetic), Gumbel variates
within 2e-6 of the exact -log(-log u) (fp64 here). The device evaluates
-log u as -ln2 * lg2.approx(u) for u <= 3/4 and by the atanh series of
t = 1 - u above, then -ln2 * lg2.approx of that; half of the bound is the
rounding of the fp32 result itself (half an ulp is 0.95e-6 at |g| near 16,
the largest variate of the 23-bit grid), and 1.6e-6 is the largest error
seen over 10^6 draws. A GPU and an oracle draw can then differ only where
the oracle's top two noised values are within about 4e-6, inside the 1e-5
near-tie rule."""
import numpy as np
import pytest

import oracle
from gpu_util import require_gpu

pytestmark = pytest.mark.gpu


def test_noise_matches_oracle():
    torch = require_gpu()
    from verify_dspark_markov_step_gb300 import _lib
    from verify_dspark_markov_step_gb300.step import to_device
    r = np.random.default_rng(5)
    n = 1_000_000
    seed = r.integers(0, 2**63, n, dtype=np.int64).astype(np.uint64) * np.uint64(5)
    pos = r.integers(-1, 2**36, n, dtype=np.int64)
    col = r.integers(0, 1 << 18, n, dtype=np.int64).astype(np.uint32)
    stream = r.choice(np.array([0, 1 << 29, 1 << 30], np.uint32), n)
    w_o, u_o, g_o = oracle.noise(seed, pos, col, stream)
    d = dict(seed=to_device(seed), pos=to_device(pos),
             col=to_device(col.view(np.int32)), stream=to_device(stream.view(np.int32)))
    word = torch.empty(n, dtype=torch.int32, device="cuda")
    u = torch.empty(n, dtype=torch.float32, device="cuda")
    g = torch.empty(n, dtype=torch.float32, device="cuda")
    _lib.noise(d["seed"], d["pos"], d["col"], d["stream"], word, u, g)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(word.cpu().numpy().view(np.uint32), w_o)
    np.testing.assert_array_equal(u.cpu().numpy(), u_o)
    gg = g.cpu().numpy().astype(np.float64)
    exact = -np.log(-np.log(u_o.astype(np.float64)))  # u is exact: 23 bits + 1/2
    err = np.abs(gg - exact)
    assert err.max() <= 2e-6, err.max()
    # the oracle's own variate is the exact one rounded once to fp32
    assert (np.abs(g_o.astype(np.float64) - exact) <=
            2.0 ** -24 * np.maximum(2.0 ** -126, np.abs(exact)) * 2).all()


def test_temperature_division_is_correctly_rounded():
    """The Markov loop's temperature step x = z / T (the FMA-corrected product
    with rn(1/T), or the IEEE division where an intermediate could leave the
    normal range) against numpy's IEEE fp32 division, bit for bit: random
    z over 2^-70..2^70 and both signs, T over 2^-35..2^35 and the usual
    0.5..1.5, and the special values (zeros, infinities, NaN, subnormals,
    the largest finite values)."""
    torch = require_gpu()
    from verify_dspark_markov_step_gb300 import _lib
    r = np.random.default_rng(9)
    n = 4_000_000
    z = (r.choice([-1.0, 1.0], n) * np.exp2(r.uniform(-70, 70, n)) *
         r.uniform(1, 2, n)).astype(np.float32)
    T = np.where(r.random(n) < 0.5, r.uniform(0.5, 1.5, n),
                 np.exp2(r.uniform(-35, 35, n))).astype(np.float32)
    sz = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, -1e-45, 1.17e-38, 3.4e38,
                   -3.4e38, 1.0, -2.5, 7.0, 1e-30, 1e30], np.float32)
    sT = np.array([1.0, 0.5, 0.7, 1.3, 3.0, 1e-20, 1e20, 2.0 ** -30, 2.0 ** 30, 0.999],
                  np.float32)
    ez, eT = np.meshgrid(sz, sT)
    z = np.concatenate([z, ez.ravel()])
    T = np.concatenate([T, eT.ravel()])
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        want = (z / T).astype(np.float32)
    zd = torch.from_numpy(z).cuda()
    Td = torch.from_numpy(T).cuda()
    xd = torch.empty_like(zd)
    _lib.temperature_divide(zd, Td, xd)
    torch.cuda.synchronize()
    got = xd.cpu().numpy()
    nan = np.isnan(want)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))
