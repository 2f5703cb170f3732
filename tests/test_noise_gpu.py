"""The device noise generator against the oracle's: Philox words and
uniforms bit-exact (pure integer and exact fp32 arithmetic), Gumbel variates
within a few fp32 ulps of max(1, |g|) (accurate fp32 logf on the device, fp64
on the host)."""
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
    go = g_o.astype(np.float64)
    # fp32 logf twice against fp64 log rounded once: a few ulps of max(1, |g|)
    # (near g = 0 the inner log's rounding dominates, so the bound is absolute)
    err = np.abs(gg - go)
    assert (err <= 4 * 2.0 ** -23 * np.maximum(1.0, np.abs(go))).all(), err.max()
