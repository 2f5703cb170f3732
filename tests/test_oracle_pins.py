"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against a library routine, a closed form, an
invariant, a special case that reduces to a textbook routine, or brute force
on a tiny input. None of these tests needs a GPU.

Passages (web pages, by title and section):
  * DSparkSpeculator API page, ``_sample_markov_chain`` / ``_sample_logits``:
    the Markov loop, bias from the previous token, noise keyed at P - 1.
  * vLLM PR #65007, Part 1, per-step list items 2-4: Gumbel-noised argmax over
    1024-column blocks; the first NaN block wins, else the first maximum.
  * vLLM PR #65007, Part 2, temperature and top-p: the smallest prefix by
    (logit, token id) whose mass reaches p, plus the row max, in 64-bit fixed
    point; Tests list: rows with 30% -inf, quarter-step ties, p up to 1-1e-7,
    rows without a finite logit, kept set equal to a float64 reference except
    within 1e-6 of p.
  * Philox4x32-10: Salmon et al., "Parallel random numbers: as easy as 1, 2, 3".
"""
import math
import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest
from scipy import stats

from verify_dspark_markov_step_gb300 import workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))


# ----------------------------------------------------------------------------
# Noise: Philox, uniform, Gumbel
# ----------------------------------------------------------------------------
def _triton_philox(key, ctr):
    pytest.importorskip("triton")
    with tempfile.TemporaryDirectory() as td:
        inp = os.path.join(td, "in.npz")
        outp = os.path.join(td, "out.npy")
        np.savez(inp, key=key, ctr=ctr)
        env = dict(os.environ, TRITON_INTERPRET="1")
        subprocess.run([sys.executable, os.path.join(HERE, "_triton_philox.py"), inp, outp],
                       check=True, env=env, timeout=600)
        return np.load(outp)


def test_philox_matches_library_philox(orc):
    """Oracle Philox4x32-10 == Triton's tl.philox on random keys and counters,
    including all-zero and all-ones words."""
    r = np.random.default_rng(7)
    n = 4096
    key = r.integers(0, 2**32, (n, 2), dtype=np.uint64).astype(np.uint32)
    ctr = r.integers(0, 2**32, (n, 4), dtype=np.uint64).astype(np.uint32)
    key[0] = 0
    ctr[0] = 0
    key[1] = 0xFFFFFFFF
    ctr[1] = 0xFFFFFFFF
    ctr[2] = [1, 0, 0, 0]
    ours = orc.philox4x32_10(key, ctr)
    ref = _triton_philox(key, ctr)
    np.testing.assert_array_equal(ours, ref)


def test_noise_word_layout_matches_library_philox(orc):
    """The (seed, position, column, stream) -> Philox (key, counter, word)
    mapping, checked against the library Philox fed the documented layout."""
    r = np.random.default_rng(8)
    n = 1024
    seed = r.integers(0, 2**63, n, dtype=np.int64).astype(np.uint64) * np.uint64(3)
    pos = r.integers(-1, 2**40, n, dtype=np.int64)
    col = r.integers(0, 1 << 18, n, dtype=np.int64).astype(np.uint32)
    stream = r.choice(np.array([0, 1 << 29, 1 << 30], np.uint32), n)
    word, _, _ = orc.noise(seed, pos, col, stream)
    key = np.stack([seed & np.uint64(0xFFFFFFFF), seed >> np.uint64(32)], 1).astype(np.uint32)
    upos = pos.astype(np.uint64)
    ctr = np.stack([col >> np.uint32(2), (upos & np.uint64(0xFFFFFFFF)).astype(np.uint32),
                    (upos >> np.uint64(32)).astype(np.uint32), stream], 1).astype(np.uint32)
    ref = _triton_philox(key, ctr)
    np.testing.assert_array_equal(word, ref[np.arange(n), col & 3])


def test_uniform_is_open_interval_and_uniform(orc):
    n = 1_000_000
    seed = np.full(n, 12345, np.uint64)
    pos = np.arange(n, dtype=np.int64) // 997
    col = (np.arange(n) % 997).astype(np.uint32)
    _, u, _ = orc.noise(seed, pos, col, np.uint32(1 << 30))
    assert u.dtype == np.float32
    assert (u > 0).all() and (u < 1).all()
    counts, _ = np.histogram(u, bins=1000, range=(0.0, 1.0))
    assert stats.chisquare(counts).pvalue > 0.01
    # 2^-23 grid with a half-step offset: u * 2^23 - 1/2 is an integer.
    k = u.astype(np.float64) * 2.0**23 - 0.5
    assert np.all(k == np.round(k))


def test_gumbel_matches_gumbel_cdf(orc):
    """g = -log(-log u) follows the standard Gumbel law (KS test), and its
    extreme values are those of the uniform grid."""
    n = 1_000_000
    seed = np.full(n, 99, np.uint64)
    _, u, g = orc.noise(seed, np.arange(n, dtype=np.int64), np.uint32(5), np.uint32(0))
    assert stats.kstest(g.astype(np.float64), "gumbel_r").pvalue > 0.01
    # g is increasing in u
    order = np.argsort(u, kind="stable")
    assert np.all(np.diff(g[order].astype(np.float64)) >= 0)
    # extremes: u in [2^-24, 1 - 2^-24]
    assert g.max() <= -math.log(-math.log1p(-2.0**-24)) + 1e-5
    assert g.min() >= -math.log(-math.log(2.0**-24)) - 1e-5


# ----------------------------------------------------------------------------
# Winner rule
# ----------------------------------------------------------------------------
def _chi2_pvalue(counts, probs):
    """Chi-square goodness of fit of integer counts against probabilities."""
    counts = np.asarray(counts, np.float64)
    probs = np.asarray(probs, np.float64)
    exp = probs / probs.sum() * counts.sum()
    return stats.chisquare(counts, exp).pvalue


def _flat_rule(y):
    nan = np.flatnonzero(np.isnan(y))
    return int(nan[0]) if nan.size else int(np.argmax(y))


def test_argmax_constructed_cases(orc):
    y = np.zeros(5000, np.float32)
    y[10] = 100.0
    y[3000] = np.nan            # NaN in a later block beats a larger max earlier
    assert orc.block_argmax(y)[0] == 3000
    y[2100] = np.nan            # two NaNs -> lower index
    assert orc.block_argmax(y)[0] == 2100
    z = np.full(4096, -1.0, np.float32)
    z[1023] = 5.0
    z[1024] = 5.0               # tie across a block boundary -> lower index
    assert orc.block_argmax(z) == (1023, 0.0)
    z[2047] = 5.0
    assert orc.block_argmax(z)[0] == 1023
    ninf = np.full(3000, -np.inf, np.float32)
    assert orc.block_argmax(ninf)[0] == 0   # all -inf -> 0
    s = np.full(10, -3.0, np.float32)
    s[4] = -0.0
    s[2] = 0.0                  # -0 and +0 tie -> lower index
    assert orc.block_argmax(s)[0] == 2
    s[2], s[4] = -0.0, 0.0
    assert orc.block_argmax(s)[0] == 2
    p = np.zeros(2048, np.float32)
    p[1500] = np.inf
    p[600] = np.inf             # +inf ties -> lower index
    assert orc.block_argmax(p) == (600, 0.0)


def test_argmax_block_form_equals_flat_rule(orc):
    r = np.random.default_rng(3)
    for trial in range(300):
        n = int(r.integers(1, 5000))
        y = r.standard_normal(n).astype(np.float32)
        if trial % 3 == 0:
            y = np.round(y * 2) / 2  # many ties
        if trial % 5 == 0:
            y[r.integers(0, n, 1 + n // 500)] = np.nan
        if trial % 7 == 0:
            y[r.integers(0, n, n // 3 + 1)] = -np.inf
        idx, gap = orc.block_argmax(y)
        assert idx == _flat_rule(y)
        if not np.isnan(y).any() and n > 1:
            srt = np.sort(y.astype(np.float64))
            expect = srt[-1] - srt[-2] if srt[-1] != srt[-2] else 0.0
            assert gap == expect or (math.isinf(gap) and math.isinf(expect))


# ----------------------------------------------------------------------------
# Markov loop
# ----------------------------------------------------------------------------
def _bf16(x):
    return wl.f32_to_bf16_bits(np.asarray(x, np.float32))


def test_bias_projection_equals_fp64_matmul(orc):
    """x - base reproduces fp32(w2 @ w1[prev]) computed by numpy in fp64, on the
    tiny workload (greedy, so x = z = base + bias exactly)."""
    w = wl.make("tiny")
    prev = int(w.anchor[0])
    tok, gap, x = orc.markov_step(w.base[0, 0], w.w1, w.w2, prev, 0.0, 0, 0)
    e = wl.bf16_bits_to_f32(w.w1[prev]).astype(np.float64)
    bias = (wl.bf16_bits_to_f32(w.w2).astype(np.float64) @ e).astype(np.float32)
    z = (w.base[0, 0] + bias).astype(np.float32)
    ulps = np.abs(x.view(np.int32).astype(np.int64) - z.view(np.int32).astype(np.int64))
    assert (ulps <= 1).all()
    assert (ulps == 0).mean() > 0.999
    assert tok == int(np.argmax(z))          # T = 0 is the textbook argmax


def test_greedy_step_is_numpy_argmax(orc):
    w = wl.custom(4, 2, 3000, 32, seed=1, temperature=0.0)
    tokens, cache, _ = orc.markov_sample(w.base, w.w1, w.w2, w.anchor, w.req_state_idx,
                                         w.positions, w.temperature, w.seeds)
    for b in range(4):
        for i in range(2):
            assert tokens[b, i] == int(np.argmax(cache[b, i]))


def test_markov_chain_uses_previous_token():
    """w1[prev] = 64 * onehot(prev + 1), w2 = identity * 64: the bias forces the
    next token to prev + 1, so tokens walk anchor+1, anchor+2, ..."""
    import oracle as orc
    V = R = 16
    w1 = np.zeros((V, R), np.float32)
    for t in range(V):
        w1[t, (t + 1) % V] = 64.0
    w2 = np.eye(V, dtype=np.float32) * 64.0
    B, K = 3, 6
    base = np.random.default_rng(0).standard_normal((B, K, V)).astype(np.float32)
    anchor = np.array([0, 5, 15], np.int32)
    tokens, _, _ = orc.markov_sample(base, _bf16(w1), _bf16(w2), anchor,
                                     np.arange(B, dtype=np.int32),
                                     wl.default_positions(B), np.ones(B, np.float32),
                                     wl.default_seeds(B, 0))
    expect = (anchor[:, None] + 1 + np.arange(K)[None, :]) % V
    np.testing.assert_array_equal(tokens, expect)


def test_gumbel_max_is_softmax_sampling(orc):
    """K = 1 with w2 = 0 reduces the step to Gumbel-max sampling of base / T: the
    token frequencies over 10^6 independent requests match softmax(base / T)."""
    n, V, R = 1_000_000, 6, 8
    logits = np.array([0.3, -1.0, 1.7, 0.0, -0.2, 1.1], np.float32)
    T = np.float32(0.8)
    base = np.broadcast_to(logits, (n, 1, V)).copy()
    w = np.zeros((V, R), np.uint16)
    tokens, _, _ = orc.markov_sample(
        base, w, w, np.zeros(n, np.int32), np.arange(n, dtype=np.int32),
        np.arange(n, dtype=np.int64) * 3 + 1, np.full(n, T, np.float32),
        wl.default_seeds(n, 77), write_cache=False)
    counts = np.bincount(tokens[:, 0], minlength=V)
    x = logits.astype(np.float64) / float(T)
    p = np.exp(x - x.max())
    p /= p.sum()
    assert _chi2_pvalue(counts, p) > 0.01


def test_noise_is_keyed_by_position_minus_one(orc):
    """Step i of a request at P0 draws the noise of step 0 of a request at
    P0 + i (same seed, same base row, no bias)."""
    V, R, K = 2048, 8, 4
    row = np.random.default_rng(1).standard_normal(V).astype(np.float32)
    base = np.broadcast_to(row, (2, K, V)).copy()
    w = np.zeros((V, R), np.uint16)
    seeds = np.array([1234567, 1234567], np.uint64)
    pos = np.array([500, 502], np.int64)
    tok, _, _ = orc.markov_sample(base, w, w, np.zeros(2, np.int32),
                                  np.array([0, 1], np.int32), pos,
                                  np.ones(2, np.float32), seeds, write_cache=False)
    assert tok[0, 2] == tok[1, 0] and tok[0, 3] == tok[1, 1]
    assert len(set(tok[0].tolist())) > 1


def test_step_noise_uses_draft_stream_at_position_minus_one(orc):
    """With no bias, step i's token is the winner of fp32(base/T) + g, g being
    the (separately pinned) noise of the DRAFT stream at position P0 + i - 1
    ("sampling keys a draw by the position before the sampled token")."""
    V, R, K = 3000, 8, 3
    r = np.random.default_rng(2)
    base = r.standard_normal((1, K, V)).astype(np.float32)
    w = np.zeros((V, R), np.uint16)
    T = np.float32(0.85)
    seed = np.uint64(0xDEADBEEF12345)
    P0 = 777
    tok, _, _ = orc.markov_sample(base, w, w, np.zeros(1, np.int32),
                                  np.zeros(1, np.int32), np.array([P0], np.int64),
                                  np.array([T]), np.array([seed]), write_cache=False)
    cols = np.arange(V, dtype=np.uint32)
    for i in range(K):
        _, _, g = orc.noise(seed, P0 + i - 1, cols, np.uint32(1 << 30))
        y = (base[0, i] / T).astype(np.float32) + g
        assert tok[0, i] == _flat_rule(y.astype(np.float32))


def test_padding_rows_are_inert_and_row_map_routes(orc):
    w = wl.custom(4, 3, 1500, 16, seed=3, S=6, rsi=[2, -1, 0, 5],
                  row_map=[3, 0, 5, 1, 2, 4], temperature=[1.0, 0.7, 1.2, 1.0, 0.9, 0.0])
    tokens, cache, _ = orc.markov_sample(w.base, w.w1, w.w2, w.anchor, w.req_state_idx,
                                         w.positions, w.temperature, w.seeds,
                                         cache_rows=6, row_map=w.row_map)
    assert (tokens[1] == -1).all()
    written = {int(w.row_map[s]) for s in (2, 0, 5)}
    for row in range(6):
        if row in written:
            assert np.abs(cache[row]).sum() > 0
        else:
            assert (cache[row] == 0).all()
    # request 0 (slot 2, T = 1.2) lands in row_map[2] = 5; greedy slot 5 -> row 4
    t0, _, x0 = orc.markov_step(w.base[0, 0], w.w1, w.w2, w.anchor[0], 1.2,
                                w.seeds[2], w.positions[0] - 1)
    np.testing.assert_array_equal(cache[5, 0], x0)
    assert t0 == tokens[0, 0]


def test_markov_deterministic_and_teacher_forcing(orc):
    w = wl.custom(3, 4, 1200, 16, seed=4, temperature=[0.9, 1.1, 1.0])
    a = orc.markov_sample(w.base, w.w1, w.w2, w.anchor, w.req_state_idx, w.positions,
                          w.temperature, w.seeds)
    b = orc.markov_sample(w.base, w.w1, w.w2, w.anchor, w.req_state_idx, w.positions,
                          w.temperature, w.seeds)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    f = orc.markov_sample(w.base, w.w1, w.w2, w.anchor, w.req_state_idx, w.positions,
                          w.temperature, w.seeds, forced=a[0])
    np.testing.assert_array_equal(a[0], f[0])


def _torch_bf16_bits(x32):
    """fp32 -> bf16 bit patterns by torch's own conversion (round to nearest
    even), a library routine independent of the oracle's bit arithmetic."""
    torch = pytest.importorskip("torch")
    t = torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_cache_is_rounded_fp32_cache(orc):
    """The bf16 cache is the fp32 cache rounded by torch's fp32 -> bf16
    conversion (nearest even), element for element."""
    w = wl.custom(2, 2, 999, 16, seed=5, temperature=[0.75, 1.0])
    _, c32, _ = orc.markov_sample(w.base, w.w1, w.w2, w.anchor, w.req_state_idx,
                                  w.positions, w.temperature, w.seeds)
    _, c16, _ = orc.markov_sample(w.base, w.w1, w.w2, w.anchor, w.req_state_idx,
                                  w.positions, w.temperature, w.seeds, cache_bf16=True)
    np.testing.assert_array_equal(c16, _torch_bf16_bits(c32))


def _bf16_edge_row():
    """fp32 values at the edges of the fp32 -> bf16 rounding: halfway cases
    with an even and an odd kept bit, one bit above and below halfway, fp32
    subnormals, bf16's largest finite value and the values that round up to
    infinity, infinities, signed zeros, NaN; then random values."""
    bits = []
    for hi in (0x3F80, 0x3F81, 0x4123, 0x4124, 0xC0A0, 0xC0A1, 0x0001, 0x8002, 0x7F7E):
        for lo in (0x8000, 0x7FFF, 0x8001, 0x0000, 0xFFFF):
            bits.append((hi << 16) | lo)
    bits += [0x00000001, 0x80000001, 0x007FFFFF, 0x00400000, 0x00008000, 0x00018000,
             0x7F7F7FFF, 0x7F7F8000, 0x7F7FFFFF, 0xFF7F8000, 0x7F800000, 0xFF800000,
             0x00000000, 0x80000000, 0x7FC00000, 0xFFC00001, 0x7F800001]
    x = np.array(bits, np.uint32).view(np.float32)
    r = np.random.default_rng(11).standard_normal(1000).astype(np.float32) * np.float32(3)
    return np.concatenate([x, r])


@pytest.mark.parametrize("T", [1.0, 0.5])
def test_bf16_cache_rounding_edges_match_torch(orc, T):
    """With markov_w2 = 0 the bias is exactly 0 and the cached value is
    fp32(fp32(base + 0) / T); its bf16 cache equals torch's nearest-even
    conversion of that value (ties, subnormals, overflow to infinity, signed
    zeros), and NaN stays NaN."""
    row = _bf16_edge_row()
    V, R = row.size, 64
    base = row.reshape(1, 1, V)
    w1 = wl.f32_to_bf16_bits(np.random.default_rng(3).standard_normal((V, R)).astype(np.float32))
    w2 = np.zeros((V, R), np.uint16)
    args = (base, w1, w2, np.array([3], np.int32), np.array([0], np.int32),
            wl.default_positions(1), np.array([T], np.float32), wl.default_seeds(1, 0))
    with np.errstate(over="ignore", invalid="ignore"):
        x = ((row + np.float32(0.0)) / np.float32(T)).astype(np.float32)
    _, c32, _ = orc.markov_sample(*args)
    _, c16, _ = orc.markov_sample(*args, cache_bf16=True)
    nan = np.isnan(x)
    np.testing.assert_array_equal(np.isnan(c32[0, 0]), nan)
    np.testing.assert_array_equal(c32[0, 0][~nan].view(np.uint32), x[~nan].view(np.uint32))
    got = c16[0, 0]
    np.testing.assert_array_equal(np.isnan(wl.bf16_bits_to_f32(got)), nan)
    np.testing.assert_array_equal(got[~nan], _torch_bf16_bits(x)[~nan])


@pytest.mark.parametrize("cache_bf16", [False, True])
def test_cache_at_temperature_is_scaled_biased_logits(orc, cache_bf16):
    """The cache holds x = fp32(fp32(base + fp32(bias)) / T) at T = 0.5, 0.7,
    1.3 and 1 (IEEE division, numpy fp32), and z at T = 0, with the bias a
    numpy fp64 matmul rounded once; the step's gap and token are those of
    y = fp32(x + g) with g the separately pinned draft noise at P0 + i - 1
    (the pages' "processed logits": the scaled logits the draft was drawn
    from). Teacher forcing fixes each step's previous token."""
    temps = [0.5, 0.7, 1.3, 1.0, 0.0]
    B, K, V, R = len(temps), 3, 777, 64
    w = wl.custom(B, K, V, R, seed=21, temperature=temps)
    forced = np.random.default_rng(22).integers(0, V, (B, K)).astype(np.int32)
    tok, cache, gaps = orc.markov_sample(w.base, w.w1, w.w2, w.anchor, w.req_state_idx,
                                         w.positions, w.temperature, w.seeds,
                                         cache_bf16=cache_bf16, forced=forced)
    w2 = wl.bf16_bits_to_f32(w.w2).astype(np.float64)
    cols = np.arange(V, dtype=np.uint32)
    for b in range(B):
        T = np.float32(temps[b])
        prev = int(w.anchor[b])
        for i in range(K):
            bias = (w2 @ wl.bf16_bits_to_f32(w.w1[prev]).astype(np.float64)).astype(np.float32)
            z = (w.base[b, i] + bias).astype(np.float32)
            x = (z / T).astype(np.float32) if T > 0 else z
            got = cache[b, i]
            if cache_bf16:
                np.testing.assert_array_equal(got, _torch_bf16_bits(x))
            else:
                np.testing.assert_array_equal(got.view(np.uint32), x.view(np.uint32))
            if T > 0:
                _, _, g = orc.noise(w.seeds[b], w.positions[b] + i - 1, cols,
                                    orc.STREAM_DRAFT)
                y = (x + g).astype(np.float32)
            else:
                y = z
            top2 = np.sort(y.astype(np.float64))[-2:]
            assert tok[b, i] == int(np.argmax(y))
            assert gaps[b, i] == top2[1] - top2[0]
            prev = int(forced[b, i])


# ----------------------------------------------------------------------------
# Top-p
# ----------------------------------------------------------------------------
def _softmax64(x):
    x = np.where(np.isnan(x), -np.inf, x.astype(np.float64))
    m = x.max()
    e = np.exp(x - m)
    return e / e.sum()


def _brute_topp(xt, p):
    """Smallest subset of maximal total probability reaching p (fp64), by
    enumerating subsets of each size; ties in logit resolved by token id."""
    V = xt.size
    pr = _softmax64(xt)
    order = sorted(range(V), key=lambda v: (-(xt[v] if not np.isnan(xt[v]) else -np.inf), v))
    import itertools
    for m in range(1, V + 1):
        best = max(sum(pr[list(c)]) for c in itertools.combinations(range(V), m))
        if best >= p:
            return set(order[:m]), pr
    return set(order), pr


def test_topp_brute_force_tiny(orc):
    r = np.random.default_rng(11)
    checked = 0
    for trial in range(400):
        V = int(r.integers(1, 11))
        xt = r.standard_normal(V).astype(np.float32) * 2
        if trial % 4 == 1:
            xt = (np.round(xt * 4) / 4).astype(np.float32)   # quarter-step ties
        if trial % 4 == 2:
            xt[r.random(V) < 0.3] = -np.inf
        p = float(np.float32(r.choice([0.01, 0.3, 0.5, 0.8, 0.9, 0.95, 0.99, r.random()])))
        pr_keep, keep, F, Fk, slack = orc.target_probs(xt, 1.0, p)
        if np.isneginf(xt).all():
            assert keep.tolist() == [True] + [False] * (V - 1)
            continue
        ref, pr = _brute_topp(xt, p)
        if slack < 1e-6:
            continue
        assert set(np.flatnonzero(keep).tolist()) == ref, (xt, p)
        np.testing.assert_allclose(pr_keep.sum(), 1.0, rtol=1e-6)
        checked += 1
    assert checked > 300


def test_topp_float64_reference_and_never_superset(orc):
    """Rows shaped like the pages' test matrix: LM-like, quarter-step ties, 30%
    -inf, peaked, flat; p over a range including 0.9999 and 1 - 1e-7."""
    r = np.random.default_rng(12)
    V = 3000
    ps = [0.01, 0.1, 0.5, 0.9, 0.95, 0.99, 0.9999, 1 - 1e-7]
    mismatches = 0
    for kind in range(5):
        for p in ps:
            x = r.standard_normal(V).astype(np.float32) * 2
            if kind == 1:
                x = (np.round(x * 4) / 4).astype(np.float32)
            elif kind == 2:
                x[r.random(V) < 0.3] = -np.inf
            elif kind == 3:
                x[r.integers(V)] += 25.0
            elif kind == 4:
                x *= 0.01
            pf = float(np.float32(p))
            _, keep, F, Fk, slack = orc.target_probs(x, 1.0, pf)
            pr = _softmax64(x)
            order = np.lexsort((np.arange(V), -np.where(np.isneginf(x), -np.inf, x)))
            cum = np.cumsum(pr[order])
            n_ref = int(np.searchsorted(cum, pf - 0.0, side="left")) + 1
            n_ref = min(n_ref, V)
            ref = set(order[:n_ref].tolist())
            ours = set(np.flatnonzero(keep).tolist())
            if ours != ref:
                boundary = cum[n_ref - 1]
                prevb = cum[n_ref - 2] if n_ref >= 2 else 0.0
                assert min(abs(boundary - pf), abs(prevb - pf)) < 1e-6
                mismatches += 1
            assert ours <= ref | set(order[:n_ref + 1].tolist())
            assert len(ours) <= n_ref + 1
            # deterministic
            _, keep2, _, _, _ = orc.target_probs(x, 1.0, pf)
            np.testing.assert_array_equal(keep, keep2)
    assert mismatches <= 2


def test_topp_edge_values(orc):
    x = np.array([1.0, 3.0, 2.0, 3.0, -np.inf, np.nan], np.float32)
    _, keep, _, _, _ = orc.target_probs(x, 1.0, 1.0)
    assert keep.all()                                  # p >= 1: no truncation
    _, keep, _, _, _ = orc.target_probs(x, 1.0, 0.0)
    assert np.flatnonzero(keep).tolist() == [1]        # p = 0: the row max only
    _, keep, _, _, _ = orc.target_probs(x, 1.0, 0.5)
    assert np.flatnonzero(keep).tolist() == [1, 3]     # tie broken by id
    # masses that reach p exactly: "reaches p" keeps the shorter prefix
    eq = np.array([0.0, 0.0, -np.inf], np.float32)
    assert np.flatnonzero(orc.target_probs(eq, 1.0, 0.5)[1]).tolist() == [0]
    eq4 = np.zeros(4, np.float32)
    assert np.flatnonzero(orc.target_probs(eq4, 1.0, 0.25)[1]).tolist() == [0]
    assert np.flatnonzero(orc.target_probs(eq4, 1.0, 0.5)[1]).tolist() == [0, 1]
    allinf = np.full(7, -np.inf, np.float32)
    allinf[3] = np.nan
    p, keep, _, _, _ = orc.target_probs(allinf, 1.0, 0.9)
    assert p.tolist() == [1.0] + [0.0] * 6


def test_fixed_point_mass_is_order_free(orc):
    r = np.random.default_rng(13)
    x = (r.standard_normal(5000) * 3).astype(np.float32)
    perm = r.permutation(5000)
    p1, k1, F1, Fk1, _ = orc.target_probs(x, 0.7, 0.93)
    p2, k2, F2, Fk2, _ = orc.target_probs(x[perm], 0.7, 0.93)
    assert F1 == F2 and Fk1 == Fk2
    np.testing.assert_array_equal(p1[perm], p2)
    np.testing.assert_array_equal(k1[perm], k2)
    np.testing.assert_allclose(p1.astype(np.float64), np.where(k1, _softmax64(x / np.float32(0.7)), 0)
                               / _softmax64(x / np.float32(0.7))[k1].sum(), rtol=2e-6, atol=1e-12)


# ----------------------------------------------------------------------------
# Rejection sampler
# ----------------------------------------------------------------------------
def _verify_trials(orc, n, target_rows, cache_rows, T=1.0, top_p=1.0, draft=None, seed=0):
    """Run n independent one-request verifications sharing the same rows."""
    K = cache_rows.shape[0]
    V = target_rows.shape[-1]
    target = np.broadcast_to(target_rows, (n, K + 1, V)).copy()
    cache = np.broadcast_to(cache_rows, (n, K, V)).copy()
    rsi = np.arange(n, dtype=np.int32)
    return orc.rejection_sample(draft, cache, target, rsi,
                                np.arange(n, dtype=np.int64) * 5 + 3,
                                np.full(n, T, np.float32), np.full(n, top_p, np.float32),
                                wl.default_seeds(n, 100 + seed))


def test_rejection_first_token_follows_target(orc):
    """Draft d ~ q (drawn by numpy), then the first emitted token ~ p (target
    after temperature and top-p): chi-square over 10^6 trials, and the accept
    rate equals sum_v min(p_v, q_v)."""
    n, V = 1_000_000, 6
    tgt = np.array([[0.5, 1.5, -0.5, 0.0, 2.0, -1.0], [0, 0, 0, 0, 0, 0]], np.float32)
    cache = np.array([[1.0, 0.2, 0.4, -0.3, 1.8, 0.0]], np.float32)
    T, top_p = np.float32(1.3), np.float32(0.9)
    p, keep, _, _, _ = orc.target_probs(tgt[0], T, top_p)
    q = orc.draft_probs(cache[0]).astype(np.float64)
    rng = np.random.default_rng(21)
    draft = rng.choice(V, size=(n, 1), p=q / q.sum()).astype(np.int32)
    res = _verify_trials(orc, n, tgt, cache, T=T, top_p=top_p, draft=draft)
    first = res["out_tokens"][:, 0]
    counts = np.bincount(first, minlength=V)
    p64 = p.astype(np.float64)
    p64 /= p64.sum()
    nz = p64 > 0
    assert counts[~nz].sum() == 0
    assert _chi2_pvalue(counts[nz], p64[nz]) > 0.01
    acc = (res["num_accepted"] == 1).mean()
    expect = np.minimum(p64, q / q.sum()).sum()
    assert abs(acc - expect) < 4 * math.sqrt(expect * (1 - expect) / n)


def test_rejection_q_equals_p_always_accepts(orc):
    n, V, K = 2000, 50, 3
    r = np.random.default_rng(22)
    rows = (r.standard_normal((K + 1, V)) * 2).astype(np.float32)
    T = np.float32(0.9)
    cache = (rows[:K] / T).astype(np.float32)
    draft = r.integers(0, V, (n, K)).astype(np.int32)
    res = _verify_trials(orc, n, rows, cache, T=T, top_p=1.0, draft=draft)
    assert (res["num_accepted"] == K).all()
    np.testing.assert_array_equal(res["out_tokens"][:, :K], draft)
    # the bonus is a draw from p_K: its frequencies follow p_K
    pK, _, _, _, _ = orc.target_probs(rows[K], T, 1.0)
    pK = pK.astype(np.float64) / pK.astype(np.float64).sum()
    counts = np.bincount(res["out_tokens"][:, K], minlength=V).astype(np.float64)
    mask = pK * n > 20
    obs = np.append(counts[mask], counts[~mask].sum())
    exp = np.append(pK[mask], pK[~mask].sum()) * n
    assert _chi2_pvalue(obs, exp) > 0.001


def test_rejection_onehot_target_rejects_and_emits(orc):
    V = 40
    tgt = np.zeros((2, V), np.float32)
    tgt[0, 17] = 1000.0            # p one-hot at 17
    cache = np.zeros((1, V), np.float32)
    draft = np.array([[3]] * 100, np.int32)
    res = _verify_trials(orc, 100, tgt, cache, draft=draft)
    assert (res["num_accepted"] == 0).all()
    assert (res["out_tokens"][:, 0] == 17).all()
    assert (res["out_tokens"][:, 1] == -1).all()


def test_rejection_never_accepts_zero_target_mass(orc):
    """A draft token with p(d) = 0 is never accepted, also when q(d) = 0 (the
    accept probability min(1, p/q) is 0 there)."""
    V = 30
    tgt = np.zeros((2, V), np.float32)
    tgt[0, 4] = -np.inf
    cache = np.zeros((1, V), np.float32)
    cache[0, 4] = -np.inf
    res = _verify_trials(orc, 500, tgt, cache, draft=np.full((500, 1), 4, np.int32))
    assert (res["num_accepted"] == 0).all()
    assert (res["out_tokens"][:, 0] != 4).all()


def test_rejection_minus_one_draft_samples_p(orc):
    n, V = 200_000, 5
    tgt = np.array([[0.1, 1.0, -1.0, 0.5, 0.0], [0] * 5], np.float32)
    cache = np.zeros((1, V), np.float32)
    res = _verify_trials(orc, n, tgt, cache, draft=np.full((n, 1), -1, np.int32))
    assert (res["num_accepted"] == 0).all()
    p, _, _, _, _ = orc.target_probs(tgt[0], 1.0, 1.0)
    counts = np.bincount(res["out_tokens"][:, 0], minlength=V)
    assert _chi2_pvalue(counts, p) > 0.01


def test_rejection_greedy_rows(orc):
    r = np.random.default_rng(23)
    B, K, V = 50, 4, 300
    target = r.standard_normal((B, K + 1, V)).astype(np.float32)
    am = target.argmax(-1).astype(np.int32)
    draft = am[:, :K].copy()
    cut = r.integers(0, K + 1, B)
    for b in range(B):
        if cut[b] < K:
            draft[b, cut[b]] = (am[b, cut[b]] + 1) % V
    res = orc.rejection_sample(draft, None, target, np.arange(B, dtype=np.int32),
                               wl.default_positions(B), np.zeros(B, np.float32),
                               np.full(B, 0.9, np.float32), wl.default_seeds(B, 5))
    for b in range(B):
        n = int(cut[b])
        assert res["num_accepted"][b] == n
        np.testing.assert_array_equal(res["out_tokens"][b, :n + 1], am[b, :n + 1])
        assert (res["out_tokens"][b, n + 1:] == -1).all()


def test_draft_probs_is_softmax(orc):
    """q = softmax of the cached row (closed form in fp64), NaN read as -inf,
    and zero everywhere for a row without a value above -inf."""
    r = np.random.default_rng(24)
    for scale in (0.01, 1.0, 4.0, 30.0):
        c = (r.standard_normal(4000) * scale).astype(np.float32)
        c[r.random(4000) < 0.2] = -np.inf
        c[5] = np.nan
        q = orc.draft_probs(c).astype(np.float64)
        np.testing.assert_allclose(q, _softmax64(c), rtol=2e-6, atol=1e-30)
    assert (orc.draft_probs(np.full(9, -np.inf, np.float32)) == 0).all()
    bf = wl.f32_to_bf16_bits(c)
    np.testing.assert_allclose(orc.draft_probs(bf).astype(np.float64),
                               _softmax64(wl.bf16_bits_to_f32(bf)), rtol=2e-6, atol=1e-30)


def test_verifier_draws_use_documented_streams_and_positions(orc):
    """Accept uniforms come from the ACCEPT stream at P0 + k - 1, column 0; the
    bonus is the Gumbel-max draw of p_K with the TARGET stream at P0 + K - 1."""
    n, V, K = 3000, 20, 2
    r = np.random.default_rng(25)
    rows = (r.standard_normal((K + 1, V))).astype(np.float32)
    cache = (rows[:K] + r.standard_normal((K, V)).astype(np.float32) * 0.7).astype(np.float32)
    draft = r.integers(0, V, (n, K)).astype(np.int32)
    pos = np.arange(n, dtype=np.int64) * 5 + 3
    seeds = wl.default_seeds(n, 100)
    res = _verify_trials(orc, n, rows, cache, draft=draft)
    p0, _, _, _, _ = orc.target_probs(rows[0], 1.0, 1.0)
    q0 = orc.draft_probs(cache[0])
    _, u, _ = orc.noise(seeds, pos - 1, np.uint32(0), np.uint32(1 << 29))
    ratio = p0[draft[:, 0]].astype(np.float64) / q0[draft[:, 0]].astype(np.float64)
    clear = np.abs(u.astype(np.float64) - ratio) > 1e-6
    assert clear.sum() > n * 0.99
    np.testing.assert_array_equal((res["num_accepted"] >= 1)[clear], (u < ratio)[clear])
    pK, _, _, _, _ = orc.target_probs(rows[K], 1.0, 1.0)
    full = np.flatnonzero(res["num_accepted"] == K)
    assert full.size > 100
    logp = np.where(pK > 0, np.log(np.maximum(pK, 1e-45).astype(np.float64)), -np.inf)
    logp = logp.astype(np.float32)
    cols = np.arange(V, dtype=np.uint32)
    for b in full[:200]:
        tok, _ = orc.categorical(pK, seeds[b], pos[b] + K - 1)
        assert res["out_tokens"][b, K] == tok
        _, _, g = orc.noise(seeds[b], pos[b] + K - 1, cols, np.uint32(0))
        assert tok == _flat_rule((logp + g).astype(np.float32))


def _p64(xt, top_p):
    """fp64 target distribution of one scaled row with the top-p keep set
    taken by sorting (logit desc, id asc) and accumulating fp64 probabilities;
    also the cumulative masses at the kept count n and at n - 1."""
    pr = _softmax64(xt)
    if top_p >= 1.0:
        return pr, None
    order = sorted(range(xt.size), key=lambda v: (-(xt[v] if not np.isnan(xt[v]) else -np.inf), v))
    cum = np.cumsum(pr[order])
    n = int(np.searchsorted(cum, top_p, side="left")) + 1
    n = min(n, xt.size)
    keep = np.zeros(xt.size, bool)
    keep[order[:n]] = True
    p = np.where(keep, pr, 0.0)
    p /= p.sum()
    return p, (cum[n - 1], cum[n - 2] if n >= 2 else 0.0)


def test_verifier_exception_gates_against_fp64(orc):
    """The three numbers that decide which GPU/oracle differences are excused,
    recomputed directly in fp64 from the pinned noise: the accept margin
    |u - p(d)/q(d)| of every ratio test made, the top-p boundary slack
    min(|S_n - p|, |S_(n-1) - p|) of every target row used, and the top-two
    gap of the draw that produced the last emitted token (residual max(0,
    p - q), or p for the bonus). A gate that were always 0 (or taken on the
    wrong row, stream or position) fails here; the oracle's decisions agree
    with the fp64 ones wherever the fp64 margin or gap is clear of rounding."""
    B, K, V = 48, 3, 400
    temps = np.resize(np.array([1.0, 0.8, 1.25], np.float32), B)
    topps = np.resize(np.array([1.0, 0.9, 0.7, 0.95], np.float32), B)
    w = wl.custom(B, K, V, 32, seed=31, temperature=temps, top_p=topps, target_noise=0.8)
    draft, cache, _ = orc.markov_sample(w.base, w.w1, w.w2, w.anchor, w.req_state_idx,
                                        w.positions, w.temperature, w.seeds)
    res = orc.rejection_sample(draft, cache, w.target, w.req_state_idx, w.positions,
                               w.temperature, w.top_p, w.seeds)
    cols = np.arange(V, dtype=np.uint32)
    n_margin = n_slack = n_gap = 0
    for b in range(B):
        T, tp, seed, P0 = temps[b], float(topps[b]), w.seeds[b], int(w.positions[b])
        emitted_row, weights = None, None
        for k in range(K + 1):
            xt = (w.target[b, k] / T).astype(np.float32)
            p, cums = _p64(xt, tp)
            sl = res["slack"][b, k]
            if cums is not None and not np.isnan(sl):
                slack64 = min(abs(cums[0] - tp), abs(cums[1] - tp))
                assert abs(sl - slack64) < 1e-6, (b, k, sl, slack64)
                n_slack += 1
            if k == K:
                emitted_row, weights = k, p
                break
            d = int(draft[b, k])
            q = _softmax64(cache[b, k])
            _, u, _ = orc.noise(seed, P0 + k - 1, 0, orc.STREAM_ACCEPT)
            m64 = abs(float(u) - p[d] / q[d])
            mo = res["margins"][b, k]
            assert abs(mo - m64) <= 1e-6 + 1e-5 * m64, (b, k, mo, m64)
            n_margin += 1
            accepted = res["out_tokens"][b, k] == d and res["num_accepted"][b] > k
            if m64 > 1e-5:
                assert accepted == (float(u) * q[d] < p[d]), (b, k)
            if not accepted:
                emitted_row, weights = k, np.maximum(p - q, 0.0)
                break
        _, _, g = orc.noise(seed, P0 + emitted_row - 1, cols, orc.STREAM_TARGET)
        with np.errstate(divide="ignore"):
            y = np.log(weights) + g.astype(np.float64)
        top2 = np.sort(y)[-2:]
        gap64 = top2[1] - top2[0]
        assert abs(res["gaps"][b] - gap64) < 1e-4, (b, res["gaps"][b], gap64)
        if gap64 > 1e-4:
            assert res["out_tokens"][b, emitted_row] == int(np.argmax(y))
        n_gap += 1
    assert n_margin > 60 and n_slack > 40 and n_gap == B


def test_rejection_padding_and_bounds(orc):
    w = wl.custom(3, 2, 100, 8, seed=6, rsi=[1, -1, 0], S=2)
    d = wl.random_drafts(w)
    res = orc.rejection_sample(d, np.zeros((2, 2, 100), np.float32), w.target,
                               w.req_state_idx, w.positions, w.temperature, w.top_p, w.seeds)
    assert (res["out_tokens"][1] == -1).all() and res["num_accepted"][1] == 0
    bad = d.copy()
    bad[0, 0] = 100
    with pytest.raises(RuntimeError):
        orc.rejection_sample(bad, np.zeros((2, 2, 100), np.float32), w.target,
                             w.req_state_idx, w.positions, w.temperature, w.top_p, w.seeds)


# ---- the top-k variant of the Markov loop ([DSP] _sample_sequential_topk) ----

def _topk_set(row, k):
    """Brute-force top-k: value descending (NaN above every number, -0 == +0),
    token id ascending; the first k of that order."""
    vals = np.asarray(row, np.float64)
    nan = np.isnan(vals)
    key = np.where(nan, np.inf, vals)
    order = sorted(range(len(vals)), key=lambda v: (-int(nan[v]), -key[v], v))
    return set(order[:k])


def test_topk_covering_the_vocabulary_is_the_dense_loop(orc):
    w = wl.custom(3, 3, 500, 64, seed=4, temperature=[1.0, 0.0, 0.7])
    args = (w.base, w.w1, w.w2, w.anchor, w.req_state_idx, w.positions, w.temperature, w.seeds)
    t0, c0, _ = orc.markov_sample(*args)
    for k in (500, 501, 10 ** 6):
        t1, c1, _ = orc.markov_sample(*args, topk=k)
        assert np.array_equal(t0, t1) and np.array_equal(c0, c1, equal_nan=True)


def test_topk_candidates_against_brute_force(orc):
    """Every cached row is finite exactly on the brute-force top-k of its base
    row and -inf elsewhere; ties, -0/+0 and NaN columns included."""
    rng = np.random.default_rng(7)
    w = wl.custom(4, 3, 300, 64, seed=9, temperature=[1.0, 0.5, 0.0, 1.3])
    base = w.base.copy()
    base[0, 0, ::7] = 1.25                      # a run of ties
    base[1, 1, 3] = -0.0
    base[1, 1, 4] = 0.0
    base[2, 2, rng.integers(0, 300, 6)] = np.nan  # more NaNs than k in one row
    base[3, 0, [5, 17]] = np.nan
    w.base = base
    k = 5
    _, cache, _ = orc.markov_sample(w.base, w.w1, w.w2, w.anchor, w.req_state_idx,
                                    w.positions, w.temperature, w.seeds, topk=k)
    for b in range(4):
        for i in range(3):
            want = _topk_set(base[b, i], k)
            got = set(np.flatnonzero(~np.isneginf(cache[b, i])).tolist())
            assert got == want, (b, i, sorted(got), sorted(want))


def test_topk_draws_follow_the_truncated_softmax(orc):
    """One step over many slots with their own seeds: the tokens follow the
    softmax of the biased logits restricted to the top-k candidates."""
    V, R, k, N = 12, 64, 4, 20000
    w = wl.custom(1, 1, V, R, seed=3, base_std=1.0)
    base = np.repeat(w.base, N, axis=0)
    anchor = np.repeat(w.anchor, N)
    seeds = (np.arange(N, dtype=np.uint64) * np.uint64(0x9E3779B97F4A7C15)) ^ np.uint64(17)
    temp = np.ones(N, np.float32)
    tok, _, _ = orc.markov_sample(base, w.w1, w.w2, anchor, np.arange(N, dtype=np.int32),
                                  np.full(N, 100, np.int64), temp, seeds, write_cache=False,
                                  topk=k)
    # z = fp32(base + fp32(bias)), bias an fp64 dot of the bf16 weights
    w1 = wl.bf16_bits_to_f32(w.w1).astype(np.float64)
    w2 = wl.bf16_bits_to_f32(w.w2).astype(np.float64)
    bias = (w2 @ w1[int(w.anchor[0])]).astype(np.float32)
    z = (w.base[0, 0] + bias).astype(np.float32).astype(np.float64)
    cand = sorted(_topk_set(w.base[0, 0], k))
    assert set(np.unique(tok).tolist()) <= set(cand)
    p = np.exp(z[cand] - z[cand].max())
    counts = [(tok[:, 0] == c).sum() for c in cand]
    assert _chi2_pvalue(counts, p) > 1e-4


def test_threaded_oracle_is_the_single_threaded_one():
    """The OpenMP build of the oracle (requests on several host threads, the
    CPU baseline's parallel leg) returns exactly what the single-threaded
    build returns: tokens, cache, gaps, and every verifier output."""
    import oracle as orc
    orc.build()
    if not os.path.exists(orc._OMP_PATH):
        pytest.skip("gcc without OpenMP")
    w = wl.custom(12, 3, 3001, 64, seed=41, temperature=[0.9, 1.0, 0.0, 1.2] * 3,
                  top_p=[1.0, 0.9, 0.8] * 4, S=12)
    args = (w.base, w.w1, w.w2, w.anchor, w.req_state_idx, w.positions, w.temperature,
            w.seeds)
    a = orc.markov_sample(*args)
    b = orc.markov_sample(*args, threads=4)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    r1 = orc.rejection_sample(a[0], a[1], w.target, w.req_state_idx, w.positions,
                              w.temperature, w.top_p, w.seeds)
    r2 = orc.rejection_sample(a[0], a[1], w.target, w.req_state_idx, w.positions,
                              w.temperature, w.top_p, w.seeds, threads=4)
    for k in r1:
        np.testing.assert_array_equal(r1[k], r2[k])
    assert orc.threads_in_use(4) == 4
