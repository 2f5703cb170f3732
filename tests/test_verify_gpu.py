"""Parity of the CUDA rejection-sampling verifier with the CPU oracle.

Both sides get the same drafts, cache and target logits. Outputs must be
bit-exact per request, except where the oracle's accept margin or draw gap is
below 1e-5 or its top-p boundary mass is within 1e-6 of p (counted).
"""
import zlib

import numpy as np
import pytest
from scipy import stats

from parity import subset, verify_parity
from gpu_util import require_gpu, run_markov, run_verify
from verify_dspark_markov_step_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _drafted(w):
    """Drafts and cache from the GPU drafter (the inputs verification sees in
    a decode step)."""
    _, tok, cache = run_markov(w)
    return tok, cache


def test_tiny():
    w = wl.make("tiny")
    draft, cache = _drafted(w)
    st, out, nacc = run_verify(w, draft, cache)
    assert st.status_code() == 0
    exc, _ = verify_parity(w, draft, cache, out, nacc)
    assert exc == 0


def test_odd_topp_nan_temperatures():
    w = wl.make("odd")
    draft, cache = _drafted(w)
    st, out, nacc = run_verify(w, draft, cache)
    assert st.status_code() == 0
    verify_parity(w, draft, cache, out, nacc, max_exception_frac=0.13)


def test_random_drafts_with_placeholders_and_greedy():
    w = wl.custom(24, 4, 9001, 64, seed=5, S=24,
                  temperature=[0.0 if i % 5 == 0 else 0.6 + 0.05 * i for i in range(24)],
                  top_p=[1.0 if i % 3 == 0 else 0.5 + 0.02 * i for i in range(24)])
    draft = wl.random_drafts(w, seed=1, p_minus1=0.4)
    _, cache = _drafted(w)
    st, out, nacc = run_verify(w, draft, cache)
    assert st.status_code() == 0
    verify_parity(w, draft, cache, out, nacc, max_exception_frac=0.05)


def _topp_rows(kind, V, rng):
    x = (rng.standard_normal(V) * 2).astype(np.float32)
    if kind == "ties":
        x = (np.round(x * 4) / 4).astype(np.float32)
    elif kind == "ninf":
        x[rng.random(V) < 0.3] = -np.inf
    elif kind == "peaked":
        x[rng.integers(V)] += 20.0
    elif kind == "flat":
        x *= 0.01
    elif kind == "allninf":
        x[:] = -np.inf
    elif kind == "coarse_ties":
        x = rng.integers(0, 3, V).astype(np.float32)
    return x


@pytest.mark.parametrize("kind", ["lm", "ties", "ninf", "peaked", "flat", "allninf", "coarse_ties"])
def test_topp_row_kinds(kind):
    """The pages' top-p test matrix: LM-like rows, quarter-step ties, 30% -inf,
    peaked and flat rows, rows with no finite logit; p from 0.01 to 1 - 1e-7."""
    rng = np.random.default_rng(zlib.crc32(kind.encode()))
    ps = [0.01, 0.3, 0.9, 0.95, 0.9999, 1 - 1e-7, 1.0, 0.5]
    B, K, V = len(ps), 2, 7013
    w = wl.custom(B, K, V, 64, seed=11, top_p=ps, temperature=[1.0] * B)
    w.target = np.stack([np.stack([_topp_rows(kind, V, rng) for _ in range(K + 1)])
                         for _ in range(B)]).astype(np.float32)
    cache = np.stack([np.stack([_topp_rows("lm", V, rng) for _ in range(K)])
                      for _ in range(B)]).astype(np.float32)
    draft = wl.random_drafts(w, seed=2)
    st, out, nacc = run_verify(w, draft, cache)
    assert st.status_code() == 0
    verify_parity(w, draft, cache, out, nacc, max_exception_frac=0.25)


@pytest.mark.parametrize("kind", ["lm", "ties", "ninf", "peaked", "flat", "tiny", "allninf",
                                  "coarse_ties"])
def test_topp_bf16_row_kinds(kind):
    """The top-p row kinds with bf16 target rows at temperature 1, where every
    value is one of 2^16 and the select counts values exactly: LM-like rows,
    ties, -inf columns, a spike far above the rest, flat rows, rows of values
    below 2^-10 in magnitude (with their signed zeros), rows with no finite
    value, three-valued rows; p from 0.01 to 1 - 1e-7."""
    rng = np.random.default_rng(zlib.crc32(("bf16-" + kind).encode()))
    ps = [0.01, 0.3, 0.9, 0.95, 0.9999, 1 - 1e-7, 0.5]
    B, K, V = len(ps), 2, 20011
    w = wl.custom(B, K, V, 64, seed=17, top_p=ps, temperature=[1.0] * B)

    def row():
        if kind == "tiny":
            x = (rng.standard_normal(V) * 1e-3).astype(np.float32)
            x[rng.integers(V, size=8)] = 0.0
            x[rng.integers(V, size=8)] = -0.0
            return x
        return _topp_rows(kind, V, rng)

    t32 = np.stack([np.stack([row() for _ in range(K + 1)]) for _ in range(B)])
    w.target = wl.f32_to_bf16_bits(t32)
    cache = np.stack([np.stack([_topp_rows("lm", V, rng) for _ in range(K)])
                      for _ in range(B)]).astype(np.float32)
    draft = wl.random_drafts(w, seed=4)
    st, out, nacc = run_verify(w, draft, cache)
    assert st.status_code() == 0
    verify_parity(w, draft, cache, out, nacc, max_exception_frac=0.25)


@pytest.mark.parametrize("kind", ["coarse_ties", "flat", "lm"])
def test_topp_long_rows_take_every_select_path(kind):
    """Rows of 65536 values: with three distinct values (coarse_ties) or all
    values within a few distance bins (flat), every warp lists thousands of
    window values, more than its list segment holds, and the row takes the
    exact select on the whole row; LM-like rows take the two-pass select.
    Each must give the oracle's keep set (the pages' top-p test matrix at a
    vocabulary size where the passes span many tiles)."""
    rng = np.random.default_rng(zlib.crc32(("long-" + kind).encode()))
    ps = [0.3, 0.9, 0.95, 0.5]
    B, K, V = len(ps), 1, 65536
    w = wl.custom(B, K, V, 64, seed=13, top_p=ps, temperature=[1.0] * B)
    w.target = np.stack([np.stack([_topp_rows(kind, V, rng) for _ in range(K + 1)])
                         for _ in range(B)]).astype(np.float32)
    cache = np.stack([np.stack([_topp_rows("lm", V, rng) for _ in range(K)])
                      for _ in range(B)]).astype(np.float32)
    draft = wl.random_drafts(w, seed=3)
    st, out, nacc = run_verify(w, draft, cache)
    assert st.status_code() == 0
    verify_parity(w, draft, cache, out, nacc, max_exception_frac=0.25)


def test_bf16_target_and_cache():
    w = wl.custom(16, 3, 8192, 64, seed=12, base_bf16=True, cache_bf16=True,
                  target_bf16=True, top_p=0.95, temperature=1.0)
    draft, cache = _drafted(w)
    st, out, nacc = run_verify(w, draft, cache)
    assert st.status_code() == 0
    verify_parity(w, draft, cache, out, nacc, max_exception_frac=0.07)


def test_minimax_full_b32():
    w = wl.make("minimax", batch=32)
    draft, cache = _drafted(w)
    st, out, nacc = run_verify(w, draft, cache)
    assert st.status_code() == 0
    verify_parity(w, draft, cache, out, nacc)
    assert 0.2 < nacc.mean() / w.K <= 1.0


@pytest.mark.parametrize("name,batch,pick", [
    ("qwen", 256, list(range(0, 256, 8))),
    ("long", 128, list(range(0, 128, 4))),
])
def test_full_size_sampled(name, batch, pick):
    w = wl.make(name, batch=batch)
    draft, cache = _drafted(w)
    st, out, nacc = run_verify(w, draft, cache)
    assert st.status_code() == 0
    sub = subset(w, pick)
    verify_parity(sub, draft[pick], cache, out[pick], nacc[pick], max_exception_frac=0.07)
    assert ((out >= -1) & (out < w.V)).all()
    for b in range(batch):
        m = nacc[b]
        assert (out[b, :m + 1] >= 0).all() and (out[b, m + 1:] == -1).all()


def test_first_token_distribution_on_gpu():
    """Draft d ~ q (numpy), then the GPU's first emitted token ~ p: chi-square
    over 2*10^5 requests, and the accept rate equals sum(min(p, q))."""
    import oracle
    n, V = 200_000, 6
    tgt = np.array([[0.5, 1.5, -0.5, 0.0, 2.0, -1.0], [0, 0, 0, 0, 0, 0]], np.float32)
    crow = np.array([[1.0, 0.2, 0.4, -0.3, 1.8, 0.0]], np.float32)
    T, top_p = 1.3, 0.9
    p, _, _, _, _ = oracle.target_probs(tgt[0], T, top_p)
    q = oracle.draft_probs(crow[0]).astype(np.float64)
    rng = np.random.default_rng(31)
    w = wl.custom(n, 1, V, 64, seed=1, temperature=T, top_p=top_p)
    w.target = np.broadcast_to(tgt, (n, 2, V)).copy()
    cache = np.broadcast_to(crow, (n, 1, V)).copy()
    draft = rng.choice(V, size=(n, 1), p=q / q.sum()).astype(np.int32)
    counts = np.zeros(V)
    acc = 0
    for lo in range(0, n, 256):
        idx = np.arange(lo, min(n, lo + 256))
        sub = subset(w, idx)
        sub.S = len(idx)
        sub.req_state_idx = np.arange(len(idx), dtype=np.int32)
        sub.temperature = w.temperature[idx]
        sub.top_p = w.top_p[idx]
        sub.seeds = w.seeds[idx]
        sub.C = len(idx)
        _, out, nacc = run_verify(sub, draft[idx], cache[idx])
        counts += np.bincount(out[:, 0], minlength=V)
        acc += int((nacc == 1).sum())
    p64 = p.astype(np.float64) / p.sum()
    nz = p64 > 0
    assert counts[~nz].sum() == 0
    assert stats.chisquare(counts[nz], p64[nz] / p64[nz].sum() * counts.sum()).pvalue > 0.01
    expect = np.minimum(p64, q / q.sum()).sum()
    assert abs(acc / n - expect) < 4 * np.sqrt(expect * (1 - expect) / n)


def test_bad_draft_token_reports_bounds():
    w = wl.custom(3, 2, 500, 64, seed=13)
    draft = wl.random_drafts(w)
    draft[1, 0] = 500
    _, cache = _drafted(w)
    st, out, nacc = run_verify(w, draft, cache)
    assert st.status_code() == -5
    assert (out[1] == -1).all() and nacc[1] == 0
    good = [0, 2]
    verify_parity(subset(w, good), draft[good], cache, out[good], nacc[good])
