"""Parity of the CUDA Markov drafting loop with the CPU oracle.

Tokens must be bit-exact except where the oracle's top-two noised-value gap is
below 1e-5 (counted); the fp32 cache within abs 1e-4 + rel 1e-5 (NaN = NaN),
a bf16 cache within one bf16 ulp. Sizes span several 64-row tiles with a
ragged tail; the full-size workloads are checked on sampled requests, each
replayed step by step from the GPU's own previous token.
"""
import numpy as np
import pytest

from parity import markov_parity, subset
from gpu_util import require_gpu, run_markov
from verify_dspark_markov_step_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_tiny():
    w = wl.make("tiny")
    st, tok, cache = run_markov(w)
    assert st.status_code() == 0
    assert markov_parity(w, tok, cache) == 0


def _edge_values():
    """fp32 values at the edges of bf16 rounding (halfway cases with an even
    and an odd kept bit, one bit either side), fp32 subnormals, values that
    round up to infinity, infinities and signed zeros."""
    bits = []
    for hi in (0x3F80, 0x3F81, 0x4123, 0xC0A1, 0x0001, 0x7F7E):
        for lo in (0x8000, 0x7FFF, 0x8001):
            bits.append((hi << 16) | lo)
    bits += [0x00000001, 0x80000001, 0x007FFFFF, 0x7F7F7FFF, 0x7F7F8000, 0xFF7F8000,
             0x7F800000, 0xFF800000, 0x00000000, 0x80000000]
    return np.array(bits, np.uint32).view(np.float32)


@pytest.mark.parametrize("base_bf16,cache_bf16", [(False, False), (False, True), (True, True)])
def test_zero_bias_cache_is_bit_identical(base_bf16, cache_bf16):
    """markov_w2 = 0 makes the bias exactly 0 on both sides, so the cached
    value is fp32(base / T) with nothing left to round differently: the GPU
    cache must equal the oracle's bit for bit at T = 1, 0.5, 0.7, 1.3 and 0
    (IEEE division, nearest-even bf16), NaN where the oracle has NaN."""
    temps = [1.0, 0.5, 0.7, 1.3, 0.0]
    B, K, V, R = len(temps), 3, 4097, 64
    w = wl.custom(B, K, V, R, seed=77, temperature=temps, base_bf16=False,
                  cache_bf16=cache_bf16)
    edge = _edge_values()
    base = w.base.copy()
    base[:, :, 1000:1000 + edge.size] = edge
    base[2, 1, 3000] = np.nan
    w.base = wl.f32_to_bf16_bits(base) if base_bf16 else base
    w.w2 = np.zeros_like(w.w2)
    st, tok, cache = run_markov(w)
    assert st.status_code() == 0
    import oracle
    _, cache_o, _ = oracle.markov_sample(
        w.base, w.w1, w.w2, w.anchor, w.req_state_idx, w.positions, w.temperature,
        w.seeds, cache_rows=w.C, cache_bf16=cache_bf16, forced=tok)
    if cache_bf16:
        nan_g = np.isnan(wl.bf16_bits_to_f32(cache))
        nan_o = np.isnan(wl.bf16_bits_to_f32(cache_o))
    else:
        nan_g, nan_o = np.isnan(cache), np.isnan(cache_o)
    np.testing.assert_array_equal(nan_g, nan_o)
    np.testing.assert_array_equal(cache[~nan_g], cache_o[~nan_o])
    assert markov_parity(w, tok) <= 1


def test_bounded_waits_run_out_and_the_next_call_is_clean():
    """The grid barrier waits for one arrival more than the grid makes, with
    every wait limited to 1 ms: each CTA's barrier wait runs out, then the
    waits of its MMA and copy warps (whose next step never starts); the call
    must end within a few limits with DSPARK_ERR_TIMEOUT in *status, and the
    next normal call on the same stream and workspace must give exactly what
    a fresh run gives (the pages' bounded exchange wait that raises on
    timeout instead of hanging: vLLM PR #65007, Part 1)."""
    import time
    import torch
    from verify_dspark_markov_step_gb300 import _lib
    w = wl.make("tiny", with_target=False)
    st, tok0, cache0 = run_markov(w)
    assert st.status_code() == 0
    stream = torch.cuda.Stream()
    st.status.zero_()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        _lib.markov_sample_wait_limit(st.base, st.w1, st.w2, st.anchor, st.rsi, st.pos,
                                      st.temperature, st.seeds, st.draft, 1_000_000, 1,
                                      cache=st.cache, workspace_buf=st.ws_markov,
                                      status=st.status, stream=stream)
    stream.synchronize()
    elapsed = time.perf_counter() - t0
    assert st.status_code() == -4, st.status_code()   # DSPARK_ERR_TIMEOUT
    assert elapsed < 1.0, elapsed
    # the same hook with the barrier left alone completes normally
    st.status.zero_()
    with torch.cuda.stream(stream):
        _lib.markov_sample_wait_limit(st.base, st.w1, st.w2, st.anchor, st.rsi, st.pos,
                                      st.temperature, st.seeds, st.draft, 1_000_000_000, 0,
                                      cache=st.cache, workspace_buf=st.ws_markov,
                                      status=st.status, stream=stream)
    stream.synchronize()
    assert st.status_code() == 0
    np.testing.assert_array_equal(st.draft.cpu().numpy(), tok0)
    # and the normal entry point after the timeout is bit-identical to before
    st.draft.fill_(-7)
    st.cache.zero_()
    with torch.cuda.stream(stream):
        st.markov(stream=stream)
    stream.synchronize()
    assert st.status_code() == 0
    np.testing.assert_array_equal(st.draft.cpu().numpy(), tok0)
    from verify_dspark_markov_step_gb300.step import to_numpy
    np.testing.assert_array_equal(to_numpy(st.cache), cache0)


def test_odd_vocab_nan_and_temperatures():
    w = wl.make("odd", with_target=False)
    st, tok, cache = run_markov(w)
    assert st.status_code() == 0
    exc = markov_parity(w, tok, cache)
    assert exc <= 1
    # planted NaN rows: a NaN column wins wherever the base row has one
    for b in range(w.B):
        for i in range(w.K):
            nan_cols = np.flatnonzero(np.isnan(w.base[b, i]))
            if nan_cols.size:
                assert tok[b, i] == nan_cols[0]


@pytest.mark.parametrize("B,K,V,R,kw", [
    (1, 1, 1, 64, {}),
    (3, 2, 37, 64, {}),
    (2, 3, 4097, 128, {"temperature": [0.5, 1.7]}),
    (5, 4, 6151, 192, {"temperature": [1.0, 0.0, 0.8, 1.3, 0.0]}),
    (4, 3, 3000, 256, {"S": 6, "rsi": [2, -1, 0, 5], "row_map": [3, 0, 5, 1, 2, 4],
                       "temperature": [1.0, 0.7, 1.2, 1.0, 0.9, 0.0]}),
    (3, 2, 2048, 512, {"temperature": [0.9, 1.1, 1.0]}),
    (6, 3, 5000, 64, {"base_bf16": True, "cache_bf16": True,
                      "temperature": [0.6, 1.0, 1.4, 0.0, 1.0, 0.8]}),
    # larger batches: more N columns per MMA, more epilogue columns per warp
    (8, 2, 129, 64, {}),
    (16, 3, 2053, 128, {"temperature": [0.0, 0.5, 1.0, 1.5] * 4}),
    (33, 2, 4100, 256, {"temperature": 0.9}),
    (20, 2, 3001, 192, {"S": 24, "rsi": list(range(23, 3, -1)), "temperature": 1.1}),
    (12, 2, 1500, 512, {"base_bf16": True, "cache_bf16": True}),
    (64, 1, 777, 256, {}),
    # the most draft steps the library takes
    (3, 16, 3001, 128, {"temperature": [1.0, 0.0, 0.6]}),
    # 200 tiles on a 152-SM grid: the 48 remainder tiles (the ragged last one
    # among them) are each shared by two CTAs, half the request columns each
    (20, 3, 25500, 128, {"temperature": [1.0, 0.0, 0.7, 1.3] * 5}),
    (40, 2, 25500, 64, {"base_bf16": True, "cache_bf16": True, "temperature": 0.9}),
])
def test_edge_shapes(B, K, V, R, kw):
    w = wl.custom(B, K, V, R, seed=B * 7 + V, **kw)
    st, tok, cache = run_markov(w)
    assert st.status_code() == 0
    assert markov_parity(w, tok, cache) <= 1
    for b in range(B):
        if w.req_state_idx[b] < 0:
            assert (tok[b] == -1).all()
    if w.row_map is not None:
        used = {int(w.row_map[s]) for s in w.req_state_idx if s >= 0}
        for row in range(w.C):
            if row not in used:
                assert (cache[row] == 0).all()


def test_empty_batch():
    w = wl.custom(0, 2, 100, 64, S=1)
    st, tok, _ = run_markov(w)
    assert tok.shape == (0, 2)


@pytest.mark.parametrize("B", [1, 4])
def test_minimax_full(B):
    w = wl.make("minimax", batch=B, with_target=False)
    st, tok, cache = run_markov(w)
    assert st.status_code() == 0
    assert markov_parity(w, tok, cache) <= 1


@pytest.mark.parametrize("name,batch,pick", [
    ("minimax", 32, [0, 13, 31]),
    ("long", 128, [0, 1, 77, 127]),
    ("qwen", 256, [0, 100, 255]),
])
def test_full_size_sampled(name, batch, pick):
    w = wl.make(name, batch=batch, with_target=False)
    st, tok, cache = run_markov(w)
    assert st.status_code() == 0
    sub = subset(w, pick)
    exc = markov_parity(sub, tok[pick], cache)
    assert exc <= 1
    # every request produced valid tokens
    assert ((tok >= 0) & (tok < w.V)).all()


def test_repeatable_and_graph_replay():
    import torch
    w = wl.custom(8, 5, 20011, 256, seed=3, temperature=[0.9, 1.0, 0.0, 1.2, 1.0, 0.7, 1.0, 1.1])
    from verify_dspark_markov_step_gb300.step import DecodeStep
    st = DecodeStep(w, with_target=False)
    st.markov()
    torch.cuda.synchronize()
    tok1, cache1 = st.draft.clone(), st.cache.clone()
    st.markov()
    torch.cuda.synchronize()
    assert torch.equal(st.draft, tok1) and torch.equal(st.cache, cache1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        st.markov(stream=s)
    st.draft.fill_(-7)
    st.cache.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(st.draft, tok1) and torch.equal(st.cache, cache1)


def test_out_of_range_anchor_reports_bounds():
    import torch
    w = wl.custom(3, 2, 1000, 64, seed=9)
    w.anchor = w.anchor.copy()
    w.anchor[1] = 1000                      # == V: out of range
    st, tok, _ = run_markov(w)
    assert st.status_code() == -5           # DSPARK_ERR_BOUNDS
    assert (tok[1] == -1).all()
    good = [0, 2]
    assert markov_parity(subset(w, good), tok[good], None) == 0
    torch.cuda.synchronize()
