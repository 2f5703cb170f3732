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
