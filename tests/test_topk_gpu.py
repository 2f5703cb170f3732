"""Parity of the top-k variant of the Markov loop (the "DSparkSpeculator"
page, _sample_sequential_topk) with the CPU oracle: the bias only on the
top-k base logits of each request and step, -inf elsewhere. Tokens as for the
dense loop (bit-exact but for counted near-ties); the cache exactly -inf off
the candidates and within the cache tolerance on them. The verifier then
runs unchanged on the truncated cache."""
import numpy as np
import pytest

from parity import markov_parity, verify_parity
from gpu_util import require_gpu
from verify_dspark_markov_step_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _run(w, topk):
    torch = require_gpu()
    from verify_dspark_markov_step_gb300.step import DecodeStep, to_numpy
    st = DecodeStep(w, draft_topk=topk)
    st.run()
    torch.cuda.synchronize()
    return st, st.draft.cpu().numpy(), to_numpy(st.cache)


@pytest.mark.parametrize("case", ["tiny", "odd", "bf16_rowmap", "ties", "nan_heavy", "k_over_v",
                                  "coarse_big"])
def test_topk_loop_and_verify(case):
    k = {"tiny": 7, "odd": 64, "bf16_rowmap": 100, "ties": 33, "nan_heavy": 5,
         "k_over_v": 5000, "coarse_big": 5000}[case]
    if case == "tiny":
        w = wl.make("tiny")
    elif case == "odd":
        w = wl.make("odd")
    elif case == "bf16_rowmap":
        w = wl.custom(12, 3, 30011, 192, seed=5, base_bf16=True, cache_bf16=True, S=16,
                      rsi=[15, 2, -1, 7, 0, 11, 3, 9, -1, 4, 13, 1],
                      row_map=[3, 0, 5, 1, 2, 4, 15, 14, 13, 12, 11, 10, 9, 8, 7, 6],
                      temperature=[1.0, 0.7, 0.0, 1.3] * 4, top_p=[1.0, 0.9] * 8)
    elif case == "ties":  # quarter-step base logits: long runs of equal candidates
        w = wl.custom(4, 3, 6151, 64, seed=12, temperature=[1.0, 0.5, 0.0, 1.1])
        w.base = (np.round(w.base * 4) / 4).astype(np.float32)
    elif case == "nan_heavy":  # more NaN columns than k in some rows
        w = wl.custom(3, 2, 4099, 64, seed=13, temperature=[1.0, 0.0, 0.8])
        rng = np.random.default_rng(1)
        w.base = w.base.copy()
        w.base[0, 0, rng.integers(0, 4099, 9)] = np.nan
        w.base[1, 1, [3, 4000]] = np.nan
    elif case == "coarse_big":  # three values over 65536 columns: the boundary
        # value holds far more candidates than a list keeps (the radix stages)
        w = wl.custom(2, 2, 65536, 64, seed=15, temperature=[1.0, 0.9])
        w.base = np.random.default_rng(2).integers(0, 3, w.base.shape).astype(np.float32)
    else:  # k above V: every column is a candidate (the dense loop)
        w = wl.custom(3, 2, 4099, 128, seed=14, temperature=[1.0, 0.0, 0.8])
    st, tok, cache = _run(w, k)
    assert st.status_code() == 0
    assert markov_parity(w, tok, cache, topk=k) <= 1
    for b, s in enumerate(w.req_state_idx):
        if s < 0:
            assert (tok[b] == -1).all()
    verify_parity(w, tok, cache, st.out.cpu().numpy(), st.num_accepted.cpu().numpy(),
                  max_exception_frac=0.13)


def test_topk_covering_the_vocabulary_equals_the_dense_loop():
    torch = require_gpu()
    from verify_dspark_markov_step_gb300.step import DecodeStep
    w = wl.custom(5, 3, 3001, 128, seed=15, temperature=[1.0, 0.0, 0.8, 1.2, 1.0])
    dense = DecodeStep(w)
    dense.markov()
    topk = DecodeStep(w, draft_topk=3001)
    topk.markov()
    torch.cuda.synchronize()
    assert torch.equal(dense.draft, topk.draft)
    # the dense cache comes from the tensor-core projection, the top-k one from
    # fp32 dot products: equal within the cache tolerance
    np.testing.assert_allclose(topk.cache.cpu().numpy(), dense.cache.cpu().numpy(),
                               atol=1e-4, rtol=1e-5)


def test_topk_full_vocabulary_sampled():
    """MiniMax-like vocabulary and rank, k = 1024, two requests checked in full."""
    w = wl.make("minimax", batch=4, with_target=True)
    st, tok, cache = _run(w, 1024)
    assert st.status_code() == 0
    assert markov_parity(w, tok, cache, topk=1024) <= 1
    assert ((cache != -np.inf).sum(axis=2)[:4] == 1024).all()
