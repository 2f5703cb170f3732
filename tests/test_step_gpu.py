"""A whole decode step (Markov loop + verification) through the library:
repeatability, CUDA-graph capture and replay, and parity of the chained
outputs with the oracle on the small workloads."""
import numpy as np
import pytest

from parity import markov_parity, verify_parity
from gpu_util import require_gpu
from verify_dspark_markov_step_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "odd"])
def test_decode_step_parity(name):
    torch = require_gpu()
    from verify_dspark_markov_step_gb300.step import DecodeStep, to_numpy
    w = wl.make(name)
    st = DecodeStep(w)
    st.run()
    torch.cuda.synchronize()
    assert st.status_code() == 0
    draft = st.draft.cpu().numpy()
    cache = to_numpy(st.cache)
    markov_parity(w, draft, cache)
    verify_parity(w, draft, cache, st.out.cpu().numpy(), st.num_accepted.cpu().numpy(),
                  max_exception_frac=0.13)


def test_decode_step_graph_replay_is_bitwise_stable():
    torch = require_gpu()
    from verify_dspark_markov_step_gb300.step import DecodeStep
    w = wl.custom(16, 4, 30011, 256, seed=21, temperature=[0.0, 0.8, 1.0, 1.2] * 4,
                  top_p=[1.0, 0.9, 0.95, 0.7] * 4)
    st = DecodeStep(w)
    st.run()
    torch.cuda.synchronize()
    ref = [t.clone() for t in (st.draft, st.cache, st.out, st.num_accepted)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        st.run(stream=s)
    for _ in range(5):
        st.out.fill_(-9)
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(ref, (st.draft, st.cache, st.out, st.num_accepted)):
            assert torch.equal(a, b)
    assert st.status_code() == 0


def _row_max_reference(cache, rsi, row_map, K, bf16):
    """Maximum of every cache row a request wrote, from the stored values
    (NaN read as -inf)."""
    from verify_dspark_markov_step_gb300.workloads import bf16_bits_to_f32
    x = bf16_bits_to_f32(cache) if bf16 else cache.astype(np.float32)
    out = {}
    for b, s in enumerate(rsi):
        if s < 0:
            continue
        row = s if row_map is None else row_map[s]
        for k in range(K):
            out[(b, k)] = np.float32(np.where(np.isnan(x[row, k]), -np.inf, x[row, k]).max())
    return out


@pytest.mark.parametrize("name", ["odd", "bf16_rowmap", "wide"])
def test_draft_row_statistics_from_the_loop(name):
    """The loop's cache-row statistics: the maximum equals the stored row's
    maximum exactly, and the fixed-point mass equals sum exp(x - m) of the
    stored row (fp64 here) within 1e-5 relative (fp32 partial sums of ex2
    terms); batches above 32 report them as not recorded. The verifier that
    takes them (and reads no draft row for its distribution) and the
    verifier that reads every row both match the oracle."""
    torch = require_gpu()
    from verify_dspark_markov_step_gb300 import _lib
    from verify_dspark_markov_step_gb300.step import DecodeStep, to_numpy
    if name == "odd":
        w = wl.make("odd")
    elif name == "wide":  # more than 32 requests: statistics reported as not recorded
        w = wl.custom(40, 2, 4099, 64, seed=8, temperature=0.9, top_p=0.95)
    else:
        w = wl.custom(12, 3, 30011, 192, seed=5, base_bf16=True, cache_bf16=True, S=16,
                      rsi=[15, 2, -1, 7, 0, 11, 3, 9, -1, 4, 13, 1],
                      row_map=[3, 0, 5, 1, 2, 4, 15, 14, 13, 12, 11, 10, 9, 8, 7, 6],
                      temperature=[1.0, 0.7, 0.0, 1.3] * 4, top_p=[1.0, 0.9] * 8)
    st = DecodeStep(w)
    st.run()
    torch.cuda.synchronize()
    assert st.status_code() == 0
    m_all, mass_all = _lib.row_stats_fields(st.dstats)
    m_all, mass_all = m_all.numpy(), mass_all.numpy().astype(np.float64)
    cache = to_numpy(st.cache)
    x_all = wl.bf16_bits_to_f32(cache) if w.cache_bf16 else cache
    ref = _row_max_reference(cache, w.req_state_idx, w.row_map, w.K, w.cache_bf16)
    for (b, k), m in ref.items():
        if w.B > 32:
            assert np.isnan(m_all[b, k]), (b, k, m_all[b, k])
            continue
        assert m_all[b, k] == m, (b, k, m_all[b, k], m)
        s = w.req_state_idx[b]
        row = x_all[s if w.row_map is None else w.row_map[s], k].astype(np.float64)
        row = np.where(np.isnan(row), -np.inf, row)
        want = np.exp(row - m).sum() if np.isfinite(m) else 0.0
        np.testing.assert_allclose(mass_all[b, k] * 2.0 ** -40, want, rtol=1e-5)
    draft = st.draft.cpu().numpy()
    verify_parity(w, draft, cache, st.out.cpu().numpy(), st.num_accepted.cpu().numpy())
    # the verifier reading every row
    st2 = DecodeStep(w, draft_stats=False)
    st2.draft.copy_(st.draft)
    st2.cache.copy_(st.cache)
    st2.verify()
    torch.cuda.synchronize()
    assert st2.status_code() == 0
    verify_parity(w, draft, cache, st2.out.cpu().numpy(), st2.num_accepted.cpu().numpy())


def test_largest_vocabulary_decode_step():
    """V = 2^22 - 1, the largest vocabulary the library takes: every 32-bit
    token index and the 64-bit row offsets at their extremes, a ragged last
    tile, and a top-p row over the whole vocabulary."""
    torch = require_gpu()
    from verify_dspark_markov_step_gb300.step import DecodeStep, to_numpy
    w = wl.custom(2, 2, (1 << 22) - 1, 64, seed=31, temperature=[1.0, 0.8], top_p=[1.0, 0.9])
    st = DecodeStep(w)
    st.run()
    torch.cuda.synchronize()
    assert st.status_code() == 0
    draft = st.draft.cpu().numpy()
    cache = to_numpy(st.cache)
    assert markov_parity(w, draft, cache) <= 1
    verify_parity(w, draft, cache, st.out.cpu().numpy(), st.num_accepted.cpu().numpy(),
                  max_exception_frac=0.5)
