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
