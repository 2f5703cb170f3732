"""dspark_markov_sample_static: the Markov sampling loop for callers that may
not allocate device memory (an engine plug-in handed all of its memory, a
decode loop that cannot take cudaMalloc's latency and synchronisation, a host
with no CUDA allocator). It keeps its scratch in a fixed array inside the
library, so the test checks that two calls in a row, the second on different
sizes and left-over scratch, give what dspark_markov_sample gives with a
fresh workspace: the same tokens, and caches within the parity tolerance.

This file's name sorts last so that a run stopping at its first failure has
run every other test first.
"""
import ctypes
import os
import shutil

import numpy as np
import pytest

from parity import check_cache

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _library():
    if not shutil.which("nvcc") and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from verify_dspark_markov_step_gb300 import _lib, build
    build.build()
    return _lib.lib()


def test_sizes_beyond_the_fixed_scratch_are_rejected_on_the_host():
    """The limit is checked before anything touches the device, so this runs
    without a GPU. 32 KiB fits 256 requests with 15 draft steps but not 16."""
    L = _library()
    from verify_dspark_markov_step_gb300 import _lib
    assert _lib.markov_workspace_bytes(256, 15, (1 << 22) - 1, 512) <= _lib.STATIC_SCRATCH_BYTES
    assert _lib.markov_workspace_bytes(256, 16, 200064, 256) > _lib.STATIC_SCRATCH_BYTES
    fake = ctypes.c_void_p(256)  # never dereferenced: every call below fails first

    def call(B, V, K=7, R=256, S=1, base=fake, bdt=0):
        return L.dspark_markov_sample_static(base, bdt, fake, fake, fake, fake, fake, fake, fake,
                                             None, 0, None, fake, None, B, K, V, R, S, 1, None,
                                             None)
    assert call(256, 200064, K=16) == -8           # DSPARK_ERR_SCRATCH_LIMIT
    assert _lib.status_string(-8).startswith("sizes need more scratch")
    # every argument check of dspark_markov_sample comes before the limit,
    # with its own code, also on sizes the scratch could not hold
    assert call(-1, 1000) == -1
    assert call(4, 1 << 22) == -1
    assert call(256, 200064, K=16, bdt=7) == -1    # bad dtype
    assert call(256, 200064, K=16, R=100) == -2    # unsupported markov_rank
    assert call(256, 200064, K=16, base=None) == -1
    assert call(256, 200064, K=16, base=ctypes.c_void_p(258)) == -7
    assert call(0, 200064, K=16) == 0              # empty batch: nothing to do


def _reference_and_static(w):
    """Tokens and cache from dspark_markov_sample (its own workspace) and from
    dspark_markov_sample_static, on the same inputs."""
    import torch
    from verify_dspark_markov_step_gb300 import _lib
    from verify_dspark_markov_step_gb300.step import DecodeStep, to_numpy
    st = DecodeStep(w, with_target=False)
    st.markov()
    torch.cuda.synchronize()
    assert st.status_code() == 0
    ref_tok, ref_cache = st.draft.cpu().numpy(), to_numpy(st.cache)
    st.draft.fill_(-7)
    st.cache.zero_()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.markov_sample_static(st.base, st.w1, st.w2, st.anchor, st.rsi, st.pos,
                              st.temperature, st.seeds, st.draft, cache=st.cache,
                              cache_row_map=st.row_map, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return ref_tok, ref_cache, st.draft.cpu().numpy(), to_numpy(st.cache)


@pytest.mark.gpu
def test_static_scratch_matches_the_workspace_entry_point_twice_in_a_row():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _library()
    from verify_dspark_markov_step_gb300 import workloads as wl
    # first call: ragged vocabulary with NaN columns, mixed temperatures
    w1 = wl.make("odd", with_target=False)
    # second call: more requests, another vocabulary and grid, bf16 logits and
    # cache, a row map and padding, over what the first call left behind
    w2 = wl.custom(20, 3, 30011, 192, seed=17, base_bf16=True, cache_bf16=True, S=24,
                   rsi=[23, 5, -1, 0, 7, 11, 2, 19, 3, 14, 8, -1, 1, 9, 21, 4, 6, 12, 10, 13],
                   row_map=list(range(23, -1, -1)),
                   temperature=[1.0, 0.0, 0.8, 1.3] * 6)
    for w in (w1, w2):
        ref_tok, ref_cache, tok, cache = _reference_and_static(w)
        np.testing.assert_array_equal(tok, ref_tok)
        check_cache(cache, ref_cache, w.cache_bf16)
