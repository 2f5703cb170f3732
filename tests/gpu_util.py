"""Helpers for the GPU tests: build the library once, run a workload."""
from __future__ import annotations

import numpy as np
import pytest


def require_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from verify_dspark_markov_step_gb300 import build
    build.build()
    return torch


def run_markov(w):
    import torch
    from verify_dspark_markov_step_gb300.step import DecodeStep, to_numpy
    st = DecodeStep(w, with_target=False)
    st.markov()
    torch.cuda.synchronize()
    return st, st.draft.cpu().numpy(), to_numpy(st.cache)


def run_verify(w, draft, cache):
    """Verify given host drafts and cache (numpy) on the GPU."""
    import torch
    from verify_dspark_markov_step_gb300.step import DecodeStep, to_device
    st = DecodeStep(w, draft_stats=False)  # the cache is the caller's: rows are read
    st.draft.copy_(torch.from_numpy(np.ascontiguousarray(draft, np.int32)))
    st.cache = to_device(np.ascontiguousarray(cache))
    st.verify()
    torch.cuda.synchronize()
    return st, st.out.cpu().numpy(), st.num_accepted.cpu().numpy()
