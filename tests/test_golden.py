"""Stored oracle outputs (tests/golden/, written by tests/golden/make_golden.py
from the oracle alone): the CPU test recomputes them, so a change to the
oracle's arithmetic cannot pass unnoticed; the GPU test checks the CUDA path
against the stored tokens (their decisions are far from ties: the smallest
top-two gap of the oracle's draws is recorded with them)."""
import json
import os
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")
sys.path.insert(0, GOLDEN)


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_oracle_noise_matches_stored():
    import make_golden
    got = make_golden.noise_fixture()
    want = _load("oracle_noise.json")
    assert len(got) == len(want)
    for g, w in zip(got, want):
        assert g["word"] == w["word"] and g["u_bits"] == w["u_bits"], (g, w)
        # g = -log(-log u) in fp64 rounded to fp32: allow one ulp across libm builds
        assert abs(g["g_bits"] - w["g_bits"]) <= 1, (g, w)


@pytest.mark.parametrize("name", ["tiny", "odd"])
def test_oracle_decode_matches_stored(name):
    import make_golden
    got = make_golden.decode_fixture(name)
    want = _load(f"oracle_decode_{name}.json")
    assert got["draft_tokens"] == want["draft_tokens"]
    assert got["cache_row_max_bits"] == want["cache_row_max_bits"]
    assert got["out_tokens"] == want["out_tokens"]
    assert got["num_accepted"] == want["num_accepted"]


def test_oracle_topk_matches_stored():
    import make_golden
    want = _load("oracle_topk_odd_k64.json")
    got = make_golden.topk_fixture(want["workload"], want["topk"])
    assert got["draft_tokens"] == want["draft_tokens"]
    assert got["finite_per_row"] == want["finite_per_row"]


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny", "odd"])
def test_gpu_tokens_match_stored(name):
    from gpu_util import require_gpu
    torch = require_gpu()
    from verify_dspark_markov_step_gb300 import workloads as wl
    from verify_dspark_markov_step_gb300.step import DecodeStep
    want = _load(f"oracle_decode_{name}.json")
    assert want["min_draft_gap"] > 1e-3  # far from any tie the GPU's rounding could flip
    st = DecodeStep(wl.make(name))
    st.run()
    torch.cuda.synchronize()
    assert st.status_code() == 0
    assert st.draft.cpu().numpy().tolist() == want["draft_tokens"]
    if name == "tiny":
        assert st.out.cpu().numpy().tolist() == want["out_tokens"]
        assert st.num_accepted.cpu().numpy().tolist() == want["num_accepted"]
