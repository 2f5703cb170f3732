"""Writes the fixtures in this folder from the oracle alone (no GPU code).

The pages print no worked numeric example, so these values are not the
pages': they record what the oracle computes on small seeded inputs, so that
any later change to the oracle's arithmetic shows up as a failing
tests/test_golden.py and has to be made on purpose (regenerating the files
with this script). Inputs come from the seeded generator module only.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from verify_dspark_markov_step_gb300 import workloads as wl  # noqa: E402

# (seed, position, column, stream) tuples: the draft, target and accept
# streams, columns in all four words of a block, positions around 2^32
NOISE_CASES = [
    (0, 0, 0, 0), (1, 21999, 3, 1 << 30), (0x9E3779B97F4A7C15, 22036, 200063, 0),
    (12345, (1 << 32) + 5, 7, 1 << 29), (2 ** 64 - 1, 2 ** 40, 4096, 1 << 30),
    (77, -1, 1, 0),
]


def noise_fixture():
    seed = np.array([c[0] for c in NOISE_CASES], dtype=np.uint64)
    pos = np.array([c[1] for c in NOISE_CASES], dtype=np.int64)
    col = np.array([c[2] for c in NOISE_CASES], dtype=np.uint32)
    stream = np.array([c[3] for c in NOISE_CASES], dtype=np.uint32)
    word, u, g = oracle.noise(seed, pos, col, stream)
    return [dict(seed=int(s), pos=int(p), col=int(c), stream=int(t), word=int(w),
                 u_bits=int(np.float32(uu).view(np.uint32)),
                 g_bits=int(np.float32(gg).view(np.uint32)))
            for s, p, c, t, w, uu, gg in zip(seed, pos, col, stream, word, u, g)]


def decode_fixture(name):
    w = wl.make(name)
    tok, cache, gaps = oracle.markov_sample(
        w.base, w.w1, w.w2, w.anchor, w.req_state_idx, w.positions, w.temperature,
        w.seeds, cache_rows=w.C, cache_bf16=w.cache_bf16, row_map=w.row_map)
    res = oracle.rejection_sample(tok, cache, w.target, w.req_state_idx, w.positions,
                                  w.temperature, w.top_p, w.seeds, row_map=w.row_map)
    c32 = wl.bf16_bits_to_f32(cache) if w.cache_bf16 else np.asarray(cache, np.float32)
    finite = np.where(np.isnan(c32), -np.inf, c32)
    return dict(workload=name, draft_tokens=tok.tolist(),
                min_draft_gap=float(np.min(gaps)),
                cache_row_max_bits=[[int(np.float32(v).view(np.uint32)) for v in row]
                                    for row in finite.max(axis=-1).reshape(-1, w.K)],
                out_tokens=res["out_tokens"].tolist(),
                num_accepted=res["num_accepted"].tolist())


def topk_fixture(name, k):
    w = wl.make(name, with_target=False)
    tok, cache, gaps = oracle.markov_sample(
        w.base, w.w1, w.w2, w.anchor, w.req_state_idx, w.positions, w.temperature,
        w.seeds, cache_rows=w.C, cache_bf16=w.cache_bf16, row_map=w.row_map, topk=k)
    c32 = wl.bf16_bits_to_f32(cache) if w.cache_bf16 else np.asarray(cache, np.float32)
    return dict(workload=name, topk=k, draft_tokens=tok.tolist(),
                min_draft_gap=float(np.min(gaps)),
                finite_per_row=np.isfinite(c32).sum(axis=-1).reshape(-1).tolist())


def main():
    with open(os.path.join(HERE, "oracle_noise.json"), "w") as f:
        json.dump(noise_fixture(), f, indent=1)
    for name in ("tiny", "odd"):
        with open(os.path.join(HERE, f"oracle_decode_{name}.json"), "w") as f:
            json.dump(decode_fixture(name), f, indent=1)
    with open(os.path.join(HERE, "oracle_topk_odd_k64.json"), "w") as f:
        json.dump(topk_fixture("odd", 64), f, indent=1)


if __name__ == "__main__":
    main()
