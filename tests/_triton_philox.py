"""Reference Philox4x32-10 outputs from a library: Triton's ``tl.philox``,
run on the CPU by Triton's interpreter. Used by the oracle pin tests, in a
subprocess so that TRITON_INTERPRET is set before Triton is imported.

Reads a .npz with ``key`` [n,2] uint32 and ``ctr`` [n,4] uint32; writes
``out`` [n,4] uint32 to the second path.
"""
import os
import sys

os.environ["TRITON_INTERPRET"] = "1"

import numpy as np  # noqa: E402
import torch  # noqa: E402
import triton  # noqa: E402
import triton.language as tl  # noqa: E402


@triton.jit
def _philox_kernel(seed_ptr, ctr_ptr, out_ptr, N: tl.constexpr):
    i = tl.arange(0, N)
    seed = tl.load(seed_ptr + i)
    c0 = tl.load(ctr_ptr + i * 4 + 0)
    c1 = tl.load(ctr_ptr + i * 4 + 1)
    c2 = tl.load(ctr_ptr + i * 4 + 2)
    c3 = tl.load(ctr_ptr + i * 4 + 3)
    r0, r1, r2, r3 = tl.philox(seed, c0, c1, c2, c3)
    tl.store(out_ptr + i * 4 + 0, r0)
    tl.store(out_ptr + i * 4 + 1, r1)
    tl.store(out_ptr + i * 4 + 2, r2)
    tl.store(out_ptr + i * 4 + 3, r3)


def main(inp, outp):
    d = np.load(inp)
    key = d["key"].astype(np.uint64)
    ctr = d["ctr"].astype(np.uint32)
    n = key.shape[0]
    assert n & (n - 1) == 0, "n must be a power of two"
    seed64 = (key[:, 0] | (key[:, 1] << np.uint64(32))).view(np.int64)
    seed_t = torch.from_numpy(seed64.copy())
    ctr_t = torch.from_numpy(ctr.view(np.int32).reshape(-1).copy())
    out_t = torch.zeros(n * 4, dtype=torch.int32)
    _philox_kernel[(1,)](seed_t, ctr_t, out_t, n)
    np.save(outp, out_t.numpy().view(np.uint32).reshape(n, 4))


if __name__ == "__main__":
    main(sys.argv[1], sys.argv[2])
