"""One decode step of the DSpark hot path on device tensors: the K-step Markov
drafting loop (which writes the draft tokens and the draft-logits cache) and
the rejection-sampling verification of those drafts against the target
logits. Both run in the CUDA library; this module only holds the buffers.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _lib
from .workloads import Workload


def to_device(a: np.ndarray, device="cuda", bf16_bits: bool = False) -> torch.Tensor:
    """numpy -> device tensor; uint16 arrays are bf16 bit patterns, uint64 seeds
    travel as int64 with the same bits."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    if a.dtype == np.uint64:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int64)).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def to_numpy(t: torch.Tensor) -> np.ndarray:
    """device tensor -> numpy; bf16 comes back as uint16 bit patterns."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


class DecodeStep:
    """Device buffers of one workload and the two library calls."""

    def __init__(self, w: Workload, device="cuda", with_target: bool = True,
                 draft_stats: bool = True, draft_topk: int = 0):
        self.w = w
        self.device = device
        self.base = to_device(w.base, device)
        self.w1 = to_device(w.w1, device)
        self.w2 = to_device(w.w2, device)
        self.anchor = to_device(w.anchor, device)
        self.rsi = to_device(w.req_state_idx, device)
        self.pos = to_device(w.positions, device)
        self.temperature = to_device(w.temperature, device)
        self.top_p = to_device(w.top_p, device)
        self.seeds = to_device(w.seeds, device)
        self.row_map = None if w.row_map is None else to_device(w.row_map, device)
        self.target = to_device(w.target, device) if (with_target and w.target is not None) else None
        cache_dtype = torch.bfloat16 if w.cache_bf16 else torch.float32
        self.cache = torch.zeros((w.C, w.K, w.V), dtype=cache_dtype, device=device)
        self.draft = torch.full((w.B, w.K), -1, dtype=torch.int32, device=device)
        self.out = torch.full((w.B, w.K + 1), -1, dtype=torch.int32, device=device)
        self.num_accepted = torch.zeros(w.B, dtype=torch.int32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.ws_markov = _lib.workspace(_lib.markov_workspace_bytes(w.B, w.K, w.V, w.R), device)
        self.ws_verify = _lib.workspace(_lib.verify_workspace_bytes(w.B, w.K, w.V), device)
        # statistics of the cache rows, written by the Markov loop and read by
        # the verifier instead of the rows themselves
        self.dstats = _lib.row_stats(w.B, w.K, device) if draft_stats else None
        # top-k variant of the loop (0: dense); it reports no row maxima
        self.draft_topk = int(draft_topk)
        if self.draft_topk:
            self.dstats = None
            self.ws_topk = _lib.workspace(_lib.lib().dspark_markov_topk_workspace_bytes(
                w.B, w.K, w.V, w.R, self.draft_topk), device)

    def markov(self, stream=None):
        if self.draft_topk:
            _lib.markov_sample_topk(self.base, self.w1, self.w2, self.anchor, self.rsi, self.pos,
                                    self.temperature, self.seeds, self.draft, self.draft_topk,
                                    cache=self.cache, cache_row_map=self.row_map,
                                    workspace_buf=self.ws_topk, status=self.status,
                                    stream=stream)
            return
        _lib.markov_sample(self.base, self.w1, self.w2, self.anchor, self.rsi, self.pos,
                           self.temperature, self.seeds, self.draft, cache=self.cache,
                           cache_row_map=self.row_map, workspace_buf=self.ws_markov,
                           status=self.status, stream=stream, draft_stats=self.dstats)

    def verify(self, stream=None):
        _lib.rejection_sample(self.draft, self.cache, self.target, self.rsi, self.pos,
                              self.temperature, self.top_p, self.seeds, self.out,
                              self.num_accepted, cache_row_map=self.row_map,
                              workspace_buf=self.ws_verify, status=self.status,
                              stream=stream, draft_stats=self.dstats)

    def run(self, stream=None):
        self.markov(stream)
        self.verify(stream)

    def status_code(self) -> int:
        return int(self.status.item())


def main(argv=None):
    """Run decode steps of a named synthetic workload, e.g. under a profiler:
    python -m verify_dspark_markov_step_gb300.step --config minimax --batch 32 --steps 2"""
    import argparse

    from . import build, workloads

    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="minimax")
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--steps", type=int, default=2)
    args = ap.parse_args(argv)
    build.build()
    w = workloads.make(args.config, batch=args.batch)
    st = DecodeStep(w)
    for _ in range(args.steps):
        st.run()
    torch.cuda.synchronize()
    print(f"{args.config} B={w.B}: status {st.status_code()}, mean accepted "
          f"{st.num_accepted.float().mean().item():.3f}")


if __name__ == "__main__":
    main()
