"""Seeded synthetic inputs for the Markov drafting step and the verifier.

This module only draws random data; it holds none of the method's arithmetic
(no noise generator, no bias, no softmax). Both the CUDA path's tests and the
CPU oracle read the same arrays from here. All arrays are numpy on the host:
fp32 logits as ``float32``, bf16 tensors as ``uint16`` bit patterns.

Five workloads, shaped like the ones on the pages (vocabularies 200064,
151936 and an odd 50017; K = 3, 5 or 7 draft steps; batches of 1 to 256;
markov_rank 256 with bf16 weights; prompts of about 22k tokens, which enter
only through the positions):

=========  ====  =  ======  ===  ==========================================
name       B     K  V       R    values
=========  ====  =  ======  ===  ==========================================
tiny       1     3  4096    64   base, target fp32 N(0,2^2); w N(0,0.02^2);
                                 T = 1; top_p = 1; seed 0
odd        8     5  50017   128  logits fp32 N(0,3^2), one NaN column in 1%
                                 of the rows (at least one base and one
                                 target row); T ~ U[0.5,1.5]; top_p = 0.9
minimax    1/4/32 7 200064  256  base fp32 N(0,2^2) plus 5 spiked columns per
                                 row at +8; fp32 cache; T = 1; top_p = 1
qwen       256   3  151936  256  base, target, cache bf16; base N(0,2^2),
                                 target = base + N(0,0.5^2); T = 1;
                                 top_p = 0.95; per-request seeds
long       128   7  200064  256  fp32; 256 request slots, req_state_idx the
                                 first 128 of a permutation of 0..255;
                                 identity row map; 25% greedy slots, others
                                 T ~ U[0.7,1.3]; top_p ~ U[0.8,1.0], 10% = 1
=========  ====  =  ======  ===  ==========================================

The target logits of the fp32 workloads are base + N(0, 0.5^2) (the workload
list gives no target distribution for them; this keeps the acceptance rate in
the pages' 0.6-0.8 range). Positions are P0[b] = 22000 + 37 b. Sampling seeds
are seeds[s] = 0x9E3779B97F4A7C15 * (s + 1) xor config_id (mod 2^64).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

CONFIG_IDS = {"tiny": 1, "odd": 2, "minimax": 3, "qwen": 4, "long": 5, "custom": 9}


@dataclass
class Workload:
    name: str
    B: int
    K: int
    V: int
    R: int
    S: int
    C: int
    base: np.ndarray            # [B,K,V] float32 or uint16 (bf16 bits)
    w1: np.ndarray              # [V,R] uint16 (bf16 bits): markov embedding
    w2: np.ndarray              # [V,R] uint16 (bf16 bits): markov_w2 projection
    anchor: np.ndarray          # [B] int32
    req_state_idx: np.ndarray   # [B] int32, -1 = padding request
    positions: np.ndarray       # [B] int64
    temperature: np.ndarray     # [S] float32, 0 = greedy
    top_p: np.ndarray           # [S] float32
    seeds: np.ndarray           # [S] uint64
    row_map: np.ndarray | None  # [S] int32 or None (identity)
    target: np.ndarray | None   # [B,K+1,V] float32 or uint16
    cache_bf16: bool = False
    extra: dict = field(default_factory=dict)

    @property
    def base_bf16(self) -> bool:
        return self.base.dtype == np.uint16

    @property
    def target_bf16(self) -> bool:
        return self.target is not None and self.target.dtype == np.uint16


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 data to bf16 bit patterns (nearest even) for synthetic inputs."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    out = ((bits + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = ((a.view(np.uint32)[nan] >> 16) | 0x40).astype(np.uint16)
    return out


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(config_id: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([1000 + config_id, stream])


def _normal_f32(rng, shape, std) -> np.ndarray:
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def default_seeds(S: int, config_id: int) -> np.ndarray:
    s = np.arange(1, S + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return (np.uint64(0x9E3779B97F4A7C15) * s) ^ np.uint64(config_id)


def default_positions(B: int) -> np.ndarray:
    return (22000 + 37 * np.arange(B, dtype=np.int64)).astype(np.int64)


def _spike(rng, base: np.ndarray, n_spikes: int, height: float) -> None:
    """Add `height` to n_spikes distinct random columns of every row."""
    B, K, V = base.shape
    for b in range(B):
        for k in range(K):
            cols = rng.choice(V, size=n_spikes, replace=False)
            base[b, k, cols] += np.float32(height)


def _plant_nans(rng, arr: np.ndarray, frac: float) -> list:
    """Give each row one NaN column with probability frac (at least one row)."""
    B, K, V = arr.shape
    rows = [(b, k) for b in range(B) for k in range(K) if rng.random() < frac]
    if not rows:
        rows = [(int(rng.integers(B)), int(rng.integers(K)))]
    for b, k in rows:
        arr[b, k, int(rng.integers(V))] = np.float32(np.nan)
    return rows


def make(name: str, batch: int | None = None, with_target: bool = True) -> Workload:
    """Build one of the named workloads (``batch`` selects 1/4/32 for minimax)."""
    cid = CONFIG_IDS[name]
    if name == "tiny":
        B, K, V, R = 1, 3, 4096, 64
        S = C = 1
        base = _normal_f32(_rng(cid, 1), (B, K, V), 2.0)
        target = _normal_f32(_rng(cid, 2), (B, K + 1, V), 2.0) if with_target else None
        temperature = np.ones(S, np.float32)
        top_p = np.ones(S, np.float32)
        seeds = np.zeros(S, np.uint64)
        rsi = np.arange(B, dtype=np.int32)
        row_map = None
        cache_bf16 = False
    elif name == "odd":
        B, K, V, R = 8, 5, 50017, 128
        S = C = B
        base = _normal_f32(_rng(cid, 1), (B, K, V), 3.0)
        nan_rows = _plant_nans(_rng(cid, 11), base, 0.01)
        target = None
        if with_target:
            target = _normal_f32(_rng(cid, 2), (B, K + 1, V), 3.0)
            _plant_nans(_rng(cid, 12), target, 0.01)
        temperature = _rng(cid, 3).uniform(0.5, 1.5, S).astype(np.float32)
        top_p = np.full(S, 0.9, np.float32)
        seeds = default_seeds(S, cid)
        rsi = np.arange(B, dtype=np.int32)
        row_map = None
        cache_bf16 = False
    elif name == "minimax":
        B = 32 if batch is None else int(batch)
        K, V, R = 7, 200064, 256
        S = C = B
        base = _normal_f32(_rng(cid, 1), (B, K, V), 2.0)
        _spike(_rng(cid, 4), base, 5, 8.0)
        target = None
        if with_target:
            noise = _normal_f32(_rng(cid, 2), (B, K + 1, V), 0.5)
            target = noise
            target[:, :K] += base
            target[:, K] += base[:, K - 1]
        temperature = np.ones(S, np.float32)
        top_p = np.ones(S, np.float32)
        seeds = default_seeds(S, cid)
        rsi = np.arange(B, dtype=np.int32)
        row_map = None
        cache_bf16 = False
    elif name == "qwen":
        B = 256 if batch is None else int(batch)
        K, V, R = 3, 151936, 256
        S = C = B
        base32 = _normal_f32(_rng(cid, 1), (B, K, V), 2.0)
        target = None
        if with_target:
            t32 = _normal_f32(_rng(cid, 2), (B, K + 1, V), 0.5)
            t32[:, :K] += base32
            t32[:, K] += base32[:, K - 1]
            target = f32_to_bf16_bits(t32)
            del t32
        base = f32_to_bf16_bits(base32)
        del base32
        temperature = np.ones(S, np.float32)
        top_p = np.full(S, 0.95, np.float32)
        seeds = default_seeds(S, cid)
        rsi = np.arange(B, dtype=np.int32)
        row_map = None
        cache_bf16 = True
    elif name == "long":
        B = 128 if batch is None else int(batch)
        K, V, R = 7, 200064, 256
        S = C = 256
        base = _normal_f32(_rng(cid, 1), (B, K, V), 2.0)
        _spike(_rng(cid, 4), base, 5, 8.0)
        target = None
        if with_target:
            noise = _normal_f32(_rng(cid, 2), (B, K + 1, V), 0.5)
            target = noise
            target[:, :K] += base
            target[:, K] += base[:, K - 1]
        r = _rng(cid, 3)
        rsi = r.permutation(S)[:B].astype(np.int32)
        temperature = r.uniform(0.7, 1.3, S).astype(np.float32)
        greedy = r.permutation(S)[: S // 4]
        temperature[greedy] = 0.0
        top_p = r.uniform(0.8, 1.0, S).astype(np.float32)
        top_p[r.permutation(S)[: S // 10]] = 1.0
        seeds = default_seeds(S, cid)
        row_map = np.arange(S, dtype=np.int32)
        cache_bf16 = False
    else:
        raise KeyError(name)
    rw = _rng(cid, 5)
    w1 = f32_to_bf16_bits(_normal_f32(rw, (V, R), 0.02))
    w2 = f32_to_bf16_bits(_normal_f32(rw, (V, R), 0.02))
    anchor = _rng(cid, 6).integers(0, V, B).astype(np.int32)
    return Workload(name=name, B=B, K=K, V=V, R=R, S=S, C=C, base=base, w1=w1, w2=w2,
                    anchor=anchor, req_state_idx=rsi.astype(np.int32),
                    positions=default_positions(B), temperature=temperature,
                    top_p=top_p, seeds=seeds, row_map=row_map, target=target,
                    cache_bf16=cache_bf16)


def custom(B, K, V, R, *, seed=0, base_std=2.0, w_std=0.02, base_bf16=False,
           cache_bf16=False, target_bf16=False, S=None, temperature=None,
           top_p=None, rsi=None, row_map=None, C=None, target_noise=0.5,
           spikes=0) -> Workload:
    """A free-form workload for edge cases (ragged sizes, padding, mixed rows)."""
    r = np.random.default_rng([2000, seed, B, K, V, R])
    S = B if S is None else S
    base32 = _normal_f32(r, (B, K, V), base_std)
    if spikes:
        _spike(r, base32, spikes, 8.0)
    t32 = _normal_f32(r, (B, K + 1, V), target_noise)
    t32[:, :K] += base32
    t32[:, K] += base32[:, K - 1]
    w1 = f32_to_bf16_bits(_normal_f32(r, (V, R), w_std))
    w2 = f32_to_bf16_bits(_normal_f32(r, (V, R), w_std))
    temp = (np.ones(S, np.float32) if temperature is None
            else np.broadcast_to(np.asarray(temperature, np.float32), (S,)).copy())
    tp = (np.ones(S, np.float32) if top_p is None
          else np.broadcast_to(np.asarray(top_p, np.float32), (S,)).copy())
    rsi_a = np.arange(B, dtype=np.int32) if rsi is None else np.asarray(rsi, np.int32)
    return Workload(
        name="custom", B=B, K=K, V=V, R=R, S=S, C=S if C is None else C,
        base=f32_to_bf16_bits(base32) if base_bf16 else base32,
        w1=w1, w2=w2, anchor=r.integers(0, V, B).astype(np.int32),
        req_state_idx=rsi_a, positions=default_positions(B), temperature=temp,
        top_p=tp, seeds=default_seeds(S, CONFIG_IDS["custom"] + seed),
        row_map=None if row_map is None else np.asarray(row_map, np.int32),
        target=f32_to_bf16_bits(t32) if target_bf16 else t32, cache_bf16=cache_bf16)


def random_drafts(w: Workload, seed: int = 0, p_minus1: float = 0.0) -> np.ndarray:
    """Draft tokens for verifier-only tests: uniform random ids, with -1
    placeholders from a random step on (probability p_minus1 per request)."""
    r = np.random.default_rng([3000, seed, w.B, w.K, w.V])
    d = r.integers(0, w.V, (w.B, w.K)).astype(np.int32)
    for b in range(w.B):
        if r.random() < p_minus1:
            d[b, int(r.integers(w.K)):] = -1
    return d
