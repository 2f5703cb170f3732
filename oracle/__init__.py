"""CPU oracle for the DSpark Markov drafting step and the rejection-sampling
verifier -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the CUDA library and
its Python binding) never imports, links or runs anything here, and this
package shares no code with it: the arithmetic lives in ``dspark_oracle.c``
(plain C11, fp64 for transcendentals and dot products, compiled with
``-ffp-contract=off``), and this module only marshals numpy arrays into it.
The same file is also built with ``-fopenmp``, which runs the independent
requests of a batch call on several host threads and changes nothing else.

What each function computes, and which passage of the pages it follows, is
documented beside the C function it calls.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
# The same source built with -fopenmp: the batch entry points then run their
# requests on several host threads (the CPU baseline's parallel leg).
_OMP_PATH = os.path.join(_HERE, "_build", "liboracle_omp.so")
_lock = threading.Lock()
_lib = None
_omp_lib = None

ORC_OK = 0
ORC_EINVAL = 1
ORC_EBOUNDS = 2
ORC_ENOMEM = 3

STREAM_DRAFT = 1 << 30
STREAM_TARGET = 0
STREAM_ACCEPT = 1 << 29


def _compile(path, extra, force):
    stale = (not os.path.exists(path)) or (os.path.getmtime(path) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = path + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-Wall", *extra, "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, path)


def build(force: bool = False) -> str:
    """Compile ``dspark_oracle.c`` into ``_build/liboracle.so`` with gcc, and
    the OpenMP build ``_build/liboracle_omp.so`` where gcc supports it."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    _compile(_LIB_PATH, [], force)
    try:
        _compile(_OMP_PATH, ["-fopenmp"], force)
    except (subprocess.CalledProcessError, OSError):
        pass  # no OpenMP: only the single-threaded oracle exists
    return _LIB_PATH


def _P(t):
    return ctypes.POINTER(t)


def _load(path):
    L = ctypes.CDLL(path)
    vp, i32, i64, f32, u64 = (ctypes.c_void_p, ctypes.c_int,
                              ctypes.c_int64, ctypes.c_float,
                              ctypes.c_uint64)
    L.orc_markov_sample.restype = i32
    L.orc_markov_sample.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp,
                                    vp, i32, vp, vp, vp, vp,
                                    i32, i32, i32, i32, i32, i32]
    L.orc_markov_sample_topk.restype = i32
    L.orc_markov_sample_topk.argtypes = L.orc_markov_sample.argtypes + [i32]
    L.orc_markov_step.restype = i32
    L.orc_markov_step.argtypes = [vp, i32, vp, vp, ctypes.c_int32, f32,
                                  u64, i64, i32, i32, vp, vp, vp]
    L.orc_rejection_sample.restype = i32
    L.orc_rejection_sample.argtypes = [vp, vp, i32, vp, vp, i32, vp, vp,
                                       vp, vp, vp, vp, vp, vp, vp, vp,
                                       i32, i32, i32, i32, i32]
    L.orc_philox_batch.restype = i32
    L.orc_philox_batch.argtypes = [i64, vp, vp, vp]
    L.orc_noise_batch.restype = i32
    L.orc_noise_batch.argtypes = [i64, vp, vp, vp, vp, vp, vp, vp]
    L.orc_block_argmax.restype = i32
    L.orc_block_argmax.argtypes = [vp, i64, vp, vp]
    L.orc_target_probs.restype = i32
    L.orc_target_probs.argtypes = [vp, i32, i32, f32, f32, vp, vp, vp,
                                   vp, vp]
    L.orc_draft_probs.restype = i32
    L.orc_draft_probs.argtypes = [vp, i32, i32, vp]
    L.orc_categorical.restype = i32
    L.orc_categorical.argtypes = [vp, i32, u64, i64, vp, vp]
    L.orc_threads.restype = i32
    L.orc_threads.argtypes = [i32]
    return L


def lib(threads: int = 1):
    """The single-threaded oracle library; with threads > 1 the OpenMP build
    set to that many host threads (RuntimeError if it could not be built)."""
    global _lib, _omp_lib
    with _lock:
        if threads <= 1:
            if _lib is None:
                build()
                _lib = _load(_LIB_PATH)
            return _lib
        if _omp_lib is None:
            build()
            if not os.path.exists(_OMP_PATH):
                raise RuntimeError("the OpenMP oracle could not be built (gcc -fopenmp)")
            _omp_lib = _load(_OMP_PATH)
        _omp_lib.orc_threads(int(threads))
        return _omp_lib


def threads_in_use(threads: int) -> int:
    """Host threads the oracle runs its requests on for a `threads` request."""
    return 1 if threads <= 1 else int(lib(threads).orc_threads(0))


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    """Contiguous array of the given dtype (no copy if it already is)."""
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != ORC_OK:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def _logit_array(a):
    """fp32 array -> (array, 0); uint16 (bf16 bit patterns) -> (array, 1)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, 0
    if a.dtype == np.uint16:
        return a, 1
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {a.dtype}")


# --------------------------------------------------------------------------
# Noise
# --------------------------------------------------------------------------
def philox4x32_10(key, ctr):
    """Philox4x32-10 on arrays: key [n,2] uint32, ctr [n,4] uint32 -> [n,4]."""
    key = _c(key, np.uint32).reshape(-1, 2)
    ctr = _c(ctr, np.uint32).reshape(-1, 4)
    assert key.shape[0] == ctr.shape[0]
    out = np.empty_like(ctr)
    _check(lib().orc_philox_batch(key.shape[0], _ptr(key), _ptr(ctr), _ptr(out)),
           "philox")
    return out


def noise(seed, pos, col, stream):
    """(word, u, g) for arrays of (seed, position, column, stream)."""
    seed, pos, col, stream = np.broadcast_arrays(
        np.asarray(seed, dtype=np.uint64), np.asarray(pos, dtype=np.int64),
        np.asarray(col, dtype=np.uint32), np.asarray(stream, dtype=np.uint32))
    shape = seed.shape
    seed, pos, col, stream = (_c(x.ravel(), x.dtype) for x in (seed, pos, col, stream))
    n = seed.size
    word = np.empty(n, np.uint32)
    u = np.empty(n, np.float32)
    g = np.empty(n, np.float32)
    _check(lib().orc_noise_batch(n, _ptr(seed), _ptr(pos), _ptr(col), _ptr(stream),
                                 _ptr(word), _ptr(u), _ptr(g)), "noise")
    return word.reshape(shape), u.reshape(shape), g.reshape(shape)


def block_argmax(y):
    """The drafter's winner rule on a 1-D fp32 array -> (index, top-two gap)."""
    y = _c(y, np.float32)
    idx = np.zeros(1, np.int64)
    gap = np.zeros(1, np.float64)
    _check(lib().orc_block_argmax(_ptr(y), y.size, _ptr(idx), _ptr(gap)), "argmax")
    return int(idx[0]), float(gap[0])


# --------------------------------------------------------------------------
# Markov drafting loop
# --------------------------------------------------------------------------
def markov_sample(base, w1, w2, anchor, req_state_idx, positions, temperature,
                  seeds, cache_rows=None, cache_bf16=False, row_map=None,
                  forced=None, write_cache=True, topk=0, threads=1):
    """Run the K-step Markov loop. Returns (tokens [B,K] int32, cache or None,
    gaps [B,K] float64). ``cache_rows`` is C (default S). ``topk`` > 0 runs the
    top-k variant (the bias only on the top-k base logits of each step).
    ``threads`` > 1 runs the requests on that many host threads (OpenMP)."""
    base, base_bf16 = _logit_array(base)
    B, K, V = base.shape
    w1 = _c(w1, np.uint16)
    w2 = _c(w2, np.uint16)
    R = w2.shape[1]
    anchor = _c(anchor, np.int32)
    rsi = _c(req_state_idx, np.int32)
    pos = _c(positions, np.int64)
    temp = _c(temperature, np.float32)
    seeds = _c(seeds, np.uint64)
    S = temp.shape[0]
    C = S if cache_rows is None else int(cache_rows)
    row_map = _c(row_map, np.int32)
    forced = _c(forced, np.int32)
    cache = None
    if write_cache:
        cache = np.zeros((C, K, V), np.uint16 if cache_bf16 else np.float32)
    tokens = np.empty((B, K), np.int32)
    gaps = np.empty((B, K), np.float64)
    args = (_ptr(base), base_bf16, _ptr(w1), _ptr(w2), _ptr(anchor), _ptr(rsi),
            _ptr(pos), _ptr(temp), _ptr(seeds), _ptr(cache), int(bool(cache_bf16)),
            _ptr(row_map), _ptr(forced), _ptr(tokens), _ptr(gaps), B, K, V, R, S, C)
    L = lib(threads)
    if topk:
        rc = L.orc_markov_sample_topk(*args, int(topk))
    else:
        rc = L.orc_markov_sample(*args)
    _check(rc, "markov_sample")
    return tokens, cache, gaps


def markov_step(base_row, w1, w2, prev, temperature, seed, noise_pos):
    """One Markov step of one request. Returns (token, gap, x [V] fp32)."""
    base_row, bf = _logit_array(base_row)
    V = base_row.shape[-1]
    w1 = _c(w1, np.uint16)
    w2 = _c(w2, np.uint16)
    R = w2.shape[1]
    x = np.empty(V, np.float32)
    tok = np.zeros(1, np.int32)
    gap = np.zeros(1, np.float64)
    rc = lib().orc_markov_step(_ptr(base_row), bf, _ptr(w1), _ptr(w2), int(prev),
                               float(temperature), int(seed) & (2**64 - 1),
                               int(noise_pos), V, R, _ptr(x), _ptr(tok), _ptr(gap))
    _check(rc, "markov_step")
    return int(tok[0]), float(gap[0]), x


# --------------------------------------------------------------------------
# Verifier
# --------------------------------------------------------------------------
def rejection_sample(draft_tokens, cache, target, req_state_idx, positions,
                     temperature, top_p, seeds, row_map=None, threads=1):
    """Run the verifier. Returns a dict with out_tokens [B,K+1],
    num_accepted [B], margins [B,K], gaps [B], slack [B,K+1]. ``threads`` > 1
    runs the requests on that many host threads (OpenMP)."""
    draft = _c(draft_tokens, np.int32)
    B, K = draft.shape
    target, t_bf16 = _logit_array(target)
    V = target.shape[-1]
    assert target.shape == (B, K + 1, V)
    if cache is None:
        cache_arr, c_bf16, C = None, 0, 1
    else:
        cache_arr, c_bf16 = _logit_array(cache)
        C = cache_arr.shape[0]
    rsi = _c(req_state_idx, np.int32)
    pos = _c(positions, np.int64)
    temp = _c(temperature, np.float32)
    tp = _c(top_p, np.float32)
    seeds = _c(seeds, np.uint64)
    S = temp.shape[0]
    row_map = _c(row_map, np.int32)
    out = np.empty((B, K + 1), np.int32)
    nacc = np.empty(B, np.int32)
    margins = np.empty((B, K), np.float64)
    gaps = np.empty(B, np.float64)
    slack = np.empty((B, K + 1), np.float64)
    rc = lib(threads).orc_rejection_sample(
        _ptr(draft), _ptr(cache_arr), c_bf16, _ptr(row_map), _ptr(target), t_bf16,
        _ptr(rsi), _ptr(pos), _ptr(temp), _ptr(tp), _ptr(seeds), _ptr(out),
        _ptr(nacc), _ptr(margins), _ptr(gaps), _ptr(slack), B, K, V, S, C)
    _check(rc, "rejection_sample")
    return dict(out_tokens=out, num_accepted=nacc, margins=margins, gaps=gaps,
                slack=slack)


def target_probs(row, temperature, top_p):
    """Target distribution of one row -> (p, keep, F, Fk, boundary_slack)."""
    row, bf = _logit_array(row)
    V = row.shape[-1]
    p = np.empty(V, np.float32)
    keep = np.empty(V, np.uint8)
    F = np.zeros(1, np.uint64)
    Fk = np.zeros(1, np.uint64)
    sl = np.zeros(1, np.float64)
    rc = lib().orc_target_probs(_ptr(row), bf, V, float(temperature), float(top_p),
                                _ptr(p), _ptr(keep), _ptr(F), _ptr(Fk), _ptr(sl))
    _check(rc, "target_probs")
    return p, keep.astype(bool), int(F[0]), int(Fk[0]), float(sl[0])


def draft_probs(row):
    """Draft distribution q of one cached row."""
    row, bf = _logit_array(row)
    V = row.shape[-1]
    q = np.empty(V, np.float32)
    _check(lib().orc_draft_probs(_ptr(row), bf, V, _ptr(q)), "draft_probs")
    return q


def categorical(weights, seed, noise_pos):
    """Gumbel-max draw from non-negative fp32 weights -> (index, gap)."""
    w = _c(weights, np.float32)
    idx = np.zeros(1, np.int64)
    gap = np.zeros(1, np.float64)
    _check(lib().orc_categorical(_ptr(w), w.size, int(seed) & (2**64 - 1),
                                 int(noise_pos), _ptr(idx), _ptr(gap)), "categorical")
    return int(idx[0]), float(gap[0])
