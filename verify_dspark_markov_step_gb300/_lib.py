"""Thin ctypes binding of the C ABI in ``include/dspark.h``.

Argument marshalling only: every step of the computation runs in the CUDA
library ``_build/libdspark.so``. PyTorch provides device memory and the
current stream. There is no CPU fallback: if the library cannot be loaded,
every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libdspark.so")

DSPARK_F32 = 0
DSPARK_BF16 = 1

STATUS = {
    0: "DSPARK_OK",
    -1: "DSPARK_ERR_INVALID_ARG",
    -2: "DSPARK_ERR_UNSUPPORTED",
    -3: "DSPARK_ERR_CUDA",
    -4: "DSPARK_ERR_TIMEOUT",
    -5: "DSPARK_ERR_BOUNDS",
    -6: "DSPARK_ERR_WORKSPACE",
    -7: "DSPARK_ERR_ALIGNMENT",
    -8: "DSPARK_ERR_SCRATCH_LIMIT",
}

# Every symbol include/dspark.h and include/dspark_testing.h declare.
EXPORTS = (
    "dspark_testing_markov_wait_limit",
    "dspark_testing_temperature_divide",
    "dspark_markov_workspace_bytes",
    "dspark_markov_sample",
    "dspark_markov_sample_static",
    "dspark_markov_topk_workspace_bytes",
    "dspark_markov_sample_topk",
    "dspark_verify_workspace_bytes",
    "dspark_rejection_sample",
    "dspark_noise",
    "dspark_status_string",
    "dspark_version",
)


class DsparkError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)}")


_lock = threading.Lock()
_lib = None


def lib(path: str | None = None) -> ctypes.CDLL:
    """Load libdspark.so (built by ``verify_dspark_markov_step_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"CUDA library not built: {p} is missing. Run "
                "`python -m verify_dspark_markov_step_gb300.build` (needs nvcc).")
        L = ctypes.CDLL(p)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        L.dspark_markov_workspace_bytes.restype = sz
        L.dspark_markov_workspace_bytes.argtypes = [i32, i32, i32, i32]
        L.dspark_markov_sample.restype = i32
        L.dspark_markov_sample.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp,
                                           vp, i32, i32, i32, i32, i32, i32, vp, sz, vp, vp]
        L.dspark_testing_markov_wait_limit.restype = i32
        L.dspark_testing_markov_wait_limit.argtypes = [
            vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32,
            vp, sz, vp, vp, ctypes.c_uint64, ctypes.c_uint32]
        L.dspark_testing_temperature_divide.restype = i32
        L.dspark_testing_temperature_divide.argtypes = [vp, vp, vp, i64, vp]
        L.dspark_markov_sample_static.restype = i32
        L.dspark_markov_sample_static.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                                  vp, vp, vp, i32, i32, i32, i32, i32, i32, vp,
                                                  vp]
        L.dspark_markov_topk_workspace_bytes.restype = sz
        L.dspark_markov_topk_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
        L.dspark_markov_sample_topk.restype = i32
        L.dspark_markov_sample_topk.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp,
                                                vp, i32, i32, i32, i32, i32, i32, i32, vp, sz,
                                                vp, vp]
        L.dspark_verify_workspace_bytes.restype = sz
        L.dspark_verify_workspace_bytes.argtypes = [i32, i32, i32]
        L.dspark_rejection_sample.restype = i32
        L.dspark_rejection_sample.argtypes = [vp, vp, i32, vp, vp, vp, i32, vp, vp, vp, vp, vp,
                                              vp, vp, i32, i32, i32, i32, i32, vp, sz, vp, vp]
        L.dspark_noise.restype = i32
        L.dspark_noise.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, vp]
        L.dspark_status_string.restype = ctypes.c_char_p
        L.dspark_status_string.argtypes = [i32]
        L.dspark_version.restype = i32
        L.dspark_version.argtypes = []
        if path is None:
            _lib = L
        return L


def status_string(code: int) -> str:
    return lib().dspark_status_string(int(code)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t, name, dtypes=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    return t


_BF16_LIKE = (torch.bfloat16, torch.int16)


def _logit_dtype(t, name):
    if t.dtype == torch.float32:
        return DSPARK_F32
    if t.dtype in _BF16_LIKE:
        return DSPARK_BF16
    raise TypeError(f"{name} must be float32 or bfloat16, got {t.dtype}")


def _check(code, what):
    if code != 0:
        raise DsparkError(code, what)


def markov_workspace_bytes(B, K, V, R) -> int:
    return int(lib().dspark_markov_workspace_bytes(B, K, V, R))


def verify_workspace_bytes(B, K, V) -> int:
    return int(lib().dspark_verify_workspace_bytes(B, K, V))


ROW_STATS_BYTES = 16  # sizeof(dspark_row_stats)


def row_stats(B: int, K: int, device=None) -> torch.Tensor:
    """A device buffer for [B, K] dspark_row_stats (16 bytes each: the row
    maximum as fp32 in the low word, a scratch word, the fixed-point mass)."""
    return torch.zeros((B, K, 2), dtype=torch.int64, device=device or "cuda")


def row_stats_fields(t: torch.Tensor):
    """(m [B,K] fp32, mass [B,K] int64) of a row_stats buffer, on the host."""
    a = t.cpu()
    m = a[..., 0].to(torch.int64).bitwise_and(0xFFFFFFFF).to(torch.int32).view(torch.float32)
    return m, a[..., 1]


def _stats(t, B, K, name="draft_stats"):
    if t is None:
        return None
    _dev(t, name)
    if t.numel() * t.element_size() != B * K * ROW_STATS_BYTES:
        raise ValueError(f"{name} must hold [B, K] {ROW_STATS_BYTES}-byte records")
    return t


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A device byte buffer usable as a workspace."""
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device or "cuda")


def markov_sample(base_logits, markov_w1, markov_w2, anchor_tokens, req_state_idx,
                  positions, temperature, seeds, out_tokens, cache=None,
                  cache_row_map=None, workspace_buf=None, status=None, stream=None,
                  draft_stats=None):
    """dspark_markov_sample on torch tensors (see include/dspark.h)."""
    _dev(base_logits, "base_logits", (torch.float32,) + _BF16_LIKE)
    B, K, V = base_logits.shape
    _dev(markov_w1, "markov_w1", _BF16_LIKE)
    _dev(markov_w2, "markov_w2", _BF16_LIKE)
    R = markov_w2.shape[1]
    if markov_w2.shape != (V, R) or markov_w1.shape[1] != R or markov_w1.shape[0] < V:
        raise ValueError("markov_w1 / markov_w2 must be [V, R]")
    _dev(anchor_tokens, "anchor_tokens", (torch.int32,))
    _dev(req_state_idx, "req_state_idx", (torch.int32,))
    _dev(positions, "positions", (torch.int64,))
    _dev(temperature, "temperature", (torch.float32,))
    _dev(seeds, "seeds", (torch.int64, torch.uint64) if hasattr(torch, "uint64") else (torch.int64,))
    _dev(out_tokens, "out_tokens", (torch.int32,))
    S = temperature.shape[0]
    if seeds.shape[0] != S or anchor_tokens.shape[0] != B or req_state_idx.shape[0] != B \
            or positions.shape[0] != B or tuple(out_tokens.shape) != (B, K):
        raise ValueError("inconsistent shapes")
    C = 0
    cache_dt = DSPARK_F32
    if cache is not None:
        _dev(cache, "cache", (torch.float32,) + _BF16_LIKE)
        if cache.dim() != 3 or cache.shape[1] != K or cache.shape[2] != V:
            raise ValueError("cache must be [C, K, V]")
        C = cache.shape[0]
        cache_dt = _logit_dtype(cache, "cache")
    _dev(cache_row_map, "cache_row_map", (torch.int32,))
    need = markov_workspace_bytes(B, K, V, R)
    if workspace_buf is None:
        workspace_buf = workspace(need, base_logits.device)
    _dev(status, "status", (torch.int32,))
    _stats(draft_stats, B, K)
    code = lib().dspark_markov_sample(
        _ptr(base_logits), _logit_dtype(base_logits, "base_logits"), _ptr(markov_w1),
        _ptr(markov_w2), _ptr(anchor_tokens), _ptr(req_state_idx), _ptr(positions),
        _ptr(temperature), _ptr(seeds), _ptr(cache), cache_dt, _ptr(cache_row_map),
        _ptr(out_tokens), _ptr(draft_stats), B, K, V, R, S, max(C, 1), _ptr(workspace_buf),
        workspace_buf.numel() * workspace_buf.element_size(), _ptr(status), _stream(stream))
    _check(code, "dspark_markov_sample")


def markov_sample_wait_limit(base_logits, markov_w1, markov_w2, anchor_tokens, req_state_idx,
                             positions, temperature, seeds, out_tokens, wait_limit_ns,
                             barrier_extra, cache=None, cache_row_map=None, workspace_buf=None,
                             status=None, stream=None):
    """dspark_testing_markov_wait_limit (include/dspark_testing.h): the Markov
    loop with its bounded waits shortened to wait_limit_ns and the grid
    barrier waiting for barrier_extra arrivals more than the grid makes, so
    that a test can make the waits run out."""
    B, K, V = base_logits.shape
    R = markov_w2.shape[1]
    S = temperature.shape[0]
    for t, n in ((base_logits, "base_logits"), (markov_w1, "markov_w1"),
                 (markov_w2, "markov_w2"), (anchor_tokens, "anchor_tokens"),
                 (req_state_idx, "req_state_idx"), (positions, "positions"),
                 (temperature, "temperature"), (seeds, "seeds"), (out_tokens, "out_tokens")):
        _dev(t, n)
    C, cache_dt = 0, DSPARK_F32
    if cache is not None:
        _dev(cache, "cache", (torch.float32,) + _BF16_LIKE)
        C, cache_dt = cache.shape[0], _logit_dtype(cache, "cache")
    if workspace_buf is None:
        workspace_buf = workspace(markov_workspace_bytes(B, K, V, R), base_logits.device)
    _dev(status, "status", (torch.int32,))
    code = lib().dspark_testing_markov_wait_limit(
        _ptr(base_logits), _logit_dtype(base_logits, "base_logits"), _ptr(markov_w1),
        _ptr(markov_w2), _ptr(anchor_tokens), _ptr(req_state_idx), _ptr(positions),
        _ptr(temperature), _ptr(seeds), _ptr(cache), cache_dt, _ptr(cache_row_map),
        _ptr(out_tokens), B, K, V, R, S, max(C, 1), _ptr(workspace_buf),
        workspace_buf.numel() * workspace_buf.element_size(), _ptr(status), _stream(stream),
        int(wait_limit_ns), int(barrier_extra))
    _check(code, "dspark_testing_markov_wait_limit")


# Bytes of the library's fixed scratch array (DSPARK_STATIC_SCRATCH_BYTES).
STATIC_SCRATCH_BYTES = 32 << 10


def markov_sample_static(base_logits, markov_w1, markov_w2, anchor_tokens, req_state_idx,
                         positions, temperature, seeds, out_tokens, cache=None,
                         cache_row_map=None, status=None, stream=None, draft_stats=None):
    """dspark_markov_sample_static on torch tensors: dspark_markov_sample with
    the library's fixed scratch array instead of a workspace, so that nothing
    is allocated (for callers that may not allocate device memory). Calls
    that overlap on the GPU race on that array (see include/dspark.h)."""
    _dev(base_logits, "base_logits", (torch.float32,) + _BF16_LIKE)
    B, K, V = base_logits.shape
    _dev(markov_w1, "markov_w1", _BF16_LIKE)
    _dev(markov_w2, "markov_w2", _BF16_LIKE)
    R = markov_w2.shape[1]
    if markov_w2.shape != (V, R) or markov_w1.shape[1] != R or markov_w1.shape[0] < V:
        raise ValueError("markov_w1 / markov_w2 must be [V, R]")
    for t, n, d in ((anchor_tokens, "anchor_tokens", torch.int32),
                    (req_state_idx, "req_state_idx", torch.int32),
                    (positions, "positions", torch.int64),
                    (temperature, "temperature", torch.float32),
                    (out_tokens, "out_tokens", torch.int32)):
        _dev(t, n, (d,))
    _dev(seeds, "seeds")
    S = temperature.shape[0]
    if seeds.shape[0] != S or anchor_tokens.shape[0] != B or req_state_idx.shape[0] != B \
            or positions.shape[0] != B or tuple(out_tokens.shape) != (B, K):
        raise ValueError("inconsistent shapes")
    C = 0
    cache_dt = DSPARK_F32
    if cache is not None:
        _dev(cache, "cache", (torch.float32,) + _BF16_LIKE)
        if cache.dim() != 3 or cache.shape[1] != K or cache.shape[2] != V:
            raise ValueError("cache must be [C, K, V]")
        C = cache.shape[0]
        cache_dt = _logit_dtype(cache, "cache")
    _dev(cache_row_map, "cache_row_map", (torch.int32,))
    _dev(status, "status", (torch.int32,))
    _stats(draft_stats, B, K)
    code = lib().dspark_markov_sample_static(
        _ptr(base_logits), _logit_dtype(base_logits, "base_logits"), _ptr(markov_w1),
        _ptr(markov_w2), _ptr(anchor_tokens), _ptr(req_state_idx), _ptr(positions),
        _ptr(temperature), _ptr(seeds), _ptr(cache), cache_dt, _ptr(cache_row_map),
        _ptr(out_tokens), _ptr(draft_stats), B, K, V, R, S, max(C, 1), _ptr(status),
        _stream(stream))
    _check(code, "dspark_markov_sample_static")


def markov_sample_topk(base_logits, markov_w1, markov_w2, anchor_tokens, req_state_idx,
                       positions, temperature, seeds, out_tokens, topk, cache=None,
                       cache_row_map=None, workspace_buf=None, status=None, stream=None):
    """dspark_markov_sample_topk on torch tensors: the Markov bias only on the
    top-k base logits of each request and step (see include/dspark.h)."""
    _dev(base_logits, "base_logits", (torch.float32,) + _BF16_LIKE)
    B, K, V = base_logits.shape
    _dev(markov_w1, "markov_w1", _BF16_LIKE)
    _dev(markov_w2, "markov_w2", _BF16_LIKE)
    R = markov_w2.shape[1]
    if markov_w2.shape != (V, R) or markov_w1.shape[1] != R or markov_w1.shape[0] < V:
        raise ValueError("markov_w1 / markov_w2 must be [V, R]")
    for t, n, d in ((anchor_tokens, "anchor_tokens", torch.int32),
                    (req_state_idx, "req_state_idx", torch.int32),
                    (positions, "positions", torch.int64),
                    (temperature, "temperature", torch.float32),
                    (out_tokens, "out_tokens", torch.int32)):
        _dev(t, n, (d,))
    _dev(seeds, "seeds")
    S = temperature.shape[0]
    if seeds.shape[0] != S or anchor_tokens.shape[0] != B or req_state_idx.shape[0] != B \
            or positions.shape[0] != B or tuple(out_tokens.shape) != (B, K):
        raise ValueError("inconsistent shapes")
    C = 0
    cache_dt = DSPARK_F32
    if cache is not None:
        _dev(cache, "cache", (torch.float32,) + _BF16_LIKE)
        if cache.dim() != 3 or cache.shape[1] != K or cache.shape[2] != V:
            raise ValueError("cache must be [C, K, V]")
        C = cache.shape[0]
        cache_dt = _logit_dtype(cache, "cache")
    _dev(cache_row_map, "cache_row_map", (torch.int32,))
    need = int(lib().dspark_markov_topk_workspace_bytes(B, K, V, R, int(topk)))
    if workspace_buf is None:
        workspace_buf = workspace(need, base_logits.device)
    _dev(status, "status", (torch.int32,))
    code = lib().dspark_markov_sample_topk(
        _ptr(base_logits), _logit_dtype(base_logits, "base_logits"), _ptr(markov_w1),
        _ptr(markov_w2), _ptr(anchor_tokens), _ptr(req_state_idx), _ptr(positions),
        _ptr(temperature), _ptr(seeds), _ptr(cache), cache_dt, _ptr(cache_row_map),
        _ptr(out_tokens), int(topk), B, K, V, R, S, max(C, 1), _ptr(workspace_buf),
        workspace_buf.numel() * workspace_buf.element_size(), _ptr(status), _stream(stream))
    _check(code, "dspark_markov_sample_topk")


def rejection_sample(draft_tokens, draft_cache, target_logits, req_state_idx, positions,
                     temperature, top_p, seeds, out_tokens, num_accepted,
                     cache_row_map=None, workspace_buf=None, status=None, stream=None,
                     draft_stats=None):
    """dspark_rejection_sample on torch tensors (see include/dspark.h)."""
    _dev(draft_tokens, "draft_tokens", (torch.int32,))
    B, K = draft_tokens.shape
    _dev(target_logits, "target_logits", (torch.float32,) + _BF16_LIKE)
    if target_logits.dim() != 3 or target_logits.shape[0] != B or target_logits.shape[1] != K + 1:
        raise ValueError("target_logits must be [B, K+1, V]")
    V = target_logits.shape[2]
    C = 0
    cache_dt = DSPARK_F32
    if draft_cache is not None:
        _dev(draft_cache, "draft_cache", (torch.float32,) + _BF16_LIKE)
        if draft_cache.dim() != 3 or draft_cache.shape[1] != K or draft_cache.shape[2] != V:
            raise ValueError("draft_cache must be [C, K, V]")
        C = draft_cache.shape[0]
        cache_dt = _logit_dtype(draft_cache, "draft_cache")
    for t, n, d in ((req_state_idx, "req_state_idx", torch.int32),
                    (positions, "positions", torch.int64),
                    (temperature, "temperature", torch.float32),
                    (top_p, "top_p", torch.float32),
                    (out_tokens, "out_tokens", torch.int32),
                    (num_accepted, "num_accepted", torch.int32)):
        _dev(t, n, (d,))
    _dev(seeds, "seeds")
    S = temperature.shape[0]
    if tuple(out_tokens.shape) != (B, K + 1) or num_accepted.shape[0] != B \
            or top_p.shape[0] != S or seeds.shape[0] != S:
        raise ValueError("inconsistent shapes")
    _dev(cache_row_map, "cache_row_map", (torch.int32,))
    need = verify_workspace_bytes(B, K, V)
    if workspace_buf is None:
        workspace_buf = workspace(need, target_logits.device)
    _dev(status, "status", (torch.int32,))
    _stats(draft_stats, B, K)
    code = lib().dspark_rejection_sample(
        _ptr(draft_tokens), _ptr(draft_cache), cache_dt, _ptr(cache_row_map), _ptr(draft_stats),
        _ptr(target_logits), _logit_dtype(target_logits, "target_logits"),
        _ptr(req_state_idx), _ptr(positions), _ptr(temperature), _ptr(top_p), _ptr(seeds),
        _ptr(out_tokens), _ptr(num_accepted), B, K, V, S, max(C, 1), _ptr(workspace_buf),
        workspace_buf.numel() * workspace_buf.element_size(), _ptr(status), _stream(stream))
    _check(code, "dspark_rejection_sample")


def temperature_divide(z, T, x, stream=None):
    """dspark_testing_temperature_divide on 1-D fp32 device tensors."""
    n = z.numel()
    for t, name in ((z, "z"), (T, "T"), (x, "x")):
        _dev(t, name, (torch.float32,))
        if t.numel() != n:
            raise ValueError("arrays must have equal length")
    _check(lib().dspark_testing_temperature_divide(_ptr(z), _ptr(T), _ptr(x), n,
                                                   _stream(stream)),
           "dspark_testing_temperature_divide")


def noise(seed, pos, col, stream_word, word=None, u=None, g=None, stream=None):
    """dspark_noise on 1-D device tensors of equal length."""
    n = seed.numel()
    for t, name in ((seed, "seed"), (pos, "pos"), (col, "col"), (stream_word, "stream")):
        _dev(t, name)
        if t.numel() != n:
            raise ValueError("noise arrays must have equal length")
    code = lib().dspark_noise(_ptr(seed), _ptr(pos), _ptr(col), _ptr(stream_word),
                              _ptr(word), _ptr(u), _ptr(g), n, _stream(stream))
    _check(code, "dspark_noise")
