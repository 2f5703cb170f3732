"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every function include/*.h declares, and its host-side argument checks
reject bad calls before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    inc = os.path.join(ROOT, "include")
    src = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc))
                  if f.endswith(".h"))
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(dspark_[a-z0-9_]+)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def L():
    import shutil
    if not shutil.which("nvcc") and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from verify_dspark_markov_step_gb300 import build, _lib
    build.build()
    return _lib.lib()


def test_header_declares_the_binding_exports():
    from verify_dspark_markov_step_gb300 import _lib
    assert _declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_status_strings_and_version(L):
    from verify_dspark_markov_step_gb300 import _lib
    assert _lib.status_string(0) == "ok"
    assert "range" in _lib.status_string(-5)
    assert _lib.status_string(12345) == "unknown status"
    assert L.dspark_version() >= 100


def test_workspace_sizes(L):
    from verify_dspark_markov_step_gb300 import _lib
    a = _lib.markov_workspace_bytes(32, 7, 200064, 256)
    b = _lib.markov_workspace_bytes(64, 7, 200064, 256)
    assert 0 < a < b and a % 256 == 0
    assert _lib.verify_workspace_bytes(32, 7, 200064) > 0
    assert _lib.markov_workspace_bytes(-1, 7, 10, 64) == 0


def test_argument_checks_return_before_any_launch(L):
    """Invalid sizes, dtypes, R and null pointers are rejected on the host
    (these calls never reach the CUDA runtime, so they run without a GPU)."""
    vp = ctypes.c_void_p
    fake = vp(256)          # never dereferenced: every call below fails first
    null = None
    def markov(B=1, K=1, V=10, R=64, S=1, C=1, base=fake, bdt=0, cdt=0, ws=fake, wsb=1 << 20):
        return L.dspark_markov_sample(base, bdt, fake, fake, fake, fake, fake, fake, fake,
                                      null, cdt, null, fake, null, B, K, V, R, S, C, ws, wsb,
                                      null, null)
    assert markov(B=-1) == -1
    assert markov(B=257) == -1
    assert markov(K=0) == -1
    assert markov(K=17) == -1
    assert markov(V=0) == -1
    assert markov(V=1 << 23) == -1
    assert markov(S=0) == -1
    assert markov(bdt=7) == -1
    assert markov(R=100) == -2            # unsupported rank
    assert markov(R=576) == -2
    assert markov(B=0) == 0               # empty batch: nothing to do
    assert markov(base=null) == -1
    assert markov(ws=null) == -6
    assert markov(wsb=8) == -6
    assert markov(base=vp(258)) == -7     # misaligned logits
    def verify(B=1, K=1, V=10, S=1, target=fake, tdt=0, ws=fake, wsb=1 << 20):
        return L.dspark_rejection_sample(fake, null, 0, null, null, target, tdt, fake, fake,
                                         fake, fake, fake, fake, fake, B, K, V, S, 1, ws, wsb,
                                         null, null)
    assert verify(B=300) == -1
    assert verify(tdt=3) == -1
    assert verify(target=null) == -1
    assert verify(target=vp(260)) == -7
    assert verify(wsb=4) == -6
    assert verify(B=0) == 0
    assert L.dspark_noise(fake, fake, fake, fake, null, null, null, -1, null) == -1
    assert L.dspark_noise(null, null, null, null, null, null, null, 0, null) == 0


def test_wait_limit_hook_checks_its_knobs(L):
    """The bounded-wait test hook takes limits from 0.1 ms to 2 s and at most
    one extra arrival; everything else is checked as dspark_markov_sample."""
    vp = ctypes.c_void_p
    fake, null = vp(256), None
    def hook(limit=1_000_000, extra=1, B=1, R=64, ws=fake):
        return L.dspark_testing_markov_wait_limit(
            fake, 0, fake, fake, fake, fake, fake, fake, fake, null, 0, null, fake, B, 1, 10, R,
            1, 1, ws, 1 << 20, null, null, limit, extra)
    assert hook(limit=10) == -1
    assert hook(limit=3_000_000_000) == -1
    assert hook(extra=2) == -1
    assert hook(B=300) == -1
    assert hook(R=100) == -2
    assert hook(ws=null) == -6
    assert hook(B=0) == 0


def test_missing_library_fails_loudly(tmp_path):
    """No CPU fallback: loading a library that is not there raises."""
    from verify_dspark_markov_step_gb300 import _lib
    with pytest.raises(RuntimeError, match="CUDA library not built"):
        _lib.lib(str(tmp_path / "libdspark.so"))
