"""The C ABI without a GPU: the library builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_99_gb300 import build_ext

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    path = build_ext.build()
    return ctypes.CDLL(path)


def _declared():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"PA_API\s+[\w\s\*]+?\b(pa_\w+)\s*\(", src)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    lib.pa_status_string.restype = ctypes.c_char_p
    seen = {lib.pa_status_string(i).decode() for i in range(7)}
    assert len(seen) == 7 and "ok" in seen
    assert lib.pa_status_string(99) == b"unknown status"


def test_version(lib):
    assert lib.pa_version() >= 100


FAKE = ctypes.c_void_p(0x10000)   # never dereferenced: every case below fails host checks first


def _decode(lib, **kw):
    a = dict(out=FAKE, q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, maxb=4, sl=FAKE, B=2, Hq=8, Hkv=2, d=128, bs=16,
             nb=10, scale=ctypes.c_float(0.088), qd=0, cd=0, ks=None, vs=None, ws=FAKE, wsb=ctypes.c_size_t(1 << 20),
             stream=None)
    a.update(kw)
    return lib.pa_decode(*a.values())


def test_decode_host_checks(lib):
    assert _decode(lib, d=64) == 2                         # head_dim != 128 unsupported
    for bs in (4, 12, 64):
        assert _decode(lib, bs=bs) == 2                    # block sizes other than 8, 16, 32
    assert _decode(lib, Hq=7) == 1                         # H_q not a multiple of H_kv
    assert _decode(lib, B=-1) == 1
    assert _decode(lib, B=9000) == 1                       # more sequences than supported
    assert _decode(lib, q=None) == 1                       # null pointer
    assert _decode(lib, cd=2) == 1                         # FP8 cache needs scales
    assert _decode(lib, qd=2) == 2                         # FP8 queries are not a mode
    assert _decode(lib, cd=1) == 2                         # bf16 q with fp16 cache
    assert _decode(lib, scale=ctypes.c_float(float("nan"))) == 1
    assert _decode(lib, ws=ctypes.c_void_p(0x10010)) == 1  # workspace not 256-byte aligned
    assert _decode(lib, kc=None) == 1                      # the cache is needed even for an empty batch


def test_empty_batch_is_a_no_op(lib):
    # B = 0: the per-sequence arrays may be null, nothing is launched
    assert _decode(lib, B=0, out=None, q=None, bt=None, sl=None) == 0
    assert _decode(lib, B=0, kc=None) == 1
    f = lib.pa_mixed
    f.argtypes = None
    assert f(None, None, None, FAKE, FAKE, None, 4, None, 0, 0, 0, 8, 2, 128, 16, 10, ctypes.c_float(0.088), 0, 0,
             None, None, FAKE, ctypes.c_size_t(1 << 20), None) == 0
    assert f(None, None, None, FAKE, FAKE, None, 4, None, 2, 3, 2, 8, 2, 128, 16, 10, ctypes.c_float(0.088), 0, 0,
             None, None, FAKE, ctypes.c_size_t(1 << 20), None) == 1   # B = 2 needs its arrays


def test_reshape_host_checks(lib):
    f = lib.pa_reshape_and_cache
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 64, 16, 10, 0, 0, None, None, None) == 2
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 16, 10, 0, 1, None, None, None) == 2
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 64, 10, 0, 0, None, None, None) == 2   # block size 64
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 16, 10, 0, 2, None, None, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, None, 4, 2, 128, 16, 10, 0, 0, None, None, None) == 1
    assert f(None, None, None, None, None, 0, 2, 128, 16, 10, 0, 0, None, None, None) == 0   # nothing to do
