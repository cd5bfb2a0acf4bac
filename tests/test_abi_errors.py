"""Error behaviour of the C ABI that needs no GPU: every case here is rejected by argument checks that run
before the library touches a device, with the return code include/whead.h documents. Pointers are fake,
16-byte aligned addresses that are never dereferenced (the checks fail first)."""
import ctypes

import pytest

from speculative_decoding_serial_gb300 import build
from speculative_decoding_serial_gb300 import whead as wh

FAKE = 0x10000  # aligned, never read
FAKE_ODD = 0x10004  # 4-byte aligned only


@pytest.fixture(scope="module")
def L():
    build.build()
    return wh.load()


def params(**kw):
    p = wh.WheadParams()
    p.kind, p.r, p.V, p.max_B, p.max_gamma = wh.MARKOV, 256, 151936, 1, 16
    for k, v in kw.items():
        setattr(p, k, v)
    return p


CREATE_CASES = [
    (dict(kind=2), wh.ERR_INVALID_ARG),
    (dict(V=0), wh.ERR_INVALID_ARG),
    (dict(max_B=0), wh.ERR_INVALID_ARG),
    (dict(max_B=17), wh.ERR_INVALID_ARG),
    (dict(max_gamma=0), wh.ERR_INVALID_ARG),
    (dict(max_gamma=65), wh.ERR_INVALID_ARG),
    (dict(V=1 << 24), wh.ERR_UNSUPPORTED),
    (dict(r=96), wh.ERR_UNSUPPORTED),
    (dict(r=320), wh.ERR_UNSUPPORTED),
    (dict(kind=wh.RECURRENT), wh.ERR_UNSUPPORTED),                       # recurrent without A
    (dict(flags=wh.FLAG_W_E4M3, r=192), wh.ERR_UNSUPPORTED),
    (dict(flags=wh.FLAG_W_E4M3, max_B=5), wh.ERR_UNSUPPORTED),
    (dict(v_offset=8), wh.ERR_INVALID_ARG),                              # shards start on 16-row groups
    (dict(v_offset=-16), wh.ERR_INVALID_ARG),
    (dict(e_rows=-1), wh.ERR_INVALID_ARG),
    (dict(v_offset=16, e_rows=151936), wh.ERR_INVALID_ARG),              # E shorter than the shard's rows
    (dict(v_offset=(1 << 24) - 16, V=16), wh.ERR_UNSUPPORTED),
]


@pytest.mark.parametrize("kw,code", CREATE_CASES)
def test_create_rejects(L, kw, code):
    out = ctypes.c_void_p(FAKE)
    p = params(**kw)
    assert L.whead_create(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), ctypes.byref(p), ctypes.byref(out)) == code
    assert out.value is None  # no handle on failure


def test_create_rejects_null_and_misaligned_pointers(L):
    out = ctypes.c_void_p()
    p = params()
    f, odd = ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE_ODD)
    assert L.whead_create(None, f, ctypes.byref(p), ctypes.byref(out)) == wh.ERR_INVALID_ARG
    assert L.whead_create(f, None, ctypes.byref(p), ctypes.byref(out)) == wh.ERR_INVALID_ARG
    assert L.whead_create(f, f, None, ctypes.byref(out)) == wh.ERR_INVALID_ARG
    assert L.whead_create(f, f, ctypes.byref(p), None) == wh.ERR_INVALID_ARG
    assert L.whead_create(odd, f, ctypes.byref(p), ctypes.byref(out)) == wh.ERR_INVALID_ARG
    assert L.whead_create(f, odd, ctypes.byref(p), ctypes.byref(out)) == wh.ERR_INVALID_ARG


def test_calls_on_a_null_handle(L):
    f = ctypes.c_void_p(FAKE)
    plan = wh.WheadPlan()
    assert L.whead_walk(None, f, f, 1, 1, 0.0, 0, f, None) == wh.ERR_INVALID_ARG
    assert L.whead_walk_ex(None, f, f, 1, 1, 0.0, 0, 0, f, None, None) == wh.ERR_INVALID_ARG
    assert L.whead_walk_keys(None, f, f, 1, 1, 0.0, 0, 0, f, f, None, None) == wh.ERR_INVALID_ARG
    assert L.whead_walk_host(None, f, f, 1, 1, 0.0, 0, f, None) == wh.ERR_INVALID_ARG
    assert L.whead_advance(None, f, f, f, 1) == wh.ERR_INVALID_ARG
    assert L.whead_status(None) == wh.ERR_INVALID_ARG
    assert L.whead_plan_info(None, 1, ctypes.byref(plan)) == wh.ERR_INVALID_ARG
    assert L.whead_set_trace(None, None, 0) == wh.ERR_INVALID_ARG
    assert L.whead_destroy(None) == wh.ERR_INVALID_ARG


@pytest.mark.parametrize("V,r,wq,sw,code", [
    (0, 256, FAKE, FAKE, wh.ERR_INVALID_ARG),
    (1000, 64, FAKE, FAKE, wh.ERR_UNSUPPORTED),
    (1000, 192, FAKE, FAKE, wh.ERR_UNSUPPORTED),
    (1 << 24, 256, FAKE, FAKE, wh.ERR_UNSUPPORTED),
    (1000, 256, FAKE_ODD, FAKE, wh.ERR_INVALID_ARG),
    (1000, 256, FAKE, FAKE + 2, wh.ERR_INVALID_ARG),
    (1000, 256, None, FAKE, wh.ERR_INVALID_ARG),
])
def test_quantizer_rejects(L, V, r, wq, sw, code):
    assert L.whead_quantize_w_e4m3(ctypes.c_void_p(FAKE), V, r, ctypes.c_void_p(wq) if wq else None,
                                   ctypes.c_void_p(sw), None) == code


NOALLOC_CASES = [
    (dict(), dict(B=17), wh.ERR_UNSUPPORTED),                 # more walks than the scratch array holds
    (dict(), dict(gamma=65), wh.ERR_UNSUPPORTED),
    (dict(), dict(B=0), wh.ERR_INVALID_ARG),
    (dict(), dict(T=-1.0), wh.ERR_INVALID_ARG),
    (dict(), dict(T=float("nan")), wh.ERR_INVALID_ARG),
    (dict(r=100), dict(), wh.ERR_UNSUPPORTED),
    (dict(V=1 << 24), dict(), wh.ERR_UNSUPPORTED),
    (dict(flags=wh.FLAG_W_E4M3), dict(), wh.ERR_UNSUPPORTED),  # needs a handle's quantized copy of W
    (dict(flags=wh.FLAG_FORCE_STREAM), dict(), wh.ERR_UNSUPPORTED),     # measurement modes need a handle's plans
    (dict(flags=wh.FLAG_PLACEMENT_CAPS), dict(), wh.ERR_UNSUPPORTED),
    (dict(flags=wh.FLAG_HOST_STAGE), dict(), wh.ERR_UNSUPPORTED),       # a host-buffer option; no host buffers here
    (dict(kind=wh.RECURRENT), dict(), wh.ERR_UNSUPPORTED),
    (dict(v_offset=8), dict(), wh.ERR_INVALID_ARG),
    (dict(), dict(u0=FAKE_ODD), wh.ERR_INVALID_ARG),
]


@pytest.mark.parametrize("pkw,ckw,code", NOALLOC_CASES)
def test_noalloc_rejects_before_touching_a_device(L, pkw, ckw, code):
    p = params(**pkw)
    c = dict(B=1, gamma=16, T=0.0, u0=FAKE)
    c.update(ckw)
    f = ctypes.c_void_p(FAKE)
    rc = L.whead_walk_noalloc(f, f, ctypes.byref(p), f, ctypes.c_void_p(c["u0"]), c["B"], c["gamma"], c["T"], 0, f,
                              None, None)
    assert rc == code


def test_noalloc_rejects_null_pointers(L):
    p = params()
    f = ctypes.c_void_p(FAKE)
    for args in ((None, f, ctypes.byref(p), f, f), (f, None, ctypes.byref(p), f, f), (f, f, None, f, f),
                 (f, f, ctypes.byref(p), None, f), (f, f, ctypes.byref(p), f, None)):
        assert L.whead_walk_noalloc(*args, 1, 16, 0.0, 0, f, None, None) == wh.ERR_INVALID_ARG
    assert L.whead_walk_noalloc(f, f, ctypes.byref(p), f, f, 1, 16, 0.0, 0, None, None, None) == wh.ERR_INVALID_ARG
