"""ctypes loader for the plain C oracle of the serial draft-head walk.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's CPU-baseline leg are the
only callers. The CUDA library never imports or links this module, and this module imports nothing
from the CUDA side.

The oracle follows "Weights That Stay: On-Chip Megakernels for Serial Heads in Speculative Decoding"
(abstract; Figs. 2, 7, 8) step by step: project the bf16-rounded state through W with fp64
accumulation, add the base logits in fp32, pick the smallest row holding the largest (optionally
Gumbel-perturbed) key, and advance a Markov (s <- E[x]) or recurrent (s <- tanh(A s + E[x] + c)) state.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "whead_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

MARKOV = 0
RECURRENT = 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, so x86 and Arm hosts agree bit for bit). OpenMP splits
    a step's rows over threads when the compiler has it; otherwise the oracle builds single-threaded."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        base = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        if subprocess.run(base[:3] + ["-fopenmp"] + base[3:], capture_output=True).returncode != 0:
            subprocess.run(base, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def set_threads(n: int) -> int:
    """Threads for the rows of each step's projection (1 by default); returns the number in use. The results
    are the same for every thread count."""
    return int(lib().whead_oracle_set_threads(int(n)))


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            L.whead_oracle_philox4x32_10.argtypes = [ctypes.POINTER(ctypes.c_uint32)] * 3
            L.whead_oracle_philox4x32_10.restype = None
            L.whead_oracle_noise_word.argtypes = [ctypes.c_uint64, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64]
            L.whead_oracle_noise_word.restype = ctypes.c_uint32
            L.whead_oracle_uniform.argtypes = [ctypes.c_uint32]
            L.whead_oracle_uniform.restype = ctypes.c_float
            L.whead_oracle_gumbel.argtypes = [ctypes.c_uint64, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64]
            L.whead_oracle_gumbel.restype = ctypes.c_float
            L.whead_oracle_set_threads.argtypes = [ctypes.c_int]
            L.whead_oracle_set_threads.restype = ctypes.c_int
            L.whead_oracle_bf16_round.argtypes = [ctypes.c_float]
            L.whead_oracle_bf16_round.restype = ctypes.c_uint16
            vp = ctypes.c_void_p
            L.whead_oracle_walk.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, vp, vp, vp, vp, vp, vp,
                                            ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                            ctypes.c_uint64, vp, vp, vp, vp, vp]
            L.whead_oracle_walk.restype = ctypes.c_int
            L.whead_oracle_walk_e4m3.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, vp, vp, vp, vp, vp,
                                                 vp, vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                                 ctypes.c_float, ctypes.c_uint64, vp, vp, vp, vp, vp]
            L.whead_oracle_walk_e4m3.restype = ctypes.c_int
            L.whead_oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            L.whead_oracle_e4m3_value.restype = ctypes.c_float
            L.whead_oracle_e4m3_round.argtypes = [ctypes.c_float]
            L.whead_oracle_e4m3_round.restype = ctypes.c_uint8
            L.whead_oracle_quantize_e4m3.argtypes = [vp, ctypes.c_int32, vp]
            L.whead_oracle_quantize_e4m3.restype = ctypes.c_float
            L.whead_oracle_split_e4m3.argtypes = [vp, ctypes.c_int32, vp, vp, ctypes.POINTER(ctypes.c_float),
                                                  ctypes.POINTER(ctypes.c_float)]
            L.whead_oracle_split_e4m3.restype = None
            L.whead_oracle_quantize_w_e4m3.argtypes = [vp, ctypes.c_int64, ctypes.c_int32, vp, vp]
            L.whead_oracle_quantize_w_e4m3.restype = None
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def philox4x32_10(ctr, key):
    c = (ctypes.c_uint32 * 4)(*[int(x) & 0xFFFFFFFF for x in ctr])
    k = (ctypes.c_uint32 * 2)(*[int(x) & 0xFFFFFFFF for x in key])
    o = (ctypes.c_uint32 * 4)()
    lib().whead_oracle_philox4x32_10(c, k, o)
    return [int(o[i]) for i in range(4)]


def noise_word(seed: int, b: int, tau: int, v: int) -> int:
    return int(lib().whead_oracle_noise_word(seed, b, tau, v))


def uniform(w: int) -> float:
    return float(lib().whead_oracle_uniform(w))


def gumbel(seed: int, b: int, tau: int, v: int) -> float:
    return float(lib().whead_oracle_gumbel(seed, b, tau, v))


def bf16_round(x: float) -> int:
    return int(lib().whead_oracle_bf16_round(x))


def e4m3_value(code: int) -> float:
    return float(lib().whead_oracle_e4m3_value(int(code) & 0xFF))


def e4m3_round(x: float) -> int:
    return int(lib().whead_oracle_e4m3_round(float(x)))


def quantize_e4m3(x):
    """x: float32 vector. Returns (scale, uint8 E4M3 codes)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    q = np.zeros(x.shape[0], dtype=np.uint8)
    s = lib().whead_oracle_quantize_e4m3(_ptr(x), x.shape[0], _ptr(q))
    return float(s), q


def split_e4m3(u):
    """u: float32 vector. Returns (s1, hi codes, s2, lo codes) of the two-vector representation."""
    u = np.ascontiguousarray(u, dtype=np.float32)
    hi = np.zeros(u.shape[0], dtype=np.uint8)
    lo = np.zeros(u.shape[0], dtype=np.uint8)
    s1, s2 = ctypes.c_float(), ctypes.c_float()
    lib().whead_oracle_split_e4m3(_ptr(u), u.shape[0], _ptr(hi), _ptr(lo), ctypes.byref(s1), ctypes.byref(s2))
    return float(s1.value), hi, float(s2.value), lo


def quantize_w_e4m3(W):
    """W: (V, r) uint16 bf16 bits. Returns (Wq (V, r) uint8 E4M3 codes, sw (V,) float32 row scales)."""
    W = np.ascontiguousarray(W, dtype=np.uint16)
    V, r = W.shape
    Wq = np.zeros((V, r), dtype=np.uint8)
    sw = np.zeros(V, dtype=np.float32)
    lib().whead_oracle_quantize_w_e4m3(_ptr(W), V, r, _ptr(Wq), _ptr(sw))
    return Wq, sw


def walk(kind, W, E, base, s0, *, A=None, c=None, t0=0, T=0.0, seed=0,
         want_logits=False, want_z=False, want_gap=True, want_state=False, w_e4m3=None):
    """Run the oracle walk.

    W, E: (V, r) uint16 bf16 bit patterns. base: (B, gamma, V) float32. s0: (B, r) float32.
    A: (r, r) float32 and c: (r,) float32 for the recurrent head. w_e4m3: None, or (Wq, sw) from
    quantize_w_e4m3 for the walk with E4M3 weights (W is then only used for its shape). Returns a dict with 'tokens'
    (B, gamma) int32 and, on request, 'logits' (B, gamma, V) uint16 bf16 bits, 'z' float32,
    'gap' (B, gamma) float32 and 'state' (B, gamma, r) float32 (the state after each step).
    """
    W = np.ascontiguousarray(W, dtype=np.uint16)
    E = np.ascontiguousarray(E, dtype=np.uint16)
    base = np.ascontiguousarray(base, dtype=np.float32)
    s0 = np.ascontiguousarray(s0, dtype=np.float32)
    V, r = W.shape
    B, gamma, Vb = base.shape
    assert Vb == V and E.shape == (V, r) and s0.shape == (B, r)
    if A is not None:
        A = np.ascontiguousarray(A, dtype=np.float32)
        assert A.shape == (r, r)
    if c is not None:
        c = np.ascontiguousarray(c, dtype=np.float32)
        assert c.shape == (r,)
    out = {"tokens": np.zeros((B, gamma), dtype=np.int32)}
    if want_logits:
        out["logits"] = np.zeros((B, gamma, V), dtype=np.uint16)
    if want_z:
        out["z"] = np.zeros((B, gamma, V), dtype=np.float32)
    if want_gap:
        out["gap"] = np.zeros((B, gamma), dtype=np.float32)
    if want_state:
        out["state"] = np.zeros((B, gamma, r), dtype=np.float32)
    tail = (B, gamma, int(t0), float(T), int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(out["tokens"]),
            _ptr(out.get("logits")), _ptr(out.get("z")), _ptr(out.get("gap")), _ptr(out.get("state")))
    if w_e4m3 is None:
        rc = lib().whead_oracle_walk(int(kind), V, r, _ptr(W), _ptr(E), _ptr(A), _ptr(c), _ptr(base), _ptr(s0), *tail)
    else:
        Wq = np.ascontiguousarray(w_e4m3[0], dtype=np.uint8)
        sw = np.ascontiguousarray(w_e4m3[1], dtype=np.float32)
        assert Wq.shape == (V, r) and sw.shape == (V,)
        rc = lib().whead_oracle_walk_e4m3(int(kind), V, r, _ptr(Wq), _ptr(sw), _ptr(E), _ptr(A), _ptr(c), _ptr(base),
                                          _ptr(s0), *tail)
    if rc != 0:
        raise ValueError(f"oracle walk rejected its arguments (code {rc})")
    return out
