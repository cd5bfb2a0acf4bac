"""Python binding of the whead C ABI (argument marshalling only).

Every step of the walk runs in the CUDA library libwhead.so; this module only converts torch tensors to
device pointers and the current CUDA stream to a cudaStream_t. There is no fallback: if the library is
missing or was not built for this machine, loading raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

MARKOV = 0
RECURRENT = 1

FLAG_LOGITS_F32 = 1 << 0
FLAG_FIXED_LATENT = 1 << 1
FLAG_FORCE_STREAM = 1 << 2
FLAG_PLACEMENT_CAPS = 1 << 3
FLAG_W_E4M3 = 1 << 4
FLAG_HOST_STAGE = 1 << 5
FLAG_FAULT_SKIP_ARRIVAL = 1 << 8

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_CUDA = -3
ERR_TIMEOUT = -4
ERR_NO_COOP = -5
ERR_INTERNAL = -6

# Every symbol include/whead.h declares.
EXPORTS = ("whead_create", "whead_walk", "whead_walk_ex", "whead_walk_host", "whead_status",
           "whead_plan_info", "whead_strerror", "whead_destroy", "whead_walk_noalloc",
           "whead_set_trace", "whead_quantize_w_e4m3", "whead_walk_keys", "whead_advance", "whead_plan_query")


class WheadParams(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("r", ctypes.c_int32), ("V", ctypes.c_int64),
                ("A", ctypes.c_void_p), ("c", ctypes.c_void_p), ("max_B", ctypes.c_int32),
                ("max_gamma", ctypes.c_int32), ("stream", ctypes.c_void_p), ("flags", ctypes.c_uint32),
                ("grid", ctypes.c_int32), ("timeout_us", ctypes.c_uint32), ("cap_smem", ctypes.c_int32),
                ("cap_tmem", ctypes.c_int32), ("cap_rf", ctypes.c_int32), ("v_offset", ctypes.c_int64),
                ("e_rows", ctypes.c_int64)]


class WheadPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("grid", "threads", "groups_per_cta", "smem_groups", "tmem_groups",
                                              "rf_groups", "stream_groups", "smem_bytes", "tmem_cols", "sm_count")]


class WheadError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libwhead.so (optionally building it first). Raises if it is not there."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing and _build.needs_build():
        _build.build()
    if not os.path.exists(path):
        raise ImportError(f"libwhead.so is not built ({path}); run speculative_decoding_serial_gb300.build.build()")
    L = ctypes.CDLL(path)
    vp, i32, i64, u64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
    L.whead_create.argtypes = [vp, vp, ctypes.POINTER(WheadParams), ctypes.POINTER(vp)]
    L.whead_walk.argtypes = [vp, vp, vp, i32, i32, f32, u64, vp, vp]
    L.whead_walk_ex.argtypes = [vp, vp, vp, i32, i32, f32, u64, i64, vp, vp, vp]
    L.whead_walk_host.argtypes = [vp, vp, vp, i32, i32, f32, u64, vp, vp]
    L.whead_status.argtypes = [vp]
    L.whead_set_trace.argtypes = [vp, vp, i64]
    L.whead_plan_info.argtypes = [vp, i32, ctypes.POINTER(WheadPlan)]
    L.whead_strerror.argtypes = [ctypes.c_int]
    L.whead_strerror.restype = ctypes.c_char_p
    L.whead_destroy.argtypes = [vp]
    L.whead_walk_noalloc.argtypes = [vp, vp, ctypes.POINTER(WheadParams), vp, vp, i32, i32, f32, u64, vp, vp, vp]
    L.whead_quantize_w_e4m3.argtypes = [vp, i64, i32, vp, vp, vp]
    L.whead_walk_keys.argtypes = [vp, vp, vp, i32, i32, f32, u64, i64, vp, vp, vp, vp]
    L.whead_advance.argtypes = [vp, vp, vp, vp, i32]
    L.whead_plan_query.argtypes = [i64, i32, i32, i32, i32, ctypes.c_uint32, i32, i32, ctypes.POINTER(WheadPlan), vp,
                                   vp, vp]
    for name in ("whead_create", "whead_walk", "whead_walk_ex", "whead_walk_host", "whead_status",
                 "whead_plan_info", "whead_destroy", "whead_walk_noalloc",
                 "whead_set_trace", "whead_quantize_w_e4m3", "whead_walk_keys", "whead_advance", "whead_plan_query"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


# tiers of a work-list entry (bits 8..9)
TIER_SMEM, TIER_TMEM, TIER_RF, TIER_STREAM = 0, 1, 2, 3
WARPS, MAX_WARP_GROUPS = 12, 32


def plan_query(V: int, r: int, kind: int = 0, *, max_B: int = 1, B: int = 1, e4m3: bool = False,
               sm_count: int, smem_optin: int) -> dict:
    """whead_plan_query: the placement whead_create would choose, computed on the host (no device needed).
    Returns the whead_plan fields plus "work_lists" (per warp, its entries as (group, tier, tmem_col)),
    "rf_warp_mask" and "ah_warp"."""
    pl = WheadPlan()
    wl = (ctypes.c_uint32 * (WARPS * (1 + MAX_WARP_GROUPS)))()
    mask = ctypes.c_uint32(0)
    ahw = ctypes.c_int32(0)
    _check(load().whead_plan_query(int(V), int(r), int(kind), int(max_B), int(B), FLAG_W_E4M3 if e4m3 else 0,
                                   int(sm_count), int(smem_optin), ctypes.byref(pl), ctypes.cast(wl, ctypes.c_void_p),
                                   ctypes.byref(mask), ctypes.byref(ahw)), "whead_plan_query")
    out = {n: int(getattr(pl, n)) for n, _ in WheadPlan._fields_}
    lists = []
    for w in range(WARPS):
        row = wl[w * (1 + MAX_WARP_GROUPS):(w + 1) * (1 + MAX_WARP_GROUPS)]
        lists.append([(e & 0xFF, (e >> 8) & 3, (e >> 16) & 0x3FF) for e in row[1:1 + row[0]]])
    out.update(work_lists=lists, rf_warp_mask=int(mask.value), ah_warp=int(ahw.value))
    return out


def strerror(code: int) -> str:
    return load().whead_strerror(int(code)).decode()


def _check(code: int, what: str):
    if code != OK:
        raise WheadError(code, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


class Head:
    """A serial draft head whose projection W stays on chip for each walk.

    W, E: (V, r) torch.bfloat16 CUDA tensors (borrowed: keep them alive and unchanged). For the recurrent
    head pass A (r, r) float32 and optionally c (r,) float32. All calls go to `stream` (default: the
    current torch stream at construction).
    """

    def __init__(self, W, E, *, kind=MARKOV, A=None, c=None, max_B=1, max_gamma=16, stream=None, flags=0,
                 grid=0, timeout_us=0, caps=None, v_offset=0, e_rows=0):
        import torch
        L = load()
        assert W.is_cuda and W.dtype == torch.bfloat16 and W.is_contiguous() and W.dim() == 2
        # E covers the shard's global rows (all of W's rows when the vocabulary is not sharded)
        assert E.dim() == 2 and E.shape[1] == W.shape[1] and E.shape[0] >= int(v_offset) + W.shape[0]
        assert E.dtype == torch.bfloat16 and E.is_contiguous()
        self.V, self.r = int(W.shape[0]), int(W.shape[1])
        # caps: (shared, tensor, register) most groups per CTA per tier (placement sweep); the rest stream
        if caps is not None:
            flags = int(flags) | FLAG_PLACEMENT_CAPS
        cs, ct, cr = (int(x) for x in caps) if caps is not None else (0, 0, 0)
        self.kind, self.flags = int(kind), int(flags)
        self._keep = (W, E, A, c)
        self._stream = torch.cuda.current_stream() if stream is None else stream
        p = WheadParams(kind=self.kind, r=self.r, V=self.V, A=_ptr(A), c=_ptr(c), max_B=int(max_B),
                        max_gamma=int(max_gamma), stream=ctypes.c_void_p(self._stream.cuda_stream),
                        flags=self.flags, grid=int(grid), timeout_us=int(timeout_us), cap_smem=cs, cap_tmem=ct,
                        cap_rf=cr, v_offset=int(v_offset), e_rows=int(e_rows))
        h = ctypes.c_void_p()
        _check(L.whead_create(_ptr(W), _ptr(E), ctypes.byref(p), ctypes.byref(h)), "whead_create")
        self._h = h
        self.max_B, self.max_gamma = int(max_B), int(max_gamma)

    def walk(self, base, u0, *, T=0.0, seed=0, out_tokens=None, out_logits=None):
        """base (B, gamma, V) float32, u0 (B, r) float32 CUDA tensors. Returns int32 tokens (B, gamma)."""
        return self.walk_ex(base, u0, T=T, seed=seed, t0=0, out_tokens=out_tokens, out_logits=out_logits)

    def walk_ex(self, base, s0, *, T=0.0, seed=0, t0=0, out_tokens=None, out_logits=None, out_state=None):
        import torch
        B, gamma, V = base.shape
        assert V == self.V and s0.shape == (B, self.r)
        assert base.dtype == torch.float32 and s0.dtype == torch.float32
        assert base.is_contiguous() and s0.is_contiguous()
        if out_tokens is None:
            out_tokens = torch.empty((B, gamma), dtype=torch.int32, device=base.device)
        _check(load().whead_walk_ex(self._h, _ptr(base), _ptr(s0), B, gamma, float(T), int(seed) & (2**64 - 1),
                                    int(t0), _ptr(out_tokens), _ptr(out_logits), _ptr(out_state)), "whead_walk_ex")
        return out_tokens

    def walk_keys(self, base, s0, *, T=0.0, seed=0, t0=0, out_tokens=None, out_keys=None, out_logits=None,
                  out_state=None):
        """whead_walk_ex plus each step's winning packed key: returns (tokens (B, gamma) int32, keys (B, gamma)
        int64 holding the uint64 keys' bits)."""
        import torch
        B, gamma, V = base.shape
        assert V == self.V and s0.shape == (B, self.r)
        if out_tokens is None:
            out_tokens = torch.empty((B, gamma), dtype=torch.int32, device=base.device)
        if out_keys is None:
            out_keys = torch.empty((B, gamma), dtype=torch.int64, device=base.device)
        _check(load().whead_walk_keys(self._h, _ptr(base), _ptr(s0), B, gamma, float(T), int(seed) & (2**64 - 1),
                                      int(t0), _ptr(out_tokens), _ptr(out_keys), _ptr(out_logits), _ptr(out_state)),
               "whead_walk_keys")
        return out_tokens, out_keys

    def advance(self, x, s, s_next):
        """Next state on the device for winners x (B,) int32 (global rows), from state s (B, r) into s_next."""
        _check(load().whead_advance(self._h, _ptr(x), _ptr(s), _ptr(s_next), int(x.shape[0])), "whead_advance")
        return s_next

    def walk_host(self, base, u0, *, T=0.0, seed=0, out_tokens=None, out_logits=None):
        """Synchronous walk on host (CPU) torch tensors. The walk reads the base logits in place where the GPU
        can address them (pinned memory; any host memory on Grace); u0 and the outputs are copied inside the
        call. Raises on a device-side error of the walk."""
        import torch
        B, gamma, V = base.shape
        assert V == self.V and not base.is_cuda and not u0.is_cuda
        if out_tokens is None:
            out_tokens = torch.empty((B, gamma), dtype=torch.int32)
        _check(load().whead_walk_host(self._h, _ptr(base), _ptr(u0), B, gamma, float(T), int(seed) & (2**64 - 1),
                                      _ptr(out_tokens), _ptr(out_logits)), "whead_walk_host")
        return out_tokens

    def set_trace(self, buf):
        """Phase stamps for the following walks (buf: int64 CUDA tensor, or None to turn them off)."""
        n = 0 if buf is None else buf.numel() * buf.element_size()
        _check(load().whead_set_trace(self._h, _ptr(buf), n), "whead_set_trace")
        self._trace = buf

    def status(self) -> int:
        return int(load().whead_status(self._h))

    def plan(self, B: int = 1) -> dict:
        pl = WheadPlan()
        _check(load().whead_plan_info(self._h, int(B), ctypes.byref(pl)), "whead_plan_info")
        return {n: int(getattr(pl, n)) for n, _ in WheadPlan._fields_}

    def close(self):
        if getattr(self, "_h", None):
            load().whead_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def walk_noalloc(W, E, base, u0, *, kind=MARKOV, A=None, c=None, T=0.0, seed=0, flags=0, timeout_us=0,
                 out_tokens, out_logits=None, out_status=None, stream=None, check=False):
    """The allocation-free walk (whead_walk_noalloc): every buffer, outputs included, comes from the caller.

    For callers that must not allocate device memory (an engine that owns all GPU memory in its own pool,
    or a loop that cannot afford the device synchronization of cudaMalloc). The library's scratch for this
    call is a fixed device array shared by all calls, so walks issued through this function must not
    overlap on the GPU. The first call on a device should come before any stream capture.

    out_status: a device int32 tensor that receives the walk's device status. Without it a time-out or
    internal error on the device is not reported anywhere. check=True (which needs out_status) waits for the
    stream and raises WheadError when the status is not 0.
    """
    import torch
    B, gamma, V = base.shape
    r = int(W.shape[1])
    s = torch.cuda.current_stream() if stream is None else stream
    p = WheadParams(kind=int(kind), r=r, V=int(V), A=_ptr(A), c=_ptr(c), max_B=int(B), max_gamma=int(gamma),
                    stream=ctypes.c_void_p(s.cuda_stream), flags=int(flags), grid=0, timeout_us=int(timeout_us))
    if check and out_status is None:
        raise ValueError("check=True needs out_status")
    _check(load().whead_walk_noalloc(_ptr(W), _ptr(E), ctypes.byref(p), _ptr(base), _ptr(u0), int(B), int(gamma),
                                     float(T), int(seed) & (2**64 - 1), _ptr(out_tokens), _ptr(out_logits),
                                     _ptr(out_status)), "whead_walk_noalloc")
    if check:
        s.synchronize()
        _check(int(out_status.item()), "whead_walk_noalloc (device status)")
    return out_tokens
