"""GB300 (sm_103a) self-attention forward: Python binding of libattn.so.

Argument marshalling only.  Every step of the forward pass runs in the CUDA
kernels of libattn.so; there is no CPU or PyTorch fallback.  If the library is
missing (not built), importing this module raises.

Low-level functions mirror the C ABI of ``include/attn.h`` (same names, integer
pointers); :class:`Attention` wraps a handle for torch tensors.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattn.so")

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_DEVICE_TIMEOUT, ATTN_ERR_OOM = range(6)
MASK_FULL, MASK_CAUSAL, MASK_SLIDING, MASK_CAUSAL_SLIDING, MASK_LOCAL_GLOBAL = range(5)
ATTN_BF16, ATTN_F32, ATTN_FP8_E4M3 = 0, 1, 2
TILE = 128
WORK_INTS = 8
LIST_FULL = 1 << 16  # ATTN_LIST_FULL: the FULL flag of a backward list entry
WORK_GLOBAL_COLS, WORK_GLOBAL_ROWS, WORK_HAS_GLOBAL_ROWS = 1, 2, 4

EXPORTED = ("attn_create", "attn_forward", "attn_destroy", "attn_status_string", "attn_schedule_host",
            "attn_poll_device_error", "attn_set_watchdog", "attn_forward_noalloc", "attn_selftest_exp2",
            "attn_decode_create", "attn_decode_forward", "attn_decode_poll_device_error", "attn_decode_destroy",
            "attn_decode_schedule_host", "attn_decode_set_grid_limit", "attn_set_alibi",
            "attn_decode_set_alibi", "attn_set_fp8_descale", "attn_kv_schedule_host",
            "attn_backward", "attn_bwd_dq_schedule_host", "attn_set_bias", "attn_decode_set_merge_mode",
            "attn_decode_launch_count", "attn_selftest_device_once", "attn_forward_noalloc_poll_error",
            "attn_forward_noalloc_set_watchdog", "attn_bwd_lg_lists_host")
NOALLOC_SCRATCH_BYTES = 8 << 20
DECODE_MAX_BATCH = 1024
DECODE_MAX_ROWS = 64


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {attn_status_string(status)} (status {status})")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libattn.so not built at {LIB_PATH}; run __graft_entry__.build() "
                          "(the library has no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    I, P, F, LL = ctypes.c_int, ctypes.c_void_p, ctypes.c_float, ctypes.c_longlong
    lib.attn_create.argtypes = [ctypes.POINTER(P), I, I, I, I, I, I, F, I, I, P, I]
    lib.attn_create.restype = I
    lib.attn_forward.argtypes = [P, P, P, P, P, P, P]
    lib.attn_forward.restype = I
    lib.attn_destroy.argtypes = [P]
    lib.attn_destroy.restype = I
    lib.attn_status_string.argtypes = [I]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_schedule_host.argtypes = [I, I, I, I, I, I, P, I, P, I, ctypes.POINTER(I), ctypes.POINTER(I)]
    lib.attn_schedule_host.restype = I
    lib.attn_poll_device_error.argtypes = [P, ctypes.POINTER(I)]
    lib.attn_poll_device_error.restype = I
    lib.attn_set_watchdog.argtypes = [P, LL, I]
    lib.attn_set_watchdog.restype = I
    lib.attn_set_alibi.argtypes = [P, P]
    lib.attn_set_alibi.restype = I
    lib.attn_decode_set_alibi.argtypes = [P, P]
    lib.attn_decode_set_alibi.restype = I
    lib.attn_set_fp8_descale.argtypes = [P, F, F, F]
    lib.attn_set_fp8_descale.restype = I
    lib.attn_kv_schedule_host.argtypes = [I, I, I, P, I, ctypes.POINTER(I)]
    lib.attn_kv_schedule_host.restype = I
    lib.attn_backward.argtypes = [P] * 11
    lib.attn_backward.restype = I
    lib.attn_bwd_dq_schedule_host.argtypes = [I, I, I, I, I, I, I, P, I, ctypes.POINTER(I)]
    lib.attn_bwd_dq_schedule_host.restype = I
    lib.attn_bwd_lg_lists_host.argtypes = [I, I, P, I, P, I, P, ctypes.POINTER(I)]
    lib.attn_bwd_lg_lists_host.restype = I
    lib.attn_set_bias.argtypes = [P, P, I, I, ctypes.c_long]
    lib.attn_set_bias.restype = I
    lib.attn_decode_set_merge_mode.argtypes = [P, I]
    lib.attn_decode_set_merge_mode.restype = I
    lib.attn_decode_launch_count.argtypes = [P, ctypes.POINTER(I)]
    lib.attn_decode_launch_count.restype = I
    lib.attn_forward_noalloc.argtypes = [I, I, I, I, I, F, I, I, P, I, P, P, P, P, P, P]
    lib.attn_forward_noalloc.restype = I
    lib.attn_forward_noalloc_poll_error.argtypes = [ctypes.POINTER(I)]
    lib.attn_forward_noalloc_poll_error.restype = I
    lib.attn_forward_noalloc_set_watchdog.argtypes = [ctypes.c_longlong, I]
    lib.attn_forward_noalloc_set_watchdog.restype = I
    lib.attn_selftest_exp2.argtypes = [P, P, I, P]
    lib.attn_selftest_exp2.restype = I
    lib.attn_selftest_device_once.argtypes = []
    lib.attn_selftest_device_once.restype = I
    lib.attn_decode_create.argtypes = [ctypes.POINTER(P), I, I, I, I, I, I, F, I, I]
    lib.attn_decode_create.restype = I
    lib.attn_decode_forward.argtypes = [P, P, P, P, P, P, P, P]
    lib.attn_decode_forward.restype = I
    lib.attn_decode_poll_device_error.argtypes = [P, ctypes.POINTER(I)]
    lib.attn_decode_poll_device_error.restype = I
    lib.attn_decode_destroy.argtypes = [P]
    lib.attn_decode_destroy.restype = I
    lib.attn_decode_schedule_host.argtypes = [I, I, I, I, I, I, P, I, ctypes.POINTER(I), P, P]
    lib.attn_decode_schedule_host.restype = I
    lib.attn_decode_set_grid_limit.argtypes = [P, I]
    lib.attn_decode_set_grid_limit.restype = I
    return lib


_lib = _load()


def _int_array(xs: Optional[Sequence[int]]):
    xs = list(xs or [])
    arr = (ctypes.c_int * max(len(xs), 1))(*xs)
    return arr, len(xs)


# ---------------------------------------------------------------- C ABI, same names

def attn_status_string(status: int) -> str:
    return _lib.attn_status_string(int(status)).decode()


def attn_create(B, Hq, Hkv, S, d_k, dtype, scale, kind, window=0, global_idx=None) -> int:
    """Returns a handle (int); raises AttnError on a non-OK status."""
    h = ctypes.c_void_p()
    g, ng = _int_array(global_idx)
    st = _lib.attn_create(ctypes.byref(h), int(B), int(Hq), int(Hkv), int(S), int(d_k), int(dtype),
                          float(scale), int(kind), int(window), ctypes.cast(g, ctypes.c_void_p) if ng else None, ng)
    if st != ATTN_OK:
        raise AttnError(st, "attn_create")
    return h.value


def attn_forward(handle: int, q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int = 0,
                 stream: int = 0) -> int:
    """Enqueue the forward pass; returns the status (does not raise)."""
    return _lib.attn_forward(handle, q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr or None, stream or None)


def attn_destroy(handle: int) -> int:
    return _lib.attn_destroy(handle)


def attn_poll_device_error(handle: int):
    code = ctypes.c_int(0)
    st = _lib.attn_poll_device_error(handle, ctypes.byref(code))
    return st, code.value


def _float_array(xs):
    xs = [float(x) for x in xs]
    return (ctypes.c_float * max(len(xs), 1))(*xs)


def attn_set_alibi(handle: int, slopes=None) -> int:
    """ALiBi bias -slopes[a] |i - j| on later forwards of this handle (None removes it); returns the status."""
    if slopes is None:
        return _lib.attn_set_alibi(handle, None)
    return _lib.attn_set_alibi(handle, ctypes.cast(_float_array(slopes), ctypes.c_void_p))


def attn_set_watchdog(handle: int, limit_ns: int, withhold: int = 0) -> int:
    return _lib.attn_set_watchdog(handle, int(limit_ns), int(withhold))


def attn_forward_noalloc(B, Hq, Hkv, S, d_k, scale, kind, window, global_idx, q_ptr, k_ptr, v_ptr, o_ptr,
                         lse_ptr=0, stream=0) -> int:
    """The bf16 forward pass without any device allocation (fixed library-owned scratch); returns the status.

    For callers that cannot allocate device memory.  Calls that overlap on the GPU race on the shared
    scratch; the first call on a device should come before any stream capture.
    """
    g, ng = _int_array(global_idx)
    return _lib.attn_forward_noalloc(int(B), int(Hq), int(Hkv), int(S), int(d_k), float(scale), int(kind),
                                     int(window), ctypes.cast(g, ctypes.c_void_p) if ng else None, ng,
                                     q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr or None, stream or None)


def attn_forward_noalloc_poll_error():
    """(status, code): synchronise, read and clear the error word of attn_forward_noalloc's scratch."""
    code = ctypes.c_int(0)
    st = _lib.attn_forward_noalloc_poll_error(ctypes.byref(code))
    return st, code.value


def attn_forward_noalloc_set_watchdog(limit_ns: int, withhold: int = 0) -> int:
    """Test hook: wait limit and V-withholding of attn_forward_noalloc's kernels (process-wide)."""
    return _lib.attn_forward_noalloc_set_watchdog(int(limit_ns), int(withhold))


def attn_selftest_exp2(x_ptr: int, y_ptr: int, n: int, stream: int = 0) -> int:
    """Test hook: the library's FMA-pipe exp2 applied elementwise (device float arrays)."""
    return _lib.attn_selftest_exp2(x_ptr, y_ptr, int(n), stream or None)


def attn_selftest_device_once() -> int:
    """Host-only test hook of the per-device kernel set-up registry (0 = every check held)."""
    return _lib.attn_selftest_device_once()


def attn_schedule_host(B, Hq, Hkv, S, kind, window=0, global_idx=None):
    """Host-only schedule: (items int32 [n, 8], n_first).  Raises AttnError on bad arguments."""
    g, ng = _int_array(global_idx)
    gp = ctypes.cast(g, ctypes.c_void_p) if ng else None
    n, n_first = ctypes.c_int(0), ctypes.c_int(0)
    st = _lib.attn_schedule_host(int(B), int(Hq), int(Hkv), int(S), int(kind), int(window), gp, ng, None, 0,
                                 ctypes.byref(n), ctypes.byref(n_first))
    if st != ATTN_OK:
        raise AttnError(st, "attn_schedule_host")
    items = np.zeros((max(n.value, 1), WORK_INTS), dtype=np.int32)
    st = _lib.attn_schedule_host(int(B), int(Hq), int(Hkv), int(S), int(kind), int(window), gp, ng,
                                 items.ctypes.data_as(ctypes.c_void_p), n.value, ctypes.byref(n),
                                 ctypes.byref(n_first))
    if st != ATTN_OK:
        raise AttnError(st, "attn_schedule_host")
    return items[: n.value], n_first.value


def attn_kv_schedule_host(S, kind, window=0):
    """Backward key-tile schedule (host only): int32 [n, 8].  Raises AttnError."""
    n = ctypes.c_int(0)
    st = _lib.attn_kv_schedule_host(int(S), int(kind), int(window), None, 0, ctypes.byref(n))
    if st != ATTN_OK:
        raise AttnError(st, "attn_kv_schedule_host")
    items = np.zeros((max(n.value, 1), WORK_INTS), dtype=np.int32)
    st = _lib.attn_kv_schedule_host(int(S), int(kind), int(window), items.ctypes.data_as(ctypes.c_void_p), n.value,
                                    ctypes.byref(n))
    if st != ATTN_OK:
        raise AttnError(st, "attn_kv_schedule_host")
    return items[: n.value]


def attn_bwd_lg_lists_host(S, window, globals_idx):
    """The backward's per-tile partner lists under local + global (host only): (list, offsets),
    int32 arrays; entries t | LIST_FULL.  Raises AttnError."""
    g = np.ascontiguousarray(np.asarray(list(globals_idx), dtype=np.int32).reshape(-1))
    gp = g.ctypes.data_as(ctypes.c_void_p) if g.size else None
    n = ctypes.c_int(0)
    st = _lib.attn_bwd_lg_lists_host(int(S), int(window), gp, int(g.size), None, 0, None, ctypes.byref(n))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd_lg_lists_host")
    lst = np.zeros(max(n.value, 1), dtype=np.int32)
    off = np.zeros((S + TILE - 1) // TILE + 1, dtype=np.int32)
    st = _lib.attn_bwd_lg_lists_host(int(S), int(window), gp, int(g.size), lst.ctypes.data_as(ctypes.c_void_p),
                                     n.value, off.ctypes.data_as(ctypes.c_void_p), ctypes.byref(n))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd_lg_lists_host")
    return lst[: n.value], off


def attn_bwd_dq_schedule_host(B, Hq, Hkv, S, d_k, kind, window=0):
    """Work items of the backward's dQ launch (host only): int32 [n, 8].  Raises AttnError."""
    n = ctypes.c_int(0)
    args = (int(B), int(Hq), int(Hkv), int(S), int(d_k), int(kind), int(window))
    st = _lib.attn_bwd_dq_schedule_host(*args, None, 0, ctypes.byref(n))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd_dq_schedule_host")
    items = np.zeros((max(n.value, 1), WORK_INTS), dtype=np.int32)
    st = _lib.attn_bwd_dq_schedule_host(*args, items.ctypes.data_as(ctypes.c_void_p), n.value, ctypes.byref(n))
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd_dq_schedule_host")
    return items[: n.value]


# ---------------------------------------------------------------- decode (key/value cache)

def attn_decode_create(B, Hq, Hkv, S_q, S_cap, d_k, scale, kind, window=0) -> int:
    """Returns a decode handle (int); raises AttnError on a non-OK status."""
    h = ctypes.c_void_p()
    st = _lib.attn_decode_create(ctypes.byref(h), int(B), int(Hq), int(Hkv), int(S_q), int(S_cap), int(d_k),
                                 float(scale), int(kind), int(window))
    if st != ATTN_OK:
        raise AttnError(st, "attn_decode_create")
    return h.value


def attn_decode_forward(handle: int, q_ptr: int, k_ptr: int, v_ptr: int, cache_len, o_ptr: int,
                        lse_ptr: int = 0, stream: int = 0) -> int:
    """Enqueue one decode step (cache_len: host sequence of B ints); returns the status."""
    lens, n = _int_array(cache_len)
    return _lib.attn_decode_forward(handle, q_ptr, k_ptr, v_ptr, ctypes.cast(lens, ctypes.c_void_p), o_ptr,
                                    lse_ptr or None, stream or None)


def attn_decode_poll_device_error(handle: int):
    code = ctypes.c_int(0)
    st = _lib.attn_decode_poll_device_error(handle, ctypes.byref(code))
    return st, code.value


def attn_decode_destroy(handle: int) -> int:
    return _lib.attn_decode_destroy(handle)


def attn_decode_schedule_host(B, Hkv, S_q, S_cap, kind, window, cache_len, n_sm):
    """Host-only decode work split: (n_cta, tile_prefix int32 [B + 1], share int64 [n_cta + 1]).
    CTA k takes the tile-list indices [share[k], share[k + 1]).  Raises AttnError."""
    lens, n = _int_array(cache_len)
    n_cta = ctypes.c_int(0)
    prefix = np.zeros(int(B) + 1, dtype=np.int32)
    share = np.zeros(max(1, int(n_sm)) + 1, dtype=np.int64)
    st = _lib.attn_decode_schedule_host(int(B), int(Hkv), int(S_q), int(S_cap), int(kind), int(window),
                                        ctypes.cast(lens, ctypes.c_void_p), int(n_sm), ctypes.byref(n_cta),
                                        prefix.ctypes.data_as(ctypes.c_void_p),
                                        share.ctypes.data_as(ctypes.c_void_p))
    if st != ATTN_OK:
        raise AttnError(st, "attn_decode_schedule_host")
    return n_cta.value, prefix, share[:n_cta.value + 1].copy()


class DecodeAttention:
    """A decode plan: S_q new query rows per sequence against a key/value cache.

    Q: [B, Hq, S_q, d] bf16; K, V (the cache): [B, Hkv, S_cap, d] bf16; cache_len: B host ints.
    Row i of sequence b sits at position cache_len[b] - S_q + i.  Returns (O like Q, LSE float32
    [B, Hq, S_q]).
    """

    def __init__(self, B, Hq, Hkv, S_q, S_cap, d, scale=None, kind=MASK_CAUSAL, window=0):
        import math
        self.shape = (int(B), int(Hq), int(Hkv), int(S_q), int(S_cap), int(d))
        self.scale = float(scale) if scale is not None else 1.0 / math.sqrt(d)
        self.kind, self.window = int(kind), int(window)
        self.handle = attn_decode_create(B, Hq, Hkv, S_q, S_cap, d, self.scale, self.kind, self.window)

    def close(self):
        if getattr(self, "handle", None):
            attn_decode_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __call__(self, Q, K, V, cache_len, O=None, LSE=None, stream=None, want_lse=True):
        import torch
        B, Hq, Hkv, S_q, S_cap, d = self.shape
        for name, t, shape in (("Q", Q, (B, Hq, S_q, d)), ("K", K, (B, Hkv, S_cap, d)), ("V", V, (B, Hkv, S_cap, d))):
            if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or tuple(t.shape) != shape:
                raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor of shape {shape}")
        if O is None:
            O = torch.empty_like(Q)
        if LSE is None and want_lse:
            LSE = torch.empty((B, Hq, S_q), dtype=torch.float32, device=Q.device)
        if stream is None:
            stream = torch.cuda.current_stream(Q.device)
        st = attn_decode_forward(self.handle, Q.data_ptr(), K.data_ptr(), V.data_ptr(), list(cache_len),
                                 O.data_ptr(), LSE.data_ptr() if LSE is not None else 0, stream.cuda_stream)
        if st != ATTN_OK:
            raise AttnError(st, "attn_decode_forward")
        return O, LSE

    def poll_device_error(self):
        return attn_decode_poll_device_error(self.handle)

    def set_alibi(self, slopes=None):
        """Add the ALiBi score bias -slopes[a] |t - j| (one slope per query head); None removes it."""
        if slopes is None:
            st = _lib.attn_decode_set_alibi(self.handle, None)
        else:
            if len(slopes) != self.shape[1]:
                raise ValueError("one slope per query head")
            st = _lib.attn_decode_set_alibi(self.handle, ctypes.cast(_float_array(slopes), ctypes.c_void_p))
        if st != ATTN_OK:
            raise AttnError(st, "attn_decode_set_alibi")

    def set_grid_limit(self, max_ctas: int):
        """Test hook: at most max_ctas CTAs per launch (long shares on small problems)."""
        st = _lib.attn_decode_set_grid_limit(self.handle, int(max_ctas))
        if st != ATTN_OK:
            raise AttnError(st, "attn_decode_set_grid_limit")

    def launch_count(self) -> int:
        """Kernels the last call enqueued (1, or 2 with the merge kernel)."""
        n = ctypes.c_int(0)
        st = _lib.attn_decode_launch_count(self.handle, ctypes.byref(n))
        if st != ATTN_OK:
            raise AttnError(st, "attn_decode_launch_count")
        return n.value

    def set_merge_mode(self, mode: int):
        """Where split units are merged: 0 auto, 1 in the decode kernel, 2 by the merge kernel."""
        st = _lib.attn_decode_set_merge_mode(self.handle, int(mode))
        if st != ATTN_OK:
            raise AttnError(st, "attn_decode_set_merge_mode")


# ---------------------------------------------------------------- torch convenience

class Attention:
    """A plan (handle) for one problem shape; call with CUDA torch tensors.

    Q: [B, Hq, S, d], K/V: [B, Hkv, S, d], contiguous, bf16 (or fp32 for dtype="f32").
    Returns (O, LSE) with O like Q and LSE float32 [B, Hq, S].
    """

    def __init__(self, B, Hq, Hkv, S, d, dtype="bf16", scale=None, kind=MASK_CAUSAL, window=0,
                 global_idx=None):
        import math
        self.shape = (int(B), int(Hq), int(Hkv), int(S), int(d))
        self.dtype = dtype
        self.scale = float(scale) if scale is not None else 1.0 / math.sqrt(d)
        self.kind, self.window = int(kind), int(window)
        self.global_idx = list(global_idx or [])
        code = {"bf16": ATTN_BF16, "f32": ATTN_F32, "e4m3": ATTN_FP8_E4M3}[dtype]
        self.handle = attn_create(B, Hq, Hkv, S, d, code, self.scale, self.kind, self.window, self.global_idx)

    def close(self):
        if getattr(self, "handle", None):
            attn_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __call__(self, Q, K, V, O=None, LSE=None, stream=None, want_lse=True):
        import torch
        B, Hq, Hkv, S, d = self.shape
        tdt = {"bf16": torch.bfloat16, "f32": torch.float32, "e4m3": torch.float8_e4m3fn}[self.dtype]
        for name, t, h in (("Q", Q, Hq), ("K", K, Hkv), ("V", V, Hkv)):
            if not t.is_cuda or t.dtype != tdt or not t.is_contiguous() or tuple(t.shape) != (B, h, S, d):
                raise ValueError(f"{name} must be a contiguous CUDA {tdt} tensor of shape {(B, h, S, d)}")
        if O is None:
            O = torch.empty(Q.shape, dtype=torch.bfloat16 if self.dtype == "e4m3" else Q.dtype, device=Q.device)
        if LSE is None and want_lse:
            LSE = torch.empty((B, Hq, S), dtype=torch.float32, device=Q.device)
        if stream is None:
            stream = torch.cuda.current_stream(Q.device)
        st = attn_forward(self.handle, Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(),
                          LSE.data_ptr() if LSE is not None else 0, stream.cuda_stream)
        if st != ATTN_OK:
            raise AttnError(st, "attn_forward")
        return O, LSE

    def poll_device_error(self):
        return attn_poll_device_error(self.handle)

    def set_watchdog(self, limit_ns: int, withhold: int = 0):
        st = attn_set_watchdog(self.handle, limit_ns, withhold)
        if st != ATTN_OK:
            raise AttnError(st, "attn_set_watchdog")

    def backward(self, Q, K, V, O, LSE, dO, dQ=None, dK=None, dV=None, stream=None):
        """Gradients (dQ, dK, dV) of this plan's forward for the output gradient dO (bf16 tensors;
        O and LSE from the forward call)."""
        import torch
        if dQ is None:
            dQ = torch.empty_like(Q)
        if dK is None:
            dK = torch.empty_like(K)
        if dV is None:
            dV = torch.empty_like(V)
        for name, t in (("O", O), ("dO", dO), ("dQ", dQ)):
            if t.shape != Q.shape or t.dtype != Q.dtype or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous tensor like Q")
        if stream is None:
            stream = torch.cuda.current_stream(Q.device)
        st = _lib.attn_backward(self.handle, Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), LSE.data_ptr(),
                                dO.data_ptr(), dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(), stream.cuda_stream)
        if st != ATTN_OK:
            raise AttnError(st, "attn_backward")
        return dQ, dK, dV

    def set_fp8_descale(self, descale_q: float, descale_k: float, descale_v: float):
        """Per-tensor factors of E4M3 inputs (real value = factor x stored value)."""
        st = _lib.attn_set_fp8_descale(self.handle, float(descale_q), float(descale_k), float(descale_v))
        if st != ATTN_OK:
            raise AttnError(st, "attn_set_fp8_descale")

    def set_alibi(self, slopes=None):
        """Add the ALiBi score bias -slopes[a] |i - j| (one slope per query head); None removes it."""
        if slopes is not None and len(slopes) != self.shape[1]:
            raise ValueError("one slope per query head")
        st = attn_set_alibi(self.handle, slopes)
        if st != ATTN_OK:
            raise AttnError(st, "attn_set_alibi")

    def set_bias(self, bias=None):
        """Add a bias matrix b_ij to the scores: a CUDA bf16 tensor [Bb, Hb, S, ld] (Bb in {1, B},
        Hb in {1, Hq}, ld >= S a multiple of 8; a 3-D [Hb, S, ld] or 2-D [S, ld] tensor is taken as
        Bb = 1 / Hb = 1).  The tensor is kept referenced by the plan; None removes the bias."""
        if bias is None:
            st = _lib.attn_set_bias(self.handle, None, 0, 0, 0)
            self._bias = None
        else:
            import torch
            t = bias
            while t.dim() < 4:
                t = t.unsqueeze(0)
            if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
                raise ValueError("bias must be a contiguous CUDA bf16 tensor")
            Bb, Hb, S, ld = t.shape
            if S != self.shape[3]:
                raise ValueError("bias rows must be the sequence length")
            st = _lib.attn_set_bias(self.handle, t.data_ptr(), int(Bb), int(Hb), int(ld))
            self._bias = t if st == ATTN_OK else None
        if st != ATTN_OK:
            raise AttnError(st, "attn_set_bias")
