"""ctypes binding of libdash.so (C ABI in include/dash.h).

Argument marshalling only: every step of the backward pass runs in the
library's CUDA kernels.  Tensors are torch CUDA tensors (device memory and
streams come from PyTorch); the library fails loudly if it is missing.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from .inputs import SCHEDULE_IDS

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdash.so")

OK, ERR_ARG, ERR_CUDA, ERR_LAUNCH, ERR_TIMEOUT, ERR_DEADLOCK, ERR_NOMEM, ERR_DEVICE = 0, -1, -2, -3, -4, -5, -6, -7
ERR_SCRATCH = -8
_NAMES = {0: "DASH_OK", -1: "DASH_ERR_ARG", -2: "DASH_ERR_CUDA", -3: "DASH_ERR_LAUNCH", -4: "DASH_ERR_TIMEOUT",
          -5: "DASH_ERR_DEADLOCK", -6: "DASH_ERR_NOMEM", -7: "DASH_ERR_DEVICE", -8: "DASH_ERR_SCRATCH"}

EXPORTS = (
    "dash_attn_bwd_preprocess", "dash_attn_bwd", "dash_dq_finalize", "dash_get_status", "dash_set_timeout_ns",
    "dash_release_workspaces", "dash_num_ctas", "dash_sim_schedule", "dash_sim_check_ranks",
    "dash_attn_bwd_debug", "dash_debug_tile_probe", "dash_attn_bwd_noalloc", "dash_select_schedule",
    "dash_attn_fwd", "dash_sim_schedule_band", "dash_attn_bwd_window", "dash_attn_fwd_window",
    "dash_sim_schedule_cross", "dash_attn_bwd_cross", "dash_attn_fwd_cross", "dash_head_split", "dash_key_blocks",
    "dash_noalloc_init", "dash_get_status_noalloc",
)


class DashError(RuntimeError):
    def __init__(self, code, what):
        super().__init__("%s failed: %s (%d)" % (what, _NAMES.get(code, "?"), code))
        self.code = code


class _DebugOpts(ctypes.Structure):
    _fields_ = [("order_log", ctypes.c_void_p), ("dq_partials", ctypes.c_void_p), ("cta_perm", ctypes.c_void_p),
                ("start_delay_ns", ctypes.c_void_p), ("ranks_host", ctypes.c_void_p),
                ("skip_table_check", ctypes.c_int), ("kernel_event_begin", ctypes.c_void_p),
                ("kernel_event_end", ctypes.c_void_p), ("wait_cycles", ctypes.c_void_p),
                ("event_trace", ctypes.c_void_p), ("window", ctypes.c_int), ("skv", ctypes.c_int),
                ("head_split", ctypes.c_int)]


_lib = None


def lib():
    """Load libdash.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libdash.so is not built (run: python -m tile_scheduling_persistent_gb300.build)")
    L = ctypes.CDLL(LIB_PATH)
    P, I, Z, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_double
    L.dash_attn_bwd_preprocess.argtypes = [P, P, P, I, I, I, I, P]
    L.dash_attn_bwd.argtypes = [P] * 9 + [I] * 7 + [P]
    L.dash_attn_bwd_debug.argtypes = [P] * 9 + [I] * 7 + [P, ctypes.POINTER(_DebugOpts)]
    L.dash_attn_bwd_noalloc.argtypes = [P] * 9 + [I] * 7 + [P]
    L.dash_dq_finalize.argtypes = [P, P, Z, P]
    L.dash_get_status.argtypes = [P, ctypes.POINTER(I), ctypes.POINTER(I)]
    L.dash_get_status_noalloc.argtypes = [P, ctypes.POINTER(I), ctypes.POINTER(I)]
    L.dash_noalloc_init.argtypes = []
    L.dash_set_timeout_ns.argtypes = [ctypes.c_uint64]
    L.dash_release_workspaces.argtypes = []
    L.dash_num_ctas.argtypes = [I, ctypes.POINTER(I)]
    L.dash_sim_schedule.argtypes = [I] * 7 + [D, D, ctypes.POINTER(D), P, ctypes.POINTER(ctypes.c_int64)]
    L.dash_sim_schedule_band.argtypes = [I] * 7 + [D, D, ctypes.POINTER(D), P, ctypes.POINTER(ctypes.c_int64)]
    L.dash_sim_schedule_cross.argtypes = [I] * 7 + [D, D, ctypes.POINTER(D), P, ctypes.POINTER(ctypes.c_int64)]
    L.dash_sim_check_ranks.argtypes = [I] * 7 + [P]
    L.dash_debug_tile_probe.argtypes = [P] * 6 + [I, I] + [P] * 7
    for name in EXPORTS:
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _check(rc, what):
    if rc != OK:
        raise DashError(rc, what)


def _sched(schedule):
    return SCHEDULE_IDS[schedule] if isinstance(schedule, str) else int(schedule)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t, dtype=None):
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "expected a contiguous CUDA tensor"
    if dtype is not None:
        assert t.dtype == dtype, "expected %s, got %s" % (dtype, t.dtype)
    return ctypes.c_void_p(t.data_ptr())


def attn_bwd_preprocess(o, do, delta, stream=None):
    B, H, S, D = o.shape
    _check(lib().dash_attn_bwd_preprocess(_ptr(o, torch.bfloat16), _ptr(do, torch.bfloat16),
                                          _ptr(delta, torch.float32), B, H, S, D, _stream(stream)),
           "dash_attn_bwd_preprocess")


def _bwd_args(q, k, v, o, do, lse, dq, dk, dv, causal, schedule):
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    bf, f32 = torch.bfloat16, torch.float32
    return [_ptr(q, bf), _ptr(k, bf), _ptr(v, bf), _ptr(o, bf), _ptr(do, bf), _ptr(lse, f32), _ptr(dq, f32),
            _ptr(dk, bf), _ptr(dv, bf), B, Hq, Hkv, S, D, int(bool(causal)), _sched(schedule)]


def attn_bwd(q, k, v, o, do, lse, dq, dk, dv, causal, schedule, stream=None, window=None):
    """dq (fp32 accumulator, zeroed by the library), dk, dv (bf16) <- backward.
    window: causal sliding window in tokens (needs causal=True), or None.
    k/v (and dk/dv) may be longer or shorter than q (full mask only)."""
    if k.shape[2] != q.shape[2]:
        assert not causal and window is None, "different lengths need a full mask"
        args = _bwd_args(q, k, v, o, do, lse, dq, dk, dv, causal, schedule)
        args[-3:-2] = [k.shape[2], q.shape[3]]   # (..., Sq, D, causal, sched) -> (..., Sq, Skv, D, sched)
        del args[-2]
        _check(lib().dash_attn_bwd_cross(*args, _stream(stream)), "dash_attn_bwd_cross")
        return
    if window is not None:
        assert causal, "a sliding window needs a causal mask"
        args = _bwd_args(q, k, v, o, do, lse, dq, dk, dv, causal, schedule)
        args[-2] = int(window)   # the causal flag's slot carries the window
        _check(lib().dash_attn_bwd_window(*args, _stream(stream)), "dash_attn_bwd_window")
        return
    _check(lib().dash_attn_bwd(*_bwd_args(q, k, v, o, do, lse, dq, dk, dv, causal, schedule), _stream(stream)),
           "dash_attn_bwd")


def attn_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, causal, schedule, stream=None):
    """attn_bwd for callers that cannot allocate: library scratch comes from a
    fixed device array (see dash_attn_bwd_noalloc in include/dash.h)."""
    _check(lib().dash_attn_bwd_noalloc(*_bwd_args(q, k, v, o, do, lse, dq, dk, dv, causal, schedule),
                                       _stream(stream)), "dash_attn_bwd_noalloc")


def noalloc_init():
    """Set-up of attn_bwd_noalloc on the current device (scratch address, kernels loaded)."""
    _check(lib().dash_noalloc_init(), "dash_noalloc_init")


def get_status_noalloc(stream=None):
    """(code, info) of the last attn_bwd_noalloc on the current device; synchronizes `stream`."""
    code = ctypes.c_int(0)
    info = (ctypes.c_int * 4)()
    _check(lib().dash_get_status_noalloc(_stream(stream), ctypes.byref(code), info), "dash_get_status_noalloc")
    return code.value, list(info)


def attn_bwd_debug(q, k, v, o, do, lse, dq, dk, dv, causal, schedule, stream=None, order_log=None,
                   dq_partials=None, cta_perm=None, start_delay_ns=None, ranks_host=None, skip_table_check=False,
                   kernel_events=None, wait_cycles=None, event_trace=None, window=None, head_split=None):
    """head_split: None (the library decides), True (one task per query head)
    or False (one task per key/value head group)."""
    opts = _DebugOpts()
    opts.window = int(window) if window is not None else 0
    opts.head_split = 0 if head_split is None else (1 if head_split else 2)
    opts.skv = int(k.shape[2]) if k.shape[2] != q.shape[2] else 0
    opts.wait_cycles = _ptr(wait_cycles, torch.int64)
    opts.event_trace = _ptr(event_trace, torch.int64)
    if kernel_events is not None:
        opts.kernel_event_begin = ctypes.c_void_p(kernel_events[0].cuda_event)
        opts.kernel_event_end = ctypes.c_void_p(kernel_events[1].cuda_event)
    opts.order_log = _ptr(order_log, torch.int32)
    opts.dq_partials = _ptr(dq_partials, torch.float32)
    opts.cta_perm = _ptr(cta_perm, torch.int32)
    opts.start_delay_ns = _ptr(start_delay_ns, torch.int64)
    keep = None
    if ranks_host is not None:
        keep = np.ascontiguousarray(ranks_host, dtype=np.uint16)
        opts.ranks_host = keep.ctypes.data_as(ctypes.c_void_p)
    opts.skip_table_check = int(bool(skip_table_check))
    rc = lib().dash_attn_bwd_debug(*_bwd_args(q, k, v, o, do, lse, dq, dk, dv, causal, schedule),
                                   _stream(stream), ctypes.byref(opts))
    if keep is not None:
        torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
    _check(rc, "dash_attn_bwd_debug")


def dq_finalize(dq_accum, dq, stream=None):
    assert dq_accum.numel() == dq.numel()
    _check(lib().dash_dq_finalize(_ptr(dq_accum, torch.float32), _ptr(dq, torch.bfloat16), dq.numel(),
                                  _stream(stream)), "dash_dq_finalize")


def get_status(stream=None):
    code = ctypes.c_int(0)
    info = (ctypes.c_int * 4)()
    _check(lib().dash_get_status(_stream(stream), ctypes.byref(code), info), "dash_get_status")
    return code.value, list(info)


def set_timeout_ns(ns):
    _check(lib().dash_set_timeout_ns(int(ns)), "dash_set_timeout_ns")


def release_workspaces():
    _check(lib().dash_release_workspaces(), "dash_release_workspaces")


def attn_fwd(q, k, v, o, lse, causal, stream=None, window=None):
    """o (bf16 [B,Hq,S,D]) and lse (fp32 [B,Hq,S], natural log) <- forward.
    window: causal sliding window in tokens (needs causal=True), or None."""
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    bf = torch.bfloat16
    ptrs = (_ptr(q, bf), _ptr(k, bf), _ptr(v, bf), _ptr(o, bf), _ptr(lse, torch.float32))
    if k.shape[2] != S:
        assert not causal and window is None, "different lengths need a full mask"
        _check(lib().dash_attn_fwd_cross(*ptrs, B, Hq, Hkv, S, k.shape[2], D, _stream(stream)), "dash_attn_fwd_cross")
        return
    if window is not None:
        assert causal, "a sliding window needs a causal mask"
        _check(lib().dash_attn_fwd_window(*ptrs, B, Hq, Hkv, S, D, int(window), _stream(stream)),
               "dash_attn_fwd_window")
        return
    _check(lib().dash_attn_fwd(*ptrs, B, Hq, Hkv, S, D, int(bool(causal)), _stream(stream)), "dash_attn_fwd")


def select_schedule(B, Hq, Hkv, S, D, causal):
    """Name of the deterministic schedule that schedule="auto" runs for this shape."""
    rc = lib().dash_select_schedule(B, Hq, Hkv, S, D, int(bool(causal)))
    _check(rc if rc < 0 else 0, "dash_select_schedule")
    return {v: k for k, v in SCHEDULE_IDS.items()}[rc]


def head_split(schedule, causal, B, Hq, Hkv, S, D, P, window=None, Skv=None):
    """True if the backward of this shape runs one task per query head (see
    dash_head_split); its accumulation order is then that of Hkv = Hq."""
    rc = lib().dash_head_split(_sched(schedule), int(bool(causal)), B, Hq, Hkv, S, D, int(window or 0),
                               int(Skv or 0), int(P))
    _check(rc if rc < 0 else 0, "dash_head_split")
    return rc == 1


def key_blocks(B, Hq, Hkv, Sq, Skv):
    """The number of key blocks the backward with key length Skv != Sq cuts
    the keys into (see dash_key_blocks); 1 = no split."""
    rc = lib().dash_key_blocks(int(B), int(Hq), int(Hkv), int(Sq), int(Skv))
    _check(rc if rc < 0 else 0, "dash_key_blocks")
    return rc


def task_heads(schedule, causal, B, Hq, Hkv, S, D, P, window=None, Skv=None):
    """The Hkv to simulate a backward run with: Hq when its tasks are split per
    query head, else Hkv."""
    return Hq if head_split(schedule, causal, B, Hq, Hkv, S, D, P, window, Skv) else Hkv


def num_ctas(device=None):
    dev = torch.cuda.current_device() if device is None else int(device)
    P = ctypes.c_int(0)
    _check(lib().dash_num_ctas(dev, ctypes.byref(P)), "dash_num_ctas")
    return P.value


def sim_schedule(schedule, causal, B, Hq, Hkv, n, P, c=1.0, r=1.0, turn_order=True, band=None, nkv=None):
    """Host DAG simulator: (makespan, turn order [B*Hq*n, nkv] or None, tasks).
    band: tile diagonals of a causal sliding window (None: no window);
    nkv: key/value tiles per head when they differ from n (full masks only)."""
    mk = ctypes.c_double(0.0)
    nt = ctypes.c_int64(0)
    nk = n if nkv is None else int(nkv)
    out = np.empty((B * Hq * n, nk), dtype=np.int32) if turn_order else None
    optr = out.ctypes.data_as(ctypes.c_void_p) if out is not None else None
    if nkv is not None:
        assert not causal and band is None, "S_q != S_kv needs a full mask"
        rc = lib().dash_sim_schedule_cross(_sched(schedule), B, Hq, Hkv, n, nk, P, float(c), float(r),
                                           ctypes.byref(mk), optr, ctypes.byref(nt))
    elif band is None:
        rc = lib().dash_sim_schedule(_sched(schedule), int(bool(causal)), B, Hq, Hkv, n, P, float(c), float(r),
                                     ctypes.byref(mk), optr, ctypes.byref(nt))
    else:
        assert causal, "a band needs a causal mask"
        rc = lib().dash_sim_schedule_band(_sched(schedule), B, Hq, Hkv, n, int(band), P, float(c), float(r),
                                          ctypes.byref(mk), optr, ctypes.byref(nt))
    _check(rc, "dash_sim_schedule")
    return mk.value, out, nt.value


def sim_check_ranks(schedule, causal, B, Hq, Hkv, n, P, ranks):
    arr = np.ascontiguousarray(ranks, dtype=np.uint16)
    return lib().dash_sim_check_ranks(_sched(schedule), int(bool(causal)), B, Hq, Hkv, n, P,
                                      arr.ctypes.data_as(ctypes.c_void_p))


def tile_probe(k, v, q, do, lse, delta, diag=False):
    """One pair through the kernel's building blocks; returns fp32 intermediates."""
    D = k.shape[-1]
    dev = k.device
    f = lambda *s: torch.empty(*s, dtype=torch.float32, device=dev)  # noqa: E731
    out = {name: f(128, 128) for name in ("sT", "pT", "dpT", "dsT")}
    out.update({name: f(128, D) for name in ("dv", "dk", "dq")})
    bf = torch.bfloat16
    _check(lib().dash_debug_tile_probe(_ptr(k, bf), _ptr(v, bf), _ptr(q, bf), _ptr(do, bf),
                                       _ptr(lse, torch.float32), _ptr(delta, torch.float32), D, int(bool(diag)),
                                       *[_ptr(out[n]) for n in ("sT", "pT", "dpT", "dsT", "dv", "dk", "dq")]),
           "dash_debug_tile_probe")
    return out
