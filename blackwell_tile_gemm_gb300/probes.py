"""Python binding of the probe kernels declared in include/tgemm_probes.h
(``_build/libtgemm_probes.so``, which links against libtgemm.so).

Each probe runs one of the pages' worked examples, or dumps one hardware
mapping, in a single CTA; the tests compare the results with the oracle.  The
rate probe and the SM occupier are measurement and test aids.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _PKG, _check, _stream_handle, lib

PROBE_LIB_PATH = os.path.join(_PKG, "_build", "libtgemm_probes.so")
_ready = False
_plib = None
_plock = threading.Lock()


def _L():
    global _ready, _plib
    lib()                       # the library the probes link against, loaded first
    with _plock:
        if _plib is None:
            if not os.path.exists(PROBE_LIB_PATH):
                raise RuntimeError(f"{PROBE_LIB_PATH} is missing: build with "
                                   "`python -m blackwell_tile_gemm_gb300.build`")
            _plib = ctypes.CDLL(PROBE_LIB_PATH)
    L = _plib
    if not _ready:
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        for name, args in {
            "tg_probe_add_one_v4": [vp, vp, vp],
            "tg_probe_ldmatrix_x2_interleaved": [vp, vp, vp],
            "tg_probe_ldmatrix": [vp, i32, i32, vp, vp],
            "tg_probe_stmatrix": [vp, i32, i32, vp, vp],
            "tg_probe_tma_two_boxes": [vp, vp, vp],
            "tg_probe_tma_swizzle128": [vp, i32, vp, vp],
            "tg_probe_mma_128x64x64": [vp, vp, vp, vp],
            "tg_probe_mma_ws_128x64x64": [vp, vp, vp, vp],
            "tg_probe_wait_timeout": [ctypes.c_uint64, vp],
            "tg_probe_mma_rate": [i32, i32, i32, vp, vp],
            "tg_probe_tmem_shapes": [vp, vp],
            "tg_probe_hold_sms": [i32, ctypes.c_uint64, vp],
        }.items():
            f = getattr(L, name)
            f.restype = i32
            f.argtypes = args
        _ready = True
    return L


def add_one_v4(a, b, stream=None):
    _check(_L().tg_probe_add_one_v4(a.data_ptr(), b.data_ptr(), _stream_handle(stream)),
           "tg_probe_add_one_v4")


def ldmatrix_x2_interleaved(x, out, stream=None):
    _check(_L().tg_probe_ldmatrix_x2_interleaved(x.data_ptr(), out.data_ptr(),
                                                 _stream_handle(stream)),
           "tg_probe_ldmatrix_x2_interleaved")


def ldmatrix(img, n, trans, out, stream=None):
    _check(_L().tg_probe_ldmatrix(img.data_ptr(), int(n), int(trans), out.data_ptr(),
                                  _stream_handle(stream)), "tg_probe_ldmatrix")


def stmatrix(regs, n, trans, out, stream=None):
    _check(_L().tg_probe_stmatrix(regs.data_ptr(), int(n), int(trans), out.data_ptr(),
                                  _stream_handle(stream)), "tg_probe_stmatrix")


def tma_two_boxes(a, out, stream=None):
    _check(_L().tg_probe_tma_two_boxes(a.data_ptr(), out.data_ptr(), _stream_handle(stream)),
           "tg_probe_tma_two_boxes")


def tma_swizzle128(src, rows, out, stream=None):
    _check(_L().tg_probe_tma_swizzle128(src.data_ptr(), int(rows), out.data_ptr(),
                                        _stream_handle(stream)), "tg_probe_tma_swizzle128")


def mma_128x64x64(a, b, out, stream=None):
    _check(_L().tg_probe_mma_128x64x64(a.data_ptr(), b.data_ptr(), out.data_ptr(),
                                       _stream_handle(stream)), "tg_probe_mma_128x64x64")


def tmem_shapes(out, stream=None):
    """TMEM cells per register for five tcgen05.ld shapes; out: int32 CUDA [5, 128, 8]."""
    _check(_L().tg_probe_tmem_shapes(out.data_ptr(), _stream_handle(stream)),
           "tg_probe_tmem_shapes")


def mma_ws_128x64x64(a, b, out, stream=None):
    _check(_L().tg_probe_mma_ws_128x64x64(a.data_ptr(), b.data_ptr(), out.data_ptr(),
                                          _stream_handle(stream)), "tg_probe_mma_ws_128x64x64")


def wait_timeout(timeout_ns, stream=None):
    _check(_L().tg_probe_wait_timeout(int(timeout_ns), _stream_handle(stream)),
           "tg_probe_wait_timeout")


def mma_rate(kind, iters, ctas, cycles, stream=None):
    """Back-to-back tcgen05.mma rate probe; cycles: int64 CUDA tensor [2*ctas] (cycles, ns)."""
    _check(_L().tg_probe_mma_rate(int(kind), int(iters), int(ctas), cycles.data_ptr(),
                                  _stream_handle(stream)), "tg_probe_mma_rate")


def hold_sms(blocks, ns, stream=None):
    """Occupy `blocks` SMs for `ns` nanoseconds (a test aid, see tgemm_probes.h)."""
    _check(_L().tg_probe_hold_sms(int(blocks), int(ns), _stream_handle(stream)),
           "tg_probe_hold_sms")
