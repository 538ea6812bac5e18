"""GB300-native tiled GEMM (D = A @ B.T) -- Python binding of libtgemm.so.

The binding only marshals arguments: it passes device pointers, row strides,
sizes and the current CUDA stream to the C entry points declared in
``include/tgemm.h``; every step of the computation runs in the library's
CUDA kernels.  PyTorch provides device memory and streams.  There is no
fallback: if the library is not built, the first call raises.

Entry points (same names as the C ABI):

* ``gemm_bf16(A, B, D=None, ...)``                -- bf16 x bf16 -> f32 / bf16
* ``gemm_mxfp8_blockscaled(A, B, SFA, SFB, ...)`` -- E4M3 x E8M0/32 -> f32 / bf16
* ``tile_transpose_b16(X, out=None)``             -- 16-bit transpose, bit-exact
* ``tg_device_status(stream=None)``               -- device-side error record
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libtgemm.so")

TG_OK = 0
TG_ERR_INVALID_ARG = 1
TG_ERR_MISALIGNED = 2
TG_ERR_UNSUPPORTED = 3
TG_ERR_CUDA = 4
TG_ERR_TIMEOUT = 5
TG_ERR_NO_SCRATCH = 6
TG_ERR_WORKSPACE = 7
TG_D_F32 = 0
TG_D_BF16 = 1
TG_EPI_NONE = 0
TG_EPI_ADD_SCALAR = 1
TG_EPI_SILU_AFFINE = 2
TG_EPI_BIAS_COL = 3
TG_EPI_BIAS_COL_SILU = 4
TG_EPI_AFFINE = 5
TG_FLAG_CTA_PAIR = 1
TG_FLAG_MULTICAST = 2
TG_FLAG_GATHER_TMA = 4
TG_CALL_GEMM_BF16 = 0
TG_CALL_GEMM_MXFP8 = 1
TG_CALL_GEMM_MXFP4 = 2
TG_CALL_GEMM_NVFP4 = 3
TG_CALL_GEMM_BF16_SKINNY = 4
TG_CALL_GEMM_BF16_GATHER = 5
TG_CLOCK_BF16 = 0
TG_CLOCK_MXFP8 = 1
TG_CLOCK_MXFP4 = 2
TG_CLOCK_NVFP4 = 3

_lock = threading.Lock()
_lib = None


class tg_epilogue(ctypes.Structure):
    """The C ABI's epilogue description (include/tgemm.h)."""
    _fields_ = [("op", ctypes.c_int), ("alpha", ctypes.c_float), ("beta", ctypes.c_float),
                ("bias", ctypes.c_void_p)]


# The no-op epilogue, shared (the C calls only read it).
_EPI_NONE = tg_epilogue(0, 0.0, 0.0, None)


class TgError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        msg = status_string(code) if _lib is not None else str(code)
        detail = ""
        if code == TG_ERR_CUDA and _lib is not None:
            detail = f" (cudaError {_lib.tg_last_cuda_error()})"
        super().__init__(f"{what}: {msg}{detail} [status {code}]")


def lib() -> ctypes.CDLL:
    """The loaded libtgemm.so (raises if it has not been built)."""
    global _lib
    L = _lib
    if L is not None:
        return L
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m blackwell_tile_gemm_gb300.build` "
                "(the package has no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint
        L.gemm_bf16.restype = i32
        L.gemm_bf16.argtypes = [vp, i64, vp, i64, vp, i64, i64, i64, i64, i32, i32,
                                ctypes.c_float, u32, vp]
        L.gemm_mxfp8_blockscaled.restype = i32
        L.gemm_mxfp8_blockscaled.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, vp, i64,
                                             i64, i64, i64, i32, i32, ctypes.c_float, u32, vp]
        L.gemm_bf16_ex.restype = i32
        L.gemm_bf16_ex.argtypes = [vp, i64, vp, i64, vp, i64, i64, i64, i64, i32,
                                   ctypes.POINTER(tg_epilogue), u32, vp]
        L.gemm_mxfp8_blockscaled_ex.restype = i32
        L.gemm_mxfp8_blockscaled_ex.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, vp, i64,
                                                i64, i64, i64, i32, ctypes.POINTER(tg_epilogue),
                                                u32, vp]
        L.gemm_bf16_skinny.restype = i32
        L.gemm_bf16_skinny.argtypes = [vp, i64, vp, i64, vp, i64, i64, i64, i64, i32,
                                       ctypes.POINTER(tg_epilogue), i32, vp]
        L.gemm_bf16_gather.restype = i32
        L.gemm_bf16_gather.argtypes = [vp, i64, i64, vp, i64, vp, i64, vp, i64, i64, i64, i32,
                                       ctypes.POINTER(tg_epilogue), u32, vp]
        L.tg_gemm_tail_split.restype = i32
        L.tg_gemm_tail_split.argtypes = [i64, i64, i64, u32]
        L.tg_gemm_multicast.restype = i32
        L.tg_gemm_multicast.argtypes = [vp, vp, i64, i64, i64, u32]
        L.tg_workspace_bytes.restype = i64
        L.tg_workspace_bytes.argtypes = [i32, i64, i64, i64, i64, i64, i32, i32, u32]
        L.tg_reserve_workspace.restype = i32
        L.tg_reserve_workspace.argtypes = [vp, i64]
        L.tg_workspace_alloc_count.restype = ctypes.c_uint64
        L.tg_workspace_alloc_count.argtypes = []
        L.tg_gemm_repitch.restype = i32
        L.tg_gemm_repitch.argtypes = [i64, i64, i64, i64, i64, u32]
        L.tg_skinny_split_count.restype = i32
        L.tg_skinny_split_count.argtypes = [i64, i64, i32]
        for name in ("gemm_mxfp4_blockscaled", "gemm_nvfp4_blockscaled"):
            getattr(L, name).restype = i32
            getattr(L, name).argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, i64, i64,
                                         i64, i32, ctypes.POINTER(tg_epilogue), u32, vp]
        L.gemm_mxfp8_blockscaled_noalloc.restype = i32
        L.gemm_mxfp8_blockscaled_noalloc.argtypes = list(L.gemm_mxfp8_blockscaled.argtypes)
        L.tile_transpose_b16.restype = i32
        L.tile_transpose_b16.argtypes = [vp, i64, vp, i64, i64, i64, vp]
        L.tg_device_status.restype = i32
        L.tg_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        L.tg_kernel_clock_record.restype = i32
        L.tg_kernel_clock_record.argtypes = [i32]
        L.tg_kernel_clock_read.restype = i32
        L.tg_kernel_clock_read.argtypes = [i32, ctypes.POINTER(ctypes.c_double),
                                           ctypes.POINTER(ctypes.c_uint64)]
        L.tg_set_wait_timeout_ns.restype = i32
        L.tg_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
        L.tg_status_string.restype = ctypes.c_char_p
        L.tg_status_string.argtypes = [i32]
        L.tg_last_cuda_error.restype = i32
        L.tg_last_cuda_error.argtypes = []
        L.tg_version.restype = i32
        L.tg_version.argtypes = []
        _lib = L
        return L


def status_string(code: int) -> str:
    return lib().tg_status_string(int(code)).decode()


def _stream_handle(stream):
    import torch
    if stream is None:
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:       # the current stream's handle without a Stream object
            return ctypes.c_void_p(raw(torch.cuda.current_device()))
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int, what: str) -> None:
    if rc != TG_OK:
        raise TgError(rc, what)


def _rows(t, name):
    shape = t.shape
    if len(shape) != 2:
        raise ValueError(f"{name} must be 2-D")
    rows, cols = shape
    st = t.stride()
    if rows > 0 and cols > 0 and st[1] != 1:
        raise ValueError(f"{name} must have unit inner stride")
    return st[0] if rows > 1 else max(cols, 1)


def _ld(t, name, mult):
    """Row stride in elements; a single-row tensor may report any stride."""
    ld = _rows(t, name)
    if t.shape[0] <= 1:
        ld = -(-max(t.shape[1], 1) // mult) * mult
    return ld


def _d_code(dtype):
    import torch
    if dtype == torch.float32:
        return TG_D_F32
    if dtype == torch.bfloat16:
        return TG_D_BF16
    raise ValueError(f"D must be float32 or bfloat16, got {dtype}")


def _flags(cta_pair, multicast):
    return (TG_FLAG_CTA_PAIR if cta_pair else 0) | (TG_FLAG_MULTICAST if multicast else 0)


def make_epilogue(epilogue_add=None, silu_affine=None, bias=None, bias_silu=False,
                  affine=None):
    """Build the C epilogue description from keyword choices (at most one op).

    epilogue_add=s: D = acc + s;  silu_affine=(scale, shift): D = silu(acc) *
    scale + shift;  affine=(scale, shift): D = acc * scale + shift;
    bias=<f32 CUDA tensor [N]>: D = acc + bias[j], or with bias_silu=True
    D = silu(acc + bias[j]).
    """
    if epilogue_add is None and silu_affine is None and bias is None and affine is None:
        return _EPI_NONE
    chosen = [epilogue_add is not None, silu_affine is not None, bias is not None,
              affine is not None]
    if sum(chosen) > 1:
        raise ValueError("choose one epilogue")
    if epilogue_add is not None:
        return tg_epilogue(TG_EPI_ADD_SCALAR, float(epilogue_add), 0.0, None)
    if affine is not None:
        scale, shift = affine
        return tg_epilogue(TG_EPI_AFFINE, float(scale), float(shift), None)
    if silu_affine is not None:
        scale, shift = silu_affine
        return tg_epilogue(TG_EPI_SILU_AFFINE, float(scale), float(shift), None)
    if bias is not None:
        import torch
        if bias.dtype != torch.float32 or bias.dim() != 1 or not bias.is_contiguous():
            raise TypeError("bias must be a contiguous float32 vector")
        return tg_epilogue(TG_EPI_BIAS_COL_SILU if bias_silu else TG_EPI_BIAS_COL, 0.0, 0.0,
                           bias.data_ptr())
    return tg_epilogue(TG_EPI_NONE, 0.0, 0.0, None)


def gemm_bf16(A, B, D=None, *, out_dtype=None, epilogue_add=None, silu_affine=None, bias=None,
              bias_silu=False, affine=None, cta_pair=False, multicast=False, stream=None):
    """D[M,N] = A[M,K] @ B[N,K].T (+ epilogue_add), bf16 inputs, f32 accumulation.

    A, B: CUDA bfloat16 tensors with unit inner stride.  D: optional output
    (float32 or bfloat16, [M, N]); otherwise allocated with ``out_dtype``
    (default float32).  ``cta_pair`` selects the two-CTA (cta_group::2) kernel;
    ``multicast`` runs clusters of two units (single CTAs, or pairs with
    ``cta_pair``) on vertically adjacent tiles that share the B tile.
    Epilogue keywords: see ``make_epilogue``.
    """
    import torch
    M, K = A.shape
    N, K2 = B.shape
    if K2 != K:
        raise ValueError("A is [M, K] and B is [N, K]")
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("gemm_bf16 takes bfloat16 A and B")
    if D is None:
        D = torch.empty((M, N), dtype=out_dtype or torch.float32, device=A.device)
    if tuple(D.shape) != (M, N):
        raise ValueError("D must be [M, N]")
    if bias is not None and bias.shape[0] != N:
        raise ValueError("bias must have N elements")
    epi = make_epilogue(epilogue_add, silu_affine, bias, bias_silu, affine)
    rc = lib().gemm_bf16_ex(A.data_ptr(), _ld(A, "A", 8), B.data_ptr(), _ld(B, "B", 8),
                            D.data_ptr(), _ld(D, "D", 8), M, N, K, _d_code(D.dtype),
                            ctypes.byref(epi), _flags(cta_pair, multicast), _stream_handle(stream))
    _check(rc, "gemm_bf16")
    return D


def gemm_mxfp8_blockscaled(A, B, SFA, SFB, D=None, *, out_dtype=None, epilogue_add=None,
                           silu_affine=None, bias=None, bias_silu=False, affine=None,
                           cta_pair=False, multicast=False, stream=None):
    """Block-scaled MXFP8 product: D = (A * 2^(SFA-127)) @ (B * 2^(SFB-127)).T.

    A: [M, K], B: [N, K] E4M3FN bytes (torch.float8_e4m3fn or uint8); SFA:
    [M, K/32], SFB: [N, K/32] E8M0 bytes (uint8).  D float32 or bfloat16
    (default bfloat16).
    """
    import torch
    M, K = A.shape
    N, K2 = B.shape
    if K2 != K:
        raise ValueError("A is [M, K] and B is [N, K]")
    for name, t in (("A", A), ("B", B), ("SFA", SFA), ("SFB", SFB)):
        if t.element_size() != 1:
            raise TypeError(f"{name} must hold 1-byte elements")
    if tuple(SFA.shape) != (M, K // 32) or tuple(SFB.shape) != (N, K // 32):
        raise ValueError("SFA must be [M, K/32] and SFB [N, K/32]")
    if D is None:
        D = torch.empty((M, N), dtype=out_dtype or torch.bfloat16, device=A.device)
    if tuple(D.shape) != (M, N):
        raise ValueError("D must be [M, N]")
    if bias is not None and bias.shape[0] != N:
        raise ValueError("bias must have N elements")
    epi = make_epilogue(epilogue_add, silu_affine, bias, bias_silu, affine)
    rc = lib().gemm_mxfp8_blockscaled_ex(
        A.data_ptr(), _ld(A, "A", 16), B.data_ptr(), _ld(B, "B", 16),
        SFA.data_ptr(), _ld(SFA, "SFA", 1), SFB.data_ptr(), _ld(SFB, "SFB", 1),
        D.data_ptr(), _ld(D, "D", 8), M, N, K, _d_code(D.dtype), ctypes.byref(epi),
        _flags(cta_pair, multicast), _stream_handle(stream))
    _check(rc, "gemm_mxfp8_blockscaled")
    return D


def gemm_bf16_skinny(A, B, D=None, *, out_dtype=None, epilogue_add=None, silu_affine=None,
                     bias=None, bias_silu=False, affine=None, split_k=0, stream=None):
    """D = A @ B.T (+ epilogue) for few rows of A (1 <= M <= 128).

    Same operands as ``gemm_bf16``; the kernel is built for reading B once
    from HBM (operands swapped, K split into ``split_k`` pieces reduced with
    TMA reduce-add; 0 = automatic).  D float32 or bfloat16 (default float32).
    """
    import torch
    M, K = A.shape
    N, K2 = B.shape
    if K2 != K:
        raise ValueError("A is [M, K] and B is [N, K]")
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("A and B must be bfloat16")
    if D is None:
        D = torch.empty((M, N), dtype=out_dtype or torch.float32, device=A.device)
    if tuple(D.shape) != (M, N):
        raise ValueError("D must be [M, N]")
    if bias is not None and bias.shape[0] != N:
        raise ValueError("bias must have N elements")
    epi = make_epilogue(epilogue_add, silu_affine, bias, bias_silu, affine)
    rc = lib().gemm_bf16_skinny(A.data_ptr(), _ld(A, "A", 8), B.data_ptr(), _ld(B, "B", 8),
                                D.data_ptr(), _ld(D, "D", 8), M, N, K, _d_code(D.dtype),
                                ctypes.byref(epi), int(split_k), _stream_handle(stream))
    _check(rc, "gemm_bf16_skinny")
    return D


def gemm_bf16_gather(A, row_idx, B, D=None, *, out_dtype=None, epilogue_add=None,
                     silu_affine=None, bias=None, bias_silu=False, affine=None, cta_pair=False,
                     gather_tma=False, stream=None):
    """D[i] = A[row_idx[i]] @ B.T (+ epilogue): rows of A gathered by index.

    A: bfloat16 [a_rows, K]; row_idx: int32 CUDA vector [M] (indices outside
    [0, a_rows) give zero rows); B: bfloat16 [N, K].  D float32 or bfloat16
    [M, N] (default float32).  ``gather_tma`` loads the rows inside the GEMM
    with TMA gather4 instead of gathering them into the workspace first.
    """
    import torch
    a_rows, K = A.shape
    N, K2 = B.shape
    if K2 != K:
        raise ValueError("A is [a_rows, K] and B is [N, K]")
    if row_idx.dtype != torch.int32 or row_idx.dim() != 1 or not row_idx.is_contiguous():
        raise TypeError("row_idx must be a contiguous int32 vector")
    M = row_idx.shape[0]
    if D is None:
        D = torch.empty((M, N), dtype=out_dtype or torch.float32, device=A.device)
    if tuple(D.shape) != (M, N):
        raise ValueError("D must be [M, N]")
    if bias is not None and bias.shape[0] != N:
        raise ValueError("bias must have N elements")
    epi = make_epilogue(epilogue_add, silu_affine, bias, bias_silu, affine)
    rc = lib().gemm_bf16_gather(A.data_ptr(), _ld(A, "A", 8), a_rows, row_idx.data_ptr(), M,
                                B.data_ptr(), _ld(B, "B", 8), D.data_ptr(), _ld(D, "D", 8), N, K,
                                _d_code(D.dtype), ctypes.byref(epi),
                                _flags(cta_pair, False) | (TG_FLAG_GATHER_TMA if gather_tma else 0),
                                _stream_handle(stream))
    _check(rc, "gemm_bf16_gather")
    return D


def gemm_tail_split(M: int, N: int, K: int, cta_pair: bool = False) -> int:
    """K pieces per tile of a last, partial wave that gemm_bf16 uses (1: none)."""
    r = lib().tg_gemm_tail_split(int(M), int(N), int(K), TG_FLAG_CTA_PAIR if cta_pair else 0)
    if r < 0:
        raise TgError(-r, "tg_gemm_tail_split")
    return r


def _addr(x):
    """Device address of a tensor, or an integer address as given."""
    return int(x) if isinstance(x, int) else x.data_ptr()


def gemm_multicast(A, B, M: int, N: int, K: int, cta_pair: bool = False,
                   multicast: bool = False) -> bool:
    """Whether gemm_bf16 runs multicast clusters for these operands (tensors or
    raw addresses), sizes and flags; False unless A and B are allocations of
    the current device.  Reads pointer attributes only."""
    r = lib().tg_gemm_multicast(_addr(A), _addr(B), int(M), int(N), int(K),
                                _flags(cta_pair, multicast))
    if r < 0:
        raise TgError(-r, "tg_gemm_multicast")
    return bool(r)


def workspace_bytes(call: int, M: int, N: int, K: int, lda: int = 0, ldb: int = 0,
                    d_dtype: int = TG_D_F32, epi_op: int = TG_EPI_NONE, flags: int = 0) -> int:
    """Stream workspace bytes one call of kind ``call`` (TG_CALL_*) needs."""
    r = lib().tg_workspace_bytes(int(call), int(M), int(N), int(K), int(lda), int(ldb),
                                 int(d_dtype), int(epi_op), int(flags))
    if r < 0:
        raise TgError(int(-r), "tg_workspace_bytes")
    return int(r)


def reserve_workspace(nbytes: int, stream=None) -> None:
    """Allocate the stream's workspace (>= nbytes) and tail scratch now; later
    calls on the stream then neither allocate nor synchronise."""
    _check(lib().tg_reserve_workspace(_stream_handle(stream), int(nbytes)), "tg_reserve_workspace")


def workspace_alloc_count() -> int:
    """Device allocations the library has made since it was loaded."""
    return int(lib().tg_workspace_alloc_count())


def gemm_repitch(M: int, N: int, K: int, lda: int, ldb: int, cta_pair: bool = False,
                 multicast: bool = False) -> int:
    """Operands gemm_bf16 copies to a 128-byte row pitch first (for operands in
    the current device's memory): bit 0 A, bit 1 B."""
    r = lib().tg_gemm_repitch(int(M), int(N), int(K), int(lda), int(ldb),
                              _flags(cta_pair, multicast))
    if r < 0:
        raise TgError(-r, "tg_gemm_repitch")
    return r


def skinny_split_count(N: int, K: int, split_k: int = 0) -> int:
    """K pieces gemm_bf16_skinny uses on the current device."""
    r = lib().tg_skinny_split_count(int(N), int(K), int(split_k))
    if r < 0:
        raise TgError(-r, "tg_skinny_split_count")
    return r


def _gemm_fp4(fn_name, block, A, B, SFA, SFB, D, out_dtype, epi_kw, cta_pair, stream):
    import torch
    M, Kh = A.shape
    N, Kh2 = B.shape
    K = 2 * Kh
    if Kh2 != Kh:
        raise ValueError("A is [M, K/2] and B is [N, K/2] packed bytes")
    for name, t in (("A", A), ("B", B), ("SFA", SFA), ("SFB", SFB)):
        if t.element_size() != 1:
            raise TypeError(f"{name} must hold 1-byte elements")
    if tuple(SFA.shape) != (M, K // block) or tuple(SFB.shape) != (N, K // block):
        raise ValueError(f"SFA must be [M, K/{block}] and SFB [N, K/{block}]")
    if D is None:
        D = torch.empty((M, N), dtype=out_dtype or torch.bfloat16, device=A.device)
    if tuple(D.shape) != (M, N):
        raise ValueError("D must be [M, N]")
    if epi_kw.get("bias") is not None and epi_kw["bias"].shape[0] != N:
        raise ValueError("bias must have N elements")
    epi = make_epilogue(**epi_kw)
    rc = getattr(lib(), fn_name)(
        A.data_ptr(), _ld(A, "A", 16), B.data_ptr(), _ld(B, "B", 16),
        SFA.data_ptr(), _ld(SFA, "SFA", 1), SFB.data_ptr(), _ld(SFB, "SFB", 1),
        D.data_ptr(), _ld(D, "D", 8), M, N, K, _d_code(D.dtype), ctypes.byref(epi),
        _flags(cta_pair, False), _stream_handle(stream))
    _check(rc, fn_name)
    return D


def gemm_mxfp4_blockscaled(A, B, SFA, SFB, D=None, *, out_dtype=None, epilogue_add=None,
                           silu_affine=None, bias=None, bias_silu=False, affine=None,
                           cta_pair=False, stream=None):
    """Block-scaled MXFP4 product: D = (a * 2^(SFA-127)) @ (b * 2^(SFB-127)).T.

    A: [M, K/2], B: [N, K/2] uint8 of packed FP4 E2M1 (element 2i in the low
    nibble of byte i); SFA: [M, K/32], SFB: [N, K/32] E8M0 bytes.  D float32
    or bfloat16 (default bfloat16).  Epilogue keywords: see ``make_epilogue``.
    """
    return _gemm_fp4("gemm_mxfp4_blockscaled", 32, A, B, SFA, SFB, D, out_dtype,
                     dict(epilogue_add=epilogue_add, silu_affine=silu_affine, bias=bias,
                          bias_silu=bias_silu, affine=affine), cta_pair, stream)


def gemm_nvfp4_blockscaled(A, B, SFA, SFB, D=None, *, out_dtype=None, epilogue_add=None,
                           silu_affine=None, bias=None, bias_silu=False, affine=None,
                           cta_pair=False, stream=None):
    """Block-scaled NVFP4 product: D = (a * ue4m3(SFA)) @ (b * ue4m3(SFB)).T.

    A, B: packed E2M1 as for ``gemm_mxfp4_blockscaled``; SFA: [M, K/16],
    SFB: [N, K/16] UE4M3 bytes (sign bit clear).  A per-tensor scale goes in
    ``affine=(scale, 0.0)``.
    """
    return _gemm_fp4("gemm_nvfp4_blockscaled", 16, A, B, SFA, SFB, D, out_dtype,
                     dict(epilogue_add=epilogue_add, silu_affine=silu_affine, bias=bias,
                          bias_silu=bias_silu, affine=affine), cta_pair, stream)


def gemm_mxfp8_blockscaled_noalloc(A, B, SFA, SFB, D, *, epilogue_add=None, cta_pair=False,
                                   multicast=False, stream=None):
    """``gemm_mxfp8_blockscaled`` for callers that must not allocate device memory.

    Same arguments and result, except that D must be supplied (this call
    allocates nothing, not even its output).  The scale rearrangement uses a
    fixed 8 MiB scratch array built into the library instead of an allocated
    workspace; problems that need more raise TgError(TG_ERR_NO_SCRATCH).
    Calls that may overlap on the GPU share that scratch and race.
    """
    M, K = A.shape
    N = B.shape[0]
    if tuple(D.shape) != (M, N):
        raise ValueError("D must be [M, N]")
    epi = TG_EPI_NONE if epilogue_add is None else TG_EPI_ADD_SCALAR
    rc = lib().gemm_mxfp8_blockscaled_noalloc(
        A.data_ptr(), _ld(A, "A", 16), B.data_ptr(), _ld(B, "B", 16),
        SFA.data_ptr(), _ld(SFA, "SFA", 1), SFB.data_ptr(), _ld(SFB, "SFB", 1),
        D.data_ptr(), _ld(D, "D", 8), M, N, K, _d_code(D.dtype), epi,
        float(epilogue_add or 0.0), _flags(cta_pair, multicast), _stream_handle(stream))
    _check(rc, "gemm_mxfp8_blockscaled_noalloc")
    return D


def tile_transpose_b16(X, out=None, *, stream=None):
    """out[j, i] = X[i, j] for any 16-bit dtype (bits moved unchanged)."""
    import torch
    rows, cols = X.shape
    if X.element_size() != 2:
        raise TypeError("tile_transpose_b16 moves 16-bit elements")
    if out is None:
        out = torch.empty((cols, rows), dtype=X.dtype, device=X.device)
    if tuple(out.shape) != (cols, rows) or out.element_size() != 2:
        raise ValueError("out must be [cols, rows] of a 16-bit dtype")
    rc = lib().tile_transpose_b16(X.data_ptr(), _ld(X, "X", 8), out.data_ptr(),
                                  _ld(out, "out", 8), rows, cols, _stream_handle(stream))
    _check(rc, "tile_transpose_b16")
    return out


def tg_device_status(stream=None):
    """Synchronise the stream; return (status, site) and clear the record."""
    site = ctypes.c_uint32(0)
    rc = lib().tg_device_status(_stream_handle(stream), ctypes.byref(site))
    return int(rc), int(site.value)


def kernel_clock_record(enable: bool = True) -> None:
    """Start (clearing the sums) or stop recording the SM clock of the GEMM
    kernels on the current device; synchronises the device."""
    _check(lib().tg_kernel_clock_record(1 if enable else 0), "tg_kernel_clock_record")


def kernel_clock_read(kind: int):
    """(average SM MHz, MMA units) of the recorded launches of `kind`
    (TG_CLOCK_BF16, _MXFP8, _MXFP4, _NVFP4); synchronises the device."""
    mhz = ctypes.c_double(0.0)
    units = ctypes.c_uint64(0)
    _check(lib().tg_kernel_clock_read(int(kind), ctypes.byref(mhz), ctypes.byref(units)),
           "tg_kernel_clock_read")
    return float(mhz.value), int(units.value)


def tg_set_wait_timeout_ns(ns: int) -> None:
    _check(lib().tg_set_wait_timeout_ns(int(ns)), "tg_set_wait_timeout_ns")
