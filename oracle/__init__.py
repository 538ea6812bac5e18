"""Plain CPU oracle for the tiled contraction D = A @ B.T and its data moves.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  The CUDA
library and its Python binding never import it, and it imports nothing from
them: the two sides share no code, only the seeded input generators.

Contents, each following the page it cites (TVM TIRx documentation):

* ``gemm_bf16`` / ``gemm_mxfp8`` / ``gemm_mxfp4`` / ``gemm_nvfp4`` -- float64
  triple loop in ``tg_oracle.c`` ("tcgen05.mma", section "Examples": B stored
  as (N, K), result a @ b.T; block scaling from section "Weight-stationary
  and block scaling", with .scale_vec::1X / 2X / 4X).
* ``transpose_b16`` -- out[j, i] = in[i, j] on raw 16-bit patterns.
* ``ldmatrix_image`` -- the register image of ``ldmatrix.m8n8.xN[.trans]``
  ("ldmatrix / stmatrix", sections "Address providers and result owners"
  and "Parameterized layouts").
* ``ldmatrix_address_row`` -- which row address each lane supplies.
* ``swizzle128`` -- the 128-byte swizzle permutation ("Explicit CUDA tile
  patterns", section "Shared matrix descriptors").
* ``tmem_register_coord`` -- the tcgen05.ld/st register images ("Explicit
  CUDA tile patterns", section "TMEM transfers").
* ``add_one`` -- the elementwise example ("Tile Operands and Execution").
* ``apply_epilogue`` -- the fused elementwise epilogues (``silu_affine`` from
  "Explicit CUDA tile patterns", section "Scalar compositions"; a constant; a
  per-column bias), in float64 on the float64 contraction.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tg_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libtgoracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``tg_oracle.c`` with gcc (OpenMP, no fast-math) and return the path."""
    if not force and os.path.exists(_LIB_PATH) and (
        os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    ):
        return _LIB_PATH
    os.makedirs(_BUILD_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = [
        "gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
        "-fno-fast-math", "-std=c11", "-o", tmp, _SRC, "-lm",
    ]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, dp = ctypes.c_int64, ctypes.c_void_p
        lib.tgo_bf16_to_f64.restype = ctypes.c_double
        lib.tgo_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.tgo_e4m3fn_to_f64.restype = ctypes.c_double
        lib.tgo_e4m3fn_to_f64.argtypes = [ctypes.c_uint8]
        lib.tgo_e8m0_to_f64.restype = ctypes.c_double
        lib.tgo_e8m0_to_f64.argtypes = [ctypes.c_uint8]
        lib.tgo_e2m1_to_f64.restype = ctypes.c_double
        lib.tgo_e2m1_to_f64.argtypes = [ctypes.c_uint8]
        lib.tgo_ue4m3_to_f64.restype = ctypes.c_double
        lib.tgo_ue4m3_to_f64.argtypes = [ctypes.c_uint8]
        for name in ("tgo_decode_bf16", "tgo_decode_e4m3fn", "tgo_decode_e8m0",
                     "tgo_decode_e2m1", "tgo_decode_ue4m3"):
            getattr(lib, name).restype = None
            getattr(lib, name).argtypes = [dp, i64, dp]
        lib.tgo_gemm_bf16.restype = ctypes.c_int
        lib.tgo_gemm_bf16.argtypes = [dp, i64, dp, i64, i64, i64, i64,
                                      ctypes.c_double, dp, i64, dp, i64, dp, dp]
        lib.tgo_gemm_mxfp8.restype = ctypes.c_int
        lib.tgo_gemm_mxfp8.argtypes = [dp, i64, dp, i64, dp, i64, dp, i64,
                                       i64, i64, i64, ctypes.c_double,
                                       dp, i64, dp, i64, dp, dp]
        lib.tgo_gemm_fp4.restype = ctypes.c_int
        lib.tgo_gemm_fp4.argtypes = [dp, i64, dp, i64, dp, i64, dp, i64,
                                     i64, i64, i64, ctypes.c_int, ctypes.c_double,
                                     dp, i64, dp, i64, dp, dp]
        lib.tgo_transpose_b16.restype = ctypes.c_int
        lib.tgo_transpose_b16.argtypes = [dp, i64, dp, i64, i64, i64]
        lib.tgo_num_threads.restype = ctypes.c_int
        lib.tgo_num_threads.argtypes = []
        lib.tgo_set_num_threads.restype = None
        lib.tgo_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().tgo_num_threads())


def set_num_threads(n: int) -> None:
    _load().tgo_set_num_threads(int(n))


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def decode_bf16(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _load().tgo_decode_bf16(_ptr(b), b.size, _ptr(out))
    return out


def decode_e4m3fn(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint8)
    out = np.empty(b.shape, dtype=np.float64)
    _load().tgo_decode_e4m3fn(_ptr(b), b.size, _ptr(out))
    return out


def decode_e8m0(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint8)
    out = np.empty(b.shape, dtype=np.float64)
    _load().tgo_decode_e8m0(_ptr(b), b.size, _ptr(out))
    return out


def decode_e2m1(nibbles: np.ndarray) -> np.ndarray:
    """E2M1 values of the low 4 bits of each byte."""
    b = np.ascontiguousarray(nibbles, dtype=np.uint8)
    out = np.empty(b.shape, dtype=np.float64)
    _load().tgo_decode_e2m1(_ptr(b), b.size, _ptr(out))
    return out


def decode_ue4m3(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint8)
    out = np.empty(b.shape, dtype=np.float64)
    _load().tgo_decode_ue4m3(_ptr(b), b.size, _ptr(out))
    return out


# ---------------------------------------------------------------------------
# The contraction
# ---------------------------------------------------------------------------

def _index_list(idx, bound):
    if idx is None:
        return None, bound
    arr = np.ascontiguousarray(np.asarray(idx, dtype=np.int64).reshape(-1))
    return arr, arr.size


def gemm_bf16(A: np.ndarray, B: np.ndarray, add: float = 0.0, rows=None, cols=None):
    """float64 oracle of D = A @ B.T (+ add) over raw bf16 bit patterns.

    A: uint16 [M, K] (any row stride, unit inner stride); B: uint16 [N, K].
    rows / cols select output rows / columns (default: all).
    Returns (ref, mag), float64 [len(rows), len(cols)], where
    mag = sum_k |a_ik * b_jk| (the tolerance scale).
    """
    A = np.asarray(A)
    B = np.asarray(B)
    if A.dtype != np.uint16 or B.dtype != np.uint16:
        raise TypeError("gemm_bf16 oracle takes uint16 bf16 bit patterns")
    if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[1]:
        raise ValueError("A must be [M, K] and B [N, K]")
    if A.strides[1] != 2:
        A = np.ascontiguousarray(A)
    if B.strides[1] != 2:
        B = np.ascontiguousarray(B)
    M, K = A.shape
    N = B.shape[0]
    r, nr = _index_list(rows, M)
    c, nc = _index_list(cols, N)
    ref = np.empty((nr, nc), dtype=np.float64)
    mag = np.empty((nr, nc), dtype=np.float64)
    rc = _load().tgo_gemm_bf16(_ptr(A), A.strides[0] // 2, _ptr(B), B.strides[0] // 2,
                               M, N, K, float(add), _ptr(r), nr, _ptr(c), nc,
                               _ptr(ref), _ptr(mag))
    if rc != 0:
        raise ValueError(f"tgo_gemm_bf16 rejected its arguments (code {rc})")
    return ref, mag


def gemm_mxfp8(A, B, SFA, SFB, add: float = 0.0, rows=None, cols=None):
    """float64 oracle of the block-scaled product over raw E4M3FN / E8M0 bytes.

    A: uint8 [M, K]; B: uint8 [N, K]; SFA: uint8 [M, K/32]; SFB: uint8 [N, K/32].
    a_ik = e4m3(A_ik) * 2^(SFA[i, k//32] - 127), likewise b; D = a @ b.T (+ add).
    """
    arrs = []
    for X in (A, B, SFA, SFB):
        X = np.asarray(X)
        if X.dtype != np.uint8 or X.ndim != 2:
            raise TypeError("gemm_mxfp8 oracle takes 2-D uint8 arrays")
        if X.strides[1] != 1:
            X = np.ascontiguousarray(X)
        arrs.append(X)
    A, B, SFA, SFB = arrs
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K or K % 32 or SFA.shape != (M, K // 32) or SFB.shape != (N, K // 32):
        raise ValueError("shape mismatch for the block-scaled product")
    r, nr = _index_list(rows, M)
    c, nc = _index_list(cols, N)
    ref = np.empty((nr, nc), dtype=np.float64)
    mag = np.empty((nr, nc), dtype=np.float64)
    rc = _load().tgo_gemm_mxfp8(_ptr(A), A.strides[0], _ptr(B), B.strides[0],
                                _ptr(SFA), SFA.strides[0], _ptr(SFB), SFB.strides[0],
                                M, N, K, float(add), _ptr(r), nr, _ptr(c), nc,
                                _ptr(ref), _ptr(mag))
    if rc != 0:
        raise ValueError(f"tgo_gemm_mxfp8 rejected its arguments (code {rc})")
    return ref, mag


FP4_MX, FP4_NV = 0, 1     # scale kinds: E8M0 per 32 (MXFP4), UE4M3 per 16 (NVFP4)


def gemm_fp4(A, B, SFA, SFB, scale_kind: int, add: float = 0.0, rows=None, cols=None):
    """float64 oracle of the block-scaled FP4 product over raw bytes.

    A: uint8 [M, K/2] packed E2M1 (element 2i in the low nibble of byte i);
    B: uint8 [N, K/2].  scale_kind FP4_MX: SFA uint8 [M, K/32] E8M0;
    FP4_NV: SFA uint8 [M, K/16] UE4M3 (SFB likewise).
    a_ik = e2m1(A_ik) * scale(SFA[i, k // block]), likewise b; D = a @ b.T (+ add).
    """
    block = {FP4_MX: 32, FP4_NV: 16}[scale_kind]
    arrs = []
    for X in (A, B, SFA, SFB):
        X = np.asarray(X)
        if X.dtype != np.uint8 or X.ndim != 2:
            raise TypeError("gemm_fp4 oracle takes 2-D uint8 arrays")
        if X.strides[1] != 1:
            X = np.ascontiguousarray(X)
        arrs.append(X)
    A, B, SFA, SFB = arrs
    M, K = A.shape[0], 2 * A.shape[1]
    N = B.shape[0]
    if B.shape[1] != K // 2 or K % block or SFA.shape != (M, K // block) or \
            SFB.shape != (N, K // block):
        raise ValueError("shape mismatch for the block-scaled FP4 product")
    r, nr = _index_list(rows, M)
    c, nc = _index_list(cols, N)
    ref = np.empty((nr, nc), dtype=np.float64)
    mag = np.empty((nr, nc), dtype=np.float64)
    rc = _load().tgo_gemm_fp4(_ptr(A), A.strides[0], _ptr(B), B.strides[0],
                              _ptr(SFA), SFA.strides[0], _ptr(SFB), SFB.strides[0],
                              M, N, K, int(scale_kind), float(add), _ptr(r), nr, _ptr(c), nc,
                              _ptr(ref), _ptr(mag))
    if rc != 0:
        raise ValueError(f"tgo_gemm_fp4 rejected its arguments (code {rc})")
    return ref, mag


def gemm_mxfp4(A, B, SFA, SFB, add: float = 0.0, rows=None, cols=None):
    """MXFP4: packed E2M1 operands, one E8M0 scale per 32 K elements."""
    return gemm_fp4(A, B, SFA, SFB, FP4_MX, add, rows, cols)


def gemm_nvfp4(A, B, SFA, SFB, add: float = 0.0, rows=None, cols=None):
    """NVFP4: packed E2M1 operands, one UE4M3 scale per 16 K elements."""
    return gemm_fp4(A, B, SFA, SFB, FP4_NV, add, rows, cols)


def transpose_b16(X: np.ndarray) -> np.ndarray:
    """out[j, i] = X[i, j] on raw 16-bit patterns (plain double loop in C)."""
    X = np.asarray(X)
    if X.dtype != np.uint16 or X.ndim != 2:
        raise TypeError("transpose_b16 oracle takes a 2-D uint16 array")
    if X.strides[1] != 2:
        X = np.ascontiguousarray(X)
    rows, cols = X.shape
    out = np.empty((cols, rows), dtype=np.uint16)
    rc = _load().tgo_transpose_b16(_ptr(X), X.strides[0] // 2, _ptr(out), rows, rows, cols)
    if rc != 0:
        raise ValueError(f"tgo_transpose_b16 rejected its arguments (code {rc})")
    return out


# Epilogue operation codes (the values of the library's C ABI, restated).
EPI_NONE, EPI_ADD_SCALAR, EPI_SILU_AFFINE, EPI_BIAS_COL, EPI_BIAS_COL_SILU = 0, 1, 2, 3, 4
EPI_AFFINE = 5


def silu(x: np.ndarray) -> np.ndarray:
    """silu(x) = x / (1 + exp(-x)), in float64 (the pages' silu_affine body)."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def apply_epilogue(ref: np.ndarray, op: int, alpha: float = 0.0, beta: float = 0.0,
                   bias=None, cols=None) -> np.ndarray:
    """The fused epilogue on a float64 result block ``ref`` [rows, ncols].

    NONE: ref; ADD_SCALAR: ref + alpha; SILU_AFFINE: silu(ref) * alpha + beta;
    BIAS_COL: ref + bias[j]; BIAS_COL_SILU: silu(ref + bias[j]);
    AFFINE: ref * alpha + beta (e.g. a per-tensor scale of NVFP4 operands).  ``bias`` is
    the full per-column vector (length N); ``cols`` lists which columns the
    block holds (default: all, in order).
    """
    ref = np.asarray(ref, dtype=np.float64)
    if op == EPI_NONE:
        return ref.copy()
    if op == EPI_ADD_SCALAR:
        return ref + float(alpha)
    if op == EPI_SILU_AFFINE:
        return silu(ref) * float(alpha) + float(beta)
    if op == EPI_AFFINE:
        return ref * float(alpha) + float(beta)
    if op in (EPI_BIAS_COL, EPI_BIAS_COL_SILU):
        b = np.asarray(bias, dtype=np.float64)
        b = b if cols is None else b[np.asarray(cols)]
        x = ref + b[None, :]
        return x if op == EPI_BIAS_COL else silu(x)
    raise ValueError(f"unknown epilogue op {op}")


def add_one(a: np.ndarray) -> np.ndarray:
    """The elementwise example of "Tile Operands and Execution": B = A + 1."""
    return np.asarray(a) + np.asarray(a).dtype.type(1)


# ---------------------------------------------------------------------------
# Layout models (pure Python, tiny inputs)
# ---------------------------------------------------------------------------

def swizzle128(offset: int) -> int:
    """Byte offset after the 128B swizzle (descriptor mode 3 / TMA swizzle 3).

    "Explicit CUDA tile patterns", section "Shared matrix descriptors": mode 3
    permutes a byte offset as offset ^ ((offset >> 3) & 112).
    """
    return offset ^ ((offset >> 3) & 112)


def ldmatrix_address_row(lane: int, n: int) -> tuple[int, int]:
    """(matrix, row) whose shared address lane ``lane`` supplies for an .xN issue.

    "ldmatrix / stmatrix", section "Code generation": lane l supplies row l % 8
    of matrix (l // 8) % N; the first 8*N lanes are the real providers.
    """
    return (lane // 8) % n, lane % 8


def ldmatrix_image(shared_matrix: np.ndarray, trans: bool = False) -> np.ndarray:
    """Register words received by each lane from ``ldmatrix.m8n8.xN[.trans].b16``.

    shared_matrix: uint16 [N, 8, 8] -- matrix i, row j, 16-bit column c.
    Returns uint32 [32, N]: entry [l, i] is the word of matrix i that lane l
    owns.  Register word (i, j, w) belongs to lane 4*j + w ("Address
    providers and result owners"); its two halves h = 0 (low 16 bits) and
    h = 1 (high) are register_image[i, j, 2w+h], which equals
    shared_matrix[i, j, 2w+h] without .trans and shared_matrix[i, 2w+h, j]
    with .trans ("Parameterized layouts").
    """
    sm = np.asarray(shared_matrix, dtype=np.uint16)
    n = sm.shape[0]
    if sm.shape != (n, 8, 8) or n not in (1, 2, 4):
        raise ValueError("shared_matrix must be [N, 8, 8] with N in {1, 2, 4}")
    out = np.zeros((32, n), dtype=np.uint32)
    for i in range(n):
        for j in range(8):
            for w in range(4):
                halves = []
                for h in range(2):
                    if trans:
                        halves.append(int(sm[i, 2 * w + h, j]))
                    else:
                        halves.append(int(sm[i, j, 2 * w + h]))
                out[4 * j + w, i] = halves[0] | (halves[1] << 16)
    return out


def stmatrix_image(registers: np.ndarray, trans: bool = False) -> np.ndarray:
    """Shared matrices written by ``stmatrix.m8n8.xN[.trans].b16``.

    The inverse of ``ldmatrix_image``: registers uint32 [32, N] (lane l's
    word i) -> uint16 [N, 8, 8].  stmatrix "uses the corresponding register
    image as input and each provider's shared row address as output".
    """
    reg = np.asarray(registers, dtype=np.uint32)
    n = reg.shape[1]
    sm = np.zeros((n, 8, 8), dtype=np.uint16)
    for i in range(n):
        for j in range(8):
            for w in range(4):
                word = int(reg[4 * j + w, i])
                for h in range(2):
                    half = (word >> (16 * h)) & 0xFFFF
                    if trans:
                        sm[i, 2 * w + h, j] = half
                    else:
                        sm[i, j, 2 * w + h] = half
    return sm


def tmem_register_coord(shape: str, lane: int, reg: int) -> tuple[int, int]:
    """(row, column) of TMEM that register ``reg`` of lane ``lane`` maps to.

    "Explicit CUDA tile patterns", section "TMEM transfers", for the four
    tcgen05.ld/st shapes, within the executing warp's 32-lane slab.
    """
    l, r = lane, reg
    if shape == "32x32b":
        return l, r
    if shape == "16x64b":
        return l // 4 + 8 * (l % 2), l // 2 % 2 + 2 * r
    if shape == "16x128b":
        return l // 4 + 8 * (r % 2), l % 4 + 4 * (r // 2)
    if shape == "16x256b":
        return l // 4 + 8 * (r // 2 % 2), r % 2 + 2 * (l % 4) + 8 * (r // 4)
    raise ValueError(f"unknown tcgen05.ld shape {shape!r}")


def tmem_register_coord_16x32bx2(lane: int, reg: int, split_lanes: int,
                                 split_cols: int) -> tuple[int, int]:
    """(row, column) of TMEM for tcgen05.ld .16x32bx2, relative to the first
    access region's base, when the second region starts ``split_lanes`` lanes
    and ``split_cols`` columns further (imm_half_splitoff = split_lanes << 16 |
    split_cols).

    "Explicit CUDA tile patterns", section "TMEM transfers": lane l owns
    (access l // 16, row l % 16, column r); each access region is 16 rows by
    N columns and the second is offset by the immediate alone (no implicit
    sixteen-row offset).
    """
    access, row = divmod(lane, 16)
    if access == 0:
        return row, reg
    return split_lanes + row, split_cols + reg


def block_scale_tmem_slot(row: int, sf: int = 0, replica: int = 0) -> tuple[int, int]:
    """(TMEM lane, byte column) holding scale ``sf`` of scale row ``row``.

    "tcgen05.mma", section "Weight-stationary and block scaling": scale row r
    uses lane r % 32 and byte-column 4 * (r // 32) + sf, with four replicas
    spaced 32 lanes apart (``replica`` 0..3 selects one).
    """
    if not 0 <= replica < 4:
        raise ValueError("four replicas, 32 lanes apart")
    return 32 * replica + row % 32, 4 * (row // 32) + sf
