"""Seeded synthetic inputs for the GEMM and transpose workloads.

This module is shared by the tests, the benchmark and the smoke check; it
holds no arithmetic of the contraction itself, only sampling and the
rounding of sampled float32 values into the stored formats (bfloat16,
FP8 E4M3FN, E8M0 scale bytes).  It imports neither the CUDA binding nor the
oracle.

Every workload draws from ``numpy.random.default_rng(seed)``; the recipes:

=====  ========================================================================
name   recipe
=====  ========================================================================
tiny   M=N=128, K=256; A, B ~ U[-1, 1) -> bf16; fp32 D            (seed 1)
sq4k   M=N=K=4096; A, B ~ N(0, 1) -> bf16; bf16 D                 (seed 2)
sq8k   M=N=K=8192; A, B ~ N(0, 1)/sqrt(8192) -> bf16; fp32 D      (seed 3)
mx8k   M=N=K=8192; A, B = E4M3(clamp(N(0, 1), +-448)); SFA, SFB bytes
       127 + U{-4..4} (scale 2^U{-4..4}) per 32 K elements; bf16 D (seed 4)
ragged M=4000, N=3000, K=1000; A, B ~ U[-1, 1) -> bf16; D = A B^T + 1,
       fp32 D                                                      (seed 5)
tr8k   8192 x 8192 random 16-bit patterns (NaN patterns included)  (seed 6)
=====  ========================================================================
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


# ---------------------------------------------------------------------------
# Rounding sampled float32 values into the stored formats
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); uint16 bits.

    Inputs are finite samples; NaN/Inf handling is not needed here.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_e4m3fn_bits(x: np.ndarray) -> np.ndarray:
    """Round to FP8 E4M3FN (nearest, ties to even), saturating at +-448; uint8 bits.

    Normal numbers: value = (1 + f/8) * 2^(e-7), e in 1..15 (e=15,f=7 is NaN);
    subnormals: value = f/8 * 2^-6.
    """
    v = np.clip(np.asarray(x, dtype=np.float64), -448.0, 448.0)
    sign = (v < 0) | ((v == 0) & np.signbit(v))
    a = np.abs(v)
    code = np.zeros(a.shape, dtype=np.int64)
    sub = a < 2.0 ** -6
    # Subnormal range: quantum 2^-9; a result of 8 quanta is the smallest
    # normal, whose code (exponent field 1, fraction 0) is also 8.
    code[sub] = np.rint(a[sub] / 2.0 ** -9).astype(np.int64)
    nrm = ~sub
    mant, expo = np.frexp(a[nrm])          # a = mant * 2^expo, mant in [0.5, 1)
    e = expo - 1                           # a = (2*mant) * 2^e, 2*mant in [1, 2)
    q = np.rint((2.0 * mant - 1.0) * 8.0).astype(np.int64)
    carry = q == 8
    e = e + carry
    q = np.where(carry, 0, q)
    code[nrm] = ((e + 7) << 3) | q
    return (code | (sign.astype(np.int64) << 7)).astype(np.uint8)


# ---------------------------------------------------------------------------
# Samplers
# ---------------------------------------------------------------------------

def bf16_uniform(rng: np.random.Generator, shape, lo=-1.0, hi=1.0) -> np.ndarray:
    return f32_to_bf16_bits(rng.uniform(lo, hi, size=shape).astype(np.float32))


def bf16_normal(rng: np.random.Generator, shape, scale=1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return f32_to_bf16_bits(x)


def bf16_quarter_integers(rng: np.random.Generator, shape) -> np.ndarray:
    """randint(-4, 5) / 4, exact in bf16 (the data of the tcgen05.mma example)."""
    return f32_to_bf16_bits((rng.integers(-4, 5, size=shape) / 4).astype(np.float32))


def e4m3_normal(rng: np.random.Generator, shape) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return f32_to_e4m3fn_bits(x)


def e8m0_scales(rng: np.random.Generator, shape, lo=-4, hi=4) -> np.ndarray:
    """E8M0 bytes 127 + U{lo..hi}, i.e. scales 2^U{lo..hi}."""
    return (127 + rng.integers(lo, hi + 1, size=shape)).astype(np.uint8)


# E2M1 magnitudes by 3-bit code (exponent bias 1, one fraction bit).
_E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def f32_to_e2m1_codes(x: np.ndarray) -> np.ndarray:
    """Round to FP4 E2M1 (nearest, ties to the even code), saturating at +-6;
    one 4-bit code per uint8 (sign in bit 3).  NaN encodes as 0."""
    x = np.asarray(x, dtype=np.float32)
    # The code of |x| is the number of midpoints between neighbouring
    # magnitudes that lie below |x|; on an exact midpoint (between codes c and
    # c+1) the even code wins.  All midpoints are multiples of 1/4, so with
    # q = 4|x| (exact) and j = floor(q) the count comes from small tables.
    q = np.minimum(np.abs(x), np.float32(6.0)) * np.float32(4.0)
    q = np.where(np.isnan(q), np.float32(0.0), q)     # E2M1 has no NaN: encode 0
    j = q.astype(np.int32)
    exact = q == j
    mid_q = ((_E2M1_MAGNITUDES[:-1] + _E2M1_MAGNITUDES[1:]) * 2).astype(np.int32)
    grid = np.arange(25)
    cnt_le = (mid_q[None, :] <= grid[:, None]).sum(1).astype(np.uint8)
    cnt_lt = (mid_q[None, :] < grid[:, None]).sum(1).astype(np.uint8)
    is_mid = np.isin(grid, mid_q)
    c = np.where(exact, cnt_lt[j], cnt_le[j])
    best = (c + (exact & is_mid[j] & (c % 2 == 1))).astype(np.uint8)
    sign = (np.signbit(x) & (best != 0)).astype(np.uint8)
    return (sign << 3) | best


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """[rows, K] 4-bit codes -> [rows, K/2] bytes, element 2i in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    if c.shape[-1] % 2:
        raise ValueError("K must be even")
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """Inverse of pack_e2m1."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def e2m1_normal_packed(rng: np.random.Generator, shape, sigma: float = 2.0) -> np.ndarray:
    """Packed E2M1 of N(0, sigma^2) samples; shape is the unpacked [rows, K]."""
    x = rng.standard_normal(size=shape, dtype=np.float32) * np.float32(sigma)
    return pack_e2m1(f32_to_e2m1_codes(x))


def ue4m3_pow2_scales(rng: np.random.Generator, shape, lo=-3, hi=3) -> np.ndarray:
    """UE4M3 bytes of 2^U{lo..hi} (exact in E4M3: exponent field 7 + u, fraction 0)."""
    return ((7 + rng.integers(lo, hi + 1, size=shape)) << 3).astype(np.uint8)


def b16_bits(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    kind: str          # "bf16", "skinny", "gather", "mxfp8", "mxfp4", "nvfp4", "transpose"
    M: int
    N: int
    K: int
    seed: int
    d_dtype: str       # "f32" or "bf16" (GEMM output)
    epi_add: float     # epilogue constant (0: plain product)
    cta_pair: bool     # launch with cta_group::2 pairs
    describe: str
    multicast: bool = False   # clusters of two MMA units sharing B by TMA multicast

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K if self.kind != "transpose" else 0


WORKLOADS = {
    "tiny": Workload("tiny", "bf16", 128, 128, 256, 1, "f32", 0.0, False,
                     "bf16 GEMM 128x128x256, U[-1,1) inputs, fp32 D"),
    "sq4k": Workload("sq4k", "bf16", 4096, 4096, 4096, 2, "bf16", 0.0, False,
                     "bf16 GEMM 4096^3, N(0,1) inputs, bf16 D, 128x256 tiles"),
    "sq8k": Workload("sq8k", "bf16", 8192, 8192, 8192, 3, "f32", 0.0, True,
                     "bf16 GEMM 8192^3, N(0,1)/sqrt(K) inputs, fp32 D, CTA pairs"),
    "mx8k": Workload("mx8k", "mxfp8", 8192, 8192, 8192, 4, "bf16", 0.0, True,
                     "MXFP8 GEMM 8192^3, E4M3 x E8M0/32 inputs, bf16 D"),
    "ragged": Workload("ragged", "bf16", 4000, 3000, 1000, 5, "f32", 1.0, True,
                       "bf16 GEMM 4000x3000x1000 + 1, U[-1,1) inputs, fp32 D, "
                       "multicast clusters of two CTA pairs", multicast=True),
    "tr8k": Workload("tr8k", "transpose", 8192, 8192, 0, 6, "b16", 0.0, False,
                     "b16 transpose 8192x8192, random bit patterns"),
    "sk16_8k": Workload("sk16_8k", "skinny", 16, 8192, 8192, 9, "bf16", 0.0, False,
                        "skinny bf16 GEMM 16x8192x8192 (B read once from HBM), bf16 D"),
    "sk64_8k": Workload("sk64_8k", "skinny", 64, 8192, 8192, 10, "bf16", 0.0, False,
                        "skinny bf16 GEMM 64x8192x8192, bf16 D"),
    "moe_8k": Workload("moe_8k", "gather", 4096, 8192, 8192, 11, "bf16", 0.0, True,
                       "gathered-row bf16 GEMM: 4096 of 16384 rows of A (sorted random) x "
                       "8192x8192 B, bf16 D, CTA pairs"),
    "mxf4_8k": Workload("mxf4_8k", "mxfp4", 8192, 8192, 8192, 7, "bf16", 0.0, True,
                        "MXFP4 GEMM 8192^3, E2M1 x E8M0/32 inputs, bf16 D"),
    "nvf4_8k": Workload("nvf4_8k", "nvfp4", 8192, 8192, 8192, 8, "bf16", 0.0, True,
                        "NVFP4 GEMM 8192^3, E2M1 x UE4M3/16 inputs, bf16 D"),
}


def make_inputs(w: Workload | str, M: int | None = None, N: int | None = None,
                K: int | None = None, seed: int | None = None) -> dict:
    """Host (numpy) inputs of a workload; sizes/seed may be overridden.

    bf16:      {"A": uint16 [M,K], "B": uint16 [N,K]}
    mxfp8:     {"A": uint8 [M,K], "B": uint8 [N,K], "SFA": uint8 [M,K/32],
                "SFB": uint8 [N,K/32]}
    mxfp4:     {"A": uint8 [M,K/2] packed E2M1, "B": uint8 [N,K/2],
                "SFA": uint8 [M,K/32] E8M0, "SFB": uint8 [N,K/32]}
    nvfp4:     as mxfp4 with "SFA": uint8 [M,K/16] UE4M3, "SFB": uint8 [N,K/16]
    gather:    {"A": uint16 [4M,K], "B": uint16 [N,K], "idx": int32 [M] rows of A}
    transpose: {"X": uint16 [M,N]}
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    M = w.M if M is None else M
    N = w.N if N is None else N
    K = w.K if K is None else K
    rng = np.random.default_rng(w.seed if seed is None else seed)
    if w.kind == "transpose":
        return {"X": b16_bits(rng, (M, N))}
    if w.kind == "mxfp8":
        return {
            "A": e4m3_normal(rng, (M, K)),
            "B": e4m3_normal(rng, (N, K)),
            "SFA": e8m0_scales(rng, (M, K // 32)),
            "SFB": e8m0_scales(rng, (N, K // 32)),
        }
    if w.kind == "mxfp4":
        return {
            "A": e2m1_normal_packed(rng, (M, K)),
            "B": e2m1_normal_packed(rng, (N, K)),
            "SFA": e8m0_scales(rng, (M, K // 32), -3, 3),
            "SFB": e8m0_scales(rng, (N, K // 32), -3, 3),
        }
    if w.kind == "nvfp4":
        return {
            "A": e2m1_normal_packed(rng, (M, K)),
            "B": e2m1_normal_packed(rng, (N, K)),
            "SFA": ue4m3_pow2_scales(rng, (M, K // 16)),
            "SFB": ue4m3_pow2_scales(rng, (N, K // 16)),
        }
    if w.kind == "gather":
        # M rows gathered from an A of 4M rows (a sorted random subset, the
        # order in which a router's token list usually arrives)
        return {"A": bf16_normal(rng, (4 * M, K), 1.0 / math.sqrt(K)),
                "B": bf16_normal(rng, (N, K)),
                "idx": np.sort(rng.choice(4 * M, M, replace=False)).astype(np.int32)}
    if w.kind == "skinny":
        return {"A": bf16_normal(rng, (M, K), 1.0 / math.sqrt(K)), "B": bf16_normal(rng, (N, K))}
    if w.name in ("tiny", "ragged"):
        return {"A": bf16_uniform(rng, (M, K)), "B": bf16_uniform(rng, (N, K))}
    if w.name == "sq8k":
        s = 1.0 / math.sqrt(K)
        return {"A": bf16_normal(rng, (M, K), s), "B": bf16_normal(rng, (N, K), s)}
    return {"A": bf16_normal(rng, (M, K)), "B": bf16_normal(rng, (N, K))}
