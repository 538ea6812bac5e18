"""Pins of the CPU oracle against facts other than itself (no GPU needed).

Each test checks the oracle against an independent route: exact rational
arithmetic, integer arithmetic, a library bit cast, closed-form special
cases (identity, one-hot, power-of-two scaling), or the worked examples the
pages print (fixtures under tests/golden/).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from blackwell_tile_gemm_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
BF16_ONE = 0x3F80


def _bf16_exact(bits):
    """Exact value of bf16 bits via a float32 bit cast (independent of the oracle)."""
    f = synth.bf16_bits_to_f32(np.asarray(bits, dtype=np.uint16))
    return [[Fraction(float(v)) for v in row] for row in np.atleast_2d(f)]


def _e4m3_exact_via_torch(bits):
    torch = pytest.importorskip("torch")
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits,value", [
    (0x3F80, 1.0), (0xBFC0, -1.5), (0x4000, 2.0), (0x3E80, 0.25),
    (0x7F7F, (2 - 2 ** -7) * 2.0 ** 127), (0x0080, 2.0 ** -126),
    (0x0001, 2.0 ** -133), (0x007F, 127 * 2.0 ** -133),
])
def test_bf16_known_values(oracle, bits, value):
    assert oracle.decode_bf16(np.array([bits]))[0] == value


def test_bf16_specials(oracle):
    v = oracle.decode_bf16(np.array([0x8000, 0x7F80, 0xFF80, 0x7FC0, 0xFFFF], dtype=np.uint16))
    assert v[0] == 0.0 and math.copysign(1.0, v[0]) == -1.0
    assert v[1] == math.inf and v[2] == -math.inf
    assert math.isnan(v[3]) and math.isnan(v[4])


def test_bf16_all_patterns_match_bitcast(oracle):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    mine = oracle.decode_bf16(bits)
    with np.errstate(invalid="ignore"):
        lib = synth.bf16_bits_to_f32(bits).astype(np.float64)
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], lib[~nan])
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(lib[~nan]))


@pytest.mark.parametrize("bits,value", [
    (0x38, 1.0), (0xB8, -1.0), (0x7E, 448.0), (0xFE, -448.0), (0x01, 2.0 ** -9),
    (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6), (0x78, 256.0), (0x3C, 1.5), (0x30, 0.5),
])
def test_e4m3_known_values(oracle, bits, value):
    assert oracle.decode_e4m3fn(np.array([bits], dtype=np.uint8))[0] == value


def test_e4m3_specials(oracle):
    v = oracle.decode_e4m3fn(np.array([0x7F, 0xFF, 0x80, 0x00], dtype=np.uint8))
    assert math.isnan(v[0]) and math.isnan(v[1])
    assert v[2] == 0.0 and math.copysign(1.0, v[2]) == -1.0 and v[3] == 0.0
    finite = oracle.decode_e4m3fn(np.arange(256, dtype=np.uint32).astype(np.uint8))
    assert np.isnan(finite).sum() == 2   # only S.1111.111; E4M3FN has no infinities


def test_e4m3_all_patterns_match_torch(oracle):
    bits = np.arange(256, dtype=np.uint32).astype(np.uint8)
    mine = oracle.decode_e4m3fn(bits)
    lib = _e4m3_exact_via_torch(bits)
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], lib[~nan])


def test_e8m0_values(oracle):
    v = oracle.decode_e8m0(np.array([127, 0, 254, 130, 120, 255], dtype=np.uint8))
    assert list(v[:5]) == [1.0, 2.0 ** -127, 2.0 ** 127, 8.0, 2.0 ** -7]
    assert math.isnan(v[5])


# ---------------------------------------------------------------------------
# the bf16 contraction
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 1, 0), (3, 5, 7, 1), (8, 8, 8, 2), (4, 9, 33, 3)])
def test_gemm_bf16_matches_exact_rationals(oracle, M, N, K, seed):
    rng = np.random.default_rng(seed)
    # Mixed magnitudes so that rounding order would matter if it were wrong.
    A = synth.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32)
                               * np.float32(2.0) ** rng.integers(-20, 20, (M, K)).astype(np.float32))
    B = synth.f32_to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32))
    ref, mag = oracle.gemm_bf16(A, B)
    a, b = _bf16_exact(A), _bf16_exact(B)
    for i in range(M):
        for j in range(N):
            exact = sum((a[i][k] * b[j][k] for k in range(K)), Fraction(0))
            emag = sum((abs(a[i][k] * b[j][k]) for k in range(K)), Fraction(0))
            bound = K * 2.0 ** -52 * float(emag)
            assert abs(Fraction(ref[i, j]) - exact) <= Fraction(bound)
            assert abs(Fraction(mag[i, j]) - emag) <= Fraction(bound)


def test_gemm_bf16_quarter_integers_are_exact(oracle):
    rng = np.random.default_rng(0)
    M, N, K = 37, 29, 300
    qa = rng.integers(-4, 5, (M, K))
    qb = rng.integers(-4, 5, (N, K))
    A = synth.f32_to_bf16_bits((qa / 4).astype(np.float32))
    B = synth.f32_to_bf16_bits((qb / 4).astype(np.float32))
    ref, mag = oracle.gemm_bf16(A, B)
    assert np.array_equal(ref * 16, (qa @ qb.T).astype(np.float64))
    assert np.array_equal(mag * 16, (np.abs(qa) @ np.abs(qb).T).astype(np.float64))


def test_gemm_bf16_identity(oracle):
    rng = np.random.default_rng(4)
    M, K = 19, 24
    A = synth.bf16_normal(rng, (M, K))
    eye = np.zeros((K, K), dtype=np.uint16)
    eye[np.arange(K), np.arange(K)] = BF16_ONE
    ref, _ = oracle.gemm_bf16(A, eye)          # D = A @ I.T = A
    assert np.array_equal(ref, synth.bf16_bits_to_f32(A).astype(np.float64))


def test_gemm_bf16_one_hot_locates_every_output(oracle):
    # A[i, k] = 1 and B[j, k] = 1 give exactly one nonzero, at D[i, j]; a
    # transposed operand or a swapped index would move or lose it.
    M, N, K = 5, 7, 3
    for i, j, k in [(0, 0, 0), (4, 6, 2), (2, 5, 1), (3, 1, 2)]:
        A = np.zeros((M, K), dtype=np.uint16)
        B = np.zeros((N, K), dtype=np.uint16)
        A[i, k] = BF16_ONE
        B[j, k] = BF16_ONE
        ref, _ = oracle.gemm_bf16(A, B)
        want = np.zeros((M, N))
        want[i, j] = 1.0
        assert np.array_equal(ref, want)
        B2 = np.zeros((N, K), dtype=np.uint16)
        B2[j, (k + 1) % K] = BF16_ONE            # different k: no contribution
        ref2, _ = oracle.gemm_bf16(A, B2)
        assert not ref2.any()


def test_gemm_bf16_epilogue_add_and_selection(oracle):
    rng = np.random.default_rng(5)
    A = synth.bf16_uniform(rng, (13, 40))
    B = synth.bf16_uniform(rng, (11, 40))
    ref0, mag0 = oracle.gemm_bf16(A, B)
    ref1, mag1 = oracle.gemm_bf16(A, B, add=1.0)
    assert np.array_equal(ref1, ref0 + 1.0) and np.array_equal(mag1, mag0)
    rows, cols = [12, 0, 5], [10, 3]
    sub, submag = oracle.gemm_bf16(A, B, rows=rows, cols=cols)
    assert np.array_equal(sub, ref0[np.ix_(rows, cols)])
    assert np.array_equal(submag, mag0[np.ix_(rows, cols)])


def test_gemm_bf16_strided_operands(oracle):
    rng = np.random.default_rng(6)
    big = synth.bf16_uniform(rng, (10, 64))
    A = big[:, :40]                         # row stride 64, K = 40
    B = synth.bf16_uniform(rng, (7, 40))
    ref, _ = oracle.gemm_bf16(A, B)
    ref_c, _ = oracle.gemm_bf16(np.ascontiguousarray(A), B)
    assert np.array_equal(ref, ref_c)


def test_gemm_thread_count_does_not_change_results(oracle):
    rng = np.random.default_rng(7)
    A = synth.bf16_normal(rng, (64, 96))
    B = synth.bf16_normal(rng, (48, 96))
    n = oracle.num_threads()
    oracle.set_num_threads(1)
    r1, m1 = oracle.gemm_bf16(A, B)
    oracle.set_num_threads(max(n, 2))
    r2, m2 = oracle.gemm_bf16(A, B)
    oracle.set_num_threads(n)
    assert np.array_equal(r1, r2) and np.array_equal(m1, m2)


def test_gemm_rejects_bad_shapes(oracle):
    with pytest.raises(ValueError):
        oracle.gemm_bf16(np.zeros((2, 3), np.uint16), np.zeros((2, 4), np.uint16))
    with pytest.raises(ValueError):
        oracle.gemm_bf16(np.zeros((2, 3), np.uint16), np.zeros((2, 3), np.uint16), rows=[2])


# ---------------------------------------------------------------------------
# the block-scaled contraction
# ---------------------------------------------------------------------------

def _quarter_e4m3(rng, shape):
    return synth.f32_to_e4m3fn_bits((rng.integers(-4, 5, shape) / 4).astype(np.float32))


def test_mxfp8_unit_scales_equal_bf16_product(oracle):
    rng = np.random.default_rng(8)
    M, N, K = 9, 6, 96
    A = synth.e4m3_normal(rng, (M, K))
    B = synth.e4m3_normal(rng, (N, K))
    ones_a = np.full((M, K // 32), 127, np.uint8)
    ones_b = np.full((N, K // 32), 127, np.uint8)
    ref, mag = oracle.gemm_mxfp8(A, B, ones_a, ones_b)
    # Every E4M3 value is exact in bf16; convert through torch, not the oracle.
    Ab = synth.f32_to_bf16_bits(_e4m3_exact_via_torch(A).astype(np.float32))
    Bb = synth.f32_to_bf16_bits(_e4m3_exact_via_torch(B).astype(np.float32))
    ref2, mag2 = oracle.gemm_bf16(Ab, Bb)
    assert np.array_equal(ref, ref2) and np.array_equal(mag, mag2)


def test_mxfp8_matches_exact_rationals(oracle):
    rng = np.random.default_rng(9)
    M, N, K = 3, 4, 64
    A = synth.e4m3_normal(rng, (M, K))
    B = synth.e4m3_normal(rng, (N, K))
    SFA = synth.e8m0_scales(rng, (M, K // 32))
    SFB = synth.e8m0_scales(rng, (N, K // 32))
    ref, mag = oracle.gemm_mxfp8(A, B, SFA, SFB)
    av, bv = _e4m3_exact_via_torch(A), _e4m3_exact_via_torch(B)
    for i in range(M):
        for j in range(N):
            terms = [Fraction(float(av[i, k])) * Fraction(2) ** (int(SFA[i, k // 32]) - 127)
                     * Fraction(float(bv[j, k])) * Fraction(2) ** (int(SFB[j, k // 32]) - 127)
                     for k in range(K)]
            exact = sum(terms, Fraction(0))
            emag = sum((abs(t) for t in terms), Fraction(0))
            bound = Fraction(K * 2.0 ** -52 * float(emag))
            assert abs(Fraction(ref[i, j]) - exact) <= bound
            assert abs(Fraction(mag[i, j]) - emag) <= bound


def test_mxfp8_raising_one_block_scale_doubles_that_block(oracle):
    rng = np.random.default_rng(10)
    M, N, K = 6, 5, 128
    A, B = _quarter_e4m3(rng, (M, K)), _quarter_e4m3(rng, (N, K))
    SFA = np.full((M, K // 32), 127, np.uint8)
    SFB = np.full((N, K // 32), 127, np.uint8)
    base, _ = oracle.gemm_mxfp8(A, B, SFA, SFB)
    i, kb = 4, 2
    only = np.zeros_like(A)
    only[i, 32 * kb:32 * kb + 32] = A[i, 32 * kb:32 * kb + 32]
    contrib, _ = oracle.gemm_mxfp8(only, B, SFA, SFB)
    SFA2 = SFA.copy()
    SFA2[i, kb] += 1
    raised, _ = oracle.gemm_mxfp8(A, B, SFA2, SFB)
    assert np.array_equal(raised, base + contrib)
    assert np.array_equal(np.delete(raised, i, 0), np.delete(base, i, 0))


def test_mxfp8_uniform_scale_is_power_of_two_factor(oracle):
    rng = np.random.default_rng(11)
    M, N, K = 7, 3, 64
    A, B = synth.e4m3_normal(rng, (M, K)), synth.e4m3_normal(rng, (N, K))
    SFB = synth.e8m0_scales(rng, (N, K // 32))
    base, bmag = oracle.gemm_mxfp8(A, B, np.full((M, 2), 127, np.uint8), SFB)
    for s in (-5, 3):
        r, m = oracle.gemm_mxfp8(A, B, np.full((M, 2), 127 + s, np.uint8), SFB)
        assert np.array_equal(r, base * 2.0 ** s) and np.array_equal(m, bmag * 2.0 ** s)


# ---------------------------------------------------------------------------
# FP4 (E2M1) block-scaled products: .scale_vec::2X (MXFP4) and ::4X (NVFP4)
# ---------------------------------------------------------------------------

# The OCP MX E2M1 element table, code 0..15 (sign in bit 3).
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
              -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_all_codes(oracle):
    v = oracle.decode_e2m1(np.arange(16, dtype=np.uint8))
    assert list(v) == E2M1_TABLE
    assert all(math.copysign(1, a) == math.copysign(1, b) for a, b in zip(v, E2M1_TABLE))
    # only the low nibble is read
    assert list(oracle.decode_e2m1(np.arange(16, dtype=np.uint8) | 0xA0)) == E2M1_TABLE


def test_ue4m3_matches_torch_e4m3_for_positive_codes(oracle):
    bits = np.arange(0, 0x7F, dtype=np.uint8)
    assert np.array_equal(oracle.decode_ue4m3(bits), _e4m3_exact_via_torch(bits))
    assert np.isnan(oracle.decode_ue4m3(np.array([0x7F, 0x80, 0xB8, 0xFF], np.uint8))).all()
    assert list(oracle.decode_ue4m3(np.array([0x38, 0x40, 0x30, 0x7E], np.uint8))) == \
        [1.0, 2.0, 0.5, 448.0]


def test_e2m1_encoder_round_trip_and_ties(oracle):
    codes = np.arange(16, dtype=np.uint8)
    vals = np.array(E2M1_TABLE, dtype=np.float32)
    assert np.array_equal(oracle.decode_e2m1(synth.f32_to_e2m1_codes(vals)), vals)
    # midpoints round to the code with a zero fraction bit; beyond 6 saturates
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 9.0], dtype=np.float32)
    assert list(oracle.decode_e2m1(synth.f32_to_e2m1_codes(mids))) == \
        [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0]
    packed = synth.pack_e2m1(codes.reshape(2, 8))
    assert packed.shape == (2, 4) and packed[0, 0] == 0x10 and packed[1, 3] == 0xFE
    assert np.array_equal(synth.unpack_e2m1(packed), codes.reshape(2, 8))


def _unpack_python(packed, K):
    """Element k of each row: low nibble of byte k // 2 for even k, else high."""
    rows = []
    for r in range(packed.shape[0]):
        rows.append([(int(packed[r, k // 2]) >> (4 * (k % 2))) & 0xF for k in range(K)])
    return rows


@pytest.mark.parametrize("kind,block", [(0, 32), (1, 16)])
def test_fp4_matches_exact_rationals(oracle, kind, block):
    rng = np.random.default_rng(30 + kind)
    M, N, K = 3, 4, 64
    A = synth.e2m1_normal_packed(rng, (M, K))
    B = synth.e2m1_normal_packed(rng, (N, K))
    if kind == 0:
        SFA, SFB = synth.e8m0_scales(rng, (M, K // 32)), synth.e8m0_scales(rng, (N, K // 32))
        scale = lambda b: Fraction(2) ** (int(b) - 127)                       # noqa: E731
    else:
        SFA = synth.ue4m3_pow2_scales(rng, (M, K // 16))
        SFB = np.array(rng.integers(0x20, 0x50, size=(N, K // 16)), np.uint8)   # any finite
        lib = _e4m3_exact_via_torch(np.arange(256, dtype=np.uint8))
        scale = lambda b: Fraction(float(lib[int(b)]))                       # noqa: E731
    ref, mag = oracle.gemm_fp4(A, B, SFA, SFB, kind)
    ua, ub = _unpack_python(A, K), _unpack_python(B, K)
    for i in range(M):
        for j in range(N):
            terms = [Fraction(E2M1_TABLE[ua[i][k]]) * scale(SFA[i, k // block]) *
                     Fraction(E2M1_TABLE[ub[j][k]]) * scale(SFB[j, k // block])
                     for k in range(K)]
            exact = sum(terms, Fraction(0))
            emag = sum((abs(t) for t in terms), Fraction(0))
            bound = Fraction(K * 2.0 ** -52 * float(emag))
            assert abs(Fraction(ref[i, j]) - exact) <= bound
            assert abs(Fraction(mag[i, j]) - emag) <= bound


def test_fp4_unit_scales_equal_bf16_product(oracle):
    rng = np.random.default_rng(32)
    M, N, K = 9, 6, 128
    A = synth.e2m1_normal_packed(rng, (M, K))
    B = synth.e2m1_normal_packed(rng, (N, K))
    table = np.array(E2M1_TABLE, dtype=np.float32)
    # every E2M1 value is exact in bf16: decode with the table, not the oracle
    Ab = synth.f32_to_bf16_bits(table[synth.unpack_e2m1(A)])
    Bb = synth.f32_to_bf16_bits(table[synth.unpack_e2m1(B)])
    want, wmag = oracle.gemm_bf16(Ab, Bb)
    mx = oracle.gemm_mxfp4(A, B, np.full((M, K // 32), 127, np.uint8),
                           np.full((N, K // 32), 127, np.uint8))
    nv = oracle.gemm_nvfp4(A, B, np.full((M, K // 16), 0x38, np.uint8),
                           np.full((N, K // 16), 0x38, np.uint8))
    for ref, mag in (mx, nv):
        assert np.array_equal(ref, want) and np.array_equal(mag, wmag)


def test_fp4_nibble_order_one_hot(oracle):
    # A row 0 holds 1.0 at element 1 only (high nibble of byte 0); B row j
    # holds 2.0 at element j only.  Then D[0, j] = 2 for j == 1, else 0.
    K = 32
    A = np.zeros((1, K // 2), np.uint8)
    A[0, 0] = 0x20
    B = synth.pack_e2m1(np.eye(4, K, dtype=np.uint8) * 4)
    ref, _ = oracle.gemm_mxfp4(A, B, np.full((1, 1), 127, np.uint8), np.full((4, 1), 127, np.uint8))
    assert list(ref[0]) == [0.0, 2.0, 0.0, 0.0]


@pytest.mark.parametrize("kind,block,two", [(0, 32, 128), (1, 16, 0x40)])
def test_fp4_doubling_one_block_scale(oracle, kind, block, two):
    rng = np.random.default_rng(33 + kind)
    M, N, K = 5, 4, 128
    A, B = synth.e2m1_normal_packed(rng, (M, K)), synth.e2m1_normal_packed(rng, (N, K))
    one = 127 if kind == 0 else 0x38
    SFA = np.full((M, K // block), one, np.uint8)
    SFB = np.full((N, K // block), one, np.uint8)
    base, _ = oracle.gemm_fp4(A, B, SFA, SFB, kind)
    i, kb = 3, 1
    codes = synth.unpack_e2m1(A)
    only = np.zeros_like(codes)
    only[i, block * kb:block * (kb + 1)] = codes[i, block * kb:block * (kb + 1)]
    contrib, _ = oracle.gemm_fp4(synth.pack_e2m1(only), B, SFA, SFB, kind)
    SFA2 = SFA.copy()
    SFA2[i, kb] = two
    raised, _ = oracle.gemm_fp4(A, B, SFA2, SFB, kind)
    assert np.array_equal(raised, base + contrib)
    assert np.array_equal(np.delete(raised, i, 0), np.delete(base, i, 0))


def test_fp4_rejects_bad_shapes(oracle):
    A = np.zeros((4, 16), np.uint8)
    with pytest.raises(ValueError):
        oracle.gemm_mxfp4(A, A, np.zeros((4, 2), np.uint8), np.zeros((4, 1), np.uint8))
    with pytest.raises(ValueError):
        oracle.gemm_nvfp4(A, A, np.zeros((4, 1), np.uint8), np.zeros((4, 1), np.uint8))


# ---------------------------------------------------------------------------
# data movement and layout models
# ---------------------------------------------------------------------------

def test_transpose_b16(oracle):
    rng = np.random.default_rng(12)
    X = synth.b16_bits(rng, (37, 53))
    T = oracle.transpose_b16(X)
    assert T.shape == (53, 37) and np.array_equal(T, X.T)
    assert np.array_equal(oracle.transpose_b16(T), X)


def test_ldmatrix_worked_example_matches_page(oracle):
    # Compose the page's interleaved example from the oracle's .x2 model:
    # S_std[k, m, r, w] = SM[2r+m, w, k]; repeat k writes slot 8k + 2m.
    x = np.arange(128, dtype=np.uint32).reshape(16, 4, 2)
    raw = np.full((32, 12), 4294966519, dtype=np.uint32)
    for k in range(2):
        words = np.array([[[x[2 * r + m, w, k] for w in range(4)] for r in range(8)]
                          for m in range(2)], dtype=np.uint32)            # [2, 8, 4] b32
        halves = words.view(np.uint16).reshape(2, 8, 8)                   # low half first
        img = oracle.ldmatrix_image(halves, trans=False)                  # [32, 2]
        for m in range(2):
            raw[:, 8 * k + 2 * m] = img[:, m]
    golden = np.loadtxt(os.path.join(GOLDEN, "ldmatrix_x2_interleaved.txt"), dtype=np.uint64)
    assert np.array_equal(raw.astype(np.uint64), golden)


def test_ldmatrix_trans_identity(oracle):
    rng = np.random.default_rng(13)
    sm = rng.integers(0, 1 << 16, (4, 8, 8), dtype=np.uint32).astype(np.uint16)
    t = oracle.ldmatrix_image(sm, trans=True)
    assert np.array_equal(t, oracle.ldmatrix_image(sm.transpose(0, 2, 1), trans=False))
    for lane in range(32):
        j, w = lane // 4, lane % 4
        for i in range(4):
            lo, hi = int(t[lane, i]) & 0xFFFF, int(t[lane, i]) >> 16
            assert lo == sm[i, 2 * w, j] and hi == sm[i, 2 * w + 1, j]
    for n in (1, 2):
        assert np.array_equal(oracle.ldmatrix_image(sm[:n], True), t[:, :n])


def test_stmatrix_inverts_ldmatrix(oracle):
    rng = np.random.default_rng(14)
    sm = rng.integers(0, 1 << 16, (2, 8, 8), dtype=np.uint32).astype(np.uint16)
    for trans in (False, True):
        assert np.array_equal(oracle.stmatrix_image(oracle.ldmatrix_image(sm, trans), trans), sm)


def test_ldmatrix_address_providers(oracle):
    for n in (1, 2, 4):
        provided = {oracle.ldmatrix_address_row(l, n) for l in range(32)}
        assert provided == {(i, r) for i in range(n) for r in range(8)}
        assert [oracle.ldmatrix_address_row(l, n) for l in range(8 * n)] == \
            [(l // 8, l % 8) for l in range(8 * n)]


def test_swizzle128_permutes_chunks_across_rows(oracle):
    # Within each 1024-byte period the swizzle is a bijection that keeps
    # bytes inside their 16-byte chunk and row, and puts chunk c of the 8
    # rows of a period at 8 distinct chunk positions (conflict-free columns).
    for base in (0, 1024, 5 * 1024):
        img = [oracle.swizzle128(base + o) for o in range(1024)]
        assert sorted(img) == list(range(base, base + 1024))
        for o in range(1024):
            s = img[o] - base
            assert s // 128 == o // 128 and s % 16 == o % 16
        for c in range(8):
            assert len({(oracle.swizzle128(base + 128 * r + 16 * c) - base) % 128 // 16
                        for r in range(8)}) == 8
    assert all(oracle.swizzle128(o) == o for o in range(128))


@pytest.mark.parametrize("shape,rows,regs_per_x", [
    ("32x32b", 32, 1), ("16x64b", 16, 1), ("16x128b", 16, 2), ("16x256b", 16, 4)])
def test_tmem_register_images_are_bijections(oracle, shape, rows, regs_per_x):
    # An .xN access moves 32 * regs_per_x * N b32 cells of a (rows, C) block;
    # every (lane, register) pair must land on a distinct cell of it.
    for nrep in (1, 2, 4):
        n_regs = regs_per_x * nrep
        cells = [oracle.tmem_register_coord(shape, l, r) for l in range(32) for r in range(n_regs)]
        C = 32 * n_regs // rows
        assert len(set(cells)) == len(cells) == rows * C
        assert {c[0] for c in cells} == set(range(rows))
        assert {c[1] for c in cells} == set(range(C))


def test_tmem_16x32bx2_matches_the_page_example(oracle):
    # The page's .16x32bx2.x4 example with imm_half_splitoff = (16 << 16) + 8
    # reads memory[:, :16, :4] and memory[:, 16:32, 8:12]: lanes 0..15 the
    # first block, lanes 16..31 the second, four registers each.
    cells = {(l, r): oracle.tmem_register_coord_16x32bx2(l, r, 16, 8)
             for l in range(32) for r in range(4)}
    low = {cells[(l, r)] for l in range(16) for r in range(4)}
    high = {cells[(l, r)] for l in range(16, 32) for r in range(4)}
    assert low == {(i, j) for i in range(16) for j in range(4)}
    assert high == {(i, j) for i in range(16, 32) for j in range(8, 12)}
    # no implicit sixteen-row offset: a zero lane offset reuses rows 0..15
    assert oracle.tmem_register_coord_16x32bx2(16, 0, 0, 8) == (0, 8)


def test_block_scale_slots_cover_128_rows(oracle):
    slots = [oracle.block_scale_tmem_slot(r) for r in range(128)]
    assert len(set(slots)) == 128
    assert {s[0] for s in slots} == set(range(32))
    assert {s[1] for s in slots} == {0, 4, 8, 12}


def test_block_scale_slots_match_the_page_rows(oracle):
    # Rows of the "tcgen05.mma" block-scaling rule written out by hand in the
    # fixture: lane r % 32 plus the four 32-lane replicas, byte column
    # 4 * (r // 32) + sf.  A transposed map (lane (r // 4) % 32, byte 4 * (r % 4))
    # or a missing replica fails here.
    rows = np.loadtxt(os.path.join(GOLDEN, "block_scale_tmem_slots.txt"), dtype=np.int64)
    assert rows.shape[1] == 7 and len(rows) >= 16
    for r, sf, l0, l1, l2, l3, col in rows:
        got = [oracle.block_scale_tmem_slot(int(r), int(sf), q) for q in range(4)]
        assert got == [(int(l0), int(col)), (int(l1), int(col)), (int(l2), int(col)),
                       (int(l3), int(col))], (r, sf)
    with pytest.raises(ValueError):
        oracle.block_scale_tmem_slot(0, 0, 4)


def test_ldmatrix_address_providers_match_the_page_example(oracle):
    # The x2 operand-specification example: with S_std[k, m, r, w] =
    # SM[2r + m, w, k], lanes 0..15 supply the fixture's original rows and
    # lanes 16..31 repeat addresses that lanes 0..15 supply.
    table = np.loadtxt(os.path.join(GOLDEN, "ldmatrix_x2_address_providers.txt"),
                       dtype=np.int64)
    assert table.shape == (16, 4)
    def sm_row(lane):
        m, r = oracle.ldmatrix_address_row(lane, 2)
        return 2 * r + m
    for lane, m, r, orig in table:
        assert oracle.ldmatrix_address_row(int(lane), 2) == (int(m), int(r))
        assert sm_row(int(lane)) == int(orig)
    valid = {int(o) for o in table[:, 3]}
    assert valid == set(range(16))
    assert all(sm_row(lane) in valid for lane in range(16, 32))


def test_add_one_worked_example(oracle):
    a = np.arange(768, dtype=np.float32).reshape(2, 32, 3, 4)
    golden = np.loadtxt(os.path.join(GOLDEN, "add_one_2x32x3x4.txt"), dtype=np.float32)
    assert np.array_equal(oracle.add_one(a).reshape(-1), golden.reshape(-1))


# ---------------------------------------------------------------------------
# fused epilogues
# ---------------------------------------------------------------------------

def test_silu_matches_library_logistic(oracle):
    special = pytest.importorskip("scipy.special")
    x = np.concatenate([np.linspace(-40, 40, 2001), [0.0, 1e-8, -1e-8, 700.0, -700.0]])
    assert np.allclose(oracle.silu(x), x * special.expit(x), rtol=1e-14, atol=1e-300)
    assert oracle.silu(np.array([0.0]))[0] == 0.0


def test_silu_reflection_identity(oracle):
    # silu(-x) = -x * sigmoid(-x) = silu(x) - x
    x = np.linspace(-30, 30, 601)
    assert np.allclose(oracle.silu(-x), oracle.silu(x) - x, rtol=1e-12, atol=1e-12)


def test_epilogue_ops_closed_forms(oracle):
    rng = np.random.default_rng(20)
    ref = rng.standard_normal((5, 7)) * 3
    bias = rng.standard_normal(11)
    cols = [0, 3, 4, 6, 8, 9, 10]
    assert np.array_equal(oracle.apply_epilogue(ref, oracle.EPI_NONE), ref)
    assert np.array_equal(oracle.apply_epilogue(ref, oracle.EPI_ADD_SCALAR, 1.0), ref + 1)
    sa = oracle.apply_epilogue(ref, oracle.EPI_SILU_AFFINE, 2.0, 1.0)
    assert np.allclose(sa, 2 * ref / (1 + np.exp(-ref)) + 1, rtol=1e-15)
    bc = oracle.apply_epilogue(ref, oracle.EPI_BIAS_COL, bias=bias, cols=cols)
    for jj, j in enumerate(cols):
        assert np.array_equal(bc[:, jj], ref[:, jj] + bias[j])
    bs = oracle.apply_epilogue(ref, oracle.EPI_BIAS_COL_SILU, bias=bias, cols=cols)
    assert np.allclose(bs, oracle.silu(bc), rtol=0, atol=0)
    # the add-one example is the ADD_SCALAR op with alpha = 1
    a = np.arange(768, dtype=np.float64).reshape(64, 12)
    assert np.array_equal(oracle.apply_epilogue(a, oracle.EPI_ADD_SCALAR, 1.0), a + 1)


def test_epilogue_affine_closed_form(oracle):
    ref = np.arange(12, dtype=np.float64).reshape(3, 4) - 5
    out = oracle.apply_epilogue(ref, oracle.EPI_AFFINE, 0.25, -2.0)
    assert np.array_equal(out, ref / 4 - 2)
