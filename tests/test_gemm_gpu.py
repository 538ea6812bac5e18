"""GPU parity of gemm_bf16 and gemm_mxfp8_blockscaled against the oracle.

Small cases are compared on every element; the 4096^3 and 8192^3 workloads
run in the launch configuration the benchmark times and are compared on
seeded samples of full rows and full columns (tile edges included).
Tolerance per element: |D - ref| <= 1e-5 * sum|a b| + 1e-6 (f32 D) or
8e-3 * sum|a b| + 1e-3 (bf16 D); cases with exactly representable partial
sums are compared bit for bit.
"""
import numpy as np
import pytest

from blackwell_tile_gemm_gb300 import synth
from tests._gpu import (assert_within, dev_bf16, dev_u8, edge_sample, host_values, sample_indices,
                        torch_cuda)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tg():
    torch_cuda()
    import blackwell_tile_gemm_gb300 as m
    m.lib()
    return m


# `pair`: False = single CTA, True = CTA pair, "mc" = clusters of two pairs
# sharing the B tile by multicast, "mc1" = clusters of two single CTAs sharing it.
def run_bf16(tg, A, B, out_dtype="f32", add=None, pair=False, ld_pad=0):
    torch = torch_cuda()
    M, K = A.shape
    N = B.shape[0]
    dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    if ld_pad:
        Dfull = torch.full((M, N + ld_pad), float("nan"), dtype=dt, device="cuda")
        D = Dfull[:, :N]
    else:
        D = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
    tg.gemm_bf16(dev_bf16(A), dev_bf16(B), D, epilogue_add=add, cta_pair=pair in (True, "mc"),
                 multicast=pair in ("mc", "mc1"))
    assert tg.tg_device_status()[0] == tg.TG_OK
    return D


def run_mx(tg, A, B, SFA, SFB, out_dtype="bf16", add=None, pair=False):
    torch = torch_cuda()
    dt = torch.float32 if out_dtype == "f32" else torch.bfloat16
    D = torch.full((A.shape[0], B.shape[0]), float("nan"), dtype=dt, device="cuda")
    tg.gemm_mxfp8_blockscaled(dev_u8(A), dev_u8(B), dev_u8(SFA), dev_u8(SFB), D,
                              epilogue_add=add, cta_pair=bool(pair), multicast=pair == "mc")
    assert tg.tg_device_status()[0] == tg.TG_OK
    return D


def quarter_bits(rng, shape):
    return synth.f32_to_bf16_bits((rng.integers(-4, 5, shape) / 4).astype(np.float32))


# ------------------------------------------------------------------ bf16, small

@pytest.mark.parametrize("pair", [False, True, "mc", "mc1"])
def test_tiny_workload_full(tg, oracle, pair):
    x = synth.make_inputs("tiny")
    D = run_bf16(tg, x["A"], x["B"], "f32", pair=pair)
    ref, mag = oracle.gemm_bf16(x["A"], x["B"])
    assert_within(host_values(D), ref, mag, False, "tiny")


@pytest.mark.parametrize("pair", [False, True, "mc", "mc1"])
@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (384, 256, 1024), (128, 256, 64)])
def test_quarter_integers_bit_exact(tg, oracle, pair, M, N, K):
    rng = np.random.default_rng(M + N + K)
    A, B = quarter_bits(rng, (M, K)), quarter_bits(rng, (N, K))
    D = run_bf16(tg, A, B, "f32", pair=pair)
    ref, _ = oracle.gemm_bf16(A, B)
    assert np.array_equal(host_values(D), ref)


@pytest.mark.parametrize("pair", [False, True, "mc", "mc1"])
def test_one_hot_across_tile_edges(tg, pair):
    M, N, K = 512, 512, 192
    one = 0x3F80
    for i, j, k in [(0, 0, 0), (127, 255, 63), (128, 256, 64), (255, 511, 191), (300, 17, 100),
                    (511, 300, 128)]:
        A = np.zeros((M, K), np.uint16)
        B = np.zeros((N, K), np.uint16)
        A[i, k] = one
        B[j, k] = one
        got = host_values(run_bf16(tg, A, B, "f32", pair=pair))
        want = np.zeros((M, N))
        want[i, j] = 1.0
        assert np.array_equal(got, want), (i, j, k)


def test_identity(tg):
    rng = np.random.default_rng(8)
    M, K = 256, 256
    A = synth.bf16_normal(rng, (M, K))
    eye = np.zeros((K, K), np.uint16)
    eye[np.arange(K), np.arange(K)] = 0x3F80
    got = host_values(run_bf16(tg, A, eye, "f32"))
    assert np.array_equal(got, synth.bf16_bits_to_f32(A).astype(np.float64))


@pytest.mark.parametrize("pair", [False, True, "mc", "mc1"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,K", [(1, 8, 16), (33, 40, 40), (130, 264, 72), (300, 520, 1000),
                                   (129, 8, 8)])
def test_ragged_small(tg, oracle, pair, out, M, N, K):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    A, B = synth.bf16_uniform(rng, (M, K)), synth.bf16_uniform(rng, (N, K))
    D = run_bf16(tg, A, B, out, add=1.0, pair=pair, ld_pad=8)
    ref, mag = oracle.gemm_bf16(A, B, add=1.0)
    assert_within(host_values(D), ref, mag, out == "bf16", f"ragged {M}x{N}x{K}")


def test_k_zero_gives_epilogue_of_zero(tg):
    torch = torch_cuda()
    A = torch.empty((5, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((7, 0), dtype=torch.bfloat16, device="cuda")
    D = torch.full((5, 8), float("nan"), device="cuda")[:, :7]
    tg.gemm_bf16(A, B, D, epilogue_add=2.5)
    assert torch.equal(D, torch.full((5, 7), 2.5, device="cuda"))


def test_ragged_equals_zero_padded_bit_exact(tg):
    # Out-of-range box elements read zero, so the ragged product equals the
    # same data zero-padded to tile multiples, bit for bit.
    rng = np.random.default_rng(5)
    M, N, K = 200, 300, 104           # K rows of 208 bytes: a legal stride, ragged K tail
    A, B = synth.bf16_uniform(rng, (M, K)), synth.bf16_uniform(rng, (N, K))
    Ap = np.zeros((256, 128), np.uint16)
    Bp = np.zeros((512, 128), np.uint16)
    Ap[:M, :K] = A
    Bp[:N, :K] = B
    d1 = host_values(run_bf16(tg, A, B, "f32"))
    d2 = host_values(run_bf16(tg, Ap, Bp, "f32"))[:M, :N]
    assert np.array_equal(d1, d2)


def test_repeat_runs_are_bit_identical(tg):
    rng = np.random.default_rng(6)
    A, B = synth.bf16_normal(rng, (512, 1024)), synth.bf16_normal(rng, (768, 1024))
    d1 = host_values(run_bf16(tg, A, B, "f32"))
    d2 = host_values(run_bf16(tg, A, B, "f32"))
    assert np.array_equal(d1, d2)


@pytest.mark.parametrize("pair", [False, True, "mc"])
def test_ragged_workload_full(tg, oracle, pair):
    # M=4000, N=3000, K=1000, D = A B^T + 1 in f32, every element, in single
    # CTAs (multicast clusters, chosen for this short K), CTA pairs and
    # multicast clusters of two pairs (the workload's launch).  Rows of 2000
    # bytes: both operands take the re-pitch copy first, except in the pair
    # clusters, which read them in place.
    x = synth.make_inputs("ragged")
    want = 0 if pair == "mc" else 3
    assert tg.gemm_repitch(4000, 3000, 1000, 1000, 1000, cta_pair=bool(pair),
                           multicast=pair == "mc") == want
    D = run_bf16(tg, x["A"], x["B"], "f32", add=1.0, pair=pair)
    ref, mag = oracle.gemm_bf16(x["A"], x["B"], add=1.0)
    assert_within(host_values(D), ref, mag, False, f"ragged 4000x3000x1000 ({pair})")


@pytest.mark.parametrize("pair", [False, True, "mc"])
def test_repitch_matches_aligned_strides_bit_for_bit(tg, pair):
    # The same operands at lda = 1000 (re-pitched; pair clusters: read in
    # place) and lda = 1024 (used in place) give the same bits: where rows
    # live does not change the arithmetic.
    torch = torch_cuda()
    x = synth.make_inputs("ragged")
    M, N, K = 4000, 3000, 1000
    assert tg.gemm_repitch(M, N, K, 1024, 1024) == 0
    Ap = torch.zeros((M, 1024), dtype=torch.bfloat16, device="cuda")
    Bp = torch.zeros((N, 1024), dtype=torch.bfloat16, device="cuda")
    Ap[:, :K] = dev_bf16(x["A"])
    Bp[:, :K] = dev_bf16(x["B"])
    D1 = torch.full((M, N), float("nan"), device="cuda")
    D2 = torch.full((M, N), float("nan"), device="cuda")
    kw = dict(cta_pair=bool(pair), multicast=pair == "mc")
    tg.gemm_bf16(dev_bf16(x["A"]), dev_bf16(x["B"]), D1, epilogue_add=1.0, **kw)
    tg.gemm_bf16(Ap[:, :K], Bp[:, :K], D2, epilogue_add=1.0, **kw)
    assert tg.tg_device_status()[0] == tg.TG_OK
    assert torch.equal(D1, D2)


def test_repitch_odd_k_never_reads_row_padding(tg, oracle):
    # K = 1003 of a 1016-element row stride (16-byte rows) with NaN in the
    # gap; the copy takes exactly K elements per row.
    torch = torch_cuda()
    rng = np.random.default_rng(181)
    M, N, K, ld = 2600, 2600, 1003, 1016
    assert tg.gemm_repitch(M, N, K, ld, ld) == 3
    A = np.full((M, ld), 0x7FC0, np.uint16)
    B = np.full((N, ld), 0x7FC0, np.uint16)
    A[:, :K] = synth.bf16_uniform(rng, (M, K))
    B[:, :K] = synth.bf16_uniform(rng, (N, K))
    D = torch.full((M, N), float("nan"), device="cuda")
    tg.gemm_bf16(dev_bf16(A)[:, :K], dev_bf16(B)[:, :K], D)
    assert tg.tg_device_status()[0] == tg.TG_OK
    got = host_values(D)
    rows = sample_indices(M, 64, 21, 128)
    ref, mag = oracle.gemm_bf16(A[:, :K], B[:, :K], rows=rows)
    assert_within(got[rows], ref, mag, False, "re-pitched odd K rows")
    cols = sample_indices(N, 64, 22, 256)
    ref, mag = oracle.gemm_bf16(A[:, :K], B[:, :K], cols=cols)
    assert_within(got[:, cols], ref, mag, False, "re-pitched odd K cols")


def test_block_scaled_calls_on_two_streams(tg, oracle):
    # Two MXFP8 products of different shapes issued on two streams with no
    # ordering between them: each stream has its own scale-image workspace.
    torch = torch_cuda()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    xs = [synth.make_inputs("mx8k", M=1024, N=768, K=1024, seed=191),
          synth.make_inputs("mx8k", M=640, N=1024, K=2048, seed=192)]
    ins = [[dev_u8(x[k]) for k in ("A", "B", "SFA", "SFB")] for x in xs]
    Ds = [torch.full((1024, 768), float("nan"), device="cuda"),
          torch.full((640, 1024), float("nan"), device="cuda")]
    torch.cuda.synchronize()
    for _ in range(3):
        for s, g, D in zip((s1, s2), ins, Ds):
            with torch.cuda.stream(s):
                tg.gemm_mxfp8_blockscaled(*g, D, stream=s)
    torch.cuda.synchronize()
    assert tg.tg_device_status()[0] == tg.TG_OK
    for x, D in zip(xs, Ds):
        ref, mag = oracle.gemm_mxfp8(x["A"], x["B"], x["SFA"], x["SFB"])
        assert_within(host_values(D), ref, mag, False, "two streams")


@pytest.mark.slow
def test_sq4k_workload_every_element(tg, oracle):
    # 4096^3, bf16 D, single-CTA 128 x 256 tiles (the workload's own kernel):
    # every element of D against the float64 oracle.
    w = synth.WORKLOADS["sq4k"]
    assert not w.cta_pair
    x = synth.make_inputs("sq4k")
    got = host_values(run_bf16(tg, x["A"], x["B"], "bf16", pair=False))
    ref, mag = oracle.gemm_bf16(x["A"], x["B"])
    assert_within(got, ref, mag, True, "sq4k every element")


@pytest.mark.slow
def test_sq8k_workload_sampled(tg, oracle):
    # 8192^3 in CTA pairs, f32 D: 256 full rows and 256 full columns of D,
    # including every row and column on either side of each 128 boundary
    # (CTA rows of a pair, B halves, tile edges).
    w = synth.WORKLOADS["sq8k"]
    x = synth.make_inputs("sq8k")
    got = host_values(run_bf16(tg, x["A"], x["B"], "f32", pair=True))
    rows = edge_sample(w.M, 256, 11)
    cols = edge_sample(w.N, 256, 12)
    assert rows.size == 256 and cols.size == 256
    ref, mag = oracle.gemm_bf16(x["A"], x["B"], rows=rows)
    assert_within(got[rows], ref, mag, False, "sq8k rows")
    ref, mag = oracle.gemm_bf16(x["A"], x["B"], cols=cols)
    assert_within(got[:, cols], ref, mag, False, "sq8k cols")


# ------------------------------------------------------------------ MXFP8

def mx_quarter(rng, shape):
    return synth.f32_to_e4m3fn_bits((rng.integers(-4, 5, shape) / 4).astype(np.float32))


@pytest.mark.parametrize("pair", [False, True, "mc"])
def test_mx_small_full(tg, oracle, pair):
    x = synth.make_inputs("mx8k", M=256, N=512, K=512, seed=40)
    D = run_mx(tg, x["A"], x["B"], x["SFA"], x["SFB"], "bf16", pair=pair)
    ref, mag = oracle.gemm_mxfp8(x["A"], x["B"], x["SFA"], x["SFB"])
    assert_within(host_values(D), ref, mag, True, "mx small")
    D = run_mx(tg, x["A"], x["B"], x["SFA"], x["SFB"], "f32", pair=pair)
    assert_within(host_values(D), ref, mag, False, "mx small f32")


@pytest.mark.parametrize("pair", [False, True, "mc"])
def test_mx_unit_scales_quarter_integers_bit_exact(tg, oracle, pair):
    rng = np.random.default_rng(41)
    M, N, K = 256, 256, 384
    A, B = mx_quarter(rng, (M, K)), mx_quarter(rng, (N, K))
    SFA = np.full((M, K // 32), 127, np.uint8)
    SFB = np.full((N, K // 32), 127, np.uint8)
    got = host_values(run_mx(tg, A, B, SFA, SFB, "f32", pair=pair))
    ref, _ = oracle.gemm_mxfp8(A, B, SFA, SFB)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("pair", [False, True, "mc"])
def test_mx_scales_reach_every_row_and_block(tg, oracle, pair):
    # Distinct power-of-two scales per (row, K block) on exact data: the
    # product is exact, so any misplaced scale byte changes some output.
    rng = np.random.default_rng(42)
    M, N, K = 256, 512, 256
    A, B = mx_quarter(rng, (M, K)), mx_quarter(rng, (N, K))
    SFA = synth.e8m0_scales(rng, (M, K // 32), -3, 3)
    SFB = synth.e8m0_scales(rng, (N, K // 32), -3, 3)
    got = host_values(run_mx(tg, A, B, SFA, SFB, "f32", pair=pair))
    ref, _ = oracle.gemm_mxfp8(A, B, SFA, SFB)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("pair", [False, True, "mc"])
@pytest.mark.parametrize("M,N,K", [(1, 16, 32), (100, 72, 96), (300, 264, 160)])
def test_mx_ragged(tg, oracle, pair, M, N, K):
    x = synth.make_inputs("mx8k", M=M, N=N, K=K, seed=M + N + K)
    D = run_mx(tg, x["A"], x["B"], x["SFA"], x["SFB"], "f32", add=1.0, pair=pair)
    ref, mag = oracle.gemm_mxfp8(x["A"], x["B"], x["SFA"], x["SFB"], add=1.0)
    assert_within(host_values(D), ref, mag, False, f"mx ragged {M}x{N}x{K}")


@pytest.mark.slow
def test_mx8k_workload_sampled(tg, oracle):
    w = synth.WORKLOADS["mx8k"]
    x = synth.make_inputs("mx8k")
    got = host_values(run_mx(tg, x["A"], x["B"], x["SFA"], x["SFB"], "bf16", pair=True))
    rows = edge_sample(w.M, 256, 13)
    cols = edge_sample(w.N, 256, 14)
    ref, mag = oracle.gemm_mxfp8(x["A"], x["B"], x["SFA"], x["SFB"], rows=rows)
    assert_within(got[rows], ref, mag, True, "mx8k rows")
    ref, mag = oracle.gemm_mxfp8(x["A"], x["B"], x["SFA"], x["SFB"], cols=cols)
    assert_within(got[:, cols], ref, mag, True, "mx8k cols")


# ------------------------------------------------------- outside D, outside K

@pytest.mark.parametrize("pair", [False, True, "mc", "mc1"])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("M,N,K", [(1, 1, 64), (37, 13, 72), (129, 250, 64), (260, 300, 200),
                                   (300, 67, 128), (128, 192, 64)])
def test_d_window_leaves_surroundings(tg, oracle, pair, out, M, N, K):
    # D is a window of a NaN-filled buffer with 40 more rows and a padded row
    # stride: the GEMM writes the window and nothing around it, whether the
    # tile edge, the column edge N or a 16-byte boundary falls inside a box.
    torch = torch_cuda()
    rng = np.random.default_rng(M * 11 + N * 5 + K)
    A, B = synth.bf16_uniform(rng, (M, K)), synth.bf16_uniform(rng, (N, K))
    dt = torch.float32 if out == "f32" else torch.bfloat16
    ldd = (N + 1 + 7) // 8 * 8
    Dfull = torch.full((M + 40, ldd), float("nan"), dtype=dt, device="cuda")
    tg.gemm_bf16(dev_bf16(A), dev_bf16(B), Dfull[:M, :N], epilogue_add=1.0,
                 cta_pair=pair in (True, "mc"), multicast=pair in ("mc", "mc1"))
    assert tg.tg_device_status()[0] == tg.TG_OK
    got = host_values(Dfull)
    ref, mag = oracle.gemm_bf16(A, B, add=1.0)
    assert_within(got[:M, :N], ref, mag, out == "bf16", f"window {M}x{N}x{K}")
    assert np.all(np.isnan(got[:M, N:])) and np.all(np.isnan(got[M:, :]))


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_mx_d_window_leaves_surroundings(tg, oracle, out):
    torch = torch_cuda()
    M, N, K = 140, 37, 96
    x = synth.make_inputs("mx8k", M=M, N=N, K=K, seed=171)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    Dfull = torch.full((M + 40, 48), float("nan"), dtype=dt, device="cuda")
    tg.gemm_mxfp8_blockscaled(dev_u8(x["A"]), dev_u8(x["B"]), dev_u8(x["SFA"]), dev_u8(x["SFB"]),
                              Dfull[:M, :N])
    assert tg.tg_device_status()[0] == tg.TG_OK
    got = host_values(Dfull)
    ref, mag = oracle.gemm_mxfp8(x["A"], x["B"], x["SFA"], x["SFB"])
    assert_within(got[:M, :N], ref, mag, out == "bf16", "mx window")
    assert np.all(np.isnan(got[:M, N:])) and np.all(np.isnan(got[M:, :]))


@pytest.mark.parametrize("pair", [False, True])
def test_odd_k_never_reads_row_padding(tg, oracle, pair):
    # K = 100 of a 104-element row stride; elements K..103 hold NaN, which
    # would reach D if any load took them.
    torch = torch_cuda()
    rng = np.random.default_rng(172)
    M, N, K = 200, 72, 100
    A = np.full((M, 104), 0x7FC0, np.uint16)
    B = np.full((N, 104), 0x7FC0, np.uint16)
    A[:, :K] = synth.bf16_uniform(rng, (M, K))
    B[:, :K] = synth.bf16_uniform(rng, (N, K))
    D = torch.full((M, N), float("nan"), device="cuda")
    tg.gemm_bf16(dev_bf16(A)[:, :K], dev_bf16(B)[:, :K], D, cta_pair=pair)
    assert tg.tg_device_status()[0] == tg.TG_OK
    ref, mag = oracle.gemm_bf16(A[:, :K], B[:, :K])
    assert_within(host_values(D), ref, mag, False, "odd K")
