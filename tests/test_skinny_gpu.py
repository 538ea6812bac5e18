"""GPU parity of gemm_bf16_skinny (few rows of A against a large B; operands
swapped, split-K pieces added with TMA reduce-add) against the oracle.

Tolerances as for gemm_bf16.  Split-K adds partial sums in a run-dependent
order; with quarter-integer inputs every partial and total is exact in f32,
so those cases are compared bit for bit whatever the split.
"""
import numpy as np
import pytest

from blackwell_tile_gemm_gb300 import synth
from tests._gpu import (BF16_ATOL, BF16_RTOL, F32_ATOL, F32_RTOL, assert_within, dev_bf16,
                        host_values, sample_indices, torch_cuda)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tg():
    torch_cuda()
    import blackwell_tile_gemm_gb300 as m
    m.lib()
    return m


def run(tg, A, B, out="f32", split_k=0, **epi):
    torch = torch_cuda()
    dt = torch.float32 if out == "f32" else torch.bfloat16
    D = torch.full((A.shape[0], B.shape[0]), float("nan"), dtype=dt, device="cuda")
    tg.gemm_bf16_skinny(dev_bf16(A), dev_bf16(B), D, split_k=split_k, **epi)
    assert tg.tg_device_status()[0] == tg.TG_OK
    return D


def quarter_bits(rng, shape):
    return synth.f32_to_bf16_bits((rng.integers(-4, 5, shape) / 4).astype(np.float32))


@pytest.mark.parametrize("M", [1, 16, 17, 33, 64, 100, 128])
@pytest.mark.parametrize("split_k", [0, 1, 3])
def test_skinny_exact_any_split(tg, oracle, M, split_k):
    rng = np.random.default_rng(M * 7 + split_k)
    N, K = 264, 1000
    A, B = quarter_bits(rng, (M, K)), quarter_bits(rng, (N, K))
    got = host_values(run(tg, A, B, "f32", split_k))
    ref, _ = oracle.gemm_bf16(A, B)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (8, 1000, 200), (64, 520, 4160), (128, 256, 512)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_skinny_uniform_inputs(tg, oracle, M, N, K, out):
    x = synth.make_inputs("tiny", M=M, N=N, K=K, seed=M + N + K)
    got = host_values(run(tg, x["A"], x["B"], out))
    ref, mag = oracle.gemm_bf16(x["A"], x["B"])
    assert_within(got, ref, mag, out == "bf16", f"skinny {M}x{N}x{K} {out}")


CASES = [("add", 1, lambda b: dict(epilogue_add=0.75), 1.0, (0.75, 0.0)),
         ("affine", 5, lambda b: dict(affine=(0.5, -1.25)), 0.5, (0.5, -1.25)),
         ("silu_affine", 2, lambda b: dict(silu_affine=(2.0, 1.0)), 2.2, (2.0, 1.0)),
         ("bias", 3, lambda b: dict(bias=b), 1.0, (0.0, 0.0)),
         ("bias_silu", 4, lambda b: dict(bias=b, bias_silu=True), 1.1, (0.0, 0.0))]


@pytest.mark.parametrize("name,op,kw,lip,ab", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_skinny_epilogues(tg, oracle, name, op, kw, lip, ab, out):
    torch = torch_cuda()
    rng = np.random.default_rng(op + 90)
    M, N, K = 40, 392, 704
    A, B = synth.bf16_uniform(rng, (M, K)), synth.bf16_uniform(rng, (N, K))
    bias_np = (rng.standard_normal(N) * 4).astype(np.float32)
    bias = torch.from_numpy(bias_np).cuda()
    got = host_values(run(tg, A, B, out, 3, **kw(bias)))
    ref, mag = oracle.gemm_bf16(A, B)
    want = oracle.apply_epilogue(ref, op, ab[0], ab[1], bias=bias_np)
    rtol, atol = (BF16_RTOL, BF16_ATOL) if out == "bf16" else (F32_RTOL, F32_ATOL)
    eps = 2.0 ** -8 if out == "bf16" else 2.0 ** -21
    tol = lip * (rtol * mag + atol) + eps * np.abs(want)
    assert np.all(np.abs(got - want) <= tol), name


def test_skinny_single_piece_is_deterministic(tg):
    rng = np.random.default_rng(95)
    A, B = synth.bf16_uniform(rng, (48, 2048)), synth.bf16_uniform(rng, (640, 2048))
    d1 = host_values(run(tg, A, B, "f32", 1))
    d2 = host_values(run(tg, A, B, "f32", 1))
    assert np.array_equal(d1, d2)


def test_skinny_split_count_query(tg):
    assert tg.skinny_split_count(8192, 8192, 1) == 1
    assert tg.skinny_split_count(8192, 8192, 7) == 7
    assert tg.skinny_split_count(8192, 128, 5) == 2         # K = 2 stages of 64
    assert tg.skinny_split_count(8192, 8192, 0) >= 2        # 64 tiles < SMs


def test_skinny_k_zero_and_rejections(tg):
    torch = torch_cuda()
    A = torch.empty((5, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((8, 0), dtype=torch.bfloat16, device="cuda")
    D = torch.full((5, 8), float("nan"), device="cuda")
    tg.gemm_bf16_skinny(A, B, D, epilogue_add=1.5)
    assert torch.all(D == 1.5)
    big = torch.zeros((129, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tg.TgError):
        tg.gemm_bf16_skinny(big, W)


@pytest.mark.slow
@pytest.mark.parametrize("M", [16, 64])
def test_skinny_8k_sampled(tg, oracle, M):
    rng = np.random.default_rng(96 + M)
    N = K = 8192
    A = synth.bf16_normal(rng, (M, K), 1.0 / np.sqrt(K))
    B = synth.bf16_normal(rng, (N, K))
    got = host_values(run(tg, A, B, "bf16"))
    cols = sample_indices(N, 128, 97, 128)
    ref, mag = oracle.gemm_bf16(A, B, cols=cols)
    assert_within(got[:, cols], ref, mag, True, f"skinny 8k M={M}")


@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("M,N", [(3, 13), (20, 130), (64, 257)])
def test_d_window_leaves_surroundings(tg, oracle, out, M, N):
    # D is a window of a buffer whose padding holds -0.0: neither a store nor
    # a reduce-add (which would turn -0.0 into +0.0) may touch it.
    torch = torch_cuda()
    rng = np.random.default_rng(M * 13 + N)
    K = 320
    A, B = synth.bf16_uniform(rng, (M, K)), synth.bf16_uniform(rng, (N, K))
    dt = torch.float32 if out == "f32" else torch.bfloat16
    ldd = (N + 1 + 7) // 8 * 8
    Dfull = torch.full((M + 8, ldd), -0.0, dtype=dt, device="cuda")
    tg.gemm_bf16_skinny(dev_bf16(A), dev_bf16(B), Dfull[:M, :N], split_k=3)
    assert tg.tg_device_status()[0] == tg.TG_OK
    got = host_values(Dfull)
    ref, mag = oracle.gemm_bf16(A, B)
    assert_within(got[:M, :N], ref, mag, out == "bf16", f"skinny window {M}x{N}")
    for pad in (got[:M, N:], got[M:, :]):
        assert np.all(pad == 0) and np.all(np.signbit(pad))


def test_odd_k_never_reads_row_padding(tg, oracle):
    torch = torch_cuda()
    rng = np.random.default_rng(173)
    M, N, K = 9, 200, 100
    A = np.full((M, 104), 0x7FC0, np.uint16)
    B = np.full((N, 104), 0x7FC0, np.uint16)
    A[:, :K] = synth.bf16_uniform(rng, (M, K))
    B[:, :K] = synth.bf16_uniform(rng, (N, K))
    D = torch.full((M, N), float("nan"), device="cuda")
    tg.gemm_bf16_skinny(dev_bf16(A)[:, :K], dev_bf16(B)[:, :K], D)
    assert tg.tg_device_status()[0] == tg.TG_OK
    ref, mag = oracle.gemm_bf16(A[:, :K], B[:, :K])
    assert_within(host_values(D), ref, mag, False, "skinny odd K")
