"""GPU parity of gemm_bf16_gather: D[i] = A[row_idx[i]] @ B^T against the
oracle evaluated on the same rows, through both paths: rows gathered into a
workspace before the dense kernel (default) and the A tile loaded inside the
GEMM by TMA tile::gather4 (gather_tma=True).

Indices may repeat and come in any order; indices outside A give zero rows
(D = epilogue(0)).  Tolerances as for gemm_bf16; quarter-integer inputs are
compared bit for bit.
"""
import numpy as np
import pytest

from blackwell_tile_gemm_gb300 import synth
from tests._gpu import assert_within, dev_bf16, host_values, sample_indices, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tg():
    torch_cuda()
    import blackwell_tile_gemm_gb300 as m
    m.lib()
    return m


def run(tg, A, idx, B, out="f32", pair=False, tma=False, **epi):
    torch = torch_cuda()
    dt = torch.float32 if out == "f32" else torch.bfloat16
    D = torch.full((len(idx), B.shape[0]), float("nan"), dtype=dt, device="cuda")
    ti = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).cuda()
    tg.gemm_bf16_gather(dev_bf16(A), ti, dev_bf16(B), D, cta_pair=pair, gather_tma=tma, **epi)
    assert tg.tg_device_status()[0] == tg.TG_OK
    return D


def quarter_bits(rng, shape):
    return synth.f32_to_bf16_bits((rng.integers(-4, 5, shape) / 4).astype(np.float32))


@pytest.mark.parametrize("tma", [False, True])
@pytest.mark.parametrize("pair", [False, True])
def test_gather_exact_permutation_with_repeats(tg, oracle, pair, tma):
    rng = np.random.default_rng(110 + pair)
    a_rows, M, N, K = 700, 520, 264, 384
    A, B = quarter_bits(rng, (a_rows, K)), quarter_bits(rng, (N, K))
    idx = rng.integers(0, a_rows, M)
    idx[:16] = idx[0]                     # repeats
    got = host_values(run(tg, A, idx, B, "f32", pair, tma))
    ref, _ = oracle.gemm_bf16(A, B, rows=idx)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("tma", [False, True])
@pytest.mark.parametrize("pair", [False, True])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("M", [1, 129, 300])
def test_gather_uniform(tg, oracle, pair, out, M, tma):
    rng = np.random.default_rng(120 + M + pair)
    a_rows, N, K = 1000, 392, 520
    A, B = synth.bf16_uniform(rng, (a_rows, K)), synth.bf16_uniform(rng, (N, K))
    idx = rng.permutation(a_rows)[:M]
    got = host_values(run(tg, A, idx, B, out, pair, tma, epilogue_add=0.5))
    ref, mag = oracle.gemm_bf16(A, B, add=0.5, rows=idx)
    assert_within(got, ref, mag, out == "bf16", f"gather M={M} {out}")


@pytest.mark.parametrize("tma", [False, True])
@pytest.mark.parametrize("pair", [False, True])
def test_gather_out_of_range_indices_give_epilogue_of_zero(tg, oracle, pair, tma):
    rng = np.random.default_rng(130)
    a_rows, N, K = 200, 256, 256
    A, B = quarter_bits(rng, (a_rows, K)), quarter_bits(rng, (N, K))
    idx = np.array([5, -1, a_rows, 7, 2 ** 31 - 1, -2 ** 31, 199, 0], dtype=np.int64)
    got = host_values(run(tg, A, idx, B, "f32", pair, tma, epilogue_add=2.0))
    valid = (idx >= 0) & (idx < a_rows)
    ref, _ = oracle.gemm_bf16(A, B, add=2.0, rows=idx[valid])
    assert np.array_equal(got[valid], ref)
    assert np.all(got[~valid] == 2.0)


def test_gather_odd_k(tg, oracle):
    rng = np.random.default_rng(135)
    # K not a multiple of 8; lda padded to 104 with NaN, which no load may take.
    a_rows, M, N, K = 90, 70, 40, 100
    A = np.full((a_rows, 104), 0x7FC0, np.uint16)
    A[:, :K] = synth.bf16_uniform(rng, (a_rows, K))
    B = np.full((N, 104), 0x7FC0, np.uint16)
    B[:, :K] = synth.bf16_uniform(rng, (N, K))
    torch = torch_cuda()
    idx = rng.integers(0, a_rows, M)
    for tma in (False, True):
        D = torch.full((M, N), float("nan"), device="cuda")
        tg.gemm_bf16_gather(dev_bf16(A)[:, :K], torch.from_numpy(idx.astype(np.int32)).cuda(),
                            dev_bf16(B)[:, :K], D, gather_tma=tma)
        ref, mag = oracle.gemm_bf16(A[:, :K], B[:, :K], rows=idx)
        assert_within(host_values(D), ref, mag, False, f"odd K tma={tma}")


def test_gather_k_zero_and_rejections(tg):
    torch = torch_cuda()
    A = torch.empty((4, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((8, 0), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros(3, dtype=torch.int32, device="cuda")
    D = torch.full((3, 8), float("nan"), device="cuda")
    tg.gemm_bf16_gather(A, idx, B, D, epilogue_add=-1.0)
    assert torch.all(D == -1.0)
    with pytest.raises(TypeError):
        tg.gemm_bf16_gather(A, idx.to(torch.int64), B)


@pytest.mark.slow
@pytest.mark.parametrize("tma", [False, True])
def test_gather_moe_shape_sampled(tg, oracle, tma):
    # 4096 tokens of 16384 routed to one expert of 8192 x 8192 (bf16 D, pairs)
    rng = np.random.default_rng(140)
    a_rows, M, N, K = 16384, 4096, 8192, 8192
    A = synth.bf16_normal(rng, (a_rows, K), 1.0 / np.sqrt(K))
    B = synth.bf16_normal(rng, (N, K))
    idx = np.sort(rng.choice(a_rows, M, replace=False))
    got = host_values(run(tg, A, idx, B, "bf16", True, tma))
    rows = sample_indices(M, 64, 141, 256)
    ref, mag = oracle.gemm_bf16(A, B, rows=idx[rows])
    assert_within(got[rows], ref, mag, True, "gather moe rows")
