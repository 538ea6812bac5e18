"""Extreme shapes for every GEMM entry point: very long K (counters of the
K loop and of the scale images), very many tiles along one side (tile
indices, raster bands, persistent strides), and single rows / columns.
Inputs are quarter integers with small K-sums, so f32 results are exact and
compared bit for bit where the product allows it.
"""
import numpy as np
import pytest

from blackwell_tile_gemm_gb300 import synth
from tests._gpu import assert_within, dev_bf16, dev_u8, host_values, torch_cuda

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def tg():
    torch_cuda()
    import blackwell_tile_gemm_gb300 as m
    m.lib()
    return m


def sparse_quarters(rng, shape, density=0.02):
    # mostly zeros, a few quarter integers: long sums stay small and exact
    v = (rng.integers(-4, 5, shape) / 4) * (rng.random(shape) < density)
    return synth.f32_to_bf16_bits(v.astype(np.float32))


def f32(torch, shape):
    return torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")


@pytest.mark.parametrize("pair", [False, True])
def test_long_k(tg, oracle, pair):
    torch = torch_cuda()
    rng = np.random.default_rng(150)
    M, N, K = 256, 256, 1 << 18           # 4096 stages of 64
    A, B = sparse_quarters(rng, (M, K)), sparse_quarters(rng, (N, K))
    D = f32(torch, (M, N))
    tg.gemm_bf16(dev_bf16(A), dev_bf16(B), D, cta_pair=pair)
    ref, _ = oracle.gemm_bf16(A, B)
    assert np.array_equal(host_values(D), ref)


def test_long_k_skinny(tg, oracle):
    torch = torch_cuda()
    rng = np.random.default_rng(151)
    M, N, K = 3, 384, 1 << 18
    A, B = sparse_quarters(rng, (M, K)), sparse_quarters(rng, (N, K))
    D = f32(torch, (M, N))
    tg.gemm_bf16_skinny(dev_bf16(A), dev_bf16(B), D)
    ref, _ = oracle.gemm_bf16(A, B)
    assert np.array_equal(host_values(D), ref)


@pytest.mark.parametrize("pair", [False, True])
def test_many_row_tiles(tg, oracle, pair):
    # 1 << 17 rows: 1024 row tiles (512 pairs) over a single column tile
    torch = torch_cuda()
    rng = np.random.default_rng(152)
    M, N, K = 1 << 17, 40, 64
    A, B = sparse_quarters(rng, (M, K), 0.3), sparse_quarters(rng, (N, K), 0.3)
    D = f32(torch, (M, N))
    tg.gemm_bf16(dev_bf16(A), dev_bf16(B), D, cta_pair=pair)
    rows = np.concatenate([np.arange(0, 300), np.arange(M - 300, M), rng.integers(0, M, 400)])
    ref, _ = oracle.gemm_bf16(A, B, rows=rows)
    assert np.array_equal(host_values(D)[rows], ref)


def test_many_column_tiles(tg, oracle):
    # 1 << 17 columns: 512 column tiles of 256 over one row tile
    torch = torch_cuda()
    rng = np.random.default_rng(153)
    M, N, K = 8, 1 << 17, 64
    A, B = sparse_quarters(rng, (M, K), 0.3), sparse_quarters(rng, (N, K), 0.3)
    D = f32(torch, (M, N))
    tg.gemm_bf16(dev_bf16(A), dev_bf16(B), D)
    cols = np.concatenate([np.arange(0, 300), np.arange(N - 300, N), rng.integers(0, N, 400)])
    ref, _ = oracle.gemm_bf16(A, B, cols=cols)
    assert np.array_equal(host_values(D)[:, cols], ref)
    # and through the skinny path (many 128-row tiles of B)
    D2 = f32(torch, (M, N))
    tg.gemm_bf16_skinny(dev_bf16(A), dev_bf16(B), D2)
    assert np.array_equal(host_values(D2)[:, cols], ref)


@pytest.mark.parametrize("kind", ["mxfp8", "mxfp4", "nvfp4"])
def test_long_k_block_scaled(tg, oracle, kind):
    torch = torch_cuda()
    rng = np.random.default_rng(154)
    M, N, K = 256, 256, 1 << 16
    if kind == "mxfp8":
        v = lambda s: synth.f32_to_e4m3fn_bits(  # noqa: E731
            ((rng.integers(-4, 5, s) / 4) * (rng.random(s) < 0.05)).astype(np.float32))
        A, B = v((M, K)), v((N, K))
        blk = 32
    else:
        v = lambda s: synth.pack_e2m1(synth.f32_to_e2m1_codes(  # noqa: E731
            ((rng.integers(-4, 5, s) / 2) * (rng.random(s) < 0.05)).astype(np.float32)))
        A, B = v((M, K)), v((N, K))
        blk = 16 if kind == "nvfp4" else 32
    if kind == "nvfp4":
        SFA, SFB = synth.ue4m3_pow2_scales(rng, (M, K // blk)), synth.ue4m3_pow2_scales(rng, (N, K // blk))
    else:
        SFA, SFB = synth.e8m0_scales(rng, (M, K // blk), -2, 2), synth.e8m0_scales(rng, (N, K // blk), -2, 2)
    D = f32(torch, (M, N))
    fn = {"mxfp8": tg.gemm_mxfp8_blockscaled, "mxfp4": tg.gemm_mxfp4_blockscaled,
          "nvfp4": tg.gemm_nvfp4_blockscaled}[kind]
    fn(dev_u8(A), dev_u8(B), dev_u8(SFA), dev_u8(SFB), D, cta_pair=True)
    assert tg.tg_device_status()[0] == tg.TG_OK
    if kind == "mxfp8":
        ref, _ = oracle.gemm_mxfp8(A, B, SFA, SFB)
    else:
        ref, _ = oracle.gemm_fp4(A, B, SFA, SFB, oracle.FP4_MX if kind == "mxfp4" else oracle.FP4_NV)
    assert np.array_equal(host_values(D), ref)


def test_single_row_and_column(tg, oracle):
    torch = torch_cuda()
    rng = np.random.default_rng(155)
    for M, N in ((1, 8), (1, 1), (257, 1)):
        K = 520
        A, B = sparse_quarters(rng, (M, K), 0.5), sparse_quarters(rng, (N, K), 0.5)
        Npad = (N + 3) // 4 * 4
        Dfull = f32(torch, (M, Npad))
        D = Dfull[:, :N]
        for pair in (False, True):
            tg.gemm_bf16(dev_bf16(A), dev_bf16(B), D, cta_pair=pair)
            ref, _ = oracle.gemm_bf16(A, B)
            got = host_values(Dfull)
            assert np.array_equal(got[:, :N], ref)
            assert np.all(np.isnan(got[:, N:]))       # row padding untouched
