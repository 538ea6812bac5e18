"""GPU parity of the tail split: when the tiles of a dense GEMM's last wave
fill at most half of the persistent grid, each of them is cut into K pieces
run by otherwise idle units, which add their f32 partial tiles for the piece
that stores D.

Shapes are chosen through tg_gemm_tail_split so that the split really
happens on the device at hand.  Quarter-integer inputs keep every partial
and total exact, so results are compared bit for bit.
"""
import numpy as np
import pytest

from blackwell_tile_gemm_gb300 import synth
from tests._gpu import assert_within, dev_bf16, dev_u8, host_values, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tg():
    torch_cuda()
    import blackwell_tile_gemm_gb300 as m
    m.lib()
    return m


def quarter_bits(rng, shape):
    return synth.f32_to_bf16_bits((rng.integers(-4, 5, shape) / 4).astype(np.float32))


def find_split_shape(tg, pair, K, want_full_waves=True):
    """(M, N, S) with S >= 2 pieces for gemm_bf16 on this device."""
    tm = 256 if pair else 128
    for nt in range(1, 64):
        for mt in range(1, 64):
            M, N = tm * mt, 256 * nt - 8           # ragged last column tile
            S = tg.gemm_tail_split(M, N, K, pair)
            if S >= 2:
                sms = torch_cuda().cuda.get_device_properties(0).multi_processor_count
                tiles = mt * nt
                full = tiles >= (sms // (2 if pair else 1)) // 2
                if full == want_full_waves or not want_full_waves:
                    return M, N, S
    pytest.skip("no tail-split shape found on this device")


@pytest.mark.parametrize("pair", [False, True])
def test_tail_split_exact(tg, oracle, pair):
    rng = np.random.default_rng(160 + pair)
    K = 1024
    M, N, S = find_split_shape(tg, pair, K)
    A, B = quarter_bits(rng, (M, K)), quarter_bits(rng, (N, K))
    torch = torch_cuda()
    D = torch.full((M, N), float("nan"), device="cuda")
    tg.gemm_bf16(dev_bf16(A), dev_bf16(B), D, cta_pair=pair)
    assert tg.tg_device_status()[0] == tg.TG_OK
    ref, _ = oracle.gemm_bf16(A, B)
    assert np.array_equal(host_values(D), ref), f"split {S} at {M}x{N}x{K}"
    # the same call again gives the same bits (flags were left at zero)
    D2 = torch.full((M, N), float("nan"), device="cuda")
    tg.gemm_bf16(dev_bf16(A), dev_bf16(B), D2, cta_pair=pair)
    assert torch.equal(D, D2)


def test_tail_split_without_full_waves(tg, oracle):
    # two tiles, long K: every unit is a K piece
    torch = torch_cuda()
    rng = np.random.default_rng(162)
    M, N, K = 128, 512, 4096
    assert tg.gemm_tail_split(M, N, K, False) >= 2
    A, B = quarter_bits(rng, (M, K)), quarter_bits(rng, (N, K))
    D = torch.full((M, N), float("nan"), device="cuda")
    tg.gemm_bf16(dev_bf16(A), dev_bf16(B), D)
    ref, _ = oracle.gemm_bf16(A, B)
    assert np.array_equal(host_values(D), ref)


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_tail_split_with_epilogue(tg, oracle, out):
    torch = torch_cuda()
    rng = np.random.default_rng(163)
    K = 1024
    M, N, _ = find_split_shape(tg, True, K)
    A, B = synth.bf16_uniform(rng, (M, K)), synth.bf16_uniform(rng, (N, K))
    bias_np = (rng.standard_normal(N) * 2).astype(np.float32)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    D = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
    tg.gemm_bf16(dev_bf16(A), dev_bf16(B), D, cta_pair=True,
                 bias=torch.from_numpy(bias_np).cuda(), bias_silu=True)
    ref, mag = oracle.gemm_bf16(A, B)
    want = oracle.apply_epilogue(ref, oracle.EPI_BIAS_COL_SILU, bias=bias_np)
    rtol, atol = (8e-3, 1e-3) if out == "bf16" else (1e-5, 1e-6)
    eps = 2.0 ** -8 if out == "bf16" else 2.0 ** -21
    tol = 1.1 * (rtol * mag + atol) + eps * np.abs(want)
    assert np.all(np.abs(host_values(D) - want) <= tol)


@pytest.mark.parametrize("kind", ["mxfp8", "mxfp4"])
def test_block_scaled_at_split_shapes(tg, oracle, kind):
    # Block-scaled kinds do not split (the exchange cost more than it saved);
    # their results at the shapes where bf16 splits stay exact.
    torch = torch_cuda()
    rng = np.random.default_rng(164)
    K = 2048
    M, N, _ = find_split_shape(tg, True, K)
    N = (N + 15) // 16 * 16
    if kind == "mxfp8":
        q = lambda s: synth.f32_to_e4m3fn_bits((rng.integers(-4, 5, s) / 4).astype(np.float32))  # noqa
        A, B = q((M, K)), q((N, K))
        SFA, SFB = synth.e8m0_scales(rng, (M, K // 32), -2, 2), synth.e8m0_scales(rng, (N, K // 32), -2, 2)
        fn, ref = tg.gemm_mxfp8_blockscaled, oracle.gemm_mxfp8(A, B, SFA, SFB)[0]
    else:
        q = lambda s: synth.pack_e2m1(synth.f32_to_e2m1_codes(  # noqa: E731
            (rng.integers(-4, 5, s) / 2).astype(np.float32)))
        A, B = q((M, K)), q((N, K))
        SFA, SFB = synth.e8m0_scales(rng, (M, K // 32), -2, 2), synth.e8m0_scales(rng, (N, K // 32), -2, 2)
        fn, ref = tg.gemm_mxfp4_blockscaled, oracle.gemm_mxfp4(A, B, SFA, SFB)[0]
    D = torch.full((M, N), float("nan"), device="cuda")
    fn(dev_u8(A), dev_u8(B), dev_u8(SFA), dev_u8(SFB), D, cta_pair=True)
    assert tg.tg_device_status()[0] == tg.TG_OK
    assert np.array_equal(host_values(D), ref)


def test_tail_split_gathered_rows(tg, oracle):
    torch = torch_cuda()
    rng = np.random.default_rng(165)
    K = 1024
    M, N, _ = find_split_shape(tg, True, K)
    a_rows = 2 * M
    A, B = quarter_bits(rng, (a_rows, K)), quarter_bits(rng, (N, K))
    idx = rng.integers(0, a_rows, M)
    for tma in (False, True):
        D = torch.full((M, N), float("nan"), device="cuda")
        tg.gemm_bf16_gather(dev_bf16(A), torch.from_numpy(idx.astype(np.int32)).cuda(),
                            dev_bf16(B), D, cta_pair=True, gather_tma=tma)
        ref, _ = oracle.gemm_bf16(A, B, rows=idx)
        assert np.array_equal(host_values(D), ref)


def test_tail_split_query(tg):
    assert tg.gemm_tail_split(128, 256, 64, False) == 1        # one tile, one stage
    assert tg.gemm_tail_split(512, 512, 8192, False) >= 2      # 8 tiles, long K
    # One row of tiles, 1..400 of them: the split depends on the last wave
    # only -- none where it fills more than half the units or is empty, one
    # after full waves where it is small.
    units = torch_cuda().cuda.get_device_properties(0).multi_processor_count
    splits = [tg.gemm_tail_split(128, 256 * t, 8192, False) for t in range(1, 401)]
    assert any(s == 1 for s in splits[units // 2 + 8:units - 8])
    assert any(s >= 2 for s in splits[units + 8:])
    assert all(1 <= s <= 4 for s in splits)


@pytest.mark.parametrize("pair", [False, True])
def test_tail_split_after_full_waves(tg, oracle, pair):
    # More tiles than units, a small last wave split along K: full rows
    # sampled from every 128-row block (all column tiles) match bit for bit.
    torch = torch_cuda()
    rng = np.random.default_rng(166 + pair)
    K = 1024
    units = torch.cuda.get_device_properties(0).multi_processor_count // (2 if pair else 1)
    tm = 256 if pair else 128
    shape = None
    for nt in range(4, 40):
        mt = units // nt + 1                              # just over one full wave
        M, N = tm * mt, 256 * nt - 24
        if mt * nt > units and tg.gemm_tail_split(M, N, K, pair) >= 2:
            shape = (M, N)
            break
    if shape is None:
        pytest.skip("no split-after-full-waves shape on this device")
    M, N = shape
    A, B = quarter_bits(rng, (M, K)), quarter_bits(rng, (N, K))
    D = torch.full((M, N), float("nan"), device="cuda")
    tg.gemm_bf16(dev_bf16(A), dev_bf16(B), D, cta_pair=pair)
    assert tg.tg_device_status()[0] == tg.TG_OK
    rows = np.unique(np.concatenate([np.arange(0, M, 128), np.arange(127, M, 128),
                                     rng.integers(0, M, 32)]))
    ref, _ = oracle.gemm_bf16(A, B, rows=rows)
    assert np.array_equal(host_values(D)[rows], ref), f"{M}x{N}x{K}"
