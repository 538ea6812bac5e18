"""GPU probes of each building block against the oracle and the pages'
worked examples (bit-exact unless stated)."""
import os

import numpy as np
import pytest

from blackwell_tile_gemm_gb300 import synth
from tests._gpu import dev_bf16, dev_u16, host_u16, torch_cuda

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def P():
    torch_cuda()
    from blackwell_tile_gemm_gb300 import probes
    return probes


def test_add_one_worked_example(P, oracle):
    torch = torch_cuda()
    a = torch.arange(768, dtype=torch.float32, device="cuda").reshape(2, 32, 3, 4)
    b = torch.empty_like(a)
    P.add_one_v4(a, b)
    golden = np.loadtxt(os.path.join(GOLDEN, "add_one_2x32x3x4.txt"), dtype=np.float32)
    assert np.array_equal(b.cpu().numpy().reshape(-1), golden.reshape(-1))
    assert np.array_equal(b.cpu().numpy(), oracle.add_one(a.cpu().numpy()))


def test_ldmatrix_interleaved_worked_example(P):
    torch = torch_cuda()
    x = torch.arange(128, dtype=torch.int32, device="cuda").reshape(16, 4, 2)
    out = torch.zeros((32, 12), dtype=torch.int32, device="cuda")
    P.ldmatrix_x2_interleaved(x, out)
    got = out.cpu().numpy().view(np.uint32).astype(np.uint64)
    golden = np.loadtxt(os.path.join(GOLDEN, "ldmatrix_x2_interleaved.txt"), dtype=np.uint64)
    assert np.array_equal(got, golden)


@pytest.mark.parametrize("n", [1, 2, 4])
@pytest.mark.parametrize("trans", [0, 1])
def test_ldmatrix_register_image(P, oracle, n, trans):
    torch = torch_cuda()
    rng = np.random.default_rng(100 + 10 * n + trans)
    img = synth.b16_bits(rng, (n, 8, 8))
    out = torch.zeros((32, n), dtype=torch.int32, device="cuda")
    P.ldmatrix(dev_u16(img), n, trans, out)
    got = out.cpu().numpy().view(np.uint32)
    assert np.array_equal(got, oracle.ldmatrix_image(img, trans=bool(trans)))


@pytest.mark.parametrize("n", [1, 2, 4])
@pytest.mark.parametrize("trans", [0, 1])
def test_stmatrix_shared_image(P, oracle, n, trans):
    torch = torch_cuda()
    rng = np.random.default_rng(200 + 10 * n + trans)
    regs = rng.integers(0, 1 << 32, (32, n), dtype=np.uint64).astype(np.uint32)
    out = torch.zeros((n, 8, 8), dtype=torch.int16, device="cuda")
    P.stmatrix(torch.from_numpy(regs.view(np.int32)).cuda(), n, trans, out)
    assert np.array_equal(host_u16(out), oracle.stmatrix_image(regs, trans=bool(trans)))


def test_tma_two_boxes_worked_example(P):
    torch = torch_cuda()
    x = torch.arange(256, dtype=torch.int32, device="cuda").reshape(16, 16)
    out = torch.zeros_like(x)
    P.tma_two_boxes(x, out)
    import blackwell_tile_gemm_gb300 as tg
    assert tg.tg_device_status()[0] == tg.TG_OK
    assert torch.equal(out, x)


@pytest.mark.parametrize("rows", [8, 64, 256])
def test_tma_swizzle128_image(P, oracle, rows):
    torch = torch_cuda()
    rng = np.random.default_rng(rows)
    src = synth.b16_bits(rng, (rows, 64))
    out = torch.zeros(rows * 128, dtype=torch.uint8, device="cuda")
    P.tma_swizzle128(dev_u16(src), rows, out)
    got = out.cpu().numpy()
    logical = src.view(np.uint8).reshape(-1)            # unswizzled row-major image
    want = np.empty_like(logical)
    for o in range(logical.size):
        want[oracle.swizzle128(o)] = logical[o]
    assert np.array_equal(got, want)


def _mma(P, a_bits, b_bits, ws=False):
    torch = torch_cuda()
    out = torch.full((128, 64), float("nan"), dtype=torch.float32, device="cuda")
    (P.mma_ws_128x64x64 if ws else P.mma_128x64x64)(dev_bf16(a_bits), dev_bf16(b_bits), out)
    import blackwell_tile_gemm_gb300 as tg
    assert tg.tg_device_status()[0] == tg.TG_OK
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("ws", [False, True], ids=["mma", "mma.ws"])
def test_mma_worked_example_128x64x64(P, oracle, ws):
    # The page's data: default_rng(0), randint(-4, 5) / 4 for a (128, 64) and
    # b (64, 64), B stored as (N, K); checked as a @ b.T at rtol = atol = 2e-4.
    # With .ws the M128 result uses the same TMEM layout, so the same check.
    rng = np.random.default_rng(0)
    a = synth.f32_to_bf16_bits((rng.integers(-4, 5, (128, 64)) / 4).astype(np.float32))
    b = synth.f32_to_bf16_bits((rng.integers(-4, 5, (64, 64)) / 4).astype(np.float32))
    got = _mma(P, a, b, ws)
    ref, _ = oracle.gemm_bf16(a, b)
    np.testing.assert_allclose(got, ref, rtol=2e-4, atol=2e-4)
    assert np.array_equal(got, ref)      # quarter integers: every partial sum is exact


def test_mma_one_hot_locates_tmem_rows_and_columns(P):
    # A = e_i e_k^T, B = e_j e_k^T  =>  D = e_i e_j^T: pins the descriptor
    # strides, the swizzle and the TMEM lane/column of every output.
    one = 0x3F80
    for i, j, k in [(0, 0, 0), (127, 63, 63), (31, 32, 15), (32, 31, 16), (77, 5, 40),
                    (96, 48, 33), (8, 9, 8), (1, 62, 1)]:
        a = np.zeros((128, 64), np.uint16)
        b = np.zeros((64, 64), np.uint16)
        a[i, k] = one
        b[j, k] = one
        got = _mma(P, a, b)
        want = np.zeros((128, 64))
        want[i, j] = 1.0
        assert np.array_equal(got, want), (i, j, k)


def test_mma_identity(P):
    rng = np.random.default_rng(3)
    a = synth.bf16_normal(rng, (128, 64))
    eye = np.zeros((64, 64), np.uint16)
    eye[np.arange(64), np.arange(64)] = 0x3F80
    got = _mma(P, a, eye)
    assert np.array_equal(got, synth.bf16_bits_to_f32(a).astype(np.float64))


def test_bounded_wait_reports_timeout_without_fault(P):
    torch = torch_cuda()
    import blackwell_tile_gemm_gb300 as tg
    tg.tg_device_status()                     # clear
    P.wait_timeout(2_000_000)                 # 2 ms on a barrier nothing completes
    code, site = tg.tg_device_status()
    assert code == tg.TG_ERR_TIMEOUT and site == 99
    assert tg.tg_device_status() == (tg.TG_OK, 0)
    x = torch.ones(4, device="cuda")          # the context is still usable
    assert float((x + 1).sum()) == 8.0


@pytest.mark.parametrize("kind,k", [(0, 16), (1, 32), (2, 32), (3, 64), (4, 64)])
def test_mma_rate_probe_runs(P, kind, k):
    # Back-to-back MMAs on every SM: the measured dense rate per SM and cycle
    # must be positive and not above the nominal 8192 (bf16) / 16384 (fp8) /
    # 49152 (fp4: 13.5 of 4.5 dense PFLOP/s per GPU) FLOP per SM per cycle by
    # more than timing noise.
    torch = torch_cuda()
    import blackwell_tile_gemm_gb300 as tg
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    out = torch.zeros(2 * sms, dtype=torch.int64, device="cuda")
    iters = 256
    P.mma_rate(kind, iters, sms, out)
    assert tg.tg_device_status()[0] == tg.TG_OK
    cyc = out.cpu().numpy()[0::2].astype(np.float64)
    assert np.all(cyc > 0)
    per_clk = 2 * 128 * 256 * k * 4 * iters / cyc
    nominal = {0: 8192, 1: 16384, 2: 16384}.get(kind, 49152)
    assert per_clk.max() <= 1.05 * nominal


def test_tmem_load_shapes_match_the_register_maps(P, oracle):
    # "Explicit CUDA tile patterns", TMEM transfers: each register of each
    # lane holds the TMEM cell the page's formula names, for 16x64b, 16x128b,
    # 16x256b, 32x32b and 16x32bx2 (cells hold row * 256 + column).
    torch = torch_cuda()
    out = torch.zeros((5, 128, 8), dtype=torch.int32, device="cuda")
    P.tmem_shapes(out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint32)
    for s, shape in enumerate(("16x64b", "16x128b", "16x256b", "32x32b", "16x32bx2")):
        want = np.zeros((128, 8), np.uint32)
        for t in range(128):
            w, lane = divmod(t, 32)
            for r in range(8):
                if shape == "16x32bx2":
                    row, col = oracle.tmem_register_coord_16x32bx2(lane, r, 16, 8)
                else:
                    row, col = oracle.tmem_register_coord(shape, lane, r)
                want[t, r] = (32 * w + row) * 256 + col
        assert np.array_equal(got[s], want), shape
