"""GPU parity of tile_transpose_b16: bit-exact against the oracle."""
import numpy as np
import pytest

from blackwell_tile_gemm_gb300 import synth
from tests._gpu import dev_u16, host_u16, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tg():
    torch_cuda()
    import blackwell_tile_gemm_gb300 as m
    m.lib()
    return m


@pytest.mark.parametrize("rows,cols", [(1, 1), (8, 8), (37, 53), (64, 64), (65, 129),
                                       (1000, 3), (3, 1000), (128, 4096), (257, 263)])
def test_transpose_small(tg, oracle, rows, cols):
    # Row strides are rounded up to multiples of 8 elements (16 bytes), as
    # the entry point requires; the padding must stay untouched.
    torch = torch_cuda()
    rng = np.random.default_rng(rows * 1000 + cols)
    X = synth.b16_bits(rng, (rows, cols))
    ld_in, ld_out = -(-cols // 8) * 8, -(-rows // 8) * 8
    src = torch.zeros((rows, ld_in), dtype=torch.int16, device="cuda")
    src[:, :cols] = dev_u16(X)
    dst = torch.full((cols, ld_out), 0x5A5A, dtype=torch.int16, device="cuda")
    tg.tile_transpose_b16(src[:, :cols], dst[:, :rows])
    got = host_u16(dst)
    assert np.array_equal(got[:, :rows], oracle.transpose_b16(X))
    assert np.all(got[:, rows:] == 0x5A5A)


def test_transpose_strided_and_involution(tg, oracle):
    torch = torch_cuda()
    rng = np.random.default_rng(7)
    X = synth.b16_bits(rng, (100, 200))
    big_in = torch.zeros((100, 208), dtype=torch.int16, device="cuda")
    big_in[:, :200] = dev_u16(X)
    big_out = torch.full((200, 112), -1, dtype=torch.int16, device="cuda")
    tg.tile_transpose_b16(big_in[:, :200], big_out[:, :100])
    got = host_u16(big_out)
    assert np.array_equal(got[:, :100], oracle.transpose_b16(X))
    assert np.all(got[:, 100:] == 0xFFFF)                 # padding untouched
    back = tg.tile_transpose_b16(big_out[:, :100])
    assert np.array_equal(host_u16(back), X)


@pytest.mark.slow
def test_transpose_workload_full(tg, oracle):
    x = synth.make_inputs("tr8k")["X"]
    out = tg.tile_transpose_b16(dev_u16(x))
    assert np.array_equal(host_u16(out), oracle.transpose_b16(x))
