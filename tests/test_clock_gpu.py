"""The SM clock readout of the GEMM kernels (tg_kernel_clock_record / _read).

NVML can report the maximum SM clock while a power-capped tensor kernel runs
slower; the readout takes the clock from the kernels' own cycle counter and
global timer.  The host-side argument checks run without a GPU; the GPU test
checks that recording adds per kind, stops when asked, and leaves the
results unchanged bit for bit."""
import ctypes

import numpy as np
import pytest

import blackwell_tile_gemm_gb300 as tg
from blackwell_tile_gemm_gb300 import build as tgbuild


def test_clock_read_rejects_unknown_kinds_and_null_output():
    tgbuild.build()
    L = tg.lib()
    mhz = ctypes.c_double(0.0)
    assert L.tg_kernel_clock_read(4, ctypes.byref(mhz), None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_kernel_clock_read(-1, ctypes.byref(mhz), None) == tg.TG_ERR_INVALID_ARG
    assert L.tg_kernel_clock_read(tg.TG_CLOCK_BF16, None, None) == tg.TG_ERR_INVALID_ARG


@pytest.mark.gpu
def test_clock_readout_per_kind_and_bit_identical_results():
    from tests._gpu import torch_cuda
    torch = torch_cuda()
    g = torch.Generator(device="cuda").manual_seed(5)
    A = torch.randn(2048, 2048, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(2048, 2048, device="cuda", generator=g).to(torch.bfloat16)
    D0 = torch.empty(2048, 2048, device="cuda")
    D1 = torch.empty_like(D0)
    tg.gemm_bf16(A, B, D0, cta_pair=True)                   # not recorded
    tg.kernel_clock_record(True)
    for _ in range(3):
        tg.gemm_bf16(A, B, D1, cta_pair=True)
    mhz, units = tg.kernel_clock_read(tg.TG_CLOCK_BF16)
    assert 300.0 < mhz < 3000.0, mhz
    assert units >= 3 and units % 3 == 0, units              # the same units each launch
    assert torch.equal(D0, D1)
    assert tg.kernel_clock_read(tg.TG_CLOCK_NVFP4) == (0.0, 0)

    # a block-scaled launch adds to its own kind only
    x = np.random.default_rng(6)
    mA = torch.from_numpy(x.integers(0, 0x7E, (512, 1024), dtype=np.uint8)).cuda()
    mB = torch.from_numpy(x.integers(0, 0x7E, (512, 1024), dtype=np.uint8)).cuda()
    sA = torch.full((512, 32), 127, dtype=torch.uint8, device="cuda")
    tg.gemm_mxfp8_blockscaled(mA, mB, sA, sA, cta_pair=True)
    mx_mhz, mx_units = tg.kernel_clock_read(tg.TG_CLOCK_MXFP8)
    assert 300.0 < mx_mhz < 3000.0 and mx_units > 0
    assert tg.kernel_clock_read(tg.TG_CLOCK_BF16)[1] == units

    # stopped: later launches add nothing, the sums stay readable
    tg.kernel_clock_record(False)
    tg.gemm_bf16(A, B, D1, cta_pair=True)
    assert tg.kernel_clock_read(tg.TG_CLOCK_BF16) == (mhz, units)
    assert tg.tg_device_status() == (tg.TG_OK, 0)
