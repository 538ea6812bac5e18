"""gemm_mxfp8_blockscaled_noalloc: the block-scaled GEMM for callers that must
not allocate device memory (a framework whose pool owns the device memory, a
latency-bound loop where cudaMalloc/cudaFree would synchronise the device, a
deployment that forbids allocation after start-up).  It takes its scratch
from a fixed 8 MiB array built into the library.

The GPU test calls the new entry point through the C ABI three times in a
row, on different problems (the first one's scale images nearly fill the
array), and checks each result bit for bit against the regular entry point
(gemm_mxfp8_blockscaled) on the same inputs and against the float64 oracle
within the tolerance the other parity tests use.  The file name sorts last so
that a run that stops at the first failure has already run every other test;
it also passes alone in a fresh process, where its first call performs the
per-device set-up.
"""
import ctypes

import numpy as np
import pytest

import blackwell_tile_gemm_gb300 as tg
from blackwell_tile_gemm_gb300 import build as tgbuild
from blackwell_tile_gemm_gb300 import synth

A16 = 0x10000      # a 16-byte aligned stand-in address, never dereferenced


def _raw_call(L, A, B, SFA, SFB, D, pair, stream):
    M, K = A.shape
    N = B.shape[0]
    return L.gemm_mxfp8_blockscaled_noalloc(
        A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), SFA.data_ptr(), SFA.stride(0),
        SFB.data_ptr(), SFB.stride(0), D.data_ptr(), D.stride(0), M, N, K,
        tg.TG_D_F32 if D.dtype.itemsize == 4 else tg.TG_D_BF16, tg.TG_EPI_ADD_SCALAR, 0.5,
        tg.TG_FLAG_CTA_PAIR if pair else 0, ctypes.c_void_p(stream.cuda_stream))


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 16384 x 16384 x 16384 in CTA pairs needs (128 + 128) * 128 * 512 bytes =
    # 16 MiB of scale images, twice the scratch; rejected before any CUDA call.
    tgbuild.build()
    L = tg.lib()
    rc = L.gemm_mxfp8_blockscaled_noalloc(A16, 16384, A16, 16384, A16, 512, A16, 512, A16, 16384,
                                          16384, 16384, 16384, 1, 0, 0.0, 1, None)
    assert rc == tg.TG_ERR_NO_SCRATCH
    assert "scratch" in tg.status_string(rc)


def _big_case_inputs(M, N, K, seed):
    """Random E4M3 bit patterns (NaN codes replaced by zero) and E8M0 scales
    127 + U{-4..4}: drawn directly as bytes, which is fast at these sizes."""
    rng = np.random.default_rng(seed)
    out = {}
    for name, rows in (("A", M), ("B", N)):
        x = rng.integers(0, 256, (rows, K), dtype=np.uint8)
        x[(x & 0x7F) == 0x7F] = 0
        out[name] = x
    out["SFA"] = (127 + rng.integers(-4, 5, (M, K // 32))).astype(np.uint8)
    out["SFB"] = (127 + rng.integers(-4, 5, (N, K // 32))).astype(np.uint8)
    return out


@pytest.mark.gpu
def test_noalloc_matches_allocating_entry_point_calls_in_a_row(oracle):
    """Three calls of the no-allocation entry point in a row, through the C
    ABI: each result equals the regular (allocating) entry point's bit for
    bit -- both run the same kernels on the same inputs -- and matches the
    float64 oracle within the parity tolerance.  The first problem's scale
    images fill 7.75 MiB of the 8 MiB array; the later, smaller ones run over
    what it left behind."""
    from tests._gpu import (BF16_ATOL, BF16_RTOL, F32_ATOL, F32_RTOL, dev_u8, edge_sample,
                            host_values, worst_ratio)
    from tests._gpu import torch_cuda
    torch = torch_cuda()
    L = tg.lib()
    stream = torch.cuda.current_stream()
    cases = [
        # (M, N, K, D dtype, CTA pairs, seed)
        (4096, 4096, 31744, torch.bfloat16, True, 73),   # (32 + 32) * 248 * 512 B of images
        (512, 768, 1024, torch.bfloat16, True, 71),
        (300, 264, 160, torch.float32, False, 72),
    ]
    for M, N, K, dt, pair, seed in cases:
        need = tg.workspace_bytes(tg.TG_CALL_GEMM_MXFP8, M, N, K,
                                  flags=tg.TG_FLAG_CTA_PAIR if pair else 0)
        assert need <= 8 << 20
        big = need >= (15 << 19)                         # >= 7.5 MiB
        x = _big_case_inputs(M, N, K, seed) if big else \
            synth.make_inputs("mx8k", M=M, N=N, K=K, seed=seed)
        A, B, SFA, SFB = (dev_u8(x[k]) for k in ("A", "B", "SFA", "SFB"))
        D_new = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
        D_ref = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
        torch.cuda.synchronize()
        assert _raw_call(L, A, B, SFA, SFB, D_new, pair, stream) == tg.TG_OK
        tg.gemm_mxfp8_blockscaled(A, B, SFA, SFB, D_ref, epilogue_add=0.5, cta_pair=pair)
        assert tg.tg_device_status() == (tg.TG_OK, 0)
        assert torch.equal(D_new.view(torch.int16) if dt == torch.bfloat16 else D_new.view(torch.int32),
                           D_ref.view(torch.int16) if dt == torch.bfloat16 else D_ref.view(torch.int32)), \
            (M, N, K, "differs from the allocating entry point")
        got = host_values(D_new)
        rows = edge_sample(M, 32, seed, tile=1024) if big else np.arange(M)
        cols = edge_sample(N, 32, seed + 1, tile=1024) if big else np.arange(N)
        rtol, atol = (F32_RTOL, F32_ATOL) if dt == torch.float32 else (BF16_RTOL, BF16_ATOL)
        ref, mag = oracle.gemm_mxfp8(x["A"], x["B"], x["SFA"], x["SFB"], add=0.5, rows=rows)
        ratio, idx = worst_ratio(got[rows], ref, mag, rtol, atol)
        assert ratio <= 1.0, (M, N, K, "rows", idx)
        ref, mag = oracle.gemm_mxfp8(x["A"], x["B"], x["SFA"], x["SFB"], add=0.5, cols=cols)
        ratio, idx = worst_ratio(got[:, cols], ref, mag, rtol, atol)
        assert ratio <= 1.0, (M, N, K, "cols", idx)
        del A, B, SFA, SFB, D_new, D_ref
