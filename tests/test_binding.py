"""The Python binding's own argument checks, without a GPU: each of these
calls is rejected in Python before the C library is called, so CPU tensors
stand in for device ones (nothing is ever dereferenced or launched)."""
import pytest
import torch

import blackwell_tile_gemm_gb300 as tg


@pytest.fixture(autouse=True)
def no_library(monkeypatch):
    # Any call that got past the Python checks would reach the C library
    # with host pointers; make that fail here instead.
    def refuse():
        raise AssertionError("the binding called the library")
    monkeypatch.setattr(tg, "lib", refuse)


def bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def u8(*shape):
    return torch.zeros(shape, dtype=torch.uint8)


@pytest.mark.parametrize("call,exc", [
    (lambda: tg.gemm_bf16(bf16(8, 16), bf16(8, 32)), ValueError),          # K mismatch
    (lambda: tg.gemm_bf16(torch.zeros(8, 16), bf16(8, 16)), TypeError),     # A not bf16
    (lambda: tg.gemm_bf16(bf16(8, 16), bf16(4, 16), torch.zeros(8, 8)), ValueError),  # D shape
    (lambda: tg.gemm_bf16(bf16(8, 16), bf16(4, 16), bias=torch.zeros(3)), ValueError),
    (lambda: tg.gemm_bf16(bf16(8, 16), bf16(4, 16), epilogue_add=1.0, affine=(1.0, 0.0)),
     ValueError),                                                           # two epilogues
    (lambda: tg.gemm_mxfp8_blockscaled(u8(8, 64), u8(4, 32), u8(8, 2), u8(4, 2)), ValueError),
    (lambda: tg.gemm_mxfp8_blockscaled(u8(8, 64), u8(4, 64), u8(8, 1), u8(4, 2)), ValueError),
    (lambda: tg.gemm_mxfp8_blockscaled(bf16(8, 64), u8(4, 64), u8(8, 2), u8(4, 2)), TypeError),
    (lambda: tg.gemm_mxfp4_blockscaled(u8(8, 32), u8(4, 16), u8(8, 2), u8(4, 2)), ValueError),
    (lambda: tg.gemm_nvfp4_blockscaled(u8(8, 32), u8(4, 32), u8(8, 2), u8(4, 4)), ValueError),
    (lambda: tg.gemm_bf16_skinny(bf16(4, 16), bf16(8, 32)), ValueError),
    (lambda: tg.gemm_bf16_gather(bf16(8, 16), torch.zeros(4, dtype=torch.int64), bf16(4, 16)),
     TypeError),                                                            # idx not int32
    (lambda: tg.tile_transpose_b16(torch.zeros(8, 8)), TypeError),          # 32-bit elements
    (lambda: tg.tile_transpose_b16(bf16(8, 16), bf16(8, 16)), ValueError),  # out not [16, 8]
])
def test_binding_rejects_before_calling_the_library(call, exc):
    with pytest.raises(exc):
        call()


def test_make_epilogue_builds_each_op():
    b = torch.zeros(4)
    assert tg.make_epilogue().op == tg.TG_EPI_NONE
    assert tg.make_epilogue(epilogue_add=2.0).op == tg.TG_EPI_ADD_SCALAR
    assert tg.make_epilogue(affine=(2.0, 1.0)).op == tg.TG_EPI_AFFINE
    assert tg.make_epilogue(silu_affine=(2.0, 1.0)).op == tg.TG_EPI_SILU_AFFINE
    assert tg.make_epilogue(bias=b).op == tg.TG_EPI_BIAS_COL
    assert tg.make_epilogue(bias=b, bias_silu=True).op == tg.TG_EPI_BIAS_COL_SILU
    e = tg.make_epilogue(affine=(2.5, -1.0))
    assert (e.alpha, e.beta) == (2.5, -1.0)
    with pytest.raises(TypeError):
        tg.make_epilogue(bias=torch.zeros(4, dtype=torch.float64))
