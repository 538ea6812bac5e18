"""GPU parity of the fused epilogues (the pages' silu_affine scalar
composition, a constant, a per-column bias) on both GEMM paths.

Tolerance: the epilogue is Lipschitz with constant L (1 for the additive
ops, 1.1 * |scale| for silu_affine, 1.1 for bias+silu; |silu'| <= 1.0998),
so the accumulator tolerance of the plain product carries through as
L * (rtol * sum|a b| + atol); the output rounding adds eps * |ref| with
eps = 2^-8 for bf16 D and 2^-21 for f32 D (expf and the f32 arithmetic).
"""
import numpy as np
import pytest

from blackwell_tile_gemm_gb300 import synth
from tests._gpu import (BF16_ATOL, BF16_RTOL, F32_ATOL, F32_RTOL, dev_bf16, dev_u8, host_values,
                        torch_cuda)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tg():
    torch_cuda()
    import blackwell_tile_gemm_gb300 as m
    m.lib()
    return m


CASES = [  # (name, oracle op, kwargs builder, Lipschitz constant)
    ("add", 1, lambda b: dict(epilogue_add=0.75), lambda: 1.0),
    ("silu_affine", 2, lambda b: dict(silu_affine=(2.0, 1.0)), lambda: 2.2),
    ("bias", 3, lambda b: dict(bias=b), lambda: 1.0),
    ("bias_silu", 4, lambda b: dict(bias=b, bias_silu=True), lambda: 1.1),
]


def _check(oracle, got, ref, mag, op, bias_np, lip, bf16_out, what):
    alpha, beta = {1: (0.75, 0.0), 2: (2.0, 1.0)}.get(op, (0.0, 0.0))
    want = oracle.apply_epilogue(ref, op, alpha, beta, bias=bias_np)
    rtol, atol = (BF16_RTOL, BF16_ATOL) if bf16_out else (F32_RTOL, F32_ATOL)
    eps = 2.0 ** -8 if bf16_out else 2.0 ** -21
    tol = lip * (rtol * mag + atol) + eps * np.abs(want)
    err = np.abs(got - want)
    i = np.unravel_index(int(np.argmax(err / tol)), err.shape)
    assert np.all(err <= tol), f"{what}: at {i} got {got[i]} want {want[i]} tol {tol[i]}"


@pytest.mark.parametrize("name,op,kw,lip", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("pair", [False, True, "mc", "mc1"])
def test_bf16_gemm_epilogues(tg, oracle, name, op, kw, lip, out, pair):
    torch = torch_cuda()
    rng = np.random.default_rng(op * 10 + (out == "bf16"))
    M, N, K = 300, 264, 200
    A, B = synth.bf16_uniform(rng, (M, K)), synth.bf16_uniform(rng, (N, K))
    bias_np = (rng.standard_normal(N) * 4).astype(np.float32)
    bias = torch.from_numpy(bias_np).cuda()
    dt = torch.float32 if out == "f32" else torch.bfloat16
    D = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
    tg.gemm_bf16(dev_bf16(A), dev_bf16(B), D, cta_pair=pair in (True, "mc"),
                 multicast=pair in ("mc", "mc1"), **kw(bias))
    assert tg.tg_device_status()[0] == tg.TG_OK
    ref, mag = oracle.gemm_bf16(A, B)
    _check(oracle, host_values(D), ref, mag, op, bias_np, lip(), out == "bf16", name)


@pytest.mark.parametrize("name,op,kw,lip", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("pair", [False, True])
def test_mxfp8_gemm_epilogues(tg, oracle, name, op, kw, lip, pair):
    torch = torch_cuda()
    x = synth.make_inputs("mx8k", M=256, N=320, K=256, seed=50 + op)
    bias_np = (np.random.default_rng(op).standard_normal(320) * 4).astype(np.float32)
    bias = torch.from_numpy(bias_np).cuda()
    D = torch.full((256, 320), float("nan"), dtype=torch.bfloat16, device="cuda")
    tg.gemm_mxfp8_blockscaled(*(dev_u8(x[k]) for k in ("A", "B", "SFA", "SFB")), D,
                              cta_pair=pair, **kw(bias))
    assert tg.tg_device_status()[0] == tg.TG_OK
    ref, mag = oracle.gemm_mxfp8(x["A"], x["B"], x["SFA"], x["SFB"])
    _check(oracle, host_values(D), ref, mag, op, bias_np, lip(), True, name)


def test_k_zero_applies_the_epilogue_to_zero(tg, oracle):
    torch = torch_cuda()
    bias_np = np.linspace(-3, 3, 24).astype(np.float32)
    bias = torch.from_numpy(bias_np).cuda()
    A = torch.empty((5, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((24, 0), dtype=torch.bfloat16, device="cuda")
    D = torch.full((5, 24), float("nan"), device="cuda")
    tg.gemm_bf16(A, B, D, bias=bias, bias_silu=True)
    want = oracle.apply_epilogue(np.zeros((5, 24)), oracle.EPI_BIAS_COL_SILU, bias=bias_np)
    assert np.allclose(D.cpu().numpy(), want, rtol=1e-6, atol=1e-6)
