"""GPU parity of the block-scaled FP4 GEMMs (gemm_mxfp4_blockscaled,
gemm_nvfp4_blockscaled) against the oracle.

MXFP4: packed E2M1 operands with one E8M0 scale per 32 K elements
(.kind::mxf4nvf4 .scale_vec::2X); NVFP4: one UE4M3 scale per 16
(.scale_vec::4X).  Tolerance per element as for the other products:
|D - ref| <= 1e-5 * sum|a b| + 1e-6 (f32 D) or 8e-3 * sum|a b| + 1e-3
(bf16 D).  With power-of-two scales every product is exact and, at these
sizes, so is every f32 partial sum, so those cases are compared bit for bit:
a misplaced nibble, scale byte, scale id or TMEM column changes some output.
"""
import numpy as np
import pytest

from blackwell_tile_gemm_gb300 import synth
from tests._gpu import assert_within, dev_u8, edge_sample, host_values, torch_cuda

pytestmark = pytest.mark.gpu

KINDS = {"mx": (32, "gemm_mxfp4_blockscaled", "mxf4_8k"),
         "nv": (16, "gemm_nvfp4_blockscaled", "nvf4_8k")}


@pytest.fixture(scope="module")
def tg():
    torch_cuda()
    import blackwell_tile_gemm_gb300 as m
    m.lib()
    return m


def run_fp4(tg, kind, A, B, SFA, SFB, out="bf16", pair=False, **epi):
    torch = torch_cuda()
    dt = torch.float32 if out == "f32" else torch.bfloat16
    D = torch.full((A.shape[0], B.shape[0]), float("nan"), dtype=dt, device="cuda")
    fn = getattr(tg, KINDS[kind][1])
    fn(dev_u8(A), dev_u8(B), dev_u8(SFA), dev_u8(SFB), D, cta_pair=pair, **epi)
    assert tg.tg_device_status()[0] == tg.TG_OK
    return D


def oracle_fp4(oracle, kind, x, **kw):
    return oracle.gemm_fp4(x["A"], x["B"], x["SFA"], x["SFB"],
                           oracle.FP4_MX if kind == "mx" else oracle.FP4_NV, **kw)


def inputs(kind, M, N, K, seed):
    return synth.make_inputs(KINDS[kind][2], M=M, N=N, K=K, seed=seed)


def pow2_scales(kind, rng, shape):
    if kind == "mx":
        return synth.e8m0_scales(rng, shape, -3, 3)
    return synth.ue4m3_pow2_scales(rng, shape)


@pytest.mark.parametrize("kind", ["mx", "nv"])
@pytest.mark.parametrize("pair", [False, True])
def test_fp4_one_tile_bit_exact(tg, oracle, kind, pair):
    # One 128 (256 for a pair) x 256 tile, one K stage of 256: every path of
    # the scale layout is used once.
    block = KINDS[kind][0]
    rng = np.random.default_rng(60 + pair)
    M, N, K = (256 if pair else 128), 256, 256
    x = {"A": synth.e2m1_normal_packed(rng, (M, K)), "B": synth.e2m1_normal_packed(rng, (N, K)),
         "SFA": pow2_scales(kind, rng, (M, K // block)),
         "SFB": pow2_scales(kind, rng, (N, K // block))}
    got = host_values(run_fp4(tg, kind, x["A"], x["B"], x["SFA"], x["SFB"], "f32", pair))
    ref, _ = oracle_fp4(oracle, kind, x)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("kind", ["mx", "nv"])
@pytest.mark.parametrize("pair", [False, True])
def test_fp4_several_tiles_and_stages_bit_exact(tg, oracle, kind, pair):
    block = KINDS[kind][0]
    rng = np.random.default_rng(62 + pair)
    M, N, K = 512, 768, 1024
    x = {"A": synth.e2m1_normal_packed(rng, (M, K)), "B": synth.e2m1_normal_packed(rng, (N, K)),
         "SFA": pow2_scales(kind, rng, (M, K // block)),
         "SFB": pow2_scales(kind, rng, (N, K // block))}
    got = host_values(run_fp4(tg, kind, x["A"], x["B"], x["SFA"], x["SFB"], "f32", pair))
    ref, _ = oracle_fp4(oracle, kind, x)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("kind", ["mx", "nv"])
@pytest.mark.parametrize("pair", [False, True])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_fp4_workload_recipe_small(tg, oracle, kind, pair, out):
    x = inputs(kind, 384, 512, 768, 70)
    got = host_values(run_fp4(tg, kind, x["A"], x["B"], x["SFA"], x["SFB"], out, pair))
    ref, mag = oracle_fp4(oracle, kind, x)
    assert_within(got, ref, mag, out == "bf16", f"{kind} small {out}")


@pytest.mark.parametrize("kind", ["mx", "nv"])
@pytest.mark.parametrize("pair", [False, True])
@pytest.mark.parametrize("M,N,K", [(1, 16, 64), (100, 72, 96), (300, 264, 352), (129, 264, 800)])
def test_fp4_ragged(tg, oracle, kind, pair, M, N, K):
    block = KINDS[kind][0]
    K = K // block * block
    x = inputs(kind, M, N, K, M + N + K)
    got = host_values(run_fp4(tg, kind, x["A"], x["B"], x["SFA"], x["SFB"], "f32", pair,
                              epilogue_add=1.0))
    ref, mag = oracle_fp4(oracle, kind, x, add=1.0)
    assert_within(got, ref, mag, False, f"{kind} ragged {M}x{N}x{K}")


@pytest.mark.parametrize("kind", ["mx", "nv"])
def test_fp4_affine_epilogue(tg, oracle, kind):
    # NVFP4's second-level (per-tensor) scale as D = acc * s + t.
    x = inputs(kind, 256, 256, 512, 80)
    got = host_values(run_fp4(tg, kind, x["A"], x["B"], x["SFA"], x["SFB"], "f32", True,
                              affine=(0.375, -2.0)))
    ref, mag = oracle_fp4(oracle, kind, x)
    want = oracle.apply_epilogue(ref, oracle.EPI_AFFINE, 0.375, -2.0)
    tol = 0.375 * (1e-5 * mag + 1e-6) + 2.0 ** -21 * np.abs(want) + 1e-6
    assert np.all(np.abs(got - want) <= tol)


@pytest.mark.parametrize("kind", ["mx", "nv"])
def test_fp4_k_zero_fills_epilogue(tg, kind):
    torch = torch_cuda()
    fn = getattr(tg, KINDS[kind][1])
    A = torch.empty((5, 0), dtype=torch.uint8, device="cuda")
    B = torch.empty((8, 0), dtype=torch.uint8, device="cuda")
    S = torch.empty((5, 0), dtype=torch.uint8, device="cuda")
    T = torch.empty((8, 0), dtype=torch.uint8, device="cuda")
    D = torch.full((5, 8), float("nan"), device="cuda")
    fn(A, B, S, T, D, epilogue_add=2.5)
    assert torch.all(D == 2.5)


@pytest.mark.slow
@pytest.mark.parametrize("kind", ["mx", "nv"])
def test_fp4_8k_workload_sampled(tg, oracle, kind):
    w = synth.WORKLOADS[KINDS[kind][2]]
    x = synth.make_inputs(w)
    got = host_values(run_fp4(tg, kind, x["A"], x["B"], x["SFA"], x["SFB"], "bf16", True))
    rows = edge_sample(w.M, 256, 15)
    cols = edge_sample(w.N, 256, 16)
    ref, mag = oracle_fp4(oracle, kind, x, rows=rows)
    assert_within(got[rows], ref, mag, True, f"{kind} 8k rows")
    ref, mag = oracle_fp4(oracle, kind, x, cols=cols)
    assert_within(got[:, cols], ref, mag, True, f"{kind} 8k cols")
