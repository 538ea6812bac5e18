"""Seeded random sweep of gemm_bf16 against the oracle, every element.

Each case draws a shape (ragged M, N, K, odd K included), row strides (with
NaN in any padding, which must be neither read nor written), the kernel
mode (single CTA, CTA pair, the two multicast cluster kinds), the output
type and an epilogue, so that the modes meet each other: tail splits (small
M x N with long K), the TMA-store epilogue and its ragged-column fallback,
odd K over padded rows.

Tolerance, as for the fused epilogues: the product's bound (1e-5 * sum|a b|
+ 1e-6 for f32 D, 8e-3 * sum|a b| + 1e-3 for bf16 D) times the epilogue's
Lipschitz constant, plus one rounding of the output type (2^-21 or 2^-8 of
|ref|).
"""
import numpy as np
import pytest

from blackwell_tile_gemm_gb300 import synth
from tests._gpu import dev_bf16, host_values, torch_cuda

pytestmark = pytest.mark.gpu

MODES = {"single": dict(), "pair": dict(cta_pair=True), "mc1": dict(multicast=True),
         "mc": dict(cta_pair=True, multicast=True)}


@pytest.fixture(scope="module")
def tg():
    torch_cuda()
    import blackwell_tile_gemm_gb300 as m
    m.lib()
    return m


def draw_case(seed):
    rng = np.random.default_rng(seed)
    M = int(rng.choice([int(rng.integers(1, 300)), int(rng.integers(300, 1400))]))
    N = int(rng.choice([int(rng.integers(1, 300)), int(rng.integers(300, 1400))]))
    K = int(rng.choice([int(rng.integers(1, 200)), int(rng.integers(200, 2100))]))
    pad_k = int(rng.choice([0, 0, 8, 24]))
    lda = (K + 7) // 8 * 8 + pad_k
    ldb = (K + 7) // 8 * 8 + int(rng.choice([0, 8]))
    mode = str(rng.choice(list(MODES)))
    out = str(rng.choice(["f32", "bf16"]))
    epi = str(rng.choice(["none", "add", "affine", "silu_affine", "bias", "bias_silu"]))
    return rng, M, N, K, lda, ldb, mode, out, epi


@pytest.mark.parametrize("seed", range(40))
def test_random_case(tg, oracle, seed):
    torch = torch_cuda()
    rng, M, N, K, lda, ldb, mode, out, epi = draw_case(1000 + seed)
    A = np.full((M, lda), 0x7FC0, np.uint16)
    B = np.full((N, ldb), 0x7FC0, np.uint16)
    A[:, :K] = synth.bf16_uniform(rng, (M, K))
    B[:, :K] = synth.bf16_uniform(rng, (N, K))
    bias_np = (rng.standard_normal(N) * 2).astype(np.float32)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    ldd = (N + 1 + 7) // 8 * 8
    Dfull = torch.full((M + 8, ldd), float("nan"), dtype=dt, device="cuda")
    kw = {"none": {}, "add": dict(epilogue_add=0.75), "affine": dict(affine=(1.25, -0.5)),
          "silu_affine": dict(silu_affine=(0.5, 0.25)),
          "bias": dict(bias=torch.from_numpy(bias_np).cuda()),
          "bias_silu": dict(bias=torch.from_numpy(bias_np).cuda(), bias_silu=True)}[epi]
    tg.gemm_bf16(dev_bf16(A)[:, :K], dev_bf16(B)[:, :K], Dfull[:M, :N], **MODES[mode], **kw)
    assert tg.tg_device_status()[0] == tg.TG_OK
    got = host_values(Dfull)
    ref, mag = oracle.gemm_bf16(A[:, :K], B[:, :K])
    op = {"none": (oracle.EPI_NONE, {}), "add": (oracle.EPI_ADD_SCALAR, dict(alpha=0.75)),
          "affine": (oracle.EPI_AFFINE, dict(alpha=1.25, beta=-0.5)),
          "silu_affine": (oracle.EPI_SILU_AFFINE, dict(alpha=0.5, beta=0.25)),
          "bias": (oracle.EPI_BIAS_COL, dict(bias=bias_np)),
          "bias_silu": (oracle.EPI_BIAS_COL_SILU, dict(bias=bias_np))}[epi]
    want = oracle.apply_epilogue(ref, op[0], **op[1])
    # The tolerance of the product, carried through the epilogue's slope
    # (at most |alpha| * 1.1 for SiLU), plus one rounding of the output type.
    slope = {"none": 1.0, "add": 1.0, "affine": 1.25, "silu_affine": 0.55, "bias": 1.0,
             "bias_silu": 1.1}[epi]
    rtol, atol = (8e-3, 1e-3) if out == "bf16" else (1e-5, 1e-6)
    eps = 2.0 ** -8 if out == "bf16" else 2.0 ** -21
    tol = slope * (rtol * mag + atol) + eps * np.abs(want)
    case = f"seed {seed}: {M}x{N}x{K} lda {lda} ldb {ldb} {mode} {out} {epi}"
    assert np.all(np.abs(got[:M, :N] - want) <= tol), case
    assert np.all(np.isnan(got[:M, N:])) and np.all(np.isnan(got[M:, :])), case
