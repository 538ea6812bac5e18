"""The seeded input generators: rounding into the stored formats and recipes."""
import numpy as np
import pytest

from blackwell_tile_gemm_gb300 import synth

torch = pytest.importorskip("torch")


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32),
        (rng.standard_normal(1000) * 1e-30).astype(np.float32),
        # exact ties between two bf16 neighbours (low 16 bits = 0x8000)
        (rng.integers(0, 1 << 15, 1000).astype(np.uint32) << 16 | 0x8000).view(np.float32),
    ])
    x = x[np.isfinite(x)]
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.f32_to_bf16_bits(x), want)


def test_e4m3_rounding_matches_torch():
    rng = np.random.default_rng(1)
    grid = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    vals = grid.to(torch.float64).numpy()
    fin = np.sort(np.unique(vals[np.isfinite(vals)]))
    mids = (fin[1:] + fin[:-1]) / 2                      # exact ties
    x = np.concatenate([rng.standard_normal(100000) * 8, rng.uniform(-448, 448, 10000),
                        mids, fin, rng.standard_normal(1000) * 2.0 ** -8]).astype(np.float32)
    x = np.clip(x, -448, 448)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(synth.f32_to_e4m3fn_bits(x), want)


def test_e4m3_saturates_at_448():
    got = synth.f32_to_e4m3fn_bits(np.array([1e6, -1e6, 460.0], dtype=np.float32))
    assert list(got) == [0x7E, 0xFE, 0x7E]


def test_workload_recipes_are_seeded_and_shaped():
    a = synth.make_inputs("tiny")
    b = synth.make_inputs("tiny")
    assert a["A"].shape == (128, 256) and a["B"].shape == (128, 256)
    assert np.array_equal(a["A"], b["A"]) and np.array_equal(a["B"], b["B"])
    m = synth.make_inputs("mx8k", M=64, N=32, K=128)
    assert m["A"].shape == (64, 128) and m["SFA"].shape == (64, 4) and m["SFB"].shape == (32, 4)
    assert m["SFA"].min() >= 123 and m["SFA"].max() <= 131
    r = synth.make_inputs("ragged", M=40, N=30, K=10)
    f = synth.bf16_bits_to_f32(r["A"])
    assert f.min() >= -1.0 and f.max() <= 1.0
    t = synth.make_inputs("tr8k", M=8, N=16)
    assert t["X"].shape == (8, 16) and t["X"].dtype == np.uint16
