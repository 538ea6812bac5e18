"""Helpers shared by the GPU parity tests: host<->device moves and the
tolerance check.  No arithmetic of the contraction lives here."""
import numpy as np

from blackwell_tile_gemm_gb300 import synth

# Tolerances: |D - ref| <= RTOL * sum_k |a_k b_k| + ATOL, per output element.
F32_RTOL, F32_ATOL = 1e-5, 1e-6
BF16_RTOL, BF16_ATOL = 8e-3, 1e-3


def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        import pytest
        pytest.skip("no CUDA device")
    return torch


def dev_bf16(bits: np.ndarray):
    torch = torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def dev_u8(bits: np.ndarray):
    torch = torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint8)).cuda()


def dev_u16(bits: np.ndarray):
    torch = torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def host_values(D) -> np.ndarray:
    """Device D (float32 or bfloat16) -> float64 numpy, exactly."""
    import torch
    if D.dtype == torch.float32:
        return D.cpu().numpy().astype(np.float64)
    if D.dtype == torch.bfloat16:
        bits = D.view(torch.int16).cpu().numpy().view(np.uint16)
        return synth.bf16_bits_to_f32(bits).astype(np.float64)
    raise TypeError(D.dtype)


def host_u16(X) -> np.ndarray:
    import torch
    return X.view(torch.int16).cpu().numpy().view(np.uint16)


def worst_ratio(got: np.ndarray, ref: np.ndarray, mag: np.ndarray, rtol: float, atol: float):
    """max over elements of |got - ref| / (rtol * mag + atol), and its index."""
    err = np.abs(got - ref)
    ratio = err / (rtol * mag + atol)
    if not np.all(np.isfinite(got)):
        return float("inf"), tuple(np.argwhere(~np.isfinite(got))[0])
    idx = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
    return float(ratio[idx]), tuple(int(i) for i in idx)


def assert_within(got, ref, mag, bf16_out: bool, what: str = ""):
    rtol, atol = (BF16_RTOL, BF16_ATOL) if bf16_out else (F32_RTOL, F32_ATOL)
    r, idx = worst_ratio(got, ref, mag, rtol, atol)
    assert r <= 1.0, (f"{what}: worst |D-ref|/tol = {r:.3g} at {idx}: got {got[idx]!r} "
                      f"ref {ref[idx]!r} mag {mag[idx]!r}")
    return r


def sample_indices(n: int, count: int, seed: int, tile: int) -> np.ndarray:
    """Seeded sample of indices in [0, n): tile edges, the last index, random ones."""
    rng = np.random.default_rng(seed)
    edges = [0, n - 1]
    for t in range(tile, n, tile):
        edges += [t - 1, t]
    edges = np.array(sorted(set(i for i in edges if 0 <= i < n)), dtype=np.int64)
    if edges.size > count // 2:
        edges = edges[np.linspace(0, edges.size - 1, count // 2).astype(np.int64)]
    rand = rng.choice(n, size=min(n, count - edges.size), replace=False)
    return np.unique(np.concatenate([edges, rand]).astype(np.int64))


def edge_sample(n: int, count: int, seed: int, tile: int = 128) -> np.ndarray:
    """Every index on either side of a tile boundary (multiples of `tile`), 0
    and n - 1, then seeded random indices up to `count` in all."""
    edges = {0, n - 1}
    for t in range(tile, n, tile):
        edges.update((t - 1, t))
    edges = np.array(sorted(i for i in edges if 0 <= i < n), dtype=np.int64)
    rest = np.setdiff1d(np.arange(n, dtype=np.int64), edges)
    k = max(0, min(rest.size, count - edges.size))
    rand = np.random.default_rng(seed).choice(rest, size=k, replace=False)
    return np.unique(np.concatenate([edges, rand]))
