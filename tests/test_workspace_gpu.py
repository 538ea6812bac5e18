"""GPU tests of the library's own device memory: explicit reservation, graph
capture without a reservation, the tail split beside kernels that hold SMs,
and the rule that multicast clusters only cover the current device's memory.

Every result is compared with the oracle on quarter-integer (exact) inputs,
bit for bit, or within the parity tolerance for general inputs.
"""
import numpy as np
import pytest

from blackwell_tile_gemm_gb300 import synth
from tests._gpu import assert_within, dev_bf16, dev_u8, host_values, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tg():
    torch_cuda()
    import blackwell_tile_gemm_gb300 as m
    m.lib()
    return m


def quarter_bits(rng, shape):
    return synth.f32_to_bf16_bits((rng.integers(-4, 5, shape) / 4).astype(np.float32))


def split_shape(tg, pair, K):
    """(M, N) of a bf16 product that gemm_bf16 splits along K on this device."""
    tm = 256 if pair else 128
    for nt in range(1, 40):
        for mt in range(1, 40):
            M, N = tm * mt, 256 * nt - 8
            if tg.gemm_tail_split(M, N, K, pair) >= 2:
                return M, N
    pytest.skip("no tail-split shape on this device")


def test_reserved_stream_allocates_nothing(tg, oracle):
    """After tg_reserve_workspace, every call kind on the stream runs without a
    single device allocation, and gives the oracle's result."""
    torch = torch_cuda()
    rng = np.random.default_rng(301)
    s = torch.cuda.Stream()
    # the calls below, with the workspace each one needs
    bf_M, bf_N, bf_K = 4000, 3000, 1000                 # 2000-byte rows: re-pitched
    sp_K = 1024
    sp_M, sp_N = split_shape(tg, True, sp_K)
    mx = synth.make_inputs("mx8k", M=512, N=768, K=1024, seed=302)
    f4 = synth.make_inputs("mxf4_8k", M=384, N=512, K=1024, seed=303)
    nv = synth.make_inputs("nvf4_8k", M=384, N=512, K=1024, seed=304)
    sk = dict(M=16, N=2048, K=4096)
    ga = dict(a_rows=2048, M=700, N=512, K=512)
    need = max(
        tg.workspace_bytes(tg.TG_CALL_GEMM_BF16, bf_M, bf_N, bf_K, bf_K, bf_K),
        tg.workspace_bytes(tg.TG_CALL_GEMM_MXFP8, 512, 768, 1024),
        tg.workspace_bytes(tg.TG_CALL_GEMM_MXFP4, 384, 512, 1024, flags=tg.TG_FLAG_CTA_PAIR),
        tg.workspace_bytes(tg.TG_CALL_GEMM_NVFP4, 384, 512, 1024),
        tg.workspace_bytes(tg.TG_CALL_GEMM_BF16_SKINNY, sk["M"], sk["N"], sk["K"],
                           d_dtype=tg.TG_D_BF16),
        tg.workspace_bytes(tg.TG_CALL_GEMM_BF16_GATHER, ga["M"], ga["N"], ga["K"]))
    assert need > 0
    tg.reserve_workspace(need, stream=s)
    before = tg.workspace_alloc_count()
    outs = []
    with torch.cuda.stream(s):
        A, B = synth.bf16_uniform(rng, (bf_M, bf_K)), synth.bf16_uniform(rng, (bf_N, bf_K))
        D = torch.full((bf_M, bf_N), float("nan"), device="cuda")
        tg.gemm_bf16(dev_bf16(A), dev_bf16(B), D, epilogue_add=1.0, stream=s)
        outs.append(("bf16 re-pitched", D, lambda r=np.arange(0, bf_M, 37):
                     (r, *oracle.gemm_bf16(A, B, add=1.0, rows=r)), False))
        As, Bs = quarter_bits(rng, (sp_M, sp_K)), quarter_bits(rng, (sp_N, sp_K))
        Ds = torch.full((sp_M, sp_N), float("nan"), device="cuda")
        tg.gemm_bf16(dev_bf16(As), dev_bf16(Bs), Ds, cta_pair=True, stream=s)
        Dm = torch.full((512, 768), float("nan"), device="cuda")
        tg.gemm_mxfp8_blockscaled(*(dev_u8(mx[k]) for k in ("A", "B", "SFA", "SFB")), Dm,
                                  stream=s)
        D4 = torch.full((384, 512), float("nan"), device="cuda")
        tg.gemm_mxfp4_blockscaled(*(dev_u8(f4[k]) for k in ("A", "B", "SFA", "SFB")), D4,
                                  cta_pair=True, stream=s)
        Dn = torch.full((384, 512), float("nan"), device="cuda")
        tg.gemm_nvfp4_blockscaled(*(dev_u8(nv[k]) for k in ("A", "B", "SFA", "SFB")), Dn,
                                  stream=s)
        Ak = synth.bf16_uniform(rng, (sk["M"], sk["K"]))
        Bk = synth.bf16_uniform(rng, (sk["N"], sk["K"]))
        Dk = torch.full((sk["M"], sk["N"]), float("nan"), dtype=torch.bfloat16, device="cuda")
        tg.gemm_bf16_skinny(dev_bf16(Ak), dev_bf16(Bk), Dk, stream=s)
        Ag = synth.bf16_uniform(rng, (ga["a_rows"], ga["K"]))
        Bg = synth.bf16_uniform(rng, (ga["N"], ga["K"]))
        idx = rng.integers(0, ga["a_rows"], ga["M"]).astype(np.int32)
        Dg = torch.full((ga["M"], ga["N"]), float("nan"), device="cuda")
        tg.gemm_bf16_gather(dev_bf16(Ag), torch.from_numpy(idx).cuda(), dev_bf16(Bg), Dg,
                            stream=s)
    s.synchronize()
    assert tg.workspace_alloc_count() == before, "a call on the reserved stream allocated"
    assert tg.tg_device_status(s)[0] == tg.TG_OK
    r, ref, mag = outs[0][2]()
    assert_within(host_values(outs[0][1])[r], ref, mag, False, "bf16 re-pitched")
    assert np.array_equal(host_values(Ds), oracle.gemm_bf16(As, Bs)[0]), "tail split"
    ref, mag = oracle.gemm_mxfp8(mx["A"], mx["B"], mx["SFA"], mx["SFB"])
    assert_within(host_values(Dm), ref, mag, False, "mxfp8")
    ref, mag = oracle.gemm_mxfp4(f4["A"], f4["B"], f4["SFA"], f4["SFB"])
    assert_within(host_values(D4), ref, mag, False, "mxfp4")
    ref, mag = oracle.gemm_nvfp4(nv["A"], nv["B"], nv["SFA"], nv["SFB"])
    assert_within(host_values(Dn), ref, mag, False, "nvfp4")
    ref, mag = oracle.gemm_bf16(Ak, Bk)
    assert_within(host_values(Dk), ref, mag, True, "skinny")
    ref, mag = oracle.gemm_bf16(Ag, Bg, rows=idx)
    assert_within(host_values(Dg), ref, mag, False, "gather")


def test_reserved_workspace_too_small_is_refused(tg):
    """A call that needs more workspace than its stream reserved returns
    TG_ERR_WORKSPACE before anything is launched or allocated."""
    torch = torch_cuda()
    s = torch.cuda.Stream()
    tg.reserve_workspace(0, stream=s)          # the smallest workspace (1 MiB)
    M = N = 4096
    K = 8192                                   # 2 MiB of scale images
    assert tg.workspace_bytes(tg.TG_CALL_GEMM_MXFP8, M, N, K) > (1 << 20)
    A = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    B = torch.empty((N, K), dtype=torch.uint8, device="cuda")
    SFA = torch.empty((M, K // 32), dtype=torch.uint8, device="cuda")
    SFB = torch.empty((N, K // 32), dtype=torch.uint8, device="cuda")
    D = torch.full((M, N), float("nan"), device="cuda")
    torch.cuda.synchronize()
    before = tg.workspace_alloc_count()
    with pytest.raises(tg.TgError) as ei:
        tg.gemm_mxfp8_blockscaled(A, B, SFA, SFB, D, stream=s)
    assert ei.value.code == tg.TG_ERR_WORKSPACE
    s.synchronize()
    assert tg.workspace_alloc_count() == before
    assert torch.isnan(D).all()
    # growing the reservation makes the same call run
    tg.reserve_workspace(tg.workspace_bytes(tg.TG_CALL_GEMM_MXFP8, M, N, K), stream=s)
    with torch.cuda.stream(s):
        A.zero_()
        B.zero_()
        SFA.fill_(127)
        SFB.fill_(127)
        tg.gemm_mxfp8_blockscaled(A, B, SFA, SFB, D, stream=s)
    s.synchronize()
    assert tg.tg_device_status(s)[0] == tg.TG_OK
    assert (D == 0).all()


def test_capture_without_reservation_never_allocates(tg, oracle):
    """While a stream without workspace is captured, a call that needs
    workspace returns TG_ERR_WORKSPACE (the capture stays valid) and a
    split-shape product is captured unsplit; the graph replays correctly."""
    torch = torch_cuda()
    rng = np.random.default_rng(311)
    K = 1024
    M, N = split_shape(tg, True, K)
    A, B = quarter_bits(rng, (M, K)), quarter_bits(rng, (N, K))
    dA, dB = dev_bf16(A), dev_bf16(B)
    D = torch.full((M, N), float("nan"), device="cuda")
    mx = synth.make_inputs("mx8k", M=256, N=256, K=256, seed=312)
    mx_d = [dev_u8(mx[k]) for k in ("A", "B", "SFA", "SFB")]
    Dm = torch.full((256, 256), float("nan"), device="cuda")
    # The same kernels once on another stream (per-device set-up outside the capture).
    torch.cuda.synchronize()
    warm = torch.cuda.Stream()
    with torch.cuda.stream(warm):
        tg.gemm_bf16(dA, dB, torch.empty_like(D), cta_pair=True, stream=warm)
    warm.synchronize()
    s = torch.cuda.Stream()
    before = tg.workspace_alloc_count()
    g = torch.cuda.CUDAGraph()
    codes = []
    with torch.cuda.graph(g, stream=s):
        try:
            tg.gemm_mxfp8_blockscaled(*mx_d, Dm, stream=s)
            codes.append(tg.TG_OK)
        except tg.TgError as e:
            codes.append(e.code)
        tg.gemm_bf16(dA, dB, D, cta_pair=True, stream=s)
    assert codes == [tg.TG_ERR_WORKSPACE]
    assert tg.workspace_alloc_count() == before
    g.replay()
    torch.cuda.synchronize()
    assert tg.tg_device_status()[0] == tg.TG_OK
    assert np.array_equal(host_values(D), oracle.gemm_bf16(A, B)[0])
    assert torch.isnan(Dm).all()


@pytest.mark.parametrize("pair", [False, True])
def test_tail_split_beside_kernel_holding_sms(tg, oracle, pair):
    """A split GEMM launched while another stream's kernel holds all but a
    few SMs for 60 ms: most of its CTAs start only when those SMs free up, and
    no piece waits for another, so it completes with TG_OK (even with a 5 ms
    deadline on every wait) and the exact result."""
    torch = torch_cuda()
    from blackwell_tile_gemm_gb300 import probes
    rng = np.random.default_rng(321 + pair)
    K = 2048
    M, N = split_shape(tg, pair, K)
    A, B = quarter_bits(rng, (M, K)), quarter_bits(rng, (N, K))
    dA, dB = dev_bf16(A), dev_bf16(B)
    s_hold, s_gemm = torch.cuda.Stream(), torch.cuda.Stream()
    D = torch.full((M, N), float("nan"), device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(s_gemm):     # tail scratch of this stream allocated here
        tg.gemm_bf16(dA, dB, torch.empty_like(D), cta_pair=pair, stream=s_gemm)
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tg.tg_set_wait_timeout_ns(5_000_000)
    try:
        probes.hold_sms(sms - 8, 60_000_000, stream=s_hold)
        tg.gemm_bf16(dA, dB, D, cta_pair=pair, stream=s_gemm)
        torch.cuda.synchronize()
        status = tg.tg_device_status()
    finally:
        tg.tg_set_wait_timeout_ns(2_000_000_000)
    assert status[0] == tg.TG_OK, status
    assert np.array_equal(host_values(D), oracle.gemm_bf16(A, B)[0])


def test_multicast_only_over_memory_of_this_device(tg, oracle):
    torch = torch_cuda()
    M, N, K = 4000, 3000, 1000
    a = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    b = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    ha = torch.empty((M, K), dtype=torch.bfloat16).pin_memory()
    hb = torch.empty((N, K), dtype=torch.bfloat16).pin_memory()
    # short K: chosen by itself for device operands
    assert tg.gemm_multicast(a, b, M, N, K)
    assert tg.gemm_multicast(a, b, M, N, K, cta_pair=True, multicast=True)
    # host (pinned) memory, or an address the driver does not know: plain kernel
    for x, y in ((ha, b), (a, hb), (ha, hb)):
        assert not tg.gemm_multicast(x, y, M, N, K)
        assert not tg.gemm_multicast(x, y, M, N, K, multicast=True)
        assert not tg.gemm_multicast(x, y, M, N, K, cta_pair=True, multicast=True)
    assert not tg.gemm_multicast(0x10000, b, M, N, K, multicast=True)
    # long K and pairs without the flag never multicast
    assert not tg.gemm_multicast(a, b, M, N, 4096)
    assert not tg.gemm_multicast(a, b, M, N, K, cta_pair=True)
    # the chosen multicast product equals the plain one bit for bit
    rng = np.random.default_rng(331)
    A, B = synth.bf16_uniform(rng, (M, K)), synth.bf16_uniform(rng, (N, K))
    Dm = tg.gemm_bf16(dev_bf16(A), dev_bf16(B))
    Dp = tg.gemm_bf16(dev_bf16(A), dev_bf16(B), cta_pair=True)
    assert tg.tg_device_status()[0] == tg.TG_OK
    rows = np.arange(0, M, 61)
    ref, mag = oracle.gemm_bf16(A, B, rows=rows)
    assert_within(host_values(Dm)[rows], ref, mag, False, "multicast clusters")
    assert_within(host_values(Dp)[rows], ref, mag, False, "pairs")
