"""The C-ABI library without a GPU: it loads, exports every declared entry
point, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

import blackwell_tile_gemm_gb300 as tg
from blackwell_tile_gemm_gb300 import build as tgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("tgemm.h", "tgemm_probes.h")]


@pytest.fixture(scope="module")
def L():
    tgbuild.build()
    return tg.lib()


def declared_functions(headers=HEADERS):
    names = []
    for h in headers:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_headers_declare_the_three_entry_points():
    names = declared_functions()
    for n in ("gemm_bf16", "gemm_mxfp8_blockscaled", "tile_transpose_b16", "tg_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    # tgemm.h: the product library; tgemm_probes.h: the probe library, which
    # links against it and loads without a GPU too.
    missing = [n for n in declared_functions(HEADERS[:1]) if not hasattr(L, n)]
    assert not missing, missing
    from blackwell_tile_gemm_gb300 import probes
    P = probes._L()
    missing = [n for n in declared_functions(HEADERS[1:]) if not hasattr(P, n)]
    assert not missing, missing
    # the product library carries no probe entry point
    assert not any(hasattr(L, n) for n in declared_functions(HEADERS[1:]))


def test_status_strings_and_version(L):
    assert tg.status_string(0) == "ok"
    assert "misaligned" in tg.status_string(2)
    assert L.tg_version() >= 100


def test_zero_timeout_is_rejected(L):
    assert L.tg_set_wait_timeout_ns(0) == tg.TG_ERR_INVALID_ARG


A16 = 0x10000           # a 16-byte aligned fake device address (never dereferenced)


@pytest.mark.parametrize("kw,code", [
    (dict(M=-1), tg.TG_ERR_INVALID_ARG),
    (dict(K=-5), tg.TG_ERR_INVALID_ARG),
    (dict(d_dtype=7), tg.TG_ERR_INVALID_ARG),
    (dict(epilogue=9), tg.TG_ERR_INVALID_ARG),
    (dict(flags=0x80), tg.TG_ERR_UNSUPPORTED),
    (dict(A=0), tg.TG_ERR_INVALID_ARG),
    (dict(D=0), tg.TG_ERR_INVALID_ARG),
    (dict(lda=32), tg.TG_ERR_INVALID_ARG),          # lda < K
    (dict(A=A16 + 2), tg.TG_ERR_MISALIGNED),
    (dict(D=A16 + 8), tg.TG_ERR_MISALIGNED),
    (dict(lda=68), tg.TG_ERR_MISALIGNED),           # 136 bytes, not a multiple of 16
    (dict(ldd=66, N=66), tg.TG_ERR_MISALIGNED),     # f32 D: 264 bytes
])
def test_gemm_bf16_rejects_before_launch(L, kw, code):
    a = dict(A=A16, lda=64, B=A16, ldb=64, D=A16, ldd=64, M=64, N=64, K=64, d_dtype=0,
             epilogue=0, s=0.0, flags=0)
    a.update(kw)
    rc = L.gemm_bf16(a["A"], a["lda"], a["B"], a["ldb"], a["D"], a["ldd"], a["M"], a["N"],
                     a["K"], a["d_dtype"], a["epilogue"], a["s"], a["flags"], None)
    assert rc == code


def test_empty_problems_return_ok_without_cuda(L):
    assert L.gemm_bf16(0, 0, 0, 0, 0, 0, 0, 64, 64, 0, 0, 0.0, 0, None) == tg.TG_OK
    assert L.gemm_bf16(0, 0, 0, 0, 0, 0, 64, 0, 64, 0, 0, 0.0, 0, None) == tg.TG_OK
    assert L.tile_transpose_b16(0, 0, 0, 0, 0, 5, None) == tg.TG_OK


def test_mxfp8_rejects_bad_k_and_scales(L):
    f = L.gemm_mxfp8_blockscaled
    # K not a multiple of 32
    assert f(A16, 48, A16, 48, A16, 2, A16, 2, A16, 64, 64, 64, 48, 0, 0, 0.0, 0, None) == 1
    # missing scales
    assert f(A16, 64, A16, 64, 0, 2, A16, 2, A16, 64, 64, 64, 64, 0, 0, 0.0, 0, None) == 1
    # scale row stride shorter than K/32
    assert f(A16, 64, A16, 64, A16, 1, A16, 2, A16, 64, 64, 64, 64, 0, 0, 0.0, 0, None) == 1
    # lda = 40 bytes is not a multiple of 16
    assert f(A16, 40, A16, 64, A16, 2, A16, 2, A16, 64, 64, 64, 32, 0, 0, 0.0, 0, None) == 2
    # block-scaled multicast clusters are made of CTA pairs
    assert f(A16, 64, A16, 64, A16, 2, A16, 2, A16, 64, 64, 64, 64, 0, 0, 0.0, 2, None) == 1


def test_transpose_rejects_bad_arguments(L):
    f = L.tile_transpose_b16
    assert f(A16, 12, A16 * 4, 64, 64, 12, None) == tg.TG_ERR_MISALIGNED     # ld_in % 8
    assert f(A16 + 2, 64, A16 * 4, 64, 64, 64, None) == tg.TG_ERR_MISALIGNED
    assert f(A16, 32, A16 * 4, 64, 64, 64, None) == tg.TG_ERR_INVALID_ARG    # ld_in < cols
    assert f(A16, 64, A16 + 64, 64, 64, 64, None) == tg.TG_ERR_INVALID_ARG  # overlap


@pytest.mark.parametrize("op,bias,code", [
    (6, 0, tg.TG_ERR_INVALID_ARG),                  # unknown op
    (-1, 0, tg.TG_ERR_INVALID_ARG),
    (tg.TG_EPI_BIAS_COL, 0, tg.TG_ERR_INVALID_ARG),  # bias op without a bias
    (tg.TG_EPI_BIAS_COL_SILU, A16 + 4, tg.TG_ERR_MISALIGNED),
])
def test_gemm_ex_rejects_bad_epilogues(L, op, bias, code):
    epi = tg.tg_epilogue(op, 0.0, 0.0, bias or None)
    for f, extra in ((L.gemm_bf16_ex, ()), (L.gemm_mxfp8_blockscaled_ex, (A16, 2, A16, 2))):
        head = (A16, 64, A16, 64) + extra
        assert f(*head, A16, 64, 64, 64, 64, 0, ctypes.byref(epi), 0, None) == code


def test_gemm_ex_accepts_a_null_epilogue_for_empty_problems(L):
    assert L.gemm_bf16_ex(0, 0, 0, 0, 0, 0, 0, 64, 64, 0, None, 0, None) == tg.TG_OK


def test_make_epilogue_rejects_two_ops():
    with pytest.raises(ValueError):
        tg.make_epilogue(epilogue_add=1.0, silu_affine=(1.0, 0.0))
    e = tg.make_epilogue(silu_affine=(2.0, -1.0))
    assert (e.op, e.alpha, e.beta) == (tg.TG_EPI_SILU_AFFINE, 2.0, -1.0)


@pytest.mark.parametrize("fn,block", [("gemm_mxfp4_blockscaled", 32),
                                      ("gemm_nvfp4_blockscaled", 16)])
def test_fp4_rejects_before_launch(L, fn, block):
    f = getattr(L, fn)
    ok = dict(A=A16, lda=64, B=A16, ldb=64, SFA=A16, ls=8, SFB=A16, lt=8, D=A16, ldd=64, M=64,
              N=64, K=128, d=0, flags=0)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(a["A"], a["lda"], a["B"], a["ldb"], a["SFA"], a["ls"], a["SFB"], a["lt"],
                 a["D"], a["ldd"], a["M"], a["N"], a["K"], a["d"], None, a["flags"], None)

    assert call(K=block + block // 2) == tg.TG_ERR_INVALID_ARG          # K % block
    assert call(lda=48, K=128) == tg.TG_ERR_INVALID_ARG                # lda < K/2 bytes
    assert call(lda=72, K=128) == tg.TG_ERR_MISALIGNED                 # 72 % 16
    assert call(ls=128 // block - 1) == tg.TG_ERR_INVALID_ARG          # ld_sfa < K/block
    assert call(SFB=0) == tg.TG_ERR_INVALID_ARG
    assert call(flags=3) == tg.TG_ERR_UNSUPPORTED                     # no FP4 multicast
    assert call(flags=2) == tg.TG_ERR_INVALID_ARG                     # multicast needs pairs
    assert call(M=0) == tg.TG_OK


def test_skinny_rejects_before_launch(L):
    f = L.gemm_bf16_skinny
    base = (A16, 64, A16, 64, A16, 64)
    assert f(*base, 129, 64, 64, 0, None, 0, None) == tg.TG_ERR_UNSUPPORTED    # M > 128
    assert f(*base, 16, 64, 64, 0, None, -1, None) == tg.TG_ERR_INVALID_ARG    # split_k < 0
    assert f(*base, 16, 64, 64, 7, None, 0, None) == tg.TG_ERR_INVALID_ARG     # d_dtype
    assert f(A16 + 2, 64, A16, 64, A16, 64, 16, 64, 64, 0, None, 0, None) == tg.TG_ERR_MISALIGNED
    assert f(*base, 0, 64, 64, 0, None, 0, None) == tg.TG_OK


def test_gather_rejects_before_launch(L):
    f = L.gemm_bf16_gather
    assert f(A16, 64, 100, A16, 64, A16, 64, A16, 64, 64, 64, 0, None, 2, None) \
        == tg.TG_ERR_UNSUPPORTED                                 # multicast
    assert f(A16, 64, 100, 0, 64, A16, 64, A16, 64, 64, 64, 0, None, 0, None) \
        == tg.TG_ERR_INVALID_ARG                                 # no row_idx
    assert f(A16, 64, 0, A16, 64, A16, 64, A16, 64, 64, 64, 0, None, 0, None) \
        == tg.TG_ERR_INVALID_ARG                                 # a_rows == 0
    assert f(A16, 64, -1, A16, 64, A16, 64, A16, 64, 64, 64, 0, None, 0, None) \
        == tg.TG_ERR_INVALID_ARG
    assert f(A16, 64, 100, A16, 0, A16, 64, A16, 64, 64, 64, 0, None, 0, None) == tg.TG_OK
    assert f(A16, 64, 100, A16, 64, A16, 64, A16, 64, 64, 64, 0, None, 8, None) \
        == tg.TG_ERR_UNSUPPORTED                                 # unknown flag
    # TG_FLAG_GATHER_TMA belongs to the gather call only
    assert L.gemm_bf16(A16, 64, A16, 64, A16, 64, 64, 64, 64, 0, 0, 0.0, 4, None) \
        == tg.TG_ERR_UNSUPPORTED


@pytest.mark.parametrize("shape,lds,want", [
    ((4000, 3000, 1000), (1000, 1000), 3),   # 16-byte rows, M*N/(M+N) = 1714
    ((4000, 3000, 1000), (1024, 1024), 0),   # 128-byte rows
    ((4000, 3000, 1000), (1000, 1024), 1),   # only A
    ((4000, 3000, 992), (992, 1000), 2),     # 64-byte rows of A are fine
    ((2048, 2048, 1000), (1000, 1000), 0),   # 1024 < 1250: the copy would not pay
    ((8192, 8192, 1000), (1008, 1008), 0),   # 32-byte rows: never
    ((8192, 8192, 1000), (1000, 1008), 1),
    ((4000, 3000, 104), (104, 104), 0),      # K < 128
])
def test_repitch_rule(L, shape, lds, want):
    assert tg.gemm_repitch(*shape, *lds) == want
    # the same for CTA pairs and for single-CTA multicast clusters
    assert tg.gemm_repitch(*shape, *lds, cta_pair=True) == want
    assert tg.gemm_repitch(*shape, *lds, multicast=True) == want
    # multicast clusters of two CTA pairs read badly aligned rows in place
    assert tg.gemm_repitch(*shape, *lds, cta_pair=True, multicast=True) == 0


def test_repitch_rejects_negative_sizes_and_unknown_flags(L):
    assert L.tg_gemm_repitch(-1, 8, 8, 8, 8, 0) == -tg.TG_ERR_INVALID_ARG
    assert L.tg_gemm_repitch(4000, 3000, 1000, 1000, 1000, 4) == -tg.TG_ERR_INVALID_ARG


def test_multicast_query_falls_back_for_unknown_pointers(L):
    # A fake address is no allocation of a current device (on a host without
    # a GPU there is none): the short-K product and an explicit multicast
    # request both answer "plain kernel".
    assert L.tg_gemm_multicast(A16, A16, 4000, 3000, 1000, 0) == 0
    assert L.tg_gemm_multicast(A16, A16, 4000, 3000, 1000, tg.TG_FLAG_MULTICAST) == 0
    assert L.tg_gemm_multicast(A16, A16, 8192, 8192, 8192,
                               tg.TG_FLAG_MULTICAST | tg.TG_FLAG_CTA_PAIR) == 0
    # shapes that never ask for multicast, and empty ones
    assert L.tg_gemm_multicast(A16, A16, 4000, 3000, 4096, 0) == 0
    assert L.tg_gemm_multicast(A16, A16, 4000, 3000, 0, tg.TG_FLAG_MULTICAST) == 0
    assert L.tg_gemm_multicast(A16, A16, -1, 3000, 1000, 0) == -tg.TG_ERR_INVALID_ARG
    assert L.tg_gemm_multicast(A16, A16, 64, 64, 64, 8) == -tg.TG_ERR_UNSUPPORTED


@pytest.mark.parametrize("call,shape,lds,d,epi,flags,want", [
    # re-pitched 16-byte rows: (M + N) rows of ceil(K/64)*64 bf16 elements
    (tg.TG_CALL_GEMM_BF16, (4000, 3000, 1000), (1000, 1000), 0, 0, 0, (4000 + 3000) * 1024 * 2),
    (tg.TG_CALL_GEMM_BF16, (4000, 3000, 1000), (1024, 1024), 0, 0, 0, 0),
    # scale images: (ceil(M/r)*r/128 + 2*ceil(N/256)) * ceil(K/stage) * V * 512
    (tg.TG_CALL_GEMM_MXFP8, (8192, 8192, 8192), (8192, 8192), 1, 0, 1, 4 << 20),
    (tg.TG_CALL_GEMM_MXFP8, (300, 264, 160), (160, 160), 0, 0, 0, (3 + 4) * 2 * 512),
    (tg.TG_CALL_GEMM_MXFP4, (8192, 8192, 8192), (4096, 4096), 1, 0, 1, 4 << 20),
    (tg.TG_CALL_GEMM_NVFP4, (8192, 8192, 8192), (4096, 4096), 1, 0, 1, 8 << 20),
    # skinny: f32 partial sums only for bf16 D (M * ceil(N/4)*4 * 4 bytes)
    (tg.TG_CALL_GEMM_BF16_SKINNY, (16, 8192, 8192), (8192, 8192), 1, 0, 0, 16 * 8192 * 4),
    (tg.TG_CALL_GEMM_BF16_SKINNY, (16, 8192, 8192), (8192, 8192), 0, 0, 0, 0),
    # gathered rows at a 128-byte pitch, unless gather4 loads them in the GEMM
    (tg.TG_CALL_GEMM_BF16_GATHER, (4096, 8192, 8192), (8192, 8192), 1, 0, 0, 4096 * 8192 * 2),
    (tg.TG_CALL_GEMM_BF16_GATHER, (4096, 8192, 8192), (8192, 8192), 1, 0,
     tg.TG_FLAG_GATHER_TMA, 0),
])
def test_workspace_bytes(L, call, shape, lds, d, epi, flags, want):
    assert tg.workspace_bytes(call, *shape, *lds, d, epi, flags) == want


def test_workspace_bytes_rejects_bad_requests(L):
    f = L.tg_workspace_bytes
    assert f(99, 64, 64, 64, 64, 64, 0, 0, 0) == -tg.TG_ERR_INVALID_ARG
    assert f(tg.TG_CALL_GEMM_MXFP8, 64, 64, 48, 64, 64, 0, 0, 0) == -tg.TG_ERR_INVALID_ARG
    assert f(tg.TG_CALL_GEMM_BF16_SKINNY, 129, 64, 64, 64, 64, 0, 0, 0) == -tg.TG_ERR_UNSUPPORTED
    assert f(tg.TG_CALL_GEMM_BF16, -1, 64, 64, 64, 64, 0, 0, 0) == -tg.TG_ERR_INVALID_ARG
    assert f(tg.TG_CALL_GEMM_BF16, 0, 64, 64, 64, 64, 0, 0, 0) == 0


def test_reserve_workspace_host_checks(L):
    assert L.tg_reserve_workspace(None, -1) == tg.TG_ERR_INVALID_ARG
    assert "workspace" in tg.status_string(tg.TG_ERR_WORKSPACE)
    before = L.tg_workspace_alloc_count()
    # the host checks above allocate nothing
    assert L.tg_workspace_alloc_count() == before
