"""C ABI checks that need no GPU: the library loads, exports every function the
header declares, and rejects bad arguments on the host with the documented
status codes (no device pointer is ever dereferenced on these paths)."""

import ctypes

import pytest

import fp8_block_scale_x128_gb300 as fb

OK, ARG, SHAPE, ALIGN, KIND, WS = 0, -1, -2, -3, -4, -5

# fake but well-aligned device addresses: the host checks never touch them.
# Every call below must be refused before any launch; as a second guard the
# module never runs where a GPU is visible.
P = 0x10000000
STREAM = None

pytestmark = pytest.mark.skipif(
    __import__("torch").cuda.is_available(),
    reason="fake device pointers: host-check tests run only where no GPU is visible")


@pytest.fixture(scope="module")
def L():
    fb.build()
    return fb.lib()


def test_library_exports_every_declared_function(L):
    names = fb.declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(L, n), n


def test_version_and_status_strings(L):
    assert fb.fp8bs_version() >> 16 == 1
    for s in (0, -1, -2, -3, -4, -5, -6, -7, -8, -9):
        assert fb.fp8bs_status_string(s) and fb.fp8bs_status_string(s) != "unknown status"
    assert fb.fp8bs_status_string(-99) == "unknown status"


def test_packed_weight_bytes(L):
    # 256-byte header + 16 KB per tile + scales, rounded to 256
    assert fb.fp8bs_packed_weight_bytes(5120, 4096, 0) == 256 + 40 * 32 * 16384 + 40 * 32 * 4
    assert fb.fp8bs_packed_weight_bytes(5120, 4096, 1) == 256 + 40 * 32 * 16384 + 1280
    assert fb.fp8bs_packed_weight_bytes(128, 128, 1) == 256 + 16384 + 256
    assert fb.fp8bs_packed_weight_bytes(100, 128, 0) == 0
    assert fb.fp8bs_packed_weight_bytes(128, 128, 7) == 0


def test_workspace_bytes_for_explicit_sm_count(L):
    def expect(K, sm):
        # error word, epoch words, two 64 x 128 tagged-word partial slots per
        # CTA index, then the codes and fp32 scales of up to 64 rows
        return 256 + 4096 + sm * 2 * 64 * 128 * 8 + 64 * K + 64 * (K // 128) * 4
    assert fb.fp8bs_workspace_bytes(5120, 4096, 152) == expect(4096, 152)
    assert fb.fp8bs_workspace_bytes(128, 128, 152) == expect(128, 152)
    # independent of N
    assert fb.fp8bs_workspace_bytes(16384, 4096, 152) == expect(4096, 152)
    assert fb.fp8bs_workspace_bytes(130, 128, 152) == 0
    # one n-tile's K blocks must fit 10 units per SM
    assert fb.fp8bs_workspace_bytes(128, 1520 * 128, 152) == expect(1520 * 128, 152)
    assert fb.fp8bs_workspace_bytes(128, 1521 * 128, 152) == 0
    assert fb.fp8bs_workspace_bytes(128, 128, 2000) == 0


def gemm(L, x=P, M=4, ldx=4096, packed=P, packed_bytes=1 << 30, N=5120, K=4096, kind=0, y=P,
         ldy=5120, ws=P, ws_bytes=1 << 30, xq=None, xs=None, flags=0):
    return L.fp8bs_gemm_fused(x, M, ldx, packed, packed_bytes, N, K, kind, y, ldy, ws, ws_bytes,
                              xq, xs, flags, STREAM)


@pytest.mark.parametrize("kw,status", [
    (dict(kind=2), ARG),
    (dict(M=65), SHAPE),
    (dict(M=-1), SHAPE),
    (dict(N=5000), SHAPE),
    (dict(K=4000, ldx=4000), SHAPE),
    (dict(N=0), SHAPE),
    (dict(N=(1 << 24) + 128, ldy=(1 << 24) + 128), SHAPE),
    (dict(flags=2), ARG),
    (dict(x=None), ARG),
    (dict(y=None), ARG),
    (dict(ws=None), ARG),
    (dict(packed=None), ARG),
    (dict(ldx=4088), ARG),
    (dict(ldy=5112), ARG),
    (dict(x=P + 8), ALIGN),
    (dict(ldx=4100), ALIGN),
    (dict(y=P + 2), ALIGN),
    (dict(packed=P + 16), ALIGN),
    (dict(ws=P + 16), ALIGN),
    (dict(xq=P + 4), ALIGN),
    (dict(packed_bytes=1000), WS),
])
def test_gemm_fused_host_checks(L, kw, status):
    assert gemm(L, **kw) == status


def test_gemm_fused_empty_batch_is_a_no_op(L):
    assert gemm(L, M=0, x=None, y=None) == OK


def gemm_static(L, x=P, M=4, ldx=4096, packed=P, packed_bytes=1 << 30, N=5120, K=4096, kind=0,
                y=P, ldy=5120, xq=None, xs=None, status=None, flags=0):
    return L.fp8bs_gemm_fused_static(x, M, ldx, packed, packed_bytes, N, K, kind, y, ldy, xq, xs,
                                     status, flags, STREAM)


@pytest.mark.parametrize("kw,status", [
    (dict(kind=2), ARG),
    (dict(flags=2), ARG),
    (dict(M=65), SHAPE),
    (dict(N=5000), SHAPE),
    (dict(x=None), ARG),
    (dict(packed=None), ARG),
    (dict(y=None), ARG),
    (dict(ldy=5112), ARG),
    (dict(x=P + 8), ALIGN),
    (dict(status=P + 2), ALIGN),
    (dict(packed_bytes=1000), WS),
    # one K block past the fixed scratch's limit
    (dict(K=fb.FP8BS_STATIC_MAX_K + 128, ldx=fb.FP8BS_STATIC_MAX_K + 128), WS),
])
def test_gemm_fused_static_host_checks(L, kw, status):
    assert gemm_static(L, **kw) == status


def test_gemm_fused_static_empty_batch_is_a_no_op(L):
    assert gemm_static(L, M=0, x=None, y=None) == OK


def gemm_prequant(L, xq=P, M=4, ldxq=4096, xs=P, packed=P, packed_bytes=1 << 30, N=5120, K=4096, kind=0,
                  y=P, ldy=5120, ws=P, ws_bytes=1 << 30, flags=0):
    return L.fp8bs_gemm_prequant(xq, M, ldxq, xs, packed, packed_bytes, N, K, kind, y, ldy, ws, ws_bytes,
                                 flags, STREAM)


@pytest.mark.parametrize("kw,status", [
    (dict(kind=3), ARG),
    (dict(flags=2), ARG),
    (dict(M=65), SHAPE),
    (dict(K=4000, ldxq=4000), SHAPE),
    (dict(xq=None), ARG),
    (dict(xs=None), ARG),
    (dict(ws=None), ARG),
    (dict(ldxq=4080), ARG),
    (dict(xq=P + 8), ALIGN),
    (dict(ldxq=4104), ALIGN),
    (dict(xs=P + 2), ALIGN),
    (dict(y=P + 2), ALIGN),
    (dict(packed_bytes=1000), WS),
])
def test_gemm_prequant_host_checks(L, kw, status):
    assert gemm_prequant(L, **kw) == status


def test_gemm_prequant_empty_batch_is_a_no_op(L):
    assert gemm_prequant(L, M=0, xq=None, xs=None, y=None) == OK


def test_quant_host_checks(L):
    q = L.fp8bs_quant
    assert q(P, 2, 4096, 4096, 3, P, P, STREAM) == ARG
    assert q(P, 2, 4000, 4000, 0, P, P, STREAM) == SHAPE
    assert q(P, -1, 4096, 4096, 0, P, P, STREAM) == SHAPE
    assert q(P, 0, 4096, 4096, 0, None, None, STREAM) == OK
    assert q(None, 2, 4096, 4096, 0, P, P, STREAM) == ARG
    assert q(P, 2, 4096, 2048, 0, P, P, STREAM) == ARG
    assert q(P + 8, 2, 4096, 4096, 0, P, P, STREAM) == ALIGN
    assert q(P, 2, 4096, 4100, 0, P, P, STREAM) == ALIGN
    assert q(P, 2, 4096, 4096, 0, P, P + 2, STREAM) == ALIGN


def test_rmsnorm_quant_host_checks(L):
    r = L.fp8bs_rmsnorm_quant
    nan = float("nan")
    # x, M, K, ldx, gamma, eps, kind, xq, xs, y, ldy, stream
    assert r(P, 2, 4096, 4096, P, 1e-6, 2, P, P, None, 0, STREAM) == ARG
    assert r(P, 2, 4096, 4096, P, -1e-6, 0, P, P, None, 0, STREAM) == ARG
    assert r(P, 2, 4096, 4096, P, nan, 0, P, P, None, 0, STREAM) == ARG
    assert r(P, 2, 4000, 4000, P, 1e-6, 0, P, P, None, 0, STREAM) == SHAPE
    assert r(P, 2, 16384 + 128, 16512, P, 1e-6, 0, P, P, None, 0, STREAM) == SHAPE
    assert r(P, -1, 4096, 4096, P, 1e-6, 0, P, P, None, 0, STREAM) == SHAPE
    assert r(P, 0, 4096, 4096, None, 1e-6, 0, None, None, None, 0, STREAM) == OK
    assert r(P, 2, 4096, 4096, None, 1e-6, 0, P, P, None, 0, STREAM) == ARG
    assert r(P, 2, 4096, 4096, P, 1e-6, 0, None, P, None, 0, STREAM) == ARG
    assert r(P, 2, 4096, 2048, P, 1e-6, 0, P, P, None, 0, STREAM) == ARG
    assert r(P, 2, 4096, 4096, P, 1e-6, 0, P, P, P, 2048, STREAM) == ARG
    assert r(P + 8, 2, 4096, 4096, P, 1e-6, 0, P, P, None, 0, STREAM) == ALIGN
    assert r(P, 2, 4096, 4100, P, 1e-6, 0, P, P, None, 0, STREAM) == ALIGN
    assert r(P, 2, 4096, 4096, P + 2, 1e-6, 0, P, P, None, 0, STREAM) == ALIGN
    assert r(P, 2, 4096, 4096, P, 1e-6, 0, P + 4, P, None, 0, STREAM) == ALIGN
    assert r(P, 2, 4096, 4096, P, 1e-6, 0, P, P + 2, None, 0, STREAM) == ALIGN
    assert r(P, 2, 4096, 4096, P, 1e-6, 0, P, P, P + 8, 4096, STREAM) == ALIGN
    assert r(P, 2, 4096, 4096, P, 1e-6, 0, P, P, P, 4100, STREAM) == ALIGN


def test_header_states_the_fixed_scratch_size(L):
    # the fixed scratch of fp8bs_gemm_fused_static is a workspace laid out for
    # FP8BS_STATIC_MAX_SMS CTAs and K = FP8BS_STATIC_MAX_K; the header states its size
    import re
    text = open(fb.HEADER_PATH).read()
    stated = int(re.search(r"fixed device array inside this library \(([0-9,]+) bytes", text).group(1)
                 .replace(",", ""))
    assert L.fp8bs_workspace_bytes(128, fb.FP8BS_STATIC_MAX_K, fb.FP8BS_STATIC_MAX_SMS) == stated


def test_moe_host_checks(L):
    wsb = L.fp8bs_moe_workspace_bytes
    # 256-byte error word + gate/up partials (M*S x H/512 x 2I) + down outputs (M*S x H), fp32
    assert wsb(16, 11, 4096, 256) == 256 + 16 * 11 * 8 * 512 * 4 + 16 * 11 * 4096 * 4
    assert wsb(16, 11, 4000, 256) == 0
    assert wsb(16, 11, 4096, 384) == 0
    assert wsb(100, 11, 4096, 256) == 0  # more than 1024 pairs
    n = wsb(4, 11, 4096, 256)
    m = L.fp8bs_moe_w8a16
    # x, M, H, ids, w, S, w13, s13, w2, s2, E, I, y, ws, ws_bytes, stream
    assert m(P, 4, 4096, P, P, 11, P, P, P, P, 513, 256, P, P, n - 1, STREAM) == WS
    assert m(P, 4, 4096, P, P, 11, P, P, P, P, 513, 200, P, P, n, STREAM) == SHAPE
    assert m(P, 4, 4100, P, P, 11, P, P, P, P, 513, 256, P, P, n, STREAM) == SHAPE
    assert m(P, 4, 4096, P, P, 0, P, P, P, P, 513, 256, P, P, n, STREAM) == SHAPE
    assert m(P, 4, 4096, P, P, 11, P, P, P, P, 0, 256, P, P, n, STREAM) == SHAPE
    assert m(P, 4, 4096, P, P, 11, P, P, P, P, 5000, 256, P, P, n, STREAM) == SHAPE
    assert m(P, 100, 4096, P, P, 11, P, P, P, P, 513, 256, P, P, n, STREAM) == SHAPE
    assert m(P, -1, 4096, P, P, 11, P, P, P, P, 513, 256, P, P, n, STREAM) == SHAPE
    assert m(None, 0, 4096, None, None, 11, None, None, None, None, 513, 256, None, None, 0, STREAM) == OK
    assert m(P, 4, 4096, None, P, 11, P, P, P, P, 513, 256, P, P, n, STREAM) == ARG
    assert m(P, 4, 4096, P, P, 11, P, P, P, P, 513, 256, None, P, n, STREAM) == ARG
    assert m(P + 8, 4, 4096, P, P, 11, P, P, P, P, 513, 256, P, P, n, STREAM) == ALIGN
    assert m(P, 4, 4096, P + 2, P, 11, P, P, P, P, 513, 256, P, P, n, STREAM) == ALIGN
    assert m(P, 4, 4096, P, P, 11, P + 8, P, P, P, 513, 256, P, P, n, STREAM) == ALIGN
    assert m(P, 4, 4096, P, P, 11, P, P, P + 4, P, 513, 256, P, P, n, STREAM) == ALIGN
    assert m(P, 4, 4096, P, P, 11, P, P, P, P, 513, 256, P + 4, P, n, STREAM) == ALIGN
    assert m(P, 4, 4096, P, P, 11, P, P, P, P, 513, 256, P, P + 128, n, STREAM) == ALIGN


def test_prepack_and_weight_quant_host_checks(L):
    pp = L.fp8bs_prepack_weight
    assert pp(P, 4096, P, 5120, 4096, 5, P, 1 << 30, STREAM) == ARG
    assert pp(P, 4096, P, 5100, 4096, 0, P, 1 << 30, STREAM) == SHAPE
    assert pp(P, 4096, P, 5120, 4096, 0, P + 128, 1 << 30, STREAM) == ALIGN
    assert pp(P, 4104, P, 5120, 4096, 0, P, 1 << 30, STREAM) == ALIGN
    assert pp(P, 4096, P, 5120, 4096, 0, P, 1000, STREAM) == WS
    qw = L.fp8bs_quant_weight
    assert qw(P, 256, 256, 256, 9, P, P, STREAM) == ARG
    assert qw(P, 256, 200, 256, 0, P, P, STREAM) == SHAPE
    assert qw(P + 4, 256, 256, 256, 0, P, P, STREAM) == ALIGN


def test_workspace_init_and_check_error_host_checks(L):
    assert L.fp8bs_workspace_init(None, 1024, STREAM) == ARG
    assert L.fp8bs_workspace_init(P + 16, 1024, STREAM) == ALIGN
    assert L.fp8bs_workspace_init(P, 100, STREAM) == WS
    assert L.fp8bs_check_error(None, STREAM) == ARG
    assert L.fp8bs_check_error(P + 8, STREAM) == ALIGN
    assert L.fp8bs_encode_e4m3(P, 6, P, STREAM) == SHAPE
    assert L.fp8bs_encode_e4m3(P, 0, None, STREAM) == OK
    assert L.fp8bs_encode_e4m3(P + 4, 8, P, STREAM) == ALIGN


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(fb, "_lib", None)
    monkeypatch.setattr(fb, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        fb.lib()
    assert ctypes  # keep import used
