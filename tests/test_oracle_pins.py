"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties an oracle function to an independent fact: the e4m3fn / e8m0 /
bf16 format definitions (closed forms, hand-worked values), a library routine
(torch's float8_e4m3fn and bfloat16 casts, numpy's fp64 and int64 matmul) or a
mathematical invariant.  The method being pinned is the one on the page
"[AMD] Small-M FP8 block-scale GEMM with fused activation quant for gfx950
(Qwen3.5)", section "Modifications" (1x128 activation groups with a row-amax
scale, [N/128, K/128] weight scales, x_scale * w_scale per 128-wide K block)
and its ue8m0 variant on "[Perf] [AMD] dsv4: optional e8m0 mxscale GEMM for
dense 128x128 fp8 linears (6/8)", section "Modifications".
"""

import math
import struct

import numpy as np
import pytest
import torch

import synth

E4M3_MAX = 448.0


def f32(v):
    return float(np.float32(v))


def f32_from_bits(u):
    return struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))[0]


def bits_of_f32(v):
    return struct.unpack("<I", struct.pack("<f", v))[0]


def next_up(v):
    return float(np.nextafter(np.float32(v), np.float32(np.inf)))


def next_down(v):
    return float(np.nextafter(np.float32(v), np.float32(-np.inf)))


def torch_e4m3_bytes(v_f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v_f32, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


# ---------------------------------------------------------------------------
# e4m3fn decode
# ---------------------------------------------------------------------------

def test_e4m3_decode_matches_torch_for_all_codes(oracle_mod):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle_mod.e4m3_table()
    nan_ref = np.isnan(ref)
    assert np.array_equal(nan_ref, np.isnan(got))
    assert set(np.flatnonzero(nan_ref)) == {0x7F, 0xFF}
    assert np.array_equal(ref[~nan_ref], got[~nan_ref])
    # signed zero of 0x80
    assert math.copysign(1.0, got[0x80]) == -1.0


@pytest.mark.parametrize("code,value", [
    (0x38, 1.0),            # exponent field 7 = bias
    (0x7E, 448.0),          # largest finite: 2^8 * 1.75
    (0x08, 2.0 ** -6),      # smallest normal
    (0x01, 2.0 ** -9),      # smallest subnormal
    (0x07, 7 * 2.0 ** -9),  # largest subnormal
    (0x5B, 22.0),           # 2^4 * (1 + 3/8)
    (0xFE, -448.0),
    (0xB8, -1.0),
])
def test_e4m3_decode_hand_values(oracle_mod, code, value):
    assert oracle_mod.e4m3_decode(code) == value


# ---------------------------------------------------------------------------
# e4m3fn encode
# ---------------------------------------------------------------------------

def test_e4m3_encode_roundtrips_every_finite_code(oracle_mod):
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        v = oracle_mod.e4m3_decode(c)
        assert oracle_mod.e4m3_encode(v) == c, hex(c)


def _finite_codes_sorted(oracle_mod):
    pos = sorted((oracle_mod.e4m3_decode(c), c) for c in range(0x00, 0x7F))
    return pos


def test_e4m3_encode_midpoints_go_to_even_and_neighbours_to_nearest(oracle_mod):
    pos = _finite_codes_sorted(oracle_mod)
    for (v0, c0), (v1, c1) in zip(pos, pos[1:]):
        mid = (v0 + v1) / 2.0
        assert float(np.float32(mid)) == mid  # midpoints are exact in fp32
        even = c0 if c0 % 2 == 0 else c1
        assert oracle_mod.e4m3_encode(mid) == even, (v0, v1)
        assert oracle_mod.e4m3_encode(-mid) == (even | 0x80)
        assert oracle_mod.e4m3_encode(next_down(mid)) == c0
        assert oracle_mod.e4m3_encode(next_up(mid)) == c1


def test_e4m3_encode_saturates(oracle_mod):
    for v in [448.0, next_up(448.0), 460.0, 463.99, 464.0, 500.0, 1e6, 3.0e38]:
        assert oracle_mod.e4m3_encode(v) == 0x7E
        assert oracle_mod.e4m3_encode(-v) == 0xFE


def test_e4m3_encode_tiny_values(oracle_mod):
    assert oracle_mod.e4m3_encode(2.0 ** -10) == 0x00           # tie with 0 -> even 0
    assert oracle_mod.e4m3_encode(next_up(2.0 ** -10)) == 0x01
    assert oracle_mod.e4m3_encode(3 * 2.0 ** -10) == 0x02       # 1.5 units -> even 2
    assert oracle_mod.e4m3_encode(-(2.0 ** -12)) == 0x80        # rounds to -0
    assert oracle_mod.e4m3_encode(-0.0) == 0x80
    assert oracle_mod.e4m3_encode(1e-40) == 0x00                # fp32 subnormal input


def test_e4m3_encode_matches_torch_cast_on_random_values(oracle_mod):
    rng = np.random.default_rng(7)
    # log-uniform magnitudes over the whole e4m3 range plus the subnormal range
    mags = np.exp2(rng.uniform(-14, math.log2(463.9), 20000)).astype(np.float32)
    signs = np.where(rng.random(20000) < 0.5, -1.0, 1.0).astype(np.float32)
    v = mags * signs
    ref = torch_e4m3_bytes(v)
    got = np.array([oracle_mod.e4m3_encode(t) for t in v], dtype=np.uint8)
    assert np.array_equal(ref, got)


def test_e4m3_encode_bits_range_agrees_with_scalar(oracle_mod):
    first = bits_of_f32(0.75)
    out = oracle_mod.e4m3_encode_bits(first, 4096)
    for i in range(0, 4096, 97):
        assert out[i] == oracle_mod.e4m3_encode(f32_from_bits(first + i))


# ---------------------------------------------------------------------------
# bf16 rounding of the fp64 result
# ---------------------------------------------------------------------------

def test_f64_to_bf16_matches_torch_on_fp32_values(oracle_mod):
    rng = np.random.default_rng(11)
    v = (rng.standard_normal(5000) * np.exp2(rng.uniform(-30, 30, 5000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = oracle_mod.f64_to_bf16_array(v.astype(np.float64))
    assert np.array_equal(ref, got)


def test_f64_to_bf16_rounds_once_from_fp64(oracle_mod):
    # 1 + 2^-8 + 2^-30 lies just above the midpoint of 1 and 1 + 2^-7.  Rounded
    # straight from fp64 it goes up; an fp32 detour would land on the midpoint
    # and tie to 1.0.
    assert oracle_mod.f64_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    assert oracle_mod.f64_to_bf16(1.0 + 2.0 ** -8) == 0x3F80          # exact tie -> even
    assert oracle_mod.f64_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82      # tie -> even (up)
    assert oracle_mod.f64_to_bf16(-2.5) == 0xC020
    assert oracle_mod.f64_to_bf16(2.0 ** -133) == 0x0001              # smallest subnormal
    assert oracle_mod.f64_to_bf16(2.0 ** -134) == 0x0000              # tie -> even 0
    assert oracle_mod.f64_to_bf16(3.0e38) == 0x7F62
    assert oracle_mod.f64_to_bf16(3.4e38) == 0x7F80                   # past the max: inf
    assert oracle_mod.f64_to_bf16(-0.0) == 0x8000


# ---------------------------------------------------------------------------
# e8m0 (power-of-two) scales
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("s,byte", [
    (1.0, 127), (f32(1.0000001), 128), (0.75, 127), (0.5, 126), (f32(0.50000006), 127),
    (2.0 ** -127, 0), (2.0 ** -130, 0), (0.0, 0), (2.0 ** 100, 227), (f32(449.0 / 448.0), 128),
])
def test_e8m0_ceil_hand_values(oracle_mod, s, byte):
    assert oracle_mod.e8m0_ceil(s) == byte


def test_e8m0_ceil_is_smallest_power_of_two_above(oracle_mod):
    rng = np.random.default_rng(3)
    for s in np.exp2(rng.uniform(-120, 120, 3000)).astype(np.float32):
        b = oracle_mod.e8m0_ceil(float(s))
        p = oracle_mod.e8m0_decode(b)
        assert p == 2.0 ** (b - 127)
        assert p >= float(s) > p / 2


# ---------------------------------------------------------------------------
# 1x128 activation quantisation
# ---------------------------------------------------------------------------

def bf16_row(values):
    v = np.asarray(values, dtype=np.float32).reshape(1, -1)
    return synth.f32_to_bf16_bits(v)


def test_quant_zero_group(oracle_mod):
    x = np.zeros((1, 128), dtype=np.uint16)
    x[0, 5] = 0x8000  # -0.0
    xq, xs = oracle_mod.quant_1x128(x, 0)
    assert xs[0, 0] == 0.0
    assert xq[0, 5] == 0x80 and np.count_nonzero(xq) == 1
    xq, xs = oracle_mod.quant_1x128(x, 1)
    assert xs[0, 0] == 0 and xq[0, 5] == 0x80 and np.count_nonzero(xq) == 1


def test_quant_all_equal_group(oracle_mod):
    x = bf16_row([3.0] * 128)
    xq, xs = oracle_mod.quant_1x128(x, 0)
    assert xs[0, 0] == np.float32(3.0) / np.float32(448.0)
    assert np.all(xq == 0x7E)


def test_quant_single_outlier_group(oracle_mod):
    vals = [0.5] * 128
    vals[5] = -10.0
    xq, xs = oracle_mod.quant_1x128(bf16_row(vals), 0)
    assert xs[0, 0] == np.float32(10.0) / np.float32(448.0)
    assert xq[0, 5] == 0xFE
    # 0.5 / (10/448) = 22.4 -> nearest e4m3 is 22 = 2^4 * 1.375 -> code 0x5B
    assert np.all(np.delete(xq[0], 5) == 0x5B)


def test_quant_ties_and_subnormal_codes(oracle_mod):
    # amax = 448 gives scale exactly 1, so x / scale = x.
    vals = [0.0] * 128
    vals[0] = 448.0
    vals[1] = 17.0              # midpoint of 16 (m=0) and 18 (m=1) -> 16, code 0x58
    vals[2] = 19.0              # midpoint of 18 (m=1) and 20 (m=2) -> 20, code 0x5A
    vals[3] = 2.0 ** -8         # subnormal: 2 * 2^-9 -> 0x02
    vals[4] = 3 * 2.0 ** -10    # 1.5 subnormal units -> tie -> 2 -> 0x02
    vals[5] = 2.0 ** -10        # half a unit -> tie -> 0
    vals[6] = -(5 * 2.0 ** -10)  # 2.5 units -> tie -> 2 -> 0x82
    vals[7] = -240.0            # 2^7 * 1.875 -> 0xF7
    xq, xs = oracle_mod.quant_1x128(bf16_row(vals), 0)
    assert xs[0, 0] == 1.0
    assert list(xq[0, :8]) == [0x7E, 0x58, 0x5A, 0x02, 0x02, 0x00, 0x82, 0xF7]


def test_quant_every_group_reaches_448(oracle_mod):
    x = synth.x_bf16(4, 1024, seed=5)
    xq, xs = oracle_mod.quant_1x128(x, 0)
    g = (xq & 0x7F).reshape(4, 8, 128)
    assert np.all(g.max(axis=2) == 0x7E)
    assert np.all(g <= 0x7E)


def test_quant_power_of_two_rescaling_is_exact(oracle_mod):
    x = synth.x_bf16(2, 512, seed=9)
    xq, xs = oracle_mod.quant_1x128(x, 0)
    xf = synth.bf16_bits_to_f32(x)
    for j in (-8, -3, 1, 6):
        x2 = synth.f32_to_bf16_bits(xf * np.float32(2.0 ** j))
        xq2, xs2 = oracle_mod.quant_1x128(x2, 0)
        assert np.array_equal(xq, xq2)
        assert np.array_equal(xs * np.float32(2.0 ** j), xs2)


def _torch_quant_1x128(x_bits):
    """Independent restatement through torch library routines."""
    xf = torch.from_numpy(synth.bf16_bits_to_f32(x_bits).copy())
    M, K = xf.shape
    g = xf.view(M, K // 128, 128)
    amax = g.abs().amax(dim=2, keepdim=True)
    s = amax / torch.tensor(448.0, dtype=torch.float32)
    q = torch.where(amax > 0, g / torch.where(amax > 0, s, torch.ones_like(s)), g * 0)
    codes = q.to(torch.float8_e4m3fn).view(torch.uint8).reshape(M, K).numpy()
    return codes, s.reshape(M, K // 128).numpy()


@pytest.mark.parametrize("M,K,seed", [(1, 2048, 1), (3, 4096, 2), (17, 1024, 3), (32, 512, 4)])
def test_quant_matches_torch_restatement(oracle_mod, M, K, seed):
    x = synth.x_bf16(M, K, seed=seed)
    xq, xs = oracle_mod.quant_1x128(x, 0)
    cq, cs = _torch_quant_1x128(x)
    assert np.array_equal(xs, cs)
    assert np.array_equal(xq, cq)


def test_quant_ue8m0_hand_values(oracle_mod):
    vals = [0.0] * 128
    vals[0] = 448.0
    xq, xs = oracle_mod.quant_1x128(bf16_row(vals), 1)
    assert xs[0, 0] == 127 and xq[0, 0] == 0x7E
    vals[0] = 449.0   # bf16 rounds 449 to 448, so use 450 (exact in bf16)
    vals[0] = 450.0
    xq, xs = oracle_mod.quant_1x128(bf16_row(vals), 1)
    assert xs[0, 0] == 128                  # scale 2
    assert xq[0, 0] == 0x76                 # 450 / 2 = 225 -> 224 = 2^7 * 1.75 -> 0x76


def test_quant_ue8m0_properties(oracle_mod):
    x = synth.x_bf16(5, 2048, seed=12)
    xq, xb = oracle_mod.quant_1x128(x, 1)
    xf = synth.bf16_bits_to_f32(x).reshape(5, 16, 128)
    amax = np.abs(xf).max(axis=2)
    s = (amax / np.float32(448.0)).astype(np.float32)
    p = np.exp2(xb.astype(np.float64) - 127)
    assert np.all(p >= s) and np.all(s > p / 2)
    assert np.all((xq & 0x7F) <= 0x7E)
    # codes are the torch cast of x / 2^e (exact power-of-two scaling)
    ref = torch_e4m3_bytes((xf / p[:, :, None].astype(np.float32)).reshape(5, 2048))
    assert np.array_equal(ref, xq)


# ---------------------------------------------------------------------------
# 128x128 weight quantisation (input generator)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", [0, 1])
def test_weight_quant_matches_torch_restatement(oracle_mod, kind):
    N, K = 256, 384
    w = synth.w_f32(N, K, seed=21)
    w[130, 300] = 0.5  # a large entry in block (1, 2) only
    wq, ws = oracle_mod.quant_weight_128x128(w, kind)
    t = torch.from_numpy(w).view(2, 128, 3, 128).permute(0, 2, 1, 3)
    amax = t.abs().amax(dim=(2, 3))
    s = amax / torch.tensor(448.0, dtype=torch.float32)
    if kind == 1:
        e = torch.ceil(torch.log2(s.double()))
        e = torch.where(torch.exp2(e - 1) >= s.double(), e - 1, e)  # guard log2 rounding
        sc = torch.exp2(e).float()
        assert np.array_equal(ws.astype(np.int64), (e + 127).long().numpy())
    else:
        sc = s
        assert np.array_equal(ws, s.numpy())
    q = (t / sc[:, :, None, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    ref = q.permute(0, 2, 1, 3).reshape(N, K).numpy()
    assert np.array_equal(ref, wq)
    # the big entry decides only its own block
    blk = wq[128:256, 256:384] & 0x7F
    assert (wq[130, 300] & 0x7F) == blk.max()
    if kind == 0:
        assert wq[130, 300] == 0x7E


# ---------------------------------------------------------------------------
# block-scale GEMM
# ---------------------------------------------------------------------------

def _dequant(codes, scales, kind, rows_per_block):
    vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    d = vals[codes]
    if kind == 1:
        sc = np.exp2(scales.astype(np.float64) - 127)
    else:
        sc = scales.astype(np.float64)
    sc = np.repeat(np.repeat(sc, rows_per_block, axis=0), 128, axis=1)
    return d * sc


@pytest.mark.parametrize("kind", [0, 1])
@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (2, 256, 384), (3, 128, 256), (3, 256, 128)])
def test_gemm_equals_dequantised_fp64_matmul(oracle_mod, kind, M, N, K):
    x = synth.x_bf16(M, K, seed=100 + M + K)
    w = synth.w_f32(N, K, seed=200 + N + K)
    xq, xs = oracle_mod.quant_1x128(x, kind)
    wq, ws = oracle_mod.quant_weight_128x128(w, kind)
    y, y64 = oracle_mod.gemm(xq, xs, wq, ws, kind, want_f64=True)
    xd = _dequant(xq, xs, kind, 1)
    wd = _dequant(wq, ws, kind, 128)
    ref = xd @ wd.T
    assert np.allclose(y64, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert np.array_equal(y, oracle_mod.f64_to_bf16_array(y64))


def test_gemm_integer_case_is_exact(oracle_mod):
    # codes of small integers, all scales 1: the result is an integer matmul.
    rng = np.random.default_rng(17)
    ints = np.arange(-6, 7)
    code_of = {int(v): oracle_mod.e4m3_encode(float(v)) for v in ints}
    M, N, K = 3, 256, 384
    a = rng.choice(ints, size=(M, K))
    b = rng.choice(ints, size=(N, K))
    xq = np.vectorize(code_of.get)(a).astype(np.uint8)
    wq = np.vectorize(code_of.get)(b).astype(np.uint8)
    xs = np.ones((M, K // 128), dtype=np.float32)
    ws = np.ones((N // 128, K // 128), dtype=np.float32)
    y, y64 = oracle_mod.gemm(xq, xs, wq, ws, 0, want_f64=True)
    exact = a.astype(np.int64) @ b.astype(np.int64).T
    assert np.array_equal(y64, exact.astype(np.float64))


def test_gemm_scales_index_blocks_not_transposed(oracle_mod):
    # one non-zero code and distinct per-block scales: the output picks exactly
    # xs[m, kb] * ws[n // 128, kb] for the block holding the code.
    M, N, K = 2, 256, 384
    xq = np.zeros((M, K), dtype=np.uint8)
    wq = np.zeros((N, K), dtype=np.uint8)
    xq[1, 300] = 0x38   # 1.0 at k = 300 (kb = 2)
    wq[200, 300] = 0x40  # 2.0 at n = 200 (n-block 1)
    xs = (np.arange(M * 3, dtype=np.float32).reshape(M, 3) + 1)
    ws = (np.arange(2 * 3, dtype=np.float32).reshape(2, 3) + 1) * np.float32(10)
    y, y64 = oracle_mod.gemm(xq, xs, wq, ws, 0, want_f64=True)
    expect = np.zeros((M, N))
    expect[1, 200] = 1.0 * 2.0 * xs[1, 2] * ws[1, 2]
    assert np.array_equal(y64, expect)


def test_gemm_threads_agree(oracle_mod):
    x = synth.x_bf16(4, 512, seed=31)
    w = synth.w_f32(512, 512, seed=32)
    xq, xs = oracle_mod.quant_1x128(x, 0)
    wq, ws = oracle_mod.quant_weight_128x128(w, 0)
    y1 = oracle_mod.gemm(xq, xs, wq, ws, 0, nthreads=1)
    y4 = oracle_mod.gemm(xq, xs, wq, ws, 0, nthreads=4)
    assert np.array_equal(y1, y4)


def test_linear_is_quant_then_gemm(oracle_mod):
    x = synth.x_bf16(3, 1024, seed=41)
    w = synth.w_f32(256, 1024, seed=42)
    for kind in (0, 1):
        wq, ws = oracle_mod.quant_weight_128x128(w, kind)
        y, xq, xs = oracle_mod.linear(x, wq, ws, kind)
        xq2, xs2 = oracle_mod.quant_1x128(x, kind)
        assert np.array_equal(xq, xq2) and np.array_equal(xs, xs2)
        assert np.array_equal(y, oracle_mod.gemm(xq2, xs2, wq, ws, kind))


# ---------------------------------------------------------------------------
# RMSNorm producer ("[Perf] [AMD] dsv4: optional e8m0 mxscale GEMM for dense
# 128x128 fp8 linears (6/8)", "Modifications": the fused input_norm / q_norm
# producers emit the 1x128 scales).  Reading: y = x * gamma / sqrt(mean x^2 +
# eps), rounded to bf16, then the 1x128 quant of those bf16 values.
# ---------------------------------------------------------------------------

BF16_ONE = 0x3F80


def bf16_bits(vals):
    return synth.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


def test_rmsnorm_three_four_five(oracle_mod):
    # mean of squares (9 + 16) / 128, so y = x * sqrt(128) / 5 in closed form
    x = np.zeros((1, 128), np.uint16)
    x[0, :2] = bf16_bits([3.0, 4.0])
    y64, _ = oracle_mod.rmsnorm(x, np.full(128, BF16_ONE, np.uint16), 0.0)
    assert y64[0, 0] == pytest.approx(3.0 * math.sqrt(128.0) / 5.0, rel=1e-15)
    assert y64[0, 1] == pytest.approx(4.0 * math.sqrt(128.0) / 5.0, rel=1e-15)
    assert np.all(y64[0, 2:] == 0.0)


@pytest.mark.parametrize("c", [0.375, -3.0, 1000.0])
def test_rmsnorm_constant_row_is_its_sign(oracle_mod, c):
    # every |x| equal -> rms = |x| -> y = sign(x) exactly (eps 0)
    K = 256
    x = np.tile(bf16_bits([c, -c]), (2, K // 2))
    y64, y = oracle_mod.rmsnorm(x, np.full(K, BF16_ONE, np.uint16), 0.0)
    assert np.all(y64[:, 0::2] == math.copysign(1.0, c)) and np.all(y64[:, 1::2] == -math.copysign(1.0, c))
    assert np.all(y[:, 0::2] == (0x3F80 if c > 0 else 0xBF80))


def test_rmsnorm_eps_enters_under_the_root(oracle_mod):
    # mean x^2 = 1 and eps = 3 -> rms = 2 -> y = x / 2
    K = 128
    x = np.tile(bf16_bits([1.0, -1.0]), (1, K // 2))
    y64, _ = oracle_mod.rmsnorm(x, np.full(K, BF16_ONE, np.uint16), 3.0)
    assert np.all(y64[0, 0::2] == 0.5) and np.all(y64[0, 1::2] == -0.5)


def test_rmsnorm_zero_row_is_zero(oracle_mod):
    K = 256
    x = np.zeros((1, K), np.uint16)
    x[0, 1::2] = 0x8000  # -0.0
    y64, y = oracle_mod.rmsnorm(x, synth.gamma_bf16(K, seed=3), 1e-6)
    assert np.all(y64 == 0.0) and not np.any(np.isnan(y64))
    _, xq, xs = oracle_mod.rmsnorm_quant(x, synth.gamma_bf16(K, seed=3), 1e-6)
    assert np.all(xs == 0.0) and np.all(xq[0, 0::2] == 0x00) and np.all(xq[0, 1::2] == 0x80)


def test_rmsnorm_power_of_two_scale_invariance(oracle_mod):
    # eps 0: scaling a row by 2^j scales every x and the rms by 2^j exactly
    K = 512
    x = synth.x_bf16(3, K, seed=11)
    g = synth.gamma_bf16(K, seed=12)
    xs = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(x) * np.float32(8.0))
    a, ya = oracle_mod.rmsnorm(x, g, 0.0)
    b, yb = oracle_mod.rmsnorm(xs, g, 0.0)
    assert np.array_equal(a, b) and np.array_equal(ya, yb)


def test_rmsnorm_gamma_multiplies_each_column(oracle_mod):
    # y(gamma) = gamma * y(1) column by column, against a numpy restatement of
    # the normalisation with unit weight
    K = 384
    x = synth.x_bf16(4, K, seed=21)
    g = synth.gamma_bf16(K, seed=22)
    y1, _ = oracle_mod.rmsnorm(x, np.full(K, BF16_ONE, np.uint16), 1e-6)
    yg, _ = oracle_mod.rmsnorm(x, g, 1e-6)
    gf = synth.bf16_bits_to_f32(g).astype(np.float64)
    np.testing.assert_allclose(yg, y1 * gf[None, :], rtol=1e-14, atol=0)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    ref = xf / np.sqrt(np.mean(xf * xf, axis=1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(y1, ref, rtol=1e-13, atol=0)


def test_rmsnorm_quant_is_quant_of_the_rounded_norm(oracle_mod):
    # the producer's bytes are those of the two steps in sequence, and the bf16
    # output is the fp64 value rounded to nearest even by torch's cast
    K = 640
    x = synth.x_bf16(5, K, seed=31)
    g = synth.gamma_bf16(K, seed=32)
    for kind in (0, 1):
        y, xq, xsc = oracle_mod.rmsnorm_quant(x, g, 1e-6, kind)
        y64, yb = oracle_mod.rmsnorm(x, g, 1e-6)
        assert np.array_equal(y, yb)
        t = torch.from_numpy(y64).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(y, t)
        q2, s2 = oracle_mod.quant_1x128(y, kind)
        assert np.array_equal(xq, q2) and np.array_equal(xsc, s2)
        if kind == 0:  # every non-zero group holds a byte of magnitude 0x7E
            assert np.all((xq.reshape(5, K // 128, 128) & 0x7F).max(axis=2) == 0x7E)


# ---------------------------------------------------------------------------
# Small-M FP8 block-scale MoE ("[AMD] gfx950 small-batch MoE: expert-count gate
# for the small sort and FP8 block-scale small-M kernel", "Modifications":
# e4m3 w13 / w2 with 128x128 fp32 block scales applied to each partial sum).
# Reading: a = bf16(silu(gate) * up), y = bf16(sum_s topk_w * (a . w2^T)).
# ---------------------------------------------------------------------------

def _moe_inputs(oracle_mod, M, S, E, H, I, seed):
    x = synth.x_bf16(M, H, seed=seed)
    ids, tw = synth.moe_routing(M, S, E, seed=seed + 1)
    w13, s13 = oracle_mod.quant_weight_128x128(synth.w_f32(E * 2 * I, H, seed=seed + 2), 0)
    w2, s2 = oracle_mod.quant_weight_128x128(synth.w_f32(E * H, I, seed=seed + 3), 0)
    return (x, ids, tw, w13.reshape(E, 2 * I, H), s13.reshape(E, 2 * I // 128, H // 128),
            w2.reshape(E, H, I), s2.reshape(E, H // 128, I // 128))


def _bf16_round_f64(oracle_mod, v):
    return synth.bf16_bits_to_f32(oracle_mod.f64_to_bf16_array(v)).astype(np.float64)


def test_moe_matches_dequantized_numpy_reference(oracle_mod):
    # the blocked partial sums equal numpy's matmul of the dequantised weights
    M, S, E, H, I = 3, 4, 5, 384, 256
    x, ids, tw, w13, s13, w2, s2 = _moe_inputs(oracle_mod, M, S, E, H, I, seed=41)
    _, y64 = oracle_mod.moe_w8a16(x, ids, tw, w13, s13, w2, s2, want_f64=True)
    dec = oracle_mod.e4m3_table()
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    W13 = dec[w13] * np.repeat(np.repeat(s13.astype(np.float64), 128, axis=1), 128, axis=2)
    W2 = dec[w2] * np.repeat(np.repeat(s2.astype(np.float64), 128, axis=1), 128, axis=2)
    ref = np.zeros((M, H))
    for m in range(M):
        for s in range(S):
            e = ids[m, s]
            h = W13[e] @ xf[m]
            g, u = h[:I], h[I:]
            a = _bf16_round_f64(oracle_mod, g / (1.0 + np.exp(-g)) * u)
            ref[m] += float(tw[m, s]) * (W2[e] @ a)
    np.testing.assert_allclose(y64, ref, rtol=1e-9, atol=1e-12 * np.abs(ref).max())


def test_moe_identity_weights_give_silu_closed_form(oracle_mod):
    # w13 = [I; I] (gate = up = x), w2 = I, scales 1: y = w * bf16(silu(x) * x)
    H = I = 128
    E, M, S = 1, 1, 1
    one = 0x38  # e4m3 code of 1.0
    w13 = np.zeros((E, 2 * I, H), np.uint8)
    w13[0, np.arange(I), np.arange(I)] = one
    w13[0, I + np.arange(I), np.arange(I)] = one
    w2 = np.zeros((E, H, I), np.uint8)
    w2[0, np.arange(H), np.arange(I)] = one
    s13 = np.ones((E, 2, 1), np.float32)
    s2 = np.ones((E, 1, 1), np.float32)
    xv = np.zeros(H, np.float32)
    xv[:4] = [1.0, -1.0, 2.0, 0.5]
    x = synth.f32_to_bf16_bits(xv)[None, :]
    _, y64 = oracle_mod.moe_w8a16(x, np.zeros((1, 1), np.int32), np.full((1, 1), 0.5, np.float32),
                                  w13, s13, w2, s2, want_f64=True)
    for k, v in enumerate([1.0, -1.0, 2.0, 0.5]):
        act = v * v / (1.0 + math.exp(-v))
        expect = 0.5 * float(synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(np.float32([act])))[0])
        assert y64[0, k] == pytest.approx(expect, rel=2 ** -8)
    assert np.all(y64[0, 4:] == 0.0)
    assert y64[0, 0] == pytest.approx(0.5 * 0.73046875, rel=1e-12)  # bf16(silu(1)) = 0.73046875


def test_moe_is_linear_in_the_routing_weights(oracle_mod):
    # the same expert in two slots with weights a and b equals one slot a + b;
    # zero weights give a zero output
    M, S, E, H, I = 2, 3, 4, 256, 128
    x, ids, tw, w13, s13, w2, s2 = _moe_inputs(oracle_mod, M, S, E, H, I, seed=51)
    ids2 = ids.copy()
    ids2[:, 1] = ids2[:, 0]
    w_split = tw.copy()
    w_split[:, 0], w_split[:, 1] = 0.25, 0.5
    w_one = w_split.copy()
    w_one[:, 0], w_one[:, 1] = 0.75, 0.0
    _, a = oracle_mod.moe_w8a16(x, ids2, w_split, w13, s13, w2, s2, want_f64=True)
    _, b = oracle_mod.moe_w8a16(x, ids2, w_one, w13, s13, w2, s2, want_f64=True)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-15)
    _, z = oracle_mod.moe_w8a16(x, ids, np.zeros_like(tw), w13, s13, w2, s2, want_f64=True)
    assert np.all(z == 0.0)


def test_integer_e4m3_decode_identity_used_by_the_moe_kernels(oracle_mod):
    # the MoE kernels decode a code c with integer operations only: its 7
    # magnitude bits to bf16 bits 4-10 and its sign to bit 15, which is the
    # code's value times 2^-120 for every finite code, subnormals included
    # (checked here exactly, against the oracle's decode from the format)
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue  # NaN codes
        bits = ((c & 0x7F) << 4) | ((c & 0x80) << 8)
        v = float(synth.bf16_bits_to_f32(np.array([bits], np.uint16))[0])
        assert math.ldexp(v, 120) == oracle_mod.e4m3_decode(c), hex(c)
