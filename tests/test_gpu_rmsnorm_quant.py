"""GPU parity of the fused RMSNorm + 1x128 quant producer against the CPU oracle.

The producer is the input_norm / q_norm kernel of "[Perf] [AMD] dsv4: optional
e8m0 mxscale GEMM for dense 128x128 fp8 linears (6/8)", "Modifications", which
emits the GEMM's activation scales itself.  Bar:

* the bf16 normalised rows y within bf16 rounding of the oracle's fp64 RMSNorm:
  |y - y64| <= 2^-8 |y64| elementwise (half a bf16 ulp of rounding plus the
  fp32 arithmetic), and equal to bf16(y64) for almost every element;
* the codes and scales bit-exact against the oracle's 1x128 quant of the y the
  kernel wrote, so the quant decision is taken from the same bf16 values on
  both sides.
"""

import numpy as np
import pytest
import torch

import fp8_block_scale_x128_gb300 as fb
import synth
from tests import helpers as H

pytestmark = pytest.mark.gpu

F32, UE8 = fb.FP8BS_SCALE_F32, fb.FP8BS_SCALE_UE8M0
EPS = 1e-6


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fb.build()
    fb.lib()
    return torch.device("cuda", 0)


def bf16_dev(bits: np.ndarray, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def check_against_oracle(oracle_mod, x, g, eps, kind, xq, xs, y, what=""):
    y64, y_ref = oracle_mod.rmsnorm(x, g, eps)
    yf = H.bf16_to_f32(y).astype(np.float64)
    assert np.all(np.isfinite(yf)), what
    err = np.abs(yf - y64)
    bound = np.abs(y64) * 2.0 ** -8
    bad = np.flatnonzero(err > bound)
    assert bad.size == 0, f"{what}: y off at {bad[:5]}: gpu {yf.flat[bad[0]]} ref {y64.flat[bad[0]]}"
    frac_exact = float((y == y_ref).mean())
    assert frac_exact > 0.99, f"{what}: only {frac_exact:.4f} of y equal bf16(y64)"
    q_ref, s_ref = oracle_mod.quant_1x128(y, kind)
    assert np.array_equal(xq, q_ref), what
    assert np.array_equal(xs, s_ref), what
    return frac_exact


def run(oracle_mod, dev, M, K, kind, seed, eps=EPS, ldx_pad=0, ldy_pad=0, x=None, g=None):
    x = synth.x_bf16(M, K, seed=seed) if x is None else x
    g = synth.gamma_bf16(K, seed=seed + 1) if g is None else g
    xd_full = torch.zeros((M, K + ldx_pad), dtype=torch.bfloat16, device=dev)
    xd_full[:, :K] = bf16_dev(x, dev)
    yd_full = torch.full((M, K + ldy_pad), float("nan"), dtype=torch.bfloat16, device=dev)
    xq, xs, yd = fb.fp8bs_rmsnorm_quant(xd_full[:, :K], bf16_dev(g, dev), eps, kind,
                                        y=yd_full[:, :K])
    torch.cuda.synchronize()
    if ldy_pad:
        assert torch.isnan(yd_full[:, K:].float()).all()  # nothing written past K
    y = H.torch_u16_to_np(yd)
    check_against_oracle(oracle_mod, x, g, eps, kind, xq.cpu().numpy(), xs.cpu().numpy(), y,
                         f"M={M} K={K} kind={kind}")
    return x, g, xq, xs, y


@pytest.mark.parametrize("kind", [F32, UE8])
@pytest.mark.parametrize("M,K", [(1, 128), (3, 640), (1, 2048), (4, 4096), (17, 7168), (32, 7168),
                                 (5, 8192), (2, 8320), (9, 16384), (33, 2048)])
def test_rmsnorm_quant_against_oracle(dev, oracle_mod, M, K, kind):
    # K from one group to the 16384 limit, ragged against the 16 groups a CTA
    # pass covers (640, 7168, 8320), every J variant of the kernel (1, 2, 4, 8)
    run(oracle_mod, dev, M, K, kind, seed=7000 + 13 * M + K // 128)


def test_rmsnorm_quant_strided_rows(dev, oracle_mod):
    run(oracle_mod, dev, 5, 2048, F32, seed=71, ldx_pad=64, ldy_pad=8)


def test_rmsnorm_quant_without_y_gives_the_same_bytes(dev, oracle_mod):
    M, K = 6, 4096
    x, g, xq, xs, _ = run(oracle_mod, dev, M, K, UE8, seed=81)
    xq2, xs2, y2 = fb.fp8bs_rmsnorm_quant(bf16_dev(x, dev), bf16_dev(g, dev), EPS, UE8)
    assert y2 is None
    assert torch.equal(xq, xq2) and torch.equal(xs, xs2)


def test_rmsnorm_quant_is_deterministic(dev, oracle_mod):
    M, K = 64, 7168
    x = bf16_dev(synth.x_bf16(M, K, seed=91), dev)
    g = bf16_dev(synth.gamma_bf16(K, seed=92), dev)
    a = fb.fp8bs_rmsnorm_quant(x, g, EPS, F32, want_y=True)
    for _ in range(3):
        b = fb.fp8bs_rmsnorm_quant(x, g, EPS, F32, want_y=True)
        assert all(torch.equal(p, q) for p, q in zip(a, b))


@pytest.mark.parametrize("kind", [F32, UE8])
def test_rmsnorm_quant_special_rows(dev, oracle_mod, kind):
    # a zero row (signed zeros, eps 0 -> no NaN), a row of one repeated value
    # (|y| constant: every byte of one magnitude), a row with one large
    # outlier, and a row of small values (1e-12: their squares stay normal fp32
    # numbers, the range the fp32 sum of squares covers)
    K = 1024
    x = np.zeros((4, K), np.uint16)
    x[0, 1::2] = 0x8000
    x[1] = synth.f32_to_bf16_bits(np.tile(np.float32([0.75, -0.75]), K // 2))
    x[2] = synth.x_bf16(1, K, seed=5, outliers=False)[0]
    x[2, 100] = synth.f32_to_bf16_bits(np.float32([3.0e4]))[0]
    x[3] = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(synth.x_bf16(1, K, seed=6)[0]) * np.float32(1e-12))
    g = np.full(K, 0x3F80, np.uint16)
    _, _, xq, xs, y = run(oracle_mod, dev, 4, K, kind, seed=0, eps=0.0, x=x, g=g)
    xq = xq.cpu().numpy()
    assert np.all(xq[0, 0::2] == 0x00) and np.all(xq[0, 1::2] == 0x80)
    # |y| = 1 everywhere: fp32 scale 1/448 -> every code +-448 (0x7E); ue8m0
    # scale 2^-8 (the power of two above 1/448) -> every code +-256 (0x78)
    assert np.all((xq[1] & 0x7F) == (0x7E if kind == F32 else 0x78))


def test_rmsnorm_quant_feeds_the_prequant_gemm(dev, oracle_mod):
    # the producer's codes and scales as the GEMM's input: the two-launch chain
    # RMSNorm+quant -> fp8bs_gemm_prequant against the oracle GEMM of the same
    # codes, and bit-identical to quantising the producer's y separately
    M, N, K, kind = 8, 1024, 4096, UE8
    x = synth.x_bf16(M, K, seed=101)
    g = synth.gamma_bf16(K, seed=102)
    wq, ws = H.weight(oracle_mod, N, K, kind, 103)
    packed = fb.fp8bs_prepack_weight(torch.from_numpy(wq).to(dev), torch.from_numpy(ws).to(dev), kind)
    wsp = fb.new_workspace(N, K, dev)
    xq, xs, yd = fb.fp8bs_rmsnorm_quant(bf16_dev(x, dev), bf16_dev(g, dev), EPS, kind, want_y=True)
    out = fb.fp8bs_gemm_prequant(xq, xs, packed, N, K, kind, workspace=wsp)
    assert fb.fp8bs_check_error(wsp) == 0
    xq2, xs2 = fb.fp8bs_quant(yd, kind)
    assert torch.equal(xq, xq2) and torch.equal(xs, xs2)
    y_ref = oracle_mod.gemm(xq.cpu().numpy(), xs.cpu().numpy(), wq, ws, kind, nthreads=H.threads())
    H.check_y(H.torch_u16_to_np(out), y_ref, "rmsnorm_quant -> gemm_prequant")


def test_rmsnorm_quant_full_size_sampled_rows(dev, oracle_mod):
    # the benchmark's large-M launch (16384 x 7168): every row is independent,
    # so sampled rows are checked one by one against the oracle
    M, K = 16384, 7168
    xd = synth.x_bf16_torch(M, K, seed=111, device=dev)
    g = synth.gamma_bf16(K, seed=112)
    xq, xs, yd = fb.fp8bs_rmsnorm_quant(xd, bf16_dev(g, dev), EPS, F32, want_y=True)
    torch.cuda.synchronize()
    rows = np.random.default_rng(113).choice(M, size=48, replace=False)
    rows = np.concatenate([rows, [0, M - 1]])
    idx = torch.from_numpy(rows).to(dev)
    x = H.torch_u16_to_np(xd.index_select(0, idx))
    y = H.torch_u16_to_np(yd.index_select(0, idx))
    check_against_oracle(oracle_mod, x, g, EPS, F32, xq.index_select(0, idx).cpu().numpy(),
                         xs.index_select(0, idx).cpu().numpy(), y, "16384x7168 sampled rows")


@pytest.mark.parametrize("kind", [F32, UE8])
def test_rmsnorm_quant_codes_equal_the_oracle_producer(dev, oracle_mod, kind):
    # End to end against the oracle's own producer (oracle.rmsnorm_quant, which
    # quantises its own bf16(y64)): wherever the kernel's normalised row equals
    # the oracle's in every element -- the premise, asserted first to hold for
    # most rows -- its codes and scales must equal the oracle's byte for byte.
    M, K = 96, 256
    x = synth.x_bf16(M, K, seed=9001 + kind)
    g = synth.gamma_bf16(K, seed=9002 + kind)
    yd = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    xq, xs, yd = fb.fp8bs_rmsnorm_quant(bf16_dev(x, dev), bf16_dev(g, dev), EPS, kind, y=yd)
    torch.cuda.synchronize()
    y = H.torch_u16_to_np(yd)
    y_o, q_o, s_o = oracle_mod.rmsnorm_quant(x, g, EPS, kind)
    rows = np.flatnonzero((y == y_o).all(axis=1))
    assert rows.size >= 3 * M // 4, f"premise: only {rows.size} of {M} rows have y == bf16(y64)"
    assert np.array_equal(xq.cpu().numpy()[rows], q_o[rows])
    assert np.array_equal(xs.cpu().numpy()[rows], s_o[rows])
