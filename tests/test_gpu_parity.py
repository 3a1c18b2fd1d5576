"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Bar: bit-exact for every quantised byte and scale (activation quant, weight
quant, the fused kernel's quant write-out, prepacked layout); the bf16 output
within the tolerance in tests/helpers.py.  Inputs come from synth with the
recipes of the pages' workloads; shapes span several tiles, ragged M and the
full sizes of the benchmark."""

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import fp8_block_scale_x128_gb300 as fb
import synth
from tests import helpers as H

pytestmark = pytest.mark.gpu

F32, UE8 = fb.FP8BS_SCALE_F32, fb.FP8BS_SCALE_UE8M0


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fb.build()
    fb.lib()
    return torch.device("cuda", 0)


def to_dev(a: np.ndarray, dev, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(dev)


def x_dev(x_bits: np.ndarray, dev):
    return to_dev(x_bits.view(np.int16), dev).view(torch.bfloat16)


def run_fused(oracle_mod, dev, M, N, K, kind, seed, want_quant=True, ldx_pad=0, ldy_pad=0,
              workspace=None):
    x = synth.x_bf16(M, K, seed=seed)
    wq, ws = H.weight(oracle_mod, N, K, kind, seed + 1)
    y_ref, xq_ref, xs_ref = oracle_mod.linear(x, wq, ws, kind, nthreads=H.threads())
    xd_full = torch.zeros((M, K + ldx_pad), dtype=torch.bfloat16, device=dev)
    xd_full[:, :K] = x_dev(x, dev)
    xd = xd_full[:, :K]
    packed = fb.fp8bs_prepack_weight(to_dev(wq, dev), to_dev(ws, dev), kind)
    yd_full = torch.full((M, N + ldy_pad), float("nan"), dtype=torch.bfloat16, device=dev)
    yd = yd_full[:, :N]
    xq = torch.zeros((M, K), dtype=torch.uint8, device=dev) if want_quant else None
    xs = (torch.zeros((M, K // 128), dtype=torch.uint8 if kind == UE8 else torch.float32,
                      device=dev) if want_quant else None)
    wsp = workspace if workspace is not None else fb.new_workspace(N, K, dev)
    fb.fp8bs_gemm_fused(xd, packed, N, K, kind, y=yd, workspace=wsp, xq_out=xq, xs_out=xs)
    assert fb.fp8bs_check_error(wsp) == 0
    y = H.torch_u16_to_np(yd)
    stats = H.check_y(y, y_ref, f"M={M} N={N} K={K} kind={kind}")
    if ldy_pad:
        assert torch.isnan(yd_full[:, N:].float()).all()  # nothing written past N
    if want_quant:
        assert np.array_equal(xq.cpu().numpy(), xq_ref)
        assert np.array_equal(xs.cpu().numpy(), xs_ref)
    return stats


# ---------------------------------------------------------------------------
# encoder: every fp32 bit pattern
# ---------------------------------------------------------------------------

def test_encode_e4m3_exhaustive_against_oracle(dev, oracle_mod):
    chunk = 1 << 26
    nthr = H.threads()
    sub = chunk // nthr
    pool = ThreadPoolExecutor(max_workers=nthr)
    ref = np.empty(chunk, dtype=np.uint8)
    base = torch.arange(chunk, dtype=torch.int64, device=dev)
    for start in range(0, 1 << 32, chunk):
        bits = (base + start).to(torch.int64)
        bits = torch.where(bits >= (1 << 31), bits - (1 << 32), bits).to(torch.int32)
        v = bits.view(torch.float32)
        got = fb.fp8bs_encode_e4m3(v).cpu().numpy()
        futs = [pool.submit(oracle_mod.e4m3_encode_bits, start + t * sub,
                            sub if t < nthr - 1 else chunk - t * sub, ref[t * sub:])
                for t in range(nthr)]
        for f in futs:
            f.result()
        vv = np.arange(start, start + chunk, dtype=np.uint64).astype(np.uint32).view(np.float32)
        nan = np.isnan(vv)
        bad = np.flatnonzero((got != ref) & ~nan)
        assert bad.size == 0, f"first mismatch at bits {start + int(bad[0]):#010x}: " \
                              f"gpu {got[bad[0]]:#04x} oracle {ref[bad[0]]:#04x}"
        assert np.all((got[nan] & 0x7F) == 0x7F)
    pool.shutdown()


# ---------------------------------------------------------------------------
# standalone quantisers
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", [F32, UE8])
@pytest.mark.parametrize("M,K,pad", [(1, 2048, 0), (3, 4096, 0), (9, 7168, 64), (17, 512, 8),
                                     (32, 4096, 0), (33, 256, 0), (100, 1024, 0)])
def test_quant_bit_exact(dev, oracle_mod, kind, M, K, pad):
    x = synth.x_bf16(M, K, seed=7 * M + K)
    xq_ref, xs_ref = oracle_mod.quant_1x128(x, kind)
    full = torch.zeros((M, K + pad), dtype=torch.bfloat16, device=dev)
    full[:, :K] = x_dev(x, dev)
    xq, xs = fb.fp8bs_quant(full[:, :K], kind)
    torch.cuda.synchronize()
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert np.array_equal(xs.cpu().numpy(), xs_ref)


@pytest.mark.parametrize("kind", [F32, UE8])
def test_quant_bit_exact_16m_values(dev, oracle_mod, kind):
    # 16M values: the quantiser's reciprocal fast path meets a few hundred
    # quotients within a few ulps of an e4m3 rounding boundary, where it must
    # fall back to the IEEE division
    M, K = 4096, 4096
    x = synth.x_bf16(M, K, seed=2024 + kind)
    xq_ref, xs_ref = oracle_mod.quant_1x128(x, kind)
    xq, xs = fb.fp8bs_quant(x_dev(x, dev), kind)
    assert np.array_equal(xs.cpu().numpy(), xs_ref)
    got = xq.cpu().numpy()
    bad = np.argwhere(got != xq_ref)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[0]}"


@pytest.mark.parametrize("kind", [F32, UE8])
def test_quant_special_groups(dev, oracle_mod, kind):
    K = 128 * 8
    v = np.zeros((4, K), dtype=np.float32)
    v[0, 128:256] = -0.0                        # zero group with negative zeros
    v[0, 256:384] = 3.0                         # all equal
    v[0, 384:512] = np.linspace(-1, 1, 128)     # plain
    v[0, 512] = 3.0e38                          # huge
    v[0, 513:640] = 1.0
    v[1, :128] = np.float32(2.0 ** -130)        # bf16 subnormals
    v[1, 5] = -np.float32(2.0 ** -133)
    v[1, 128:256] = np.float32(448.0)
    v[1, 129] = 17.0                            # exact tie at scale 1
    v[2] = synth.bf16_bits_to_f32(synth.x_bf16(1, K, seed=3))[0] * np.float32(1e-30)
    v[3] = synth.bf16_bits_to_f32(synth.x_bf16(1, K, seed=4))[0] * np.float32(1e30)
    x = synth.f32_to_bf16_bits(v)
    x[0, 128:256] = 0x8000
    xq_ref, xs_ref = oracle_mod.quant_1x128(x, kind)
    xq, xs = fb.fp8bs_quant(x_dev(x, dev), kind)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert np.array_equal(xs.cpu().numpy(), xs_ref)


@pytest.mark.parametrize("kind", [F32, UE8])
@pytest.mark.parametrize("N,K", [(128, 128), (256, 384), (4096, 2048)])
def test_quant_weight_bit_exact(dev, oracle_mod, kind, N, K):
    w = synth.w_f32(N, K, seed=N + K)
    w[0, 0] = 0.0
    if N >= 256:
        w[128:256, :128] = 0.0                  # an all-zero block
        w[130, 5] = -0.0
    wq_ref, ws_ref = oracle_mod.quant_weight_128x128(w, kind)
    wq, ws = fb.fp8bs_quant_weight(to_dev(w, dev), kind)
    assert np.array_equal(wq.cpu().numpy(), wq_ref)
    assert np.array_equal(ws.cpu().numpy(), ws_ref)


# ---------------------------------------------------------------------------
# prepack layout
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", [F32, UE8])
def test_prepack_layout(dev, kind):
    N, K = 384, 256
    rng = np.random.default_rng(5)
    wq = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    ws = (rng.random((N // 128, K // 128)).astype(np.float32) if kind == F32
          else rng.integers(100, 140, size=(N // 128, K // 128), dtype=np.uint8))
    packed = fb.fp8bs_prepack_weight(to_dev(wq, dev), to_dev(ws, dev), kind).cpu().numpy()
    hdr = packed[:32]
    assert hdr[:4].tobytes() == b"F8BS"
    assert int(hdr[8:16].view(np.int64)[0]) == N and int(hdr[16:24].view(np.int64)[0]) == K
    assert int(hdr[24:28].view(np.int32)[0]) == kind
    KB = K // 128
    for nt in range(N // 128):
        for kb in range(KB):
            tile = packed[256 + (nt * KB + kb) * 16384:][:16384]
            for r in range(128):
                for j in range(8):
                    off = (r // 8) * 1024 + (r % 8) * 128 + ((j ^ (r % 8)) * 16)
                    src = wq[nt * 128 + r, kb * 128 + j * 16: kb * 128 + j * 16 + 16]
                    assert np.array_equal(tile[off:off + 16], src)
    sc = packed[256 + (N // 128) * KB * 16384:]
    if kind == F32:
        assert np.array_equal(sc[:ws.size * 4].view(np.float32), ws.ravel())
    else:
        assert np.array_equal(sc[:ws.size], ws.ravel())


# ---------------------------------------------------------------------------
# fused quant + GEMM
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("kind", [F32, UE8])
@pytest.mark.parametrize("M", [1, 5, 6, 7, 16, 17, 32])
@pytest.mark.parametrize("N,K", [(128, 128), (256, 384), (384, 640), (1024, 1024), (640, 2048)])
def test_fused_small_shapes(dev, oracle_mod, kind, M, N, K):
    run_fused(oracle_mod, dev, M, N, K, kind, seed=M * 131 + N + K)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 6, 8, 12, 13])
@pytest.mark.parametrize("N,K,kind", [(128, 128, F32), (384, 640, F32), (640, 2048, UE8), (5120, 4096, F32),
                                      (4608, 4096, F32), (4096, 2048, F32), (7168, 2048, UE8),
                                      (1536, 7168, UE8), (4096, 4096, UE8)])
def test_fused_few_tokens(dev, oracle_mod, N, K, kind, M):
    # the local-quant variant (up to 6 tokens), the exchange variant with tagged
    # split-K partials (7 to 12) and with flagged ones (13) on every benchmark
    # shape and a few small ones, quant bytes included
    run_fused(oracle_mod, dev, M, N, K, kind, seed=5000 + 7 * M + N // 128 + K // 128)


def test_fused_few_tokens_strided(dev, oracle_mod):
    run_fused(oracle_mod, dev, 3, 1024, 1024, F32, seed=9, ldx_pad=64, ldy_pad=8)


@pytest.mark.parametrize("M", [1, 3, 4, 8, 9, 16, 17, 24, 32])
def test_fused_m_sweep_5120x4096(dev, oracle_mod, M):
    # the M sweep at N=5120, K=4096 with bit-exact quant bytes and scales
    run_fused(oracle_mod, dev, M, 5120, 4096, F32, seed=1000 + M)


def test_fused_smallest_4096x2048(dev, oracle_mod):
    run_fused(oracle_mod, dev, 1, 4096, 2048, F32, seed=0)


@pytest.mark.parametrize("N,K", [(5120, 4096), (4608, 4096), (4096, 2048)])
@pytest.mark.parametrize("M", [1, 4, 8, 16, 32])
def test_fused_projection_shapes(dev, oracle_mod, N, K, M):
    run_fused(oracle_mod, dev, M, N, K, F32, seed=2000 + M + N // 128)


@pytest.mark.parametrize("N,K", [(7168, 2048), (1536, 7168), (4096, 4096)])
@pytest.mark.parametrize("M", [1, 16, 32])
def test_fused_ue8m0_shapes(dev, oracle_mod, N, K, M):
    run_fused(oracle_mod, dev, M, N, K, UE8, seed=3000 + M + N // 128)


@pytest.mark.parametrize("M", [33, 40, 48, 64])
@pytest.mark.parametrize("N,K,kind", [(384, 640, F32), (5120, 4096, F32), (4096, 2048, F32),
                                      (7168, 2048, UE8), (1536, 7168, UE8), (4096, 4096, UE8)])
def test_fused_above_32_tokens(dev, oracle_mod, N, K, kind, M):
    # 33..64 tokens: the 64-token tile (one CTA per SM, deeper weight ring)
    # with the activation exchange and flagged split-K partials, quant bytes
    # included
    run_fused(oracle_mod, dev, M, N, K, kind, seed=8000 + M + N // 128 + K // 128)


@pytest.mark.parametrize("M,kind", [(4, F32), (9, F32), (17, F32), (32, UE8), (64, F32)])
def test_fused_weight_larger_than_one_launch(dev, oracle_mod, M, kind):
    # 8192 units: more than one CTA per SM can hold, so the call runs several
    # launches of whole 128-row slices
    run_fused(oracle_mod, dev, M, 16384, 8192, kind, seed=4000 + M, want_quant=False)


@pytest.mark.parametrize("kind", [F32, UE8])
@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (5, 384, 640), (9, 1024, 1024), (17, 640, 2048),
                                   (32, 5120, 4096), (3, 5120, 4096), (16, 4096, 2048),
                                   (48, 5120, 4096), (64, 1536, 7168)])
def test_prequant_gemm_against_oracle(dev, oracle_mod, kind, M, N, K):
    # the second launch of the two-launch path, fed the oracle's quantised x
    x = synth.x_bf16(M, K, seed=6000 + M + K // 128)
    xq_ref, xs_ref = oracle_mod.quant_1x128(x, kind)
    wq, ws = H.weight(oracle_mod, N, K, kind, seed=6001 + N // 128)
    y_ref = oracle_mod.gemm(xq_ref, xs_ref, wq, ws, kind, nthreads=H.threads())
    packed = fb.fp8bs_prepack_weight(to_dev(wq, dev), to_dev(ws, dev), kind)
    xs_d = to_dev(xs_ref, dev) if kind == UE8 else to_dev(xs_ref, dev)
    wsp = fb.new_workspace(N, K, dev)
    y = fb.fp8bs_gemm_prequant(to_dev(xq_ref, dev), xs_d, packed, N, K, kind, workspace=wsp)
    assert fb.fp8bs_check_error(wsp) == 0
    H.check_y(H.torch_u16_to_np(y), y_ref, f"prequant M={M} N={N} K={K} kind={kind}")


@pytest.mark.parametrize("kind", [F32, UE8])
@pytest.mark.parametrize("M", [1, 6, 7, 12, 13, 16, 17, 32, 33, 64])
def test_two_launch_path_is_bit_identical_to_fused(dev, kind, M):
    # fp8bs_quant + fp8bs_gemm_prequant runs the same MMAs, rescale and split-K
    # order as the fused call on the same x
    N, K = 5120, 4096
    x = synth.x_bf16_torch(M, K, seed=77 + M, device=dev)
    w = synth.w_f32_torch(N, K, seed=78, device=dev)
    wq, ws = fb.fp8bs_quant_weight(w, kind)
    packed = fb.fp8bs_prepack_weight(wq, ws, kind)
    wsp = fb.new_workspace(N, K, dev)
    y_fused = fb.fp8bs_gemm_fused(x, packed, N, K, kind, workspace=wsp)
    xq, xs = fb.fp8bs_quant(x, kind)
    y_two = fb.fp8bs_gemm_prequant(xq, xs, packed, N, K, kind, workspace=wsp)
    assert fb.fp8bs_check_error(wsp) == 0
    assert torch.equal(y_fused.view(torch.int16), y_two.view(torch.int16))


def test_prequant_strided_codes(dev, oracle_mod):
    M, N, K = 7, 1024, 2048
    x = synth.x_bf16(M, K, seed=41)
    xq_ref, xs_ref = oracle_mod.quant_1x128(x, F32)
    wq, ws = H.weight(oracle_mod, N, K, F32, seed=42)
    y_ref = oracle_mod.gemm(xq_ref, xs_ref, wq, ws, F32, nthreads=H.threads())
    packed = fb.fp8bs_prepack_weight(to_dev(wq, dev), to_dev(ws, dev), F32)
    xq_full = torch.zeros((M, K + 48), dtype=torch.uint8, device=dev)
    xq_full[:, :K] = to_dev(xq_ref, dev)
    y = fb.fp8bs_gemm_prequant(xq_full[:, :K], to_dev(xs_ref, dev), packed, N, K, F32)
    torch.cuda.synchronize()
    H.check_y(H.torch_u16_to_np(y), y_ref, "prequant strided")


def test_fused_strided_x_and_y(dev, oracle_mod):
    run_fused(oracle_mod, dev, 7, 640, 1024, F32, seed=11, ldx_pad=64, ldy_pad=24)


def test_fused_workspace_reused_across_shapes(dev, oracle_mod):
    ws = fb.new_workspace(16384, 8192, dev)
    for (M, N, K) in [(3, 1024, 2048), (32, 5120, 4096), (1, 384, 640), (16, 4608, 4096)]:
        run_fused(oracle_mod, dev, M, N, K, F32, seed=M + N, workspace=ws)


def _setup(oracle_mod, dev, M, N, K, kind, seed):
    x = synth.x_bf16(M, K, seed=seed)
    wq, ws = H.weight(oracle_mod, N, K, kind, seed + 1)
    packed = fb.fp8bs_prepack_weight(to_dev(wq, dev), to_dev(ws, dev), kind)
    return x, wq, ws, x_dev(x, dev), packed


def test_fused_deterministic_and_graph_replay(dev, oracle_mod):
    M, N, K = 9, 5120, 4096
    x, wq, ws, xd, packed = _setup(oracle_mod, dev, M, N, K, F32, 77)
    wsp = fb.new_workspace(N, K, dev)
    outs = []
    for _ in range(3):
        y = fb.fp8bs_gemm_fused(xd, packed, N, K, F32, workspace=wsp)
        outs.append(y.clone())
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    y_graph = torch.empty_like(outs[0])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fb.fp8bs_gemm_fused(xd, packed, N, K, F32, y=y_graph, workspace=wsp, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    y_graph.zero_()
    with torch.cuda.graph(g):
        fb.fp8bs_gemm_fused(xd, packed, N, K, F32, y=y_graph, workspace=wsp)
    for _ in range(3):
        y_graph.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y_graph.view(torch.int16), outs[0].view(torch.int16))
    assert fb.fp8bs_check_error(wsp) == 0


def test_fused_pdl_independent_calls_match_plain_launches(dev, oracle_mod):
    # back-to-back calls on different weights, launched with programmatic
    # dependent launch inside a CUDA graph, give the same bits as plain calls
    for M in (5, 17):
        N, K = 4608, 4096
        x = synth.x_bf16(M, K, seed=91 + M)
        xd = x_dev(x, dev)
        packs = []
        for c in range(4):
            wq, ws = H.weight(oracle_mod, N, K, F32, 500 + c)
            packs.append(fb.fp8bs_prepack_weight(to_dev(wq, dev), to_dev(ws, dev), F32))
        wsp = fb.new_workspace(N, K, dev)
        plain = [fb.fp8bs_gemm_fused(xd, pk, N, K, F32, workspace=wsp).clone() for pk in packs]
        ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in packs]
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for pk, y in zip(packs, ys):
                fb.fp8bs_gemm_fused(xd, pk, N, K, F32, y=y, workspace=wsp, pdl=True, stream=s)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        for a, b in zip(plain, ys):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for pk, y in zip(packs, ys):
                fb.fp8bs_gemm_fused(xd, pk, N, K, F32, y=y, workspace=wsp, pdl=True)
        for _ in range(3):
            for y in ys:
                y.zero_()
            g.replay()
            torch.cuda.synchronize()
            for a, b in zip(plain, ys):
                assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        assert fb.fp8bs_check_error(wsp) == 0


@pytest.mark.parametrize("kind,M", [(F32, 8), (F32, 24), (UE8, 8)])
def test_fused_pdl_dependent_chain(dev, oracle_mod, kind, M):
    # each layer's output is the next layer's input: with programmatic
    # dependent launch the consumer must still see the producer's y
    D, layers = 2048, 6
    x0 = synth.x_bf16(M, D, seed=7)
    packs, wts = [], []
    for layer in range(layers):
        wq, ws = H.weight(oracle_mod, D, D, kind, 600 + layer)
        wts.append((wq, ws))
        packs.append(fb.fp8bs_prepack_weight(to_dev(wq, dev), to_dev(ws, dev), kind))
    wsp = fb.new_workspace(D, D, dev)
    acts = [x_dev(x0, dev)] + [torch.empty((M, D), dtype=torch.bfloat16, device=dev)
                               for _ in range(layers)]

    def run(pdl):
        for layer in range(layers):
            fb.fp8bs_gemm_fused(acts[layer], packs[layer], D, D, kind, y=acts[layer + 1],
                                workspace=wsp, pdl=pdl)
        torch.cuda.synchronize()
        return [a.clone() for a in acts[1:]]

    plain = run(False)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for layer in range(layers):
            fb.fp8bs_gemm_fused(acts[layer], packs[layer], D, D, kind, y=acts[layer + 1],
                                workspace=wsp, pdl=True)
    for _ in range(3):
        for a in acts[1:]:
            a.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(plain, acts[1:]):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # every layer matches the oracle applied to the GPU's own input
    prev = x0
    for layer in range(layers):
        wq, ws = wts[layer]
        y_ref, _, _ = oracle_mod.linear(prev, wq, ws, kind, nthreads=H.threads())
        got = H.torch_u16_to_np(plain[layer])
        H.check_y(got, y_ref, f"layer {layer}")
        prev = got
    assert fb.fp8bs_check_error(wsp) == 0


def test_fused_rejects_mismatched_packed_weight(dev, oracle_mod):
    M, N, K = 4, 256, 512
    x, wq, ws, xd, packed = _setup(oracle_mod, dev, M, N, K, F32, 5)
    wsp = fb.new_workspace(N, K, dev)
    y = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=dev)
    # packed with fp32 scales, called as ue8m0: the device header check refuses
    fb.fp8bs_gemm_fused(xd, packed, N, K, UE8, y=y, workspace=wsp)
    assert fb.fp8bs_check_error(wsp) == -4
    assert bool((y.float() == 7.0).all())
    # called with another N: refused as well
    y2 = torch.full((M, 128), 7.0, dtype=torch.bfloat16, device=dev)
    fb.fp8bs_gemm_fused(xd, packed, 128, K, F32, y=y2, workspace=wsp)
    assert fb.fp8bs_check_error(wsp) == -4
    assert bool((y2.float() == 7.0).all())
    # and the error word was cleared: a good call reports ok
    fb.fp8bs_gemm_fused(xd, packed, N, K, F32, y=y, workspace=wsp)
    assert fb.fp8bs_check_error(wsp) == 0


def test_fused_host_errors_raise(dev, oracle_mod):
    M, N, K = 65, 256, 512
    xd = torch.zeros((M, K), dtype=torch.bfloat16, device=dev)
    packed = torch.zeros(fb.fp8bs_packed_weight_bytes(N, K, F32), dtype=torch.uint8, device=dev)
    with pytest.raises(fb.Fp8bsError) as e:
        fb.fp8bs_gemm_fused(xd, packed, N, K, F32)
    assert e.value.status == -2
    with pytest.raises(fb.Fp8bsError) as e:
        fb.fp8bs_gemm_fused(xd[:4], packed[:1000], N, K, F32)
    assert e.value.status == -5


def test_binding_uses_native_library(dev):
    maps = open(f"/proc/{os.getpid()}/maps").read()
    assert "libfp8bs.so" in maps


# ---------------------------------------------------------------------------
# special 1x128 groups through every fused variant
# ---------------------------------------------------------------------------

def _special_rows(K: int) -> list:
    """fp32 rows (later rounded to bf16) of the groups the quant treats specially,
    whole rows first, then single special groups inside otherwise normal rows.
    Returns a list of (name, fp32 row, check_row): check_row is False for the
    row whose every scale is an fp32 subnormal, where the fp32 product
    xs * ws of the rescale ("[AMD] Small-M FP8 block-scale GEMM with fused
    activation quant for gfx950 (Qwen3.5)", "Modifications": the scales are
    applied in fp32) underflows while the oracle's fp64 does not; that row is
    covered by the whole-output criterion and the bit-exact codes."""
    normal = lambda s: synth.bf16_bits_to_f32(synth.x_bf16(1, K, seed=s)[0])
    rows = []
    z = np.zeros(K, np.float32)
    z[1::2] = -0.0
    rows.append(("zero row with -0", z, True))
    rows.append(("all-equal row", np.full(K, 3.0, np.float32), True))
    rows.append(("row x 1e-30", normal(11) * np.float32(1e-30), True))
    rows.append(("row x 1e30", normal(12) * np.float32(1e30), True))
    sub = np.full(K, np.float32(2.0 ** -130), np.float32)
    sub[5::7] = -np.float32(2.0 ** -133)
    rows.append(("bf16 subnormal row", sub, False))
    tie = np.tile(np.float32([448.0, 17.0, -19.0, 21.0, -0.0, 1.0, 3.0, -448.0]), K // 8)
    rows.append(("exact e4m3 ties at scale 1", tie, True))
    r = normal(13)
    r[128:256] = -0.0                           # one zero group
    r[256:384] = 3.0                            # one all-equal group
    rows.append(("normal row, zero and all-equal groups", r, True))
    r = normal(14)
    r[0] = 3.0e38                               # one huge value in group 0
    r[1:128] = 1.0
    r[384] = -3.0e38                            # and a negative one in group 3
    rows.append(("normal row, +-3e38 groups", r, True))
    r = normal(15)
    r[128:256] = np.float32(2.0 ** -130)        # one bf16-subnormal group
    r[129] = -np.float32(2.0 ** -133)
    r[256:384] = 448.0                          # one group at scale 1 with a tie
    r[257] = 17.0
    rows.append(("normal row, subnormal and tie groups", r, True))
    return rows


@pytest.mark.parametrize("kind", [F32, UE8])
@pytest.mark.parametrize("M", [3, 9, 17, 32, 33, 48])
def test_fused_special_groups(dev, oracle_mod, kind, M):
    # M = 3 and 9: the 16-token kernel, which quantises its own groups (one and
    # several rounds); 17 and 32: the 32-token kernel, the same at its smallest
    # and largest; 33 and 48: the quant kernel, then the GEMM on its codes with
    # the 64-token tile.  Every special row goes through each variant (in
    # chunks of M rows, the rest normal rows).  Quant bytes and scales
    # bit-exact; y within the tolerance as a whole and row by row.
    N, K = 5120, 4096
    specials = _special_rows(K)
    wq, ws = H.weight(oracle_mod, N, K, kind, 901)
    packed = fb.fp8bs_prepack_weight(to_dev(wq, dev), to_dev(ws, dev), kind)
    wsp = fb.new_workspace(N, K, dev)
    for start in range(0, len(specials), M):
        chunk = specials[start:start + M]
        v = synth.bf16_bits_to_f32(synth.x_bf16(M, K, seed=900 + M + start))
        names, check = ["normal"] * M, [True] * M
        for i, (name, row, ok) in enumerate(chunk):
            v[i], names[i], check[i] = row, name, ok
        x = synth.f32_to_bf16_bits(v)
        y_ref, xq_ref, xs_ref = oracle_mod.linear(x, wq, ws, kind, nthreads=H.threads())
        assert np.all(np.isfinite(H.bf16_to_f32(y_ref)))
        xq = torch.zeros((M, K), dtype=torch.uint8, device=dev)
        xs = torch.zeros((M, K // 128), dtype=torch.uint8 if kind == UE8 else torch.float32, device=dev)
        yd = fb.fp8bs_gemm_fused(x_dev(x, dev), packed, N, K, kind, workspace=wsp, xq_out=xq, xs_out=xs)
        assert fb.fp8bs_check_error(wsp) == 0
        got_q, got_s = xq.cpu().numpy(), xs.cpu().numpy()
        for i in range(M):
            assert np.array_equal(got_q[i], xq_ref[i]), f"codes of row {i} ({names[i]})"
            assert np.array_equal(got_s[i].view(np.uint8), xs_ref[i].view(np.uint8)), \
                f"scales of row {i} ({names[i]})"
        y = H.torch_u16_to_np(yd)
        H.check_y(y, y_ref, f"special groups M={M} kind={kind} chunk {start}")
        for i in range(M):
            if check[i]:
                H.check_y(y[i:i + 1], y_ref[i:i + 1], f"row {i} ({names[i]}) M={M} kind={kind}")
