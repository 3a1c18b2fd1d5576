"""fp8bs_gemm_fused_static (the fused GEMM with the library's fixed scratch)
against fp8bs_gemm_fused with a caller-supplied workspace.

Named to be collected last, so it also runs after every other GPU test has
used the library; it sets up its own inputs and passes alone as well."""

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


def packed_weight(N, K, kind, seed, dev):
    w = synth.w_f32_torch(N, K, seed=seed, device=dev)
    wq, ws = fb.fp8bs_quant_weight(w, kind)
    return fb.fp8bs_prepack_weight(wq, ws, kind)


def quant_outs(M, K, kind, dev):
    xq = torch.zeros((M, K), dtype=torch.uint8, device=dev)
    xs = torch.zeros((M, K // 128), dtype=torch.uint8 if kind == UE8 else torch.float32,
                     device=dev)
    return xq, xs


@pytest.mark.parametrize("M,N,K,kind,pdl", [
    (5, 5120, 4096, F32, False),      # one launch, 16-token tile
    (17, 4096, 2048, UE8, False),     # one launch, 32-token tile
    (32, 1536, 7168, UE8, True),      # one launch, 32-token tile, PDL
    (24, 16384, 8192, F32, False),    # one launch, the GEMM split over n-tile slices
    (40, 5120, 4096, F32, False),     # two launches, 64-token tile
    (64, 1536, 7168, UE8, True),      # two launches, 64-token tile, PDL
])
def test_static_scratch_matches_workspace_call_twice(dev, M, N, K, kind, pdl):
    x = synth.x_bf16_torch(M, K, seed=77 * M + K, device=dev)
    packed = packed_weight(N, K, kind, seed=N + K + kind, dev=dev)
    y_ref = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    xq_ref, xs_ref = quant_outs(M, K, kind, dev)
    wsp = fb.new_workspace(N, K, dev)
    fb.fp8bs_gemm_fused(x, packed, N, K, kind, y=y_ref, workspace=wsp, xq_out=xq_ref,
                        xs_out=xs_ref)
    assert fb.fp8bs_check_error(wsp) == 0

    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    ys = [torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    outs = [quant_outs(M, K, kind, dev) for _ in range(2)]
    torch.cuda.synchronize()
    for i in range(2):  # two calls in a row on one stream share the scratch
        fb.fp8bs_gemm_fused_static(x, packed, N, K, kind, y=ys[i], xq_out=outs[i][0],
                                   xs_out=outs[i][1], status_out=status, pdl=pdl)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = H.torch_u16_to_np(y_ref)
    for i in range(2):
        H.check_y(H.torch_u16_to_np(ys[i]), ref, f"static call {i} M={M} N={N} K={K}")
        assert torch.equal(outs[i][0], xq_ref)
        assert torch.equal(outs[i][1], xs_ref)


def test_static_call_allocates_no_device_memory(dev):
    M, N, K = 9, 2048, 4096
    x = synth.x_bf16_torch(M, K, seed=5, device=dev)
    packed = packed_weight(N, K, F32, seed=6, dev=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    fb.fp8bs_gemm_fused_static(x, packed, N, K, F32, y=y)  # set-up happens here at the latest
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    for _ in range(3):
        fb.fp8bs_gemm_fused_static(x, packed, N, K, F32, y=y)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0


def test_static_rejects_k_beyond_its_scratch(dev):
    N, K = 128, fb.FP8BS_STATIC_MAX_K + 128
    x = torch.zeros((1, K), dtype=torch.bfloat16, device=dev)
    packed = torch.zeros(fb.fp8bs_packed_weight_bytes(N, K, F32), dtype=torch.uint8, device=dev)
    y = torch.full((1, N), 7.0, dtype=torch.bfloat16, device=dev)
    with pytest.raises(fb.Fp8bsError) as e:
        fb.fp8bs_gemm_fused_static(x, packed, N, K, F32, y=y)
    assert e.value.status == -5  # FP8BS_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((y.float() == 7.0).all())  # nothing was enqueued
