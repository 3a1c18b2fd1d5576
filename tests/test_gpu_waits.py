"""The fused GEMM's failure paths, driven without a GPU fault.

* A bounded wait that cannot complete: one CTA's epoch word is set apart from
  its peers', so the split-K partials it exchanges with them never carry the
  epoch the other side polls for.  With a short wait limit (the diagnostic
  setting) every such wait expires; the kernel records FP8BS_ERR_TIMEOUT,
  drains its own copies and MMAs and returns.  The test then checks that the
  device still answers and that a re-initialised workspace gives the oracle's
  result again.
* A grid that cannot be resident at once: with the library sized for four
  times the device's multiprocessors, the call is refused on the host
  (FP8BS_ERR_RESIDENCY) and nothing is launched.
* The epoch counter's wrap: epoch words seeded just below 2^32 step through
  0xFFFFFFFF and the wrap (which skips 0, the tag of a never-written word)
  with results bit-identical to the first call."""

import numpy as np
import pytest
import torch

import fp8_block_scale_x128_gb300 as fb
from tests import helpers as H
from tests.test_gpu_parity import _setup

pytestmark = pytest.mark.gpu

F32 = fb.FP8BS_SCALE_F32
GEN_OFFSET = 256      # workspace bytes: the device error word, then the epoch words
GEN_WORDS = 1024


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fb.build()
    fb.lib()
    return torch.device("cuda", 0)


@pytest.fixture(autouse=True)
def _restore_defaults():
    yield
    fb.fp8bs_debug_config(0, 0)


def _gen_words(wsp: torch.Tensor) -> torch.Tensor:
    return wsp[GEN_OFFSET:GEN_OFFSET + 4 * GEN_WORDS].view(torch.int32)


def test_bounded_wait_expiry_reports_timeout(dev, oracle_mod):
    M, N, K = 4, 5120, 4096
    x, wq, ws, xd, packed = _setup(oracle_mod, dev, M, N, K, F32, 71)
    y_ref, _, _ = oracle_mod.linear(x, wq, ws, F32, nthreads=H.threads())
    fb.fp8bs_debug_config(timeout_cycles=400_000)  # ~0.2 ms: far above a normal call's waits
    wsp = fb.new_workspace(N, K, dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    fb.fp8bs_gemm_fused(xd, packed, N, K, F32, y=y, workspace=wsp)
    assert fb.fp8bs_check_error(wsp) == 0
    y_good = y.clone()
    H.check_y(H.torch_u16_to_np(y_good), y_ref, "before the expiry")

    # CTA 0 takes another epoch than its peers: the partials of the n-tiles it
    # shares are never seen as current, on either side
    gen = _gen_words(wsp)
    gen[0] = gen[1] + 0x100
    torch.cuda.synchronize()
    fb.fp8bs_gemm_fused(xd, packed, N, K, F32, y=y, workspace=wsp)
    assert fb.fp8bs_check_error(wsp) == fb.FP8BS_ERR_TIMEOUT

    # the device still answers, and a fresh workspace gives the oracle's result
    assert float(torch.ones(8, device=dev).sum()) == 8.0
    fb.fp8bs_debug_config(0, 0)
    fb.fp8bs_workspace_init(wsp)
    y.fill_(float("nan"))
    fb.fp8bs_gemm_fused(xd, packed, N, K, F32, y=y, workspace=wsp)
    assert fb.fp8bs_check_error(wsp) == 0
    assert torch.equal(y.view(torch.int16), y_good.view(torch.int16))


def test_launch_refused_when_grid_cannot_be_resident(dev, oracle_mod):
    M, N, K = 4, 5120, 4096
    _x, _wq, _ws, xd, packed = _setup(oracle_mod, dev, M, N, K, F32, 73)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    fb.fp8bs_debug_config(0, 4 * sms)  # grids of up to 4 CTAs per multiprocessor
    wsp = fb.new_workspace(N, K, dev)
    y = torch.full((M, N), 7.0, dtype=torch.bfloat16, device=dev)
    with pytest.raises(fb.Fp8bsError) as err:
        fb.fp8bs_gemm_fused(xd, packed, N, K, F32, y=y, workspace=wsp)
    assert err.value.status == fb.FP8BS_ERR_RESIDENCY
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())           # nothing was launched
    assert fb.fp8bs_check_error(wsp) == 0


@pytest.mark.parametrize("M", [3, 17])
def test_epoch_wrap_keeps_results(dev, oracle_mod, M):
    N, K = 5120, 4096
    x, wq, ws, xd, packed = _setup(oracle_mod, dev, M, N, K, F32, 79 + M)
    y_ref, _, _ = oracle_mod.linear(x, wq, ws, F32, nthreads=H.threads())
    wsp = fb.new_workspace(N, K, dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    fb.fp8bs_gemm_fused(xd, packed, N, K, F32, y=y, workspace=wsp)
    assert fb.fp8bs_check_error(wsp) == 0
    first = y.clone()
    H.check_y(H.torch_u16_to_np(first), y_ref, f"M={M} before the wrap")
    gen = _gen_words(wsp)
    gen.fill_(-2)  # 0xFFFFFFFE: the next epochs are 0xFFFFFFFF, then 1 (0 skipped), then 2
    torch.cuda.synchronize()
    for step in range(4):
        y.fill_(float("nan"))
        fb.fp8bs_gemm_fused(xd, packed, N, K, F32, y=y, workspace=wsp)
        assert fb.fp8bs_check_error(wsp) == 0, step
        assert torch.equal(y.view(torch.int16), first.view(torch.int16)), step
    words = _gen_words(wsp).cpu().numpy().view(np.uint32)
    assert int(words.max()) == 3  # 0xFFFFFFFF, 1, 2, 3: the counter went round
