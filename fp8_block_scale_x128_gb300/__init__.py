"""Python binding of libfp8bs (small-M W8A8 FP8 block-scale linear for GB300).

Argument marshalling only: every function here turns torch tensors into the
device pointers, sizes and the cudaStream_t of the C ABI declared in
``include/fp8bs.h`` and calls it; all arithmetic runs in the library's CUDA
kernels.  There is no fallback: if the compiled library is missing, or a call
returns an error status, an exception is raised.

The names match the C entry points.  Layout and rounding rules are documented
in the header; the method is the one of "[AMD] Small-M FP8 block-scale GEMM
with fused activation quant for gfx950 (Qwen3.5)", "Modifications", with the
power-of-two variant of "[Perf] [AMD] dsv4: optional e8m0 mxscale GEMM for
dense 128x128 fp8 linears (6/8)".
"""

from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

FP8BS_SCALE_F32 = 0
FP8BS_SCALE_UE8M0 = 1
FP8BS_MAX_M = 64
FP8BS_FLAG_PDL = 1
FP8BS_STATIC_MAX_K = 16384
FP8BS_STATIC_MAX_SMS = 160

STATUS = {
    0: "FP8BS_OK", -1: "FP8BS_ERR_ARG", -2: "FP8BS_ERR_SHAPE", -3: "FP8BS_ERR_ALIGN",
    -4: "FP8BS_ERR_SCALE_KIND", -5: "FP8BS_ERR_WORKSPACE", -6: "FP8BS_ERR_CUDA",
    -7: "FP8BS_ERR_TIMEOUT", -8: "FP8BS_ERR_DEVICE", -9: "FP8BS_ERR_RESIDENCY",
}
globals().update({name: code for code, name in STATUS.items()})

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfp8bs.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "fp8bs.h")

_lock = threading.Lock()
_lib = None


class Fp8bsError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({fp8bs_status_string(status)})")


def build(force: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a)."""
    from . import native_build as _b
    return _b.build(force=force)


def use_trace_library() -> str:
    """Build the traced variant of the library (the fused kernel stamps its
    phase boundaries, read back with fp8bs_trace_read) and make lib() load it.
    Must be called before the first lib() call of the process."""
    global LIB_PATH
    from . import native_build as _b
    with _lock:
        if _lib is not None:
            raise RuntimeError("the library is already loaded")
        LIB_PATH = _b.build(trace=True)
    return LIB_PATH


def declared_functions() -> list[str]:
    """Names of the functions include/fp8bs.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8bs_[a-z0-9_]+)\s*\(", text)))


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libfp8bs.so is not built ({LIB_PATH}); call "
                               "fp8_block_scale_x128_gb300.build() first")
        L = ctypes.CDLL(LIB_PATH)
        c = ctypes
        vp, i64, sz, ci = c.c_void_p, c.c_int64, c.c_size_t, c.c_int
        sig = {
            "fp8bs_status_string": ([ci], c.c_char_p),
            "fp8bs_version": ([], ci),
            "fp8bs_encode_e4m3": ([vp, i64, vp, vp], ci),
            "fp8bs_quant": ([vp, i64, i64, i64, ci, vp, vp, vp], ci),
            "fp8bs_rmsnorm_quant": ([vp, i64, i64, i64, vp, ctypes.c_float, ci, vp, vp, vp, i64, vp], ci),
            "fp8bs_moe_workspace_bytes": ([i64, i64, i64, i64], ctypes.c_size_t),
            "fp8bs_moe_w8a16": ([vp, i64, i64, vp, vp, i64, vp, vp, vp, vp, i64, i64, vp, vp,
                                 ctypes.c_size_t, vp], ci),
            "fp8bs_quant_weight": ([vp, i64, i64, i64, ci, vp, vp, vp], ci),
            "fp8bs_packed_weight_bytes": ([i64, i64, ci], sz),
            "fp8bs_prepack_weight": ([vp, i64, vp, i64, i64, ci, vp, sz, vp], ci),
            "fp8bs_workspace_bytes": ([i64, i64, ci], sz),
            "fp8bs_workspace_init": ([vp, sz, vp], ci),
            "fp8bs_gemm_fused": ([vp, i64, i64, vp, sz, i64, i64, ci, vp, i64, vp, sz, vp, vp,
                                  c.c_uint, vp], ci),
            "fp8bs_check_error": ([vp, vp], ci),
            "fp8bs_gemm_prequant": ([vp, i64, i64, vp, vp, sz, i64, i64, ci, vp, i64, vp, sz, c.c_uint, vp],
                                    ci),
            "fp8bs_gemm_fused_static": ([vp, i64, i64, vp, sz, i64, i64, ci, vp, i64, vp, vp, vp,
                                         c.c_uint, vp], ci),
            "fp8bs_trace_read": ([vp, sz], ci),
            "fp8bs_debug_config": ([ctypes.c_longlong, ci], ci),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
        return L


def fp8bs_status_string(status: int) -> str:
    try:
        return lib().fp8bs_status_string(int(status)).decode()
    except RuntimeError:
        return STATUS.get(status, "unknown")


def fp8bs_version() -> int:
    return int(lib().fp8bs_version())


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise Fp8bsError(rc, where)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _scale_dtype(kind: int):
    return torch.uint8 if kind == FP8BS_SCALE_UE8M0 else torch.float32


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("fp8bs tensors must live on a CUDA device")


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def fp8bs_encode_e4m3(v: torch.Tensor, codes: torch.Tensor | None = None, stream=None):
    """fp32 v [n] (n % 4 == 0) -> uint8 e4m3fn codes [n] (RNE, satfinite)."""
    _require_cuda(v)
    assert v.dtype == torch.float32 and v.is_contiguous()
    if codes is None:
        codes = torch.empty(v.numel(), dtype=torch.uint8, device=v.device)
    rc = lib().fp8bs_encode_e4m3(_ptr(v), v.numel(), _ptr(codes), _stream(stream))
    _check(rc, "fp8bs_encode_e4m3")
    return codes


def fp8bs_quant(x: torch.Tensor, scale_kind: int = FP8BS_SCALE_F32, xq: torch.Tensor | None = None,
                xs: torch.Tensor | None = None, stream=None):
    """bf16 x [M, K] (row stride x.stride(0)) -> (xq uint8 [M, K], xs [M, K/128])."""
    _require_cuda(x)
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if xs is None:
        xs = torch.empty((M, K // 128), dtype=_scale_dtype(scale_kind), device=x.device)
    rc = lib().fp8bs_quant(_ptr(x), M, K, x.stride(0), int(scale_kind), _ptr(xq), _ptr(xs),
                           _stream(stream))
    _check(rc, "fp8bs_quant")
    return xq, xs


def fp8bs_rmsnorm_quant(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6,
                        scale_kind: int = FP8BS_SCALE_F32, xq: torch.Tensor | None = None,
                        xs: torch.Tensor | None = None, y: torch.Tensor | None = None,
                        want_y: bool = False, stream=None):
    """RMSNorm of bf16 x [M, K] with bf16 weight gamma [K], then the 1x128 quant.

    Returns (xq uint8 [M, K], xs [M, K/128], y bf16 [M, K] or None); y is
    written when given or when want_y."""
    _require_cuda(x, gamma)
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    assert gamma.dtype == torch.bfloat16 and gamma.dim() == 1 and gamma.is_contiguous()
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if xs is None:
        xs = torch.empty((M, K // 128), dtype=_scale_dtype(scale_kind), device=x.device)
    if y is None and want_y:
        y = torch.empty((M, K), dtype=torch.bfloat16, device=x.device)
    if y is not None:
        assert y.dtype == torch.bfloat16 and y.dim() == 2 and y.stride(1) == 1
    rc = lib().fp8bs_rmsnorm_quant(_ptr(x), M, K, x.stride(0), _ptr(gamma), float(eps),
                                   int(scale_kind), _ptr(xq), _ptr(xs),
                                   _ptr(y) if y is not None else None,
                                   y.stride(0) if y is not None else 0, _stream(stream))
    _check(rc, "fp8bs_rmsnorm_quant")
    return xq, xs, y


def fp8bs_moe_workspace_bytes(M: int, S: int, H: int, I: int) -> int:
    return int(lib().fp8bs_moe_workspace_bytes(int(M), int(S), int(H), int(I)))


def new_moe_workspace(M: int, S: int, H: int, I: int, device=None) -> torch.Tensor:
    """Allocate (with torch) a zeroed MoE workspace for up to M tokens x S slots."""
    device = device or torch.device("cuda", torch.cuda.current_device())
    n = fp8bs_moe_workspace_bytes(M, S, H, I)
    if n == 0:
        raise Fp8bsError(FP8BS_ERR_SHAPE, "fp8bs_moe_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def fp8bs_moe_w8a16(x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor,
                    w13: torch.Tensor, s13: torch.Tensor, w2: torch.Tensor, s2: torch.Tensor,
                    y: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """One small-M MoE layer: bf16 x [M, H]; int32 topk_ids and fp32 topk_w
    [M, S]; e4m3 (uint8) w13 [E, 2I, H] with fp32 s13 [E, 2I/128, H/128]; w2
    [E, H, I] with s2 [E, H/128, I/128].  Returns bf16 y [M, H]."""
    _require_cuda(x, topk_ids, topk_w, w13, s13, w2, s2, y, workspace)
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()
    assert topk_ids.dtype == torch.int32 and topk_w.dtype == torch.float32
    assert topk_ids.is_contiguous() and topk_w.is_contiguous() and topk_ids.shape == topk_w.shape
    for t in (w13, s13, w2, s2):
        assert t.is_contiguous()
    assert w13.dtype == torch.uint8 and w2.dtype == torch.uint8
    assert s13.dtype == torch.float32 and s2.dtype == torch.float32
    M, H = x.shape
    S = topk_ids.shape[1]
    E, I2, _ = w13.shape
    I = I2 // 2
    if y is None:
        y = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = new_moe_workspace(M, S, H, I, x.device)
    rc = lib().fp8bs_moe_w8a16(_ptr(x), M, H, _ptr(topk_ids), _ptr(topk_w), S, _ptr(w13), _ptr(s13),
                               _ptr(w2), _ptr(s2), E, I, _ptr(y), _ptr(workspace),
                               workspace.numel(), _stream(stream))
    _check(rc, "fp8bs_moe_w8a16")
    return y


def fp8bs_quant_weight(w: torch.Tensor, scale_kind: int = FP8BS_SCALE_F32, stream=None):
    """fp32 w [N, K] -> (wq uint8 [N, K], ws [N/128, K/128]) in 128x128 blocks."""
    _require_cuda(w)
    assert w.dtype == torch.float32 and w.dim() == 2 and w.stride(1) == 1
    N, K = w.shape
    wq = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    ws = torch.empty((N // 128, K // 128), dtype=_scale_dtype(scale_kind), device=w.device)
    rc = lib().fp8bs_quant_weight(_ptr(w), N, K, w.stride(0), int(scale_kind), _ptr(wq), _ptr(ws),
                                  _stream(stream))
    _check(rc, "fp8bs_quant_weight")
    return wq, ws


def fp8bs_packed_weight_bytes(N: int, K: int, scale_kind: int = FP8BS_SCALE_F32) -> int:
    return int(lib().fp8bs_packed_weight_bytes(int(N), int(K), int(scale_kind)))


def fp8bs_prepack_weight(wq: torch.Tensor, ws: torch.Tensor, scale_kind: int = FP8BS_SCALE_F32,
                         packed: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """wq uint8 [N, K] + ws [N/128, K/128] -> packed uint8 buffer (GB300 tile layout)."""
    _require_cuda(wq, ws)
    assert wq.dtype == torch.uint8 and wq.dim() == 2 and wq.stride(1) == 1
    assert ws.is_contiguous() and ws.dtype == _scale_dtype(scale_kind)
    N, K = wq.shape
    nbytes = fp8bs_packed_weight_bytes(N, K, scale_kind)
    if nbytes == 0:
        raise Fp8bsError(-2, "fp8bs_packed_weight_bytes")
    if packed is None:
        packed = torch.empty(nbytes, dtype=torch.uint8, device=wq.device)
    rc = lib().fp8bs_prepack_weight(_ptr(wq), wq.stride(0), _ptr(ws), N, K, int(scale_kind),
                                    _ptr(packed), packed.numel(), _stream(stream))
    _check(rc, "fp8bs_prepack_weight")
    return packed


def fp8bs_workspace_bytes(N: int, K: int, sm_count: int = 0) -> int:
    return int(lib().fp8bs_workspace_bytes(int(N), int(K), int(sm_count)))


def fp8bs_workspace_init(workspace: torch.Tensor, stream=None) -> None:
    _require_cuda(workspace)
    rc = lib().fp8bs_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream))
    _check(rc, "fp8bs_workspace_init")


def new_workspace(N: int, K: int, device=None, stream=None) -> torch.Tensor:
    """Allocate (with torch) and initialise a workspace for an N x K weight."""
    device = device or torch.device("cuda", torch.cuda.current_device())
    n = fp8bs_workspace_bytes(N, K)
    if n == 0:
        raise Fp8bsError(-2, "fp8bs_workspace_bytes")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    fp8bs_workspace_init(ws, stream)
    return ws


def fp8bs_gemm_fused(x: torch.Tensor, packed: torch.Tensor, N: int, K: int,
                     scale_kind: int = FP8BS_SCALE_F32, y: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None, xq_out: torch.Tensor | None = None,
                     xs_out: torch.Tensor | None = None, pdl: bool = False,
                     stream=None) -> torch.Tensor:
    """Y = bf16(quant(x) . W^T) for bf16 x [M <= 64, K] and a packed weight.

    pdl=True launches with programmatic dependent launch (FP8BS_FLAG_PDL); use
    it only when the work just before this call on the stream does not write
    `packed`.
    """
    _require_cuda(x, packed, y, workspace, xq_out, xs_out)
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    M = x.shape[0]
    assert x.shape[1] == K
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = new_workspace(N, K, x.device, stream)
    rc = lib().fp8bs_gemm_fused(
        _ptr(x), M, x.stride(0), _ptr(packed), packed.numel(), N, K, int(scale_kind), _ptr(y),
        y.stride(0), _ptr(workspace), workspace.numel(), _ptr(xq_out), _ptr(xs_out),
        FP8BS_FLAG_PDL if pdl else 0, _stream(stream))
    _check(rc, "fp8bs_gemm_fused")
    return y


def fp8bs_gemm_prequant(xq: torch.Tensor, xs: torch.Tensor, packed: torch.Tensor, N: int, K: int,
                        scale_kind: int = FP8BS_SCALE_F32, y: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None, pdl: bool = False,
                        stream=None) -> torch.Tensor:
    """Y = bf16(xq . W^T) with the block scales, for pre-quantised activations
    (uint8 e4m3 codes [M, K], scales [M, K/128] fp32 or uint8 e8m0): the
    second launch of the two-launch path."""
    _require_cuda(xq, xs, packed, y, workspace)
    assert xq.dtype == torch.uint8 and xq.dim() == 2 and xq.stride(1) == 1 and xq.shape[1] == K
    assert xs.is_contiguous() and xs.shape == (xq.shape[0], K // 128)
    M = xq.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device)
    if workspace is None:
        workspace = new_workspace(N, K, xq.device, stream)
    rc = lib().fp8bs_gemm_prequant(
        _ptr(xq), M, xq.stride(0), _ptr(xs), _ptr(packed), packed.numel(), N, K, int(scale_kind),
        _ptr(y), y.stride(0), _ptr(workspace), workspace.numel(), FP8BS_FLAG_PDL if pdl else 0,
        _stream(stream))
    _check(rc, "fp8bs_gemm_prequant")
    return y


def fp8bs_gemm_fused_static(x: torch.Tensor, packed: torch.Tensor, N: int, K: int,
                            scale_kind: int = FP8BS_SCALE_F32, y: torch.Tensor | None = None,
                            xq_out: torch.Tensor | None = None, xs_out: torch.Tensor | None = None,
                            status_out: torch.Tensor | None = None, pdl: bool = False,
                            stream=None) -> torch.Tensor:
    """fp8bs_gemm_fused with the library's fixed per-device scratch instead of a
    workspace (K <= FP8BS_STATIC_MAX_K).  The C call allocates nothing; pass
    `y` to keep this wrapper from allocating it.  `status_out` (int32 [1] on
    the device, optional) receives the sticky device status after the kernel.
    """
    _require_cuda(x, packed, y, xq_out, xs_out, status_out)
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    M = x.shape[0]
    assert x.shape[1] == K
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    rc = lib().fp8bs_gemm_fused_static(
        _ptr(x), M, x.stride(0), _ptr(packed), packed.numel(), N, K, int(scale_kind), _ptr(y),
        y.stride(0), _ptr(xq_out), _ptr(xs_out), _ptr(status_out),
        FP8BS_FLAG_PDL if pdl else 0, _stream(stream))
    _check(rc, "fp8bs_gemm_fused_static")
    return y


FP8BS_TRACE_CALLS, FP8BS_TRACE_CTAS, FP8BS_TRACE_POINTS = 256, 160, 64


def fp8bs_trace_read():
    """The traced library's timeline as a numpy uint64 array
    [calls][CTAs][points][2] (globaltimer ns, clock64); raises in a plain build."""
    import numpy as np
    buf = np.zeros((FP8BS_TRACE_CALLS, FP8BS_TRACE_CTAS, FP8BS_TRACE_POINTS, 2), dtype=np.uint64)
    rc = lib().fp8bs_trace_read(ctypes.c_void_p(buf.ctypes.data), buf.nbytes)
    _check(rc, "fp8bs_trace_read")
    return buf


def fp8bs_debug_config(timeout_cycles: int = 0, sm_count_override: int = 0) -> None:
    """Diagnostic overrides of the fused GEMM's launches (tests only): the
    bounded waits' limit in SM cycles and the multiprocessor count grids and
    workspaces are sized for; 0 restores each default."""
    _check(lib().fp8bs_debug_config(int(timeout_cycles), int(sm_count_override)), "fp8bs_debug_config")


def fp8bs_check_error(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(lib().fp8bs_check_error(_ptr(workspace), _stream(stream)))
