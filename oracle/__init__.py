"""CPU oracle for the small-M W8A8 FP8 block-scale linear (test infrastructure).

Only the tests, the smoke check and the CPU-baseline leg of the benchmark may
import this package.  It is a thin ctypes/numpy wrapper around ``oracle.c``,
a plain C restatement of the method written from the format definitions and
from these pages:

* "[AMD] Small-M FP8 block-scale GEMM with fused activation quant for gfx950
  (Qwen3.5)", section "Modifications" -- 1x128 activation groups, row amax,
  [N/128, K/128] fp32 weight scales, x_scale * w_scale in fp32 per K block.
* "[AMD] gfx950 small-batch MoE: expert-count gate for the small sort and FP8
  block-scale small-M kernel", section "Modifications" -- float8_e4m3fn and
  the 128x128 block scale applied to each partial sum (also the w13 / w2 of
  its small-M MoE layer).
* "[Perf] [AMD] dsv4: optional e8m0 mxscale GEMM for dense 128x128 fp8
  linears (6/8)", "Motivation" / "Modifications" -- power-of-two (e8m0)
  weight scales and ue8m0 activation scales, emitted by the fused
  input_norm / q_norm (RMSNorm) producers.

It shares no code with the CUDA library and never imports it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

SCALE_F32 = 0
SCALE_UE8M0 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_CFLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-pthread", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so with gcc (no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        c = ctypes
        vp, i64 = c.c_void_p, c.c_int64
        lib.oracle_bf16_to_f32.argtypes = [c.c_uint16]
        lib.oracle_bf16_to_f32.restype = c.c_float
        lib.oracle_f64_to_bf16.argtypes = [c.c_double]
        lib.oracle_f64_to_bf16.restype = c.c_uint16
        lib.oracle_e4m3_decode.argtypes = [c.c_uint8]
        lib.oracle_e4m3_decode.restype = c.c_double
        lib.oracle_e4m3_encode.argtypes = [c.c_float]
        lib.oracle_e4m3_encode.restype = c.c_uint8
        lib.oracle_e4m3_encode_bits.argtypes = [c.c_uint32, c.c_uint64, vp]
        lib.oracle_e4m3_encode_bits.restype = None
        lib.oracle_e8m0_decode.argtypes = [c.c_uint8]
        lib.oracle_e8m0_decode.restype = c.c_double
        lib.oracle_e8m0_ceil.argtypes = [c.c_float]
        lib.oracle_e8m0_ceil.restype = c.c_uint8
        lib.oracle_quant_1x128.argtypes = [vp, i64, i64, i64, c.c_int, vp, vp]
        lib.oracle_quant_1x128.restype = c.c_int
        lib.oracle_quant_weight_128x128.argtypes = [vp, i64, i64, c.c_int, vp, vp]
        lib.oracle_quant_weight_128x128.restype = c.c_int
        lib.oracle_gemm.argtypes = [vp, vp, vp, vp, i64, i64, i64, c.c_int, vp, vp, c.c_int]
        lib.oracle_gemm.restype = c.c_int
        lib.oracle_linear.argtypes = [vp, i64, i64, i64, vp, vp, i64, c.c_int, vp, vp, vp,
                                      c.c_int]
        lib.oracle_linear.restype = c.c_int
        lib.oracle_rmsnorm.argtypes = [vp, i64, i64, i64, vp, c.c_double, vp, vp]
        lib.oracle_rmsnorm.restype = c.c_int
        lib.oracle_rmsnorm_quant.argtypes = [vp, i64, i64, i64, vp, c.c_double, c.c_int, vp, vp,
                                             vp]
        lib.oracle_rmsnorm_quant.restype = c.c_int
        lib.oracle_moe_w8a16.argtypes = [vp, i64, i64, vp, vp, i64, vp, vp, vp, vp, i64, i64, vp,
                                         vp]
        lib.oracle_moe_w8a16.restype = c.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _scale_dtype(kind: int):
    return np.uint8 if kind == SCALE_UE8M0 else np.float32


# --------------------------------------------------------------------------
# scalar codecs
# --------------------------------------------------------------------------

def bf16_to_f32(h: int) -> float:
    return float(_load().oracle_bf16_to_f32(int(h)))


def f64_to_bf16(v: float) -> int:
    """fp64 -> bf16 bits, round to nearest even, directly from fp64."""
    return int(_load().oracle_f64_to_bf16(float(v)))


def e4m3_decode(code: int) -> float:
    return float(_load().oracle_e4m3_decode(int(code)))


def e4m3_encode(v: float) -> int:
    """Nearest e4m3fn code of the fp32 value v (RNE, saturating to +-448)."""
    return int(_load().oracle_e4m3_encode(float(np.float32(v))))


def e4m3_encode_bits(first: int, count: int, out: np.ndarray | None = None) -> np.ndarray:
    """Codes for every fp32 bit pattern first .. first+count-1."""
    if out is None:
        out = np.empty(count, dtype=np.uint8)
    assert out.dtype == np.uint8 and out.size >= count and out.flags.c_contiguous
    _load().oracle_e4m3_encode_bits(int(first), int(count), _ptr(out))
    return out


def e8m0_decode(b: int) -> float:
    return float(_load().oracle_e8m0_decode(int(b)))


def e8m0_ceil(s: float) -> int:
    """e8m0 byte of the smallest power of two >= the fp32 value s."""
    return int(_load().oracle_e8m0_ceil(float(np.float32(s))))


def e4m3_table() -> np.ndarray:
    """fp64 values of all 256 codes (NaN for 0x7F and 0xFF)."""
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def f64_to_bf16_array(v: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(v, dtype=np.float64).ravel()
    return np.array([lib.oracle_f64_to_bf16(float(t)) for t in flat],
                    dtype=np.uint16).reshape(np.shape(v))


# --------------------------------------------------------------------------
# array operations
# --------------------------------------------------------------------------

def quant_1x128(x_bf16: np.ndarray, kind: int = SCALE_F32):
    """x_bf16: uint16 [M, K] (bf16 bits).  Returns (xq uint8 [M,K], xs [M,K/128])."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x.shape
    xq = np.empty((M, K), dtype=np.uint8)
    xs = np.empty((M, K // 128), dtype=_scale_dtype(kind))
    rc = _load().oracle_quant_1x128(_ptr(x), M, K, K, int(kind), _ptr(xq), _ptr(xs))
    if rc:
        raise ValueError(f"oracle_quant_1x128 rejected shape {x.shape}")
    return xq, xs


def quant_weight_128x128(w_f32: np.ndarray, kind: int = SCALE_F32):
    """w_f32: float32 [N, K].  Returns (wq uint8 [N,K], ws [N/128, K/128])."""
    w = np.ascontiguousarray(w_f32, dtype=np.float32)
    N, K = w.shape
    wq = np.empty((N, K), dtype=np.uint8)
    ws = np.empty((N // 128, K // 128), dtype=_scale_dtype(kind))
    rc = _load().oracle_quant_weight_128x128(_ptr(w), N, K, int(kind), _ptr(wq), _ptr(ws))
    if rc:
        raise ValueError(f"oracle_quant_weight_128x128 rejected shape {w.shape}")
    return wq, ws


def gemm(xq, xs, wq, ws, kind: int = SCALE_F32, nthreads: int = 1, want_f64: bool = False):
    """Block-scale GEMM.  Returns bf16 bits uint16 [M, N] (and fp64 [M, N])."""
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    xs = np.ascontiguousarray(xs, dtype=_scale_dtype(kind))
    ws = np.ascontiguousarray(ws, dtype=_scale_dtype(kind))
    M, K = xq.shape
    N = wq.shape[0]
    assert wq.shape[1] == K and xs.shape == (M, K // 128) and ws.shape == (N // 128, K // 128)
    y = np.empty((M, N), dtype=np.uint16)
    y64 = np.empty((M, N), dtype=np.float64) if want_f64 else None
    rc = _load().oracle_gemm(_ptr(xq), _ptr(xs), _ptr(wq), _ptr(ws), M, N, K, int(kind), _ptr(y),
                             _ptr(y64) if want_f64 else None, int(nthreads))
    if rc:
        raise ValueError("oracle_gemm rejected its arguments")
    return (y, y64) if want_f64 else y


def linear(x_bf16, wq, ws, kind: int = SCALE_F32, nthreads: int = 1):
    """Quantise x in 1x128 groups, then the block-scale GEMM.  Returns (y, xq, xs)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x.shape
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    ws = np.ascontiguousarray(ws, dtype=_scale_dtype(kind))
    N = wq.shape[0]
    xq = np.empty((M, K), dtype=np.uint8)
    xs = np.empty((M, K // 128), dtype=_scale_dtype(kind))
    y = np.empty((M, N), dtype=np.uint16)
    rc = _load().oracle_linear(_ptr(x), M, K, K, _ptr(wq), _ptr(ws), N, int(kind), _ptr(xq),
                               _ptr(xs), _ptr(y), int(nthreads))
    if rc:
        raise ValueError("oracle_linear rejected its arguments")
    return y, xq, xs


def rmsnorm(x_bf16: np.ndarray, gamma_bf16: np.ndarray, eps: float):
    """RMSNorm of each row (x * gamma / sqrt(mean x^2 + eps)) in fp64.

    Returns (y fp64 [M, K], y rounded to bf16 bits uint16 [M, K])."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    g = np.ascontiguousarray(gamma_bf16, dtype=np.uint16)
    M, K = x.shape
    assert g.shape == (K,)
    y64 = np.empty((M, K), dtype=np.float64)
    y = np.empty((M, K), dtype=np.uint16)
    rc = _load().oracle_rmsnorm(_ptr(x), M, K, K, _ptr(g), float(eps), _ptr(y64), _ptr(y))
    if rc:
        raise ValueError("oracle_rmsnorm rejected its arguments")
    return y64, y


def rmsnorm_quant(x_bf16: np.ndarray, gamma_bf16: np.ndarray, eps: float, kind: int = SCALE_F32):
    """The producer: RMSNorm rounded to bf16, then the 1x128 quant.

    Returns (y bf16 bits [M, K], xq uint8 [M, K], xs [M, K/128])."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    g = np.ascontiguousarray(gamma_bf16, dtype=np.uint16)
    M, K = x.shape
    y = np.empty((M, K), dtype=np.uint16)
    xq = np.empty((M, K), dtype=np.uint8)
    xs = np.empty((M, K // 128), dtype=_scale_dtype(kind))
    rc = _load().oracle_rmsnorm_quant(_ptr(x), M, K, K, _ptr(g), float(eps), int(kind), _ptr(y),
                                      _ptr(xq), _ptr(xs))
    if rc:
        raise ValueError("oracle_rmsnorm_quant rejected its arguments")
    return y, xq, xs


def moe_w8a16(x_bf16, ids, topk_w, w13, s13, w2, s2, want_f64: bool = False):
    """Small-M FP8 block-scale MoE layer (bf16 activations, e4m3 weights with
    128x128 fp32 block scales).  x [M, H] bf16 bits; ids int32 [M, S]; topk_w
    fp32 [M, S]; w13 uint8 [E, 2I, H]; s13 fp32 [E, 2I/128, H/128]; w2 uint8
    [E, H, I]; s2 fp32 [E, H/128, I/128].  Returns y bf16 bits [M, H] (and the
    fp64 values before rounding)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    tw = np.ascontiguousarray(topk_w, dtype=np.float32)
    w13 = np.ascontiguousarray(w13, dtype=np.uint8)
    w2 = np.ascontiguousarray(w2, dtype=np.uint8)
    s13 = np.ascontiguousarray(s13, dtype=np.float32)
    s2 = np.ascontiguousarray(s2, dtype=np.float32)
    M, H = x.shape
    S = ids.shape[1]
    E, I2, _ = w13.shape
    I = I2 // 2
    assert ids.shape == (M, S) and tw.shape == (M, S) and w13.shape == (E, 2 * I, H)
    assert w2.shape == (E, H, I) and s13.shape == (E, 2 * I // 128, H // 128)
    assert s2.shape == (E, H // 128, I // 128)
    y = np.empty((M, H), dtype=np.uint16)
    y64 = np.empty((M, H), dtype=np.float64) if want_f64 else None
    rc = _load().oracle_moe_w8a16(_ptr(x), M, H, _ptr(ids), _ptr(tw), S, _ptr(w13), _ptr(s13),
                                  _ptr(w2), _ptr(s2), E, I, _ptr(y),
                                  _ptr(y64) if want_f64 else None)
    if rc:
        raise ValueError("oracle_moe_w8a16 rejected its arguments")
    return (y, y64) if want_f64 else y


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
