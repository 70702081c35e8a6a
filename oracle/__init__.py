"""CPU oracle for the NVFP4 weight-only LoRA linear path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and the
two share no code: the oracle is plain C (``qerl_oracle.c``) compiled with gcc,
wrapped here with ctypes and numpy.

bf16 tensors cross this boundary as ``numpy.uint16`` bit patterns; every
floating-point result comes back as fp64 except the FP32 tensor scale, whose
value (and the quantizer's decisions) the format fixes in single precision.

Parity unpinned (the pages cannot decide these, so both sides apply the same
reading): block-scale rounding mode (round up is the default), the tensor-scale
formula amax/(6*448), nibble order, additive noise on the norm scale, eps, the
number of noise stages and the per-step redraw of the noise.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qerl_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_qerl.so")
_lock = threading.Lock()
_lib = None

ORC_OK, ORC_ERR_SHAPE, ORC_ERR_NONFINITE = 0, 2, 4

_P = np.ctypeslib.ndpointer
_u8 = _P(dtype=np.uint8, flags="C_CONTIGUOUS")
_u16 = _P(dtype=np.uint16, flags="C_CONTIGUOUS")
_u64 = _P(dtype=np.uint64, flags="C_CONTIGUOUS")
_i64 = _P(dtype=np.int64, flags="C_CONTIGUOUS")
_f32 = _P(dtype=np.float32, flags="C_CONTIGUOUS")
_f64 = _P(dtype=np.float64, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE single semantics: no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-fopenmp", "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            i64, u8, u32, u64, f32, f64, i32 = (C.c_int64, C.c_uint8, C.c_uint32, C.c_uint64,
                                                C.c_float, C.c_double, C.c_int)
            L.orc_bf16_value.argtypes = [C.c_uint16]; L.orc_bf16_value.restype = f64
            L.orc_e4m3_value.argtypes = [u8]; L.orc_e4m3_value.restype = f64
            L.orc_e2m1_value.argtypes = [u8]; L.orc_e2m1_value.restype = f64
            L.orc_e4m3_round_up.argtypes = [f32]; L.orc_e4m3_round_up.restype = u8
            L.orc_e4m3_round_rne.argtypes = [f32]; L.orc_e4m3_round_rne.restype = u8
            L.orc_e2m1_round.argtypes = [f32]; L.orc_e2m1_round.restype = u8
            L.orc_nvfp4_quantize.argtypes = [_u16, i64, i64, i64, _u8, _u8, _f32, i32]
            L.orc_nvfp4_quantize.restype = i32
            L.orc_nvfp4_dequantize.argtypes = [_u8, _u8, f32, i64, i64, _f64]
            L.orc_nvfp4_dequantize.restype = None
            L.orc_lora_linear_fwd.argtypes = [_u16, i64, i64, i64, _u8, _u8, f32, _u16, _u16,
                                              i32, f64, _i64, i64, _f64, C.c_void_p]
            L.orc_lora_linear_fwd.restype = None
            L.orc_set_threads.argtypes = [i32]
            L.orc_set_threads.restype = None
            L.orc_e8m0_value.argtypes = [u8]; L.orc_e8m0_value.restype = f64
            L.orc_mxfp4_quantize.argtypes = [_u16, i64, i64, i64, _u8, _u8]
            L.orc_mxfp4_quantize.restype = i32
            L.orc_mxfp4_dequantize.argtypes = [_u8, _u8, i64, i64, _f64]
            L.orc_mxfp4_dequantize.restype = None
            L.orc_lora_linear_fwd_f32ab.argtypes = [_u16, i64, i64, i64, _u8, _u8, f32, _f32, _f32,
                                                    i32, f64, _i64, i64, _f64, C.c_void_p]
            L.orc_lora_linear_fwd_f32ab.restype = None
            L.orc_mxfp4_lora_linear_fwd.argtypes = [_u16, i64, i64, i64, _u8, _u8, _u16, _u16,
                                                    i32, f64, _i64, i64, _f64, C.c_void_p]
            L.orc_mxfp4_lora_linear_fwd.restype = None
            L.orc_lora_linear_bwd.argtypes = [_u16, _u16, i64, i64, i64, _u8, _u8, f32, _u16,
                                              _u16, i32, f64,
                                              C.c_void_p, i64, C.c_void_p,
                                              C.c_void_p, i64, C.c_void_p,
                                              C.c_void_p, i64, C.c_void_p]
            L.orc_lora_linear_bwd.restype = None
            L.orc_philox4x64_10.argtypes = [_u64, _u64, _u64]
            L.orc_philox4x64_10.restype = None
            L.orc_aqn_noise.argtypes = [i64, u64, u64, u32, _f64, C.c_void_p]
            L.orc_aqn_noise.restype = None
            L.orc_aqn_rmsnorm.argtypes = [_u16, i64, i64, _u16, f64, f64, u64, u64, u32,
                                          _i64, i64, _f64]
            L.orc_aqn_rmsnorm.restype = None
            L.orc_aqn_rmsnorm_mode.argtypes = [_u16, i64, i64, _u16, f64, f64, u64, u64, u32, C.c_int,
                                               _i64, i64, _f64]
            L.orc_aqn_rmsnorm_mode.restype = None
            L.orc_aqn_sigma.argtypes = [i64, i64, f64, f64, i32]
            L.orc_aqn_sigma.restype = f64
            _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


# ---------------------------------------------------------------- formats
def e4m3_value(b: int) -> float:
    return lib().orc_e4m3_value(b)


def e2m1_value(c: int) -> float:
    return lib().orc_e2m1_value(c)


def e4m3_round_up(t: float) -> int:
    return lib().orc_e4m3_round_up(t)


def e4m3_round_rne(t: float) -> int:
    return lib().orc_e4m3_round_rne(t)


def e2m1_round(q: float) -> int:
    return lib().orc_e2m1_round(q)


# ---------------------------------------------------------------- quantizer
def nvfp4_quantize(W_bits: np.ndarray, scale_mode: int = 0):
    """W_bits: uint16 [N, K] bf16 patterns -> (status, codes u8 [N,K/2],
    scales u8 [N,K/16], tensor_scale float32)."""
    W_bits = _c(W_bits, np.uint16)
    N, K = W_bits.shape
    codes = np.zeros((N, max(K // 2, 0)), np.uint8)
    scales = np.zeros((N, max(K // 16, 0)), np.uint8)
    st = np.zeros(1, np.float32)
    rc = lib().orc_nvfp4_quantize(W_bits, N, K, K, codes, scales, st, scale_mode)
    return rc, codes, scales, np.float32(st[0])


def nvfp4_dequantize(codes, scales, tensor_scale, N, K) -> np.ndarray:
    out = np.zeros((N, K), np.float64)
    lib().orc_nvfp4_dequantize(_c(codes, np.uint8), _c(scales, np.uint8),
                               float(tensor_scale), N, K, out)
    return out


# ---------------------------------------------------------------- linear
def set_threads(n: int):
    """Threads the linear forward may use (1, the default: single-threaded)."""
    lib().orc_set_threads(int(n))


def lora_linear_fwd(x_bits, codes, scales, tensor_scale, A_bits, B_bits, lora_scale,
                    rows=None, want_t=False):
    """y = x W_hat^T + s (x A^T) B^T in fp64 for the token rows ``rows``."""
    x_bits = _c(x_bits, np.uint16)
    M, K = x_bits.shape
    N = codes.shape[0]
    r = A_bits.shape[0]
    rows = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    y = np.zeros((len(rows), N), np.float64)
    t = np.zeros((len(rows), r), np.float64) if want_t else None
    lib().orc_lora_linear_fwd(x_bits, M, K, N, _c(codes, np.uint8), _c(scales, np.uint8),
                              float(tensor_scale), _c(A_bits, np.uint16), _c(B_bits, np.uint16),
                              r, float(lora_scale), rows, len(rows), y, _ptr(t))
    return (y, t) if want_t else y


def lora_linear_fwd_f32ab(x_bits, codes, scales, tensor_scale, A_f32, B_f32, lora_scale, rows=None,
                          want_t=False):
    """The forward with FP32 LoRA adapters (A [r,K], B [N,r] float32)."""
    x_bits = _c(x_bits, np.uint16)
    M, K = x_bits.shape
    N = codes.shape[0]
    r = A_f32.shape[0]
    rows = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    y = np.zeros((len(rows), N), np.float64)
    t = np.zeros((len(rows), r), np.float64) if want_t else None
    lib().orc_lora_linear_fwd_f32ab(x_bits, M, K, N, _c(codes, np.uint8), _c(scales, np.uint8),
                                    float(tensor_scale), _c(A_f32, np.float32), _c(B_f32, np.float32),
                                    r, float(lora_scale), rows, len(rows), y, _ptr(t))
    return (y, t) if want_t else y


# ---------------------------------------------------------------- MXFP4
def e8m0_value(b: int) -> float:
    return lib().orc_e8m0_value(b)


def mxfp4_quantize(W_bits: np.ndarray):
    """W_bits uint16 [N, K] -> (status, codes u8 [N,K/2], E8M0 scales u8 [N,K/32])."""
    W_bits = _c(W_bits, np.uint16)
    N, K = W_bits.shape
    codes = np.zeros((N, max(K // 2, 0)), np.uint8)
    scales = np.zeros((N, max(K // 32, 0)), np.uint8)
    rc = lib().orc_mxfp4_quantize(W_bits, N, K, K, codes, scales)
    return rc, codes, scales


def mxfp4_dequantize(codes, scales, N, K) -> np.ndarray:
    out = np.zeros((N, K), np.float64)
    lib().orc_mxfp4_dequantize(_c(codes, np.uint8), _c(scales, np.uint8), N, K, out)
    return out


def mxfp4_lora_linear_fwd(x_bits, codes, scales, A_bits, B_bits, lora_scale, rows=None, want_t=False):
    """y = x W_hat^T + s (x A^T) B^T with an MXFP4 weight, fp64."""
    x_bits = _c(x_bits, np.uint16)
    M, K = x_bits.shape
    N = codes.shape[0]
    r = A_bits.shape[0]
    rows = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    y = np.zeros((len(rows), N), np.float64)
    t = np.zeros((len(rows), r), np.float64) if want_t else None
    lib().orc_mxfp4_lora_linear_fwd(x_bits, M, K, N, _c(codes, np.uint8), _c(scales, np.uint8),
                                    _c(A_bits, np.uint16), _c(B_bits, np.uint16), r, float(lora_scale),
                                    rows, len(rows), y, _ptr(t))
    return (y, t) if want_t else y


def lora_linear_bwd(dy_bits, x_bits, codes, scales, tensor_scale, A_bits, B_bits, lora_scale,
                    dx_rows=None, dA_cols=None, dB_rows=None):
    """Returns (dx [len(dx_rows),K], dA [r,len(dA_cols)], dB [len(dB_rows),r]) in fp64.
    ``None`` index lists select every row / column."""
    dy_bits = _c(dy_bits, np.uint16)
    x_bits = _c(x_bits, np.uint16)
    M, N = dy_bits.shape
    K = x_bits.shape[1]
    r = A_bits.shape[0]
    dx_rows = np.arange(M, dtype=np.int64) if dx_rows is None else _c(dx_rows, np.int64)
    dA_cols = np.arange(K, dtype=np.int64) if dA_cols is None else _c(dA_cols, np.int64)
    dB_rows = np.arange(N, dtype=np.int64) if dB_rows is None else _c(dB_rows, np.int64)
    dx = np.zeros((len(dx_rows), K), np.float64)
    dA = np.zeros((r, len(dA_cols)), np.float64)
    dB = np.zeros((len(dB_rows), r), np.float64)
    lib().orc_lora_linear_bwd(dy_bits, x_bits, M, K, N, _c(codes, np.uint8), _c(scales, np.uint8),
                              float(tensor_scale), _c(A_bits, np.uint16), _c(B_bits, np.uint16),
                              r, float(lora_scale),
                              _ptr(dx_rows), len(dx_rows), _ptr(dx),
                              _ptr(dA_cols), len(dA_cols), _ptr(dA),
                              _ptr(dB_rows), len(dB_rows), _ptr(dB))
    return dx, dA, dB


# ---------------------------------------------------------------- AQN
def philox4x64_10(ctr, key) -> np.ndarray:
    out = np.zeros(4, np.uint64)
    lib().orc_philox4x64_10(_c(ctr, np.uint64), _c(key, np.uint64), out)
    return out


def aqn_noise(H, seed, step, layer, want_raw=False):
    z = np.zeros(H, np.float64)
    raw = np.zeros(H, np.uint64) if want_raw else None
    lib().orc_aqn_noise(H, seed, step, layer, z, _ptr(raw))
    return (z, raw) if want_raw else z


def aqn_rmsnorm(x_bits, gamma_bits, eps, sigma, seed, step, layer, rows=None, multiplicative=False):
    """Noise added to the scale (gamma + sigma z), or with multiplicative=True
    scaling it (gamma (1 + sigma z))."""
    x_bits = _c(x_bits, np.uint16)
    M, H = x_bits.shape
    rows = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    y = np.zeros((len(rows), H), np.float64)
    if multiplicative:
        lib().orc_aqn_rmsnorm_mode(x_bits, M, H, _c(gamma_bits, np.uint16), float(eps), float(sigma),
                                   seed, step, layer, 1, rows, len(rows), y)
    else:
        lib().orc_aqn_rmsnorm(x_bits, M, H, _c(gamma_bits, np.uint16), float(eps), float(sigma),
                              seed, step, layer, rows, len(rows), y)
    return y


def aqn_sigma(step, total_steps, sigma_start, sigma_end, num_stages) -> float:
    return lib().orc_aqn_sigma(step, total_steps, sigma_start, sigma_end, num_stages)
