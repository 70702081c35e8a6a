"""Python binding of libqerl, the sm_103a NVFP4 weight-only LoRA linear library.

Argument marshalling only: each function passes torch tensors' device pointers,
sizes and the current CUDA stream to the C entry point of the same name in
``include/qerl.h`` and raises ``QerlError`` on a non-OK status.  Every step of
the computation runs in the library's CUDA kernels; there is no fallback.  If
``_lib/libqerl.so`` is missing the import of the library fails loudly (run
``build()``).
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libqerl.so")

QERL_OK = 0
STATUS_NAMES = {0: "QERL_OK", 1: "QERL_ERR_INVALID_ARG", 2: "QERL_ERR_SHAPE", 3: "QERL_ERR_ALIGN",
                4: "QERL_ERR_NONFINITE", 5: "QERL_ERR_CUDA", 6: "QERL_ERR_TIMEOUT",
                7: "QERL_ERR_UNSUPPORTED_DEVICE", 8: "QERL_ERR_WORKSPACE", 9: "QERL_ERR_TOO_LARGE"}
NOALLOC_SCRATCH_BYTES = 8 << 20  # QERL_NOALLOC_SCRATCH_BYTES
SCALE_ROUND_UP, SCALE_ROUND_NEAREST_EVEN = 0, 1
OP_QUANTIZE, OP_LINEAR_FWD, OP_LINEAR_BWD, OP_AQN_RMSNORM, OP_MXFP4_FWD, OP_LINEAR_FWD_F32AB = 0, 1, 2, 3, 4, 5
ALGO_AUTO, ALGO_SIMT, ALGO_TCGEN05, ALGO_GEMV = 0, 1, 2, 3
AQN_NOISE_ADD, AQN_NOISE_MUL = 0, 1

# Every C symbol include/qerl.h declares (checked by the CPU test suite).
EXPORTED = ["qerl_nvfp4_quantize", "qerl_nvfp4_dequantize", "qerl_nvfp4_lora_linear_fwd",
            "qerl_nvfp4_lora_linear_fwd_noalloc", "qerl_nvfp4_pack_codes", "qerl_nvfp4_unpack_codes",
            "qerl_nvfp4_lora_linear_fwd_packed", "qerl_nvfp4_lora_linear_bwd_packed",
            "qerl_nvfp4_lora_linear_bwd", "qerl_aqn_rmsnorm", "qerl_aqn_rmsnorm_mode", "qerl_aqn_noise",
            "qerl_aqn_sigma",
            "qerl_workspace_bytes", "qerl_get_error", "qerl_status_string", "qerl_set_linear_algo",
            "qerl_set_launch_chaining", "qerl_lora_linear_fwd_grouped_ws_bytes",
            "qerl_nvfp4_lora_linear_fwd_grouped",
            "qerl_launch_count", "qerl_decoder_chain_ws_bytes", "qerl_decoder_chain_plan",
            "qerl_decoder_chain_run", "qerl_decoder_chain_destroy", "qerl_mxfp4_quantize",
            "qerl_mxfp4_lora_linear_fwd", "qerl_nvfp4_lora_linear_fwd_f32ab", "qerl_residual_add", "qerl_swiglu"]


class QerlError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({status_string(status)})")


class _QuantOpts(C.Structure):
    _fields_ = [("scale_round", C.c_int)]


_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    from .build import build as _build
    return _build(force=force)


def lib() -> C.CDLL:
    """The loaded libqerl.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"libqerl.so not built ({LIB_PATH}); call "
                                  "nvfp4_weight_only_quantize_gb300.build()")
            L = C.CDLL(LIB_PATH)
            vp, i64, i32, f32, u64, u32, sz = (C.c_void_p, C.c_int64, C.c_int, C.c_float, C.c_uint64,
                                               C.c_uint32, C.c_size_t)
            sig = {
                "qerl_nvfp4_quantize": ([vp, i64, i64, i64, vp, vp, vp, vp, vp, sz, vp], i32),
                "qerl_nvfp4_dequantize": ([vp, vp, vp, i64, i64, vp, i32, vp], i32),
                "qerl_nvfp4_lora_linear_fwd": ([vp, i64, i64, i64, vp, vp, vp, vp, vp, i32, f32, vp, vp, vp,
                                                sz, vp], i32),
                "qerl_nvfp4_lora_linear_fwd_noalloc": ([vp, i64, i64, i64, vp, vp, vp, vp, vp, i32, f32, vp, vp,
                                                        vp], i32),
                "qerl_nvfp4_lora_linear_bwd": ([vp, vp, i64, i64, i64, vp, vp, vp, vp, vp, i32, f32, vp, vp,
                                                vp, vp, i32, vp, sz, vp], i32),
                "qerl_nvfp4_pack_codes": ([vp, i64, i64, vp, vp], i32),
                "qerl_nvfp4_unpack_codes": ([vp, i64, i64, vp, vp], i32),
                "qerl_aqn_rmsnorm": ([vp, i64, i64, vp, f32, f32, u64, u64, u32, vp, vp, sz, vp], i32),
                "qerl_aqn_rmsnorm_mode": ([vp, i64, i64, vp, f32, f32, u64, u64, u32, i32, vp, vp, sz, vp], i32),
                "qerl_aqn_noise": ([i64, u64, u64, u32, vp, vp, vp], i32),
                "qerl_aqn_sigma": ([i64, i64, f32, f32, i32], f32),
                "qerl_workspace_bytes": ([i32, i64, i64, i64, i32], sz),
                "qerl_get_error": ([vp], i32),
                "qerl_status_string": ([i32], C.c_char_p),
                "qerl_set_linear_algo": ([i32], i32),
                "qerl_set_launch_chaining": ([i32], i32),
                "qerl_launch_count": ([], u64),
            }
            sig["qerl_lora_linear_fwd_grouped_ws_bytes"] = ([i64, i64, i32, vp, i32], sz)
            sig["qerl_nvfp4_lora_linear_fwd_grouped"] = ([vp, i64, i64, i32, f32, vp, i32, i32, vp, sz, vp], i32)
            sig["qerl_mxfp4_quantize"] = ([vp, i64, i64, i64, vp, vp, vp], i32)
            sig["qerl_mxfp4_lora_linear_fwd"] = ([vp, i64, i64, i64, vp, vp, vp, vp, i32, f32, vp, vp, vp, sz, vp], i32)
            sig["qerl_nvfp4_lora_linear_fwd_f32ab"] = ([vp, i64, i64, i64, vp, vp, vp, vp, vp, i32, f32, vp, vp, vp,
                                                        sz, vp], i32)
            sig["qerl_decoder_chain_ws_bytes"] = ([vp, i32], sz)
            sig["qerl_decoder_chain_plan"] = ([vp, i32, vp, vp, vp, vp, sz, vp], i32)
            sig["qerl_decoder_chain_run"] = ([vp, f32, u64, u64, u32, vp], i32)
            sig["qerl_decoder_chain_destroy"] = ([vp], None)
            sig["qerl_residual_add"] = ([vp, vp, i64, vp, vp], i32)
            sig["qerl_swiglu"] = ([vp, vp, i64, vp, vp], i32)
            sig["qerl_nvfp4_lora_linear_fwd_packed"] = sig["qerl_nvfp4_lora_linear_fwd"]
            sig["qerl_nvfp4_lora_linear_bwd_packed"] = sig["qerl_nvfp4_lora_linear_bwd"]
            for name, (args, res) in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().qerl_status_string(status).decode()


def _check(status: int, where: str):
    if status != QERL_OK:
        raise QerlError(status, where)


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def workspace_bytes(op: int, M: int, N: int, K: int, r: int) -> int:
    return lib().qerl_workspace_bytes(op, M, N, K, r)


def workspace(op: int, M: int, N: int, K: int, r: int, device="cuda") -> torch.Tensor:
    """A caller-owned scratch buffer of the size the library asks for."""
    return torch.empty(max(workspace_bytes(op, M, N, K, r), 1), dtype=torch.uint8, device=device)


def set_linear_algo(algo: int):
    _check(lib().qerl_set_linear_algo(algo), "qerl_set_linear_algo")


def set_launch_chaining(on: bool):
    """Programmatic dependent launches between consecutive calls (default on)."""
    _check(lib().qerl_set_launch_chaining(int(bool(on))), "qerl_set_launch_chaining")


def launch_count() -> int:
    return lib().qerl_launch_count()


def get_error(stream=None) -> int:
    return lib().qerl_get_error(_stream(stream))


# ---------------------------------------------------------------- quantizer
def qerl_nvfp4_quantize(W: torch.Tensor, scale_round: int = SCALE_ROUND_UP, out=None, ws=None, stream=None):
    """W bf16 [N, K] (row stride W.stride(0)) -> (codes u8 [N,K/2], scales u8 [N,K/16], s_t f32 [1])."""
    assert W.dtype == torch.bfloat16 and W.dim() == 2 and W.stride(1) == 1
    N, K = W.shape
    if out is None:
        out = (torch.empty(N, K // 2, dtype=torch.uint8, device=W.device),
               torch.empty(N, K // 16, dtype=torch.uint8, device=W.device),
               torch.empty(1, dtype=torch.float32, device=W.device))
    codes, scales, ts = out
    ws = workspace(OP_QUANTIZE, 0, N, K, 0, W.device) if ws is None else ws
    opts = _QuantOpts(scale_round)
    _check(lib().qerl_nvfp4_quantize(_p(W), N, K, W.stride(0), _p(codes), _p(scales), _p(ts), C.byref(opts),
                                     _p(ws), ws.numel(), _stream(stream)), "qerl_nvfp4_quantize")
    return codes, scales, ts


def qerl_nvfp4_dequantize(codes, scales, tensor_scale, N: int, K: int, apply_tensor_scale: bool = True,
                          out=None, stream=None):
    out = torch.empty(N, K, dtype=torch.bfloat16, device=codes.device) if out is None else out
    _check(lib().qerl_nvfp4_dequantize(_p(codes), _p(scales), _p(tensor_scale), N, K, _p(out),
                                       int(apply_tensor_scale), _stream(stream)), "qerl_nvfp4_dequantize")
    return out


# ---------------------------------------------------------------- linear
def _fwd(name, x, codes, scales, tensor_scale, A, B, lora_scale, y, t_out, ws, stream):
    M, K = x.shape
    N, r = B.shape
    y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device) if y is None else y
    ws = workspace(OP_LINEAR_FWD, M, N, K, r, x.device) if ws is None else ws
    _check(getattr(lib(), name)(_p(x), M, K, N, _p(codes), _p(scales), _p(tensor_scale), _p(A), _p(B), r,
                                float(lora_scale), _p(y), _p(t_out), _p(ws), ws.numel(), _stream(stream)), name)
    return y


def qerl_nvfp4_lora_linear_fwd(x, codes, scales, tensor_scale, A, B, lora_scale: float, y=None, t_out=None,
                               ws=None, stream=None):
    """y = x w_hat^T + s (x A^T) B^T.  x bf16 [M,K], A bf16 [r,K], B bf16 [N,r] -> y bf16 [M,N]."""
    return _fwd("qerl_nvfp4_lora_linear_fwd", x, codes, scales, tensor_scale, A, B, lora_scale, y, t_out, ws, stream)


def qerl_nvfp4_lora_linear_fwd_packed(x, packed_codes, scales, tensor_scale, A, B, lora_scale: float, y=None,
                                      t_out=None, ws=None, stream=None):
    """The forward with the codes in the packed layout (qerl_nvfp4_pack_codes)."""
    return _fwd("qerl_nvfp4_lora_linear_fwd_packed", x, packed_codes, scales, tensor_scale, A, B, lora_scale, y,
                t_out, ws, stream)


class _Group(C.Structure):
    _fields_ = [("N", C.c_int64), ("codes", C.c_void_p), ("scales", C.c_void_p), ("tensor_scale", C.c_void_p),
                ("A", C.c_void_p), ("B", C.c_void_p), ("y", C.c_void_p), ("t_out", C.c_void_p)]


def grouped_ws_bytes(M: int, K: int, r: int, Ns) -> int:
    arr = (C.c_int64 * len(Ns))(*Ns)
    return lib().qerl_lora_linear_fwd_grouped_ws_bytes(M, K, r, C.cast(arr, C.c_void_p), len(Ns))


def qerl_nvfp4_lora_linear_fwd_grouped(x, groups, lora_scale: float, packed: bool = False, ys=None, t_outs=None,
                                       ws=None, stream=None):
    """Linears sharing x: groups = [(codes, scales, tensor_scale, A, B), ...].  Returns [y_g]."""
    M, K = x.shape
    r = groups[0][3].shape[0]
    Ns = [g[4].shape[0] for g in groups]
    ys = [torch.empty(M, N, dtype=torch.bfloat16, device=x.device) for N in Ns] if ys is None else ys
    t_outs = [None] * len(groups) if t_outs is None else t_outs
    arr = (_Group * len(groups))()
    for i, (codes, scales, ts, A, B) in enumerate(groups):
        arr[i] = _Group(Ns[i], _p(codes), _p(scales), _p(ts), _p(A), _p(B), _p(ys[i]), _p(t_outs[i]))
    if ws is None:
        ws = torch.empty(max(grouped_ws_bytes(M, K, r, Ns), 1), dtype=torch.uint8, device=x.device)
    _check(lib().qerl_nvfp4_lora_linear_fwd_grouped(_p(x), M, K, r, float(lora_scale), C.cast(arr, C.c_void_p),
                                                    len(groups), int(bool(packed)), _p(ws), ws.numel(),
                                                    _stream(stream)), "qerl_nvfp4_lora_linear_fwd_grouped")
    return ys


def qerl_nvfp4_pack_codes(codes, out=None, stream=None):
    """Standard NVFP4 codes [N, K/2] -> the packed layout (same shape; out may be codes itself)."""
    N, half = codes.shape
    out = torch.empty_like(codes) if out is None else out
    _check(lib().qerl_nvfp4_pack_codes(_p(codes), N, 2 * half, _p(out), _stream(stream)), "qerl_nvfp4_pack_codes")
    return out


def qerl_nvfp4_unpack_codes(packed, out=None, stream=None):
    """Inverse of qerl_nvfp4_pack_codes."""
    N, half = packed.shape
    out = torch.empty_like(packed) if out is None else out
    _check(lib().qerl_nvfp4_unpack_codes(_p(packed), N, 2 * half, _p(out), _stream(stream)),
           "qerl_nvfp4_unpack_codes")
    return out


def qerl_nvfp4_lora_linear_fwd_noalloc(x, codes, scales, tensor_scale, A, B, lora_scale: float, y=None,
                                       t_out=None, stream=None):
    """The forward with the library's fixed device scratch instead of a workspace
    (for callers that cannot allocate device memory; see include/qerl.h)."""
    M, K = x.shape
    N, r = B.shape
    y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device) if y is None else y
    _check(lib().qerl_nvfp4_lora_linear_fwd_noalloc(_p(x), M, K, N, _p(codes), _p(scales), _p(tensor_scale), _p(A),
                                                    _p(B), r, float(lora_scale), _p(y), _p(t_out), _stream(stream)),
           "qerl_nvfp4_lora_linear_fwd_noalloc")
    return y


def qerl_nvfp4_lora_linear_bwd(dy, x, codes, scales, tensor_scale, A, B, lora_scale: float, t_saved=None,
                               dx=None, dA=None, dB=None, accumulate: bool = False, want=("dx", "dA", "dB"),
                               ws=None, stream=None):
    """Returns (dx bf16 [M,K], dA f32 [r,K], dB f32 [N,r]); outputs not in ``want`` are None."""
    return _bwd("qerl_nvfp4_lora_linear_bwd", dy, x, codes, scales, tensor_scale, A, B, lora_scale, t_saved, dx, dA,
                dB, accumulate, want, ws, stream)


def qerl_nvfp4_lora_linear_bwd_packed(dy, x, packed_codes, scales, tensor_scale, A, B, lora_scale: float,
                                      t_saved=None, dx=None, dA=None, dB=None, accumulate: bool = False,
                                      want=("dx", "dA", "dB"), ws=None, stream=None):
    """The backward with the codes in the packed layout."""
    return _bwd("qerl_nvfp4_lora_linear_bwd_packed", dy, x, packed_codes, scales, tensor_scale, A, B, lora_scale,
                t_saved, dx, dA, dB, accumulate, want, ws, stream)


def _bwd(name, dy, x, codes, scales, tensor_scale, A, B, lora_scale, t_saved, dx, dA, dB, accumulate, want, ws,
         stream):
    M, N = dy.shape
    K = x.shape[1]
    r = A.shape[0]
    dev = x.device
    if dx is None and "dx" in want:
        dx = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    if dA is None and "dA" in want:
        dA = torch.zeros(r, K, dtype=torch.float32, device=dev)
    if dB is None and "dB" in want:
        dB = torch.zeros(N, r, dtype=torch.float32, device=dev)
    ws = workspace(OP_LINEAR_BWD, M, N, K, r, dev) if ws is None else ws
    _check(getattr(lib(), name)(_p(dy), _p(x), M, K, N, _p(codes), _p(scales), _p(tensor_scale), _p(A), _p(B), r,
                                float(lora_scale), _p(t_saved), _p(dx), _p(dA), _p(dB), int(accumulate), _p(ws),
                                ws.numel(), _stream(stream)), name)
    return dx, dA, dB


# ---------------------------------------------------------------- format variants
def qerl_mxfp4_quantize(W: torch.Tensor, out=None, stream=None):
    """W bf16 [N, K] -> (codes u8 [N, K/2], E8M0 scales u8 [N, K/32])."""
    assert W.dtype == torch.bfloat16 and W.dim() == 2 and W.stride(1) == 1
    N, K = W.shape
    if out is None:
        out = (torch.empty(N, K // 2, dtype=torch.uint8, device=W.device),
               torch.empty(N, K // 32, dtype=torch.uint8, device=W.device))
    codes, scales = out
    _check(lib().qerl_mxfp4_quantize(_p(W), N, K, W.stride(0), _p(codes), _p(scales), _stream(stream)),
           "qerl_mxfp4_quantize")
    return codes, scales


def qerl_mxfp4_lora_linear_fwd(x, codes, scales, A, B, lora_scale: float, y=None, t_out=None, ws=None, stream=None):
    M, K = x.shape
    N, r = B.shape
    y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device) if y is None else y
    ws = workspace(OP_MXFP4_FWD, M, N, K, r, x.device) if ws is None else ws
    _check(lib().qerl_mxfp4_lora_linear_fwd(_p(x), M, K, N, _p(codes), _p(scales), _p(A), _p(B), r, float(lora_scale),
                                            _p(y), _p(t_out), _p(ws), ws.numel(), _stream(stream)),
           "qerl_mxfp4_lora_linear_fwd")
    return y


def qerl_nvfp4_lora_linear_fwd_f32ab(x, codes, scales, tensor_scale, A, B, lora_scale: float, y=None, t_out=None,
                                     ws=None, stream=None):
    """The forward with FP32 LoRA adapters A [r, K] and B [N, r] (float32)."""
    assert A.dtype == torch.float32 and B.dtype == torch.float32
    M, K = x.shape
    N, r = B.shape
    y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device) if y is None else y
    ws = workspace(OP_LINEAR_FWD_F32AB, M, N, K, r, x.device) if ws is None else ws
    _check(lib().qerl_nvfp4_lora_linear_fwd_f32ab(_p(x), M, K, N, _p(codes), _p(scales), _p(tensor_scale), _p(A),
                                                  _p(B), r, float(lora_scale), _p(y), _p(t_out), _p(ws), ws.numel(),
                                                  _stream(stream)),
           "qerl_nvfp4_lora_linear_fwd_f32ab")
    return y


# ---------------------------------------------------------------- decoder-layer glue
def qerl_residual_add(h, y, out=None, stream=None):
    """out = bf16(h + y) elementwise (bf16 tensors of one shape); out may be h."""
    assert h.shape == y.shape and h.dtype == y.dtype == torch.bfloat16
    out = torch.empty_like(h) if out is None else out
    _check(lib().qerl_residual_add(_p(h), _p(y), h.numel(), _p(out), _stream(stream)), "qerl_residual_add")
    return out


def qerl_swiglu(g, u, out=None, stream=None):
    """out = bf16(silu(g) * u) elementwise (bf16 tensors of one shape)."""
    assert g.shape == u.shape and g.dtype == u.dtype == torch.bfloat16
    out = torch.empty_like(g) if out is None else out
    _check(lib().qerl_swiglu(_p(g), _p(u), g.numel(), _p(out), _stream(stream)), "qerl_swiglu")
    return out


# ---------------------------------------------------------------- AQN
def qerl_aqn_rmsnorm(x, gamma, eps: float, sigma: float, seed: int, step: int, layer_id: int, y=None, ws=None,
                     stream=None, noise_mode: int = None):
    """noise_mode None: qerl_aqn_rmsnorm (additive); AQN_NOISE_ADD / AQN_NOISE_MUL:
    qerl_aqn_rmsnorm_mode."""
    M, H = x.shape
    y = torch.empty_like(x) if y is None else y
    ws = workspace(OP_AQN_RMSNORM, M, 0, H, 0, x.device) if ws is None else ws
    if noise_mode is None:
        _check(lib().qerl_aqn_rmsnorm(_p(x), M, H, _p(gamma), float(eps), float(sigma), seed, step, layer_id, _p(y),
                                      _p(ws), ws.numel(), _stream(stream)), "qerl_aqn_rmsnorm")
    else:
        _check(lib().qerl_aqn_rmsnorm_mode(_p(x), M, H, _p(gamma), float(eps), float(sigma), seed, step, layer_id,
                                           int(noise_mode), _p(y), _p(ws), ws.numel(), _stream(stream)),
               "qerl_aqn_rmsnorm_mode")
    return y


def qerl_aqn_noise(H: int, seed: int, step: int, layer_id: int, want_raw: bool = False, device="cuda",
                   stream=None):
    z = torch.empty(H, dtype=torch.float32, device=device)
    raw = torch.empty(H, dtype=torch.int64, device=device) if want_raw else None
    _check(lib().qerl_aqn_noise(H, seed, step, layer_id, _p(z), _p(raw), _stream(stream)), "qerl_aqn_noise")
    return (z, raw) if want_raw else z


def qerl_aqn_sigma(step: int, total_steps: int, sigma_start: float, sigma_end: float, num_stages: int) -> float:
    return lib().qerl_aqn_sigma(step, total_steps, sigma_start, sigma_end, num_stages)


# ---------------------------------------------------------------- decoder chain
class _LinW(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("scales", C.c_void_p), ("tensor_scale", C.c_void_p), ("A", C.c_void_p),
                ("B", C.c_void_p)]


CHAIN_LINEARS = ("q", "k", "v", "o", "gate", "up", "down")


class _Layer(C.Structure):
    _fields_ = [(n, _LinW) for n in CHAIN_LINEARS] + [
        ("gamma_attn", C.c_void_p), ("gamma_mlp", C.c_void_p), ("attn", C.c_void_p), ("q_out", C.c_void_p),
        ("k_out", C.c_void_p), ("v_out", C.c_void_p)]


class _Dims(C.Structure):
    _fields_ = [("M", C.c_int64), ("hidden", C.c_int64), ("q_dim", C.c_int64), ("kv_dim", C.c_int64),
                ("intermediate", C.c_int64), ("r", C.c_int), ("lora_scale", C.c_float), ("eps", C.c_float)]


def decoder_chain_ws_bytes(M, hidden, q_dim, kv_dim, intermediate, r, lora_scale, eps, n_layers) -> int:
    d = _Dims(M, hidden, q_dim, kv_dim, intermediate, r, lora_scale, eps)
    return lib().qerl_decoder_chain_ws_bytes(C.byref(d), n_layers)


class DecoderChain:
    """A planned chain of decoder layers (qerl_decoder_chain_plan / _run).

    layers: one dict per layer with the seven linears under "q", "k", "v", "o",
    "gate", "up", "down" as (packed codes, scales, tensor_scale, A, B), and
    "gamma_attn", "gamma_mlp", "attn" (bf16 [M, hidden]) and optional "q_out",
    "k_out", "v_out".  The tensors are kept referenced while the plan lives."""

    def __init__(self, layers, M, hidden, q_dim, kv_dim, intermediate, r, lora_scale, eps, x_in, x_out, ws=None):
        self._keep = [layers, x_in, x_out]
        d = _Dims(M, hidden, q_dim, kv_dim, intermediate, r, lora_scale, eps)
        n = lib().qerl_decoder_chain_ws_bytes(C.byref(d), len(layers))
        if n == 0:
            raise QerlError(2, "qerl_decoder_chain_ws_bytes")
        self.ws = torch.empty(n, dtype=torch.uint8, device=x_in.device) if ws is None else ws
        arr = (_Layer * len(layers))()
        for i, Ly in enumerate(layers):
            for nm in CHAIN_LINEARS:
                codes, scales, ts, A, B = Ly[nm]
                setattr(arr[i], nm, _LinW(_p(codes), _p(scales), _p(ts), _p(A), _p(B)))
            arr[i].gamma_attn = _p(Ly["gamma_attn"])
            arr[i].gamma_mlp = _p(Ly["gamma_mlp"])
            arr[i].attn = _p(Ly["attn"])
            arr[i].q_out = _p(Ly.get("q_out"))
            arr[i].k_out = _p(Ly.get("k_out"))
            arr[i].v_out = _p(Ly.get("v_out"))
        h = C.c_void_p()
        _check(lib().qerl_decoder_chain_plan(C.cast(arr, C.c_void_p), len(layers), C.byref(d), _p(x_in), _p(x_out),
                                             _p(self.ws), self.ws.numel(), C.byref(h)), "qerl_decoder_chain_plan")
        self._h = h

    def run(self, sigma: float, seed: int, step: int, first_layer: int = 0, stream=None):
        _check(lib().qerl_decoder_chain_run(self._h, float(sigma), seed, step, first_layer, _stream(stream)),
               "qerl_decoder_chain_run")

    def close(self):
        if self._h:
            lib().qerl_decoder_chain_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
