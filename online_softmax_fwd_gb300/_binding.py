"""ctypes binding of ``libattn.so`` (the C ABI declared in include/attn.h).

Argument marshalling only: torch tensors supply device memory and the current
CUDA stream; every step of the computation runs in the library's kernels.
There is no fallback: if the shared library is missing or cannot be loaded,
every call raises.
"""
from __future__ import annotations

import ctypes
import enum
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn.so")

_lib = None
_lock = threading.Lock()


class Status(enum.IntEnum):
    OK = 0
    INVALID_ARG = 1
    UNSUPPORTED = 2
    MISALIGNED = 3
    CUDA = 4
    TIMEOUT = 5


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = Status(status) if status in Status._value2member_map_ else status
        super().__init__(f"{what}: {self.status!r}")


_SIGNATURES = {
    # q, k, v, o, lse, B, H, N, d, causal, scale, stream
    "attn_fwd": ([ctypes.c_void_p] * 5 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_void_p], ctypes.c_int),
    # ..., scale, tau, exp2_emu16, stream
    "attn_fwd_ex": ([ctypes.c_void_p] * 5 + [ctypes.c_int] * 5
                    + [ctypes.c_float, ctypes.c_float, ctypes.c_int, ctypes.c_void_p], ctypes.c_int),
    # q, k, v, o, lse, B, H, N, d, causal, scale, stream
    "attn_fwd_2cta": ([ctypes.c_void_p] * 5 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_void_p], ctypes.c_int),
    # o_parts, lse_parts, parts, o, lse, B, H, N, d, stream
    "attn_combine": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
                     + [ctypes.c_int] * 4 + [ctypes.c_void_p], ctypes.c_int),
    # q, k, v, o, lse, rescale_log, rescale_log_bytes, B, H, N, d, causal, scale, tau, stream
    "attn_fwd_rescale_log": ([ctypes.c_void_p] * 6 + [ctypes.c_size_t] + [ctypes.c_int] * 5
                             + [ctypes.c_float, ctypes.c_float, ctypes.c_void_p], ctypes.c_int),
    "attn_mxfp8_scale_bytes": ([ctypes.c_int] * 4, ctypes.c_size_t),
    # x, x_e4m3, x_scales, B, H, N, d, role, stream
    "attn_mxfp8_quantize": ([ctypes.c_void_p] * 3 + [ctypes.c_int] * 5 + [ctypes.c_void_p], ctypes.c_int),
    # q8, q_sf, k8, k_sf, v8, v_sf, o, lse, B, H, N, d, causal, scale, stream
    "attn_fwd_mxfp8": ([ctypes.c_void_p] * 8 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_void_p], ctypes.c_int),
    # ... scale, tau, exp2_emu16, p_scaling, stream
    "attn_fwd_mxfp8_ex": ([ctypes.c_void_p] * 8 + [ctypes.c_int] * 5
                          + [ctypes.c_float, ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p],
                          ctypes.c_int),
    # q8, q_sf, k8, k_sf, v8, v_sf, o, lse, B, H, N, d, causal, scale, stream
    "attn_fwd_mxfp8_unroll_kv": ([ctypes.c_void_p] * 8 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_void_p],
                                 ctypes.c_int),
    # q8, q_sf, k8, k_sf, v8, v_sf, o, lse, rescale_log, rescale_log_bytes, B, H, N, d, causal, scale, tau, stream
    "attn_fwd_mxfp8_rescale_log": ([ctypes.c_void_p] * 9 + [ctypes.c_size_t] + [ctypes.c_int] * 5
                                   + [ctypes.c_float, ctypes.c_float, ctypes.c_void_p], ctypes.c_int),
    "attn_exp2_emulated": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong, ctypes.c_void_p], ctypes.c_int),
    "attn_fwd_host_workspace_bytes": ([ctypes.c_int] * 4, ctypes.c_size_t),
    # q, k, v, o, lse (host), B, H, N, d, causal, scale, workspace, workspace_bytes, stream
    "attn_fwd_host": ([ctypes.c_void_p] * 5 + [ctypes.c_int] * 5
                      + [ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p], ctypes.c_int),
    "attn_fwd_host_noalloc_max_workspace": ([], ctypes.c_size_t),
    # q, k, v, o, lse (host), B, H, N, d, causal, scale, stream
    "attn_fwd_host_noalloc": ([ctypes.c_void_p] * 5 + [ctypes.c_int] * 5 + [ctypes.c_float, ctypes.c_void_p],
                              ctypes.c_int),
    "attn_bwd_workspace_bytes": ([ctypes.c_int] * 4, ctypes.c_size_t),
    # q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, causal, scale, workspace, workspace_bytes, stream
    "attn_bwd": ([ctypes.c_void_p] * 9 + [ctypes.c_int] * 5
                 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p], ctypes.c_int),
    # q8, q_sf, k8, k_sf, v8, v_sf, o, do8, do_sf, lse, dq, dk, dv, B, H, N, d, causal, scale, workspace,
    # workspace_bytes, stream
    "attn_bwd_mxfp8": ([ctypes.c_void_p] * 13 + [ctypes.c_int] * 5
                       + [ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p], ctypes.c_int),
    "attn_get_device_status": ([ctypes.c_void_p], ctypes.c_int),
    "attn_selftest_wait_timeout": ([ctypes.c_longlong, ctypes.c_void_p], ctypes.c_int),
    "attn_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "attn_version": ([], ctypes.c_int),
}


def lib() -> ctypes.CDLL:
    """Load libattn.so once; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -m online_softmax_fwd_gb300.build` "
                    "(there is no CPU or PyTorch fallback)")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (argtypes, restype) in _SIGNATURES.items():
                fn = getattr(handle, name)
                fn.argtypes = argtypes
                fn.restype = restype
            _lib = handle
    return _lib


def _check(status: int, what: str) -> None:
    if status != 0:
        raise AttnError(status, what)


def _stream_handle(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _check_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor) -> tuple[int, int, int, int]:
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor [B,H,N,d]")
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError(f"q, k, v shapes differ: {tuple(q.shape)} {tuple(k.shape)} {tuple(v.shape)}")
    B, H, N, d = q.shape
    return B, H, N, d


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
             scale: float | None = None, o: torch.Tensor | None = None, lse: torch.Tensor | None = None,
             tau: float = 8.0, exp2_emu16: int = 0, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """O = softmax(scale * Q K^T [causal mask]) V and LSE, through the C ABI.

    q, k, v: contiguous CUDA bf16 [B,H,N,d]. Returns (o bf16 [B,H,N,d],
    lse float32 [B,H,N]); pass ``o`` / ``lse`` to write into existing buffers.
    ``tau`` and ``exp2_emu16`` select attn_fwd_ex (defaults = attn_fwd).
    """
    B, H, N, d = _check_qkv(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if o.shape != q.shape or o.dtype != torch.bfloat16 or not o.is_contiguous() or o.device != q.device:
        raise ValueError("o must be a contiguous bf16 tensor shaped like q on q's device")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous() or lse.device != q.device:
        raise ValueError("lse must be a contiguous float32 tensor [B,H,N] on q's device")
    h = _stream_handle(stream)
    with torch.cuda.device(q.device):
        if tau == 8.0 and exp2_emu16 == 0:
            st = lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, int(bool(causal)),
                                float(scale), h)
            _check(st, "attn_fwd")
        else:
            st = lib().attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                                   int(bool(causal)), float(scale), float(tau), int(exp2_emu16), h)
            _check(st, "attn_fwd_ex")
    return o, lse


def attn_fwd_2cta(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                  scale: float | None = None, o: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                  stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """attn_fwd on CTA pairs (d = 128, non-causal): same inputs and outputs."""
    B, H, N, d = _check_qkv(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        st = lib().attn_fwd_2cta(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, int(bool(causal)),
                                 float(scale), _stream_handle(stream))
        _check(st, "attn_fwd_2cta")
    return o, lse


def attn_combine(o_parts: torch.Tensor, lse_parts: torch.Tensor, o: torch.Tensor | None = None,
                 lse: torch.Tensor | None = None, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Merge attention results over disjoint key sets: o_parts bf16 [P,B,H,N,d],
    lse_parts float32 [P,B,H,N] (CUDA, contiguous) -> (o [B,H,N,d], lse [B,H,N])."""
    if (not o_parts.is_cuda or o_parts.dtype != torch.bfloat16 or o_parts.dim() != 5
            or not o_parts.is_contiguous()):
        raise ValueError("o_parts must be a contiguous CUDA bfloat16 tensor [P,B,H,N,d]")
    P, B, H, N, d = o_parts.shape
    if (not lse_parts.is_cuda or lse_parts.dtype != torch.float32 or tuple(lse_parts.shape) != (P, B, H, N)
            or not lse_parts.is_contiguous()):
        raise ValueError("lse_parts must be a contiguous CUDA float32 tensor [P,B,H,N]")
    if o is None:
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=o_parts.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=o_parts.device)
    with torch.cuda.device(o_parts.device):
        st = lib().attn_combine(_ptr(o_parts), _ptr(lse_parts), P, _ptr(o), _ptr(lse), B, H, N, d,
                                _stream_handle(stream))
        _check(st, "attn_combine")
    return o, lse


def attn_fwd_rescale_log(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                         scale: float | None = None, tau: float = 8.0, stream=None):
    """attn_fwd_ex (MUFU exp2) plus the rescale log: returns (o, lse, log)
    with log uint8 [B, H, N, ceil(N/128)] (bit 0 = the row's max moved at that
    key block, bit 1 = its warp rescaled O). Bytes of blocks a row's tile does
    not stream stay 0."""
    B, H, N, d = _check_qkv(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    log = torch.zeros((B, H, N, (N + 127) // 128), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        st = lib().attn_fwd_rescale_log(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(log), log.numel(), B, H,
                                        N, d, int(bool(causal)), float(scale), float(tau), _stream_handle(stream))
        _check(st, "attn_fwd_rescale_log")
    return o, lse, log


def attn_fwd_raw(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int, d: int, causal: int,
                 scale: float, stream: int, tau: float = 8.0, exp2_emu16: int = 0) -> int:
    """The C entry point with plain integers (device addresses); returns the status."""
    if tau == 8.0 and exp2_emu16 == 0:
        return lib().attn_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, stream)
    return lib().attn_fwd_ex(q, k, v, o, lse, B, H, N, d, causal, scale, tau, exp2_emu16, stream)


def attn_fwd_from_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                       scale: float | None = None, device: int | torch.device = 0,
                       o_host: torch.Tensor | None = None, lse_host: torch.Tensor | None = None,
                       workspace: dict | None = None, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """End-to-end call with host tensors through attn_fwd_host: Q, K, V (CPU
    bf16 [B,H,N,d], pinned for overlap) in, O and LSE back into host tensors;
    the library overlaps the copies with the kernels. ``workspace`` (a dict)
    keeps the device workspace between calls of the same shape. Returns after
    the results are in host memory."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous() or t.shape != q.shape:
            raise ValueError(f"{name} must be a contiguous CPU bfloat16 tensor shaped like q")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda", device) if isinstance(device, int) else device
    if o_host is None:
        o_host = torch.empty((B, H, N, d), dtype=torch.bfloat16, pin_memory=True)
    if lse_host is None:
        lse_host = torch.empty((B, H, N), dtype=torch.float32, pin_memory=True)
    need = lib().attn_fwd_host_workspace_bytes(B, H, N, d)
    ws = workspace if workspace is not None else {}
    if ws.get("key") != (need, str(dev)):
        ws.clear()
        ws["key"] = (need, str(dev))
        ws["buf"] = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        h = _stream_handle(stream)
        st = lib().attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o_host), _ptr(lse_host), B, H, N, d,
                                 int(bool(causal)), float(scale), _ptr(ws["buf"]), need, h)
        _check(st, "attn_fwd_host")
        torch.cuda.current_stream(dev).synchronize() if stream is None else torch.cuda.Stream(
            stream_ptr=h, device=dev).synchronize()
    return o_host, lse_host


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, dout: torch.Tensor,
             lse: torch.Tensor, causal: bool = False, scale: float | None = None, workspace: dict | None = None,
             stream=None) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """dQ, dK, dV (bf16 [B,H,N,d]) through the C ABI, from the forward's inputs,
    its output O and LSE, and the upstream gradient dout (all contiguous CUDA;
    bf16 except lse fp32 [B,H,N]). ``workspace`` (a dict) keeps the device
    workspace between calls of the same shape."""
    B, H, N, d = _check_qkv(q, k, v)
    for name, t in (("o", o), ("dout", dout)):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q on q's device")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous() or lse.device != q.device:
        raise ValueError("lse must be a contiguous float32 tensor [B,H,N] on q's device")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    need = lib().attn_bwd_workspace_bytes(B, H, N, d)
    ws = workspace if workspace is not None else {}
    if ws.get("key") != (need, str(q.device)):
        ws.clear()
        ws["key"] = (need, str(q.device))
        ws["buf"] = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    h = _stream_handle(stream)
    with torch.cuda.device(q.device):
        st = lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                            _ptr(dv), B, H, N, d, int(bool(causal)), float(scale), _ptr(ws["buf"]), need, h)
    _check(st, "attn_bwd")
    return dq, dk, dv


def mxfp8_scale_bytes(B: int, H: int, N: int, d: int) -> int:
    return lib().attn_mxfp8_scale_bytes(B, H, N, d)


def mxfp8_quantize(x: torch.Tensor, role: int, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """fp32 CUDA [B,H,N,128] -> (E4M3 codes uint8 [B,H,N,128], scale atoms uint8
    [B*H*ceil(N/128)*512]). role 0: Q or K of the forward (atom rows = sequence
    positions); role 1: V of the forward (rows = d columns); role 2: both
    layouts, one array after the other (Q, K and dO of attn_bwd_mxfp8)."""
    if not x.is_cuda or x.dtype != torch.float32 or x.dim() != 4 or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA float32 tensor [B,H,N,d]")
    B, H, N, d = x.shape
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    copies = 2 if role == 2 else 1
    scales = torch.empty(max(1, copies * mxfp8_scale_bytes(B, H, N, d)), dtype=torch.uint8, device=x.device)
    with torch.cuda.device(x.device):
        _check(lib().attn_mxfp8_quantize(_ptr(x), _ptr(codes), _ptr(scales), B, H, N, d, int(role),
                                         _stream_handle(stream)), "attn_mxfp8_quantize")
    return codes, scales


def attn_bwd_mxfp8(q8: torch.Tensor, q_sf: torch.Tensor, k8: torch.Tensor, k_sf: torch.Tensor, v8: torch.Tensor,
                   v_sf: torch.Tensor, o: torch.Tensor, do8: torch.Tensor, do_sf: torch.Tensor, lse: torch.Tensor,
                   causal: bool = False, scale: float | None = None, workspace: dict | None = None,
                   stream=None) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """dQ, dK, dV (bf16 [B,H,N,128]) through the C ABI from MXFP8 inputs: q8/q_sf,
    k8/k_sf and do8/do_sf from mxfp8_quantize(role=2), v8/v_sf from role 0, the
    forward's output o (bf16) and LSE (fp32 [B,H,N]). ``workspace`` (a dict)
    keeps the device workspace between calls of the same shape."""
    for name, t in (("q8", q8), ("k8", k8), ("v8", v8), ("do8", do8)):
        if not t.is_cuda or t.dtype != torch.uint8 or t.dim() != 4 or not t.is_contiguous() or t.shape != q8.shape:
            raise ValueError(f"{name} must be contiguous CUDA uint8 (E4M3 codes) shaped like q8")
    B, H, N, d = q8.shape
    need_sf = mxfp8_scale_bytes(B, H, N, d)
    for name, t, copies in (("q_sf", q_sf, 2), ("k_sf", k_sf, 2), ("v_sf", v_sf, 1), ("do_sf", do_sf, 2)):
        if not t.is_cuda or t.dtype != torch.uint8 or t.numel() < copies * need_sf:
            raise ValueError(f"{name} must be a CUDA uint8 scale array of >= {copies * need_sf} bytes")
    if o.shape != q8.shape or o.dtype != torch.bfloat16 or not o.is_contiguous() or o.device != q8.device:
        raise ValueError("o must be a contiguous bf16 tensor shaped like q8 on its device")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous() or lse.device != q8.device:
        raise ValueError("lse must be a contiguous float32 tensor [B,H,N] on q8's device")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = (torch.empty(q8.shape, dtype=torch.bfloat16, device=q8.device) for _ in range(3))
    need = lib().attn_bwd_workspace_bytes(B, H, N, d)
    ws = workspace if workspace is not None else {}
    if ws.get("key") != (need, str(q8.device)):
        ws.clear()
        ws["key"] = (need, str(q8.device))
        ws["buf"] = torch.empty(max(need, 1), dtype=torch.uint8, device=q8.device)
    h = _stream_handle(stream)
    with torch.cuda.device(q8.device):
        st = lib().attn_bwd_mxfp8(*(_ptr(t) for t in (q8, q_sf, k8, k_sf, v8, v_sf, o, do8, do_sf, lse, dq, dk, dv)),
                                  B, H, N, d, int(bool(causal)), float(scale), _ptr(ws["buf"]), need, h)
    _check(st, "attn_bwd_mxfp8")
    return dq, dk, dv


P_SCALE_BLOCK_AMAX = 0
P_SCALE_CONSTANT = 1
P_SCALE_CONSTANT_E5M2 = 2


def attn_fwd_mxfp8(q8: torch.Tensor, q_sf: torch.Tensor, k8: torch.Tensor, k_sf: torch.Tensor, v8: torch.Tensor,
                   v_sf: torch.Tensor, causal: bool = False, scale: float | None = None, o: torch.Tensor | None = None,
                   lse: torch.Tensor | None = None, tau: float = 0.0, exp2_emu16: int = 0,
                   p_scaling: int = 0, unroll_kv: bool = False, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Attention forward from MXFP8 inputs (outputs of mxfp8_quantize); tau
    defaults to 0, the FP8 setting (attn_fwd_mxfp8). p_scaling: 0 = one scale
    per 32 keys from the block amax (P_SCALE_BLOCK_AMAX), 1 = the constant 2^-8
    (P_SCALE_CONSTANT, tau <= 0.807), 2 = the same constant with P held in
    E5M2 (P_SCALE_CONSTANT_E5M2, tau <= 7.807). unroll_kv selects the unroll-KV
    schedule (attn_fwd_mxfp8_unroll_kv; tau 0, no software exp2, p_scaling 0)."""
    for name, t in (("q8", q8), ("k8", k8), ("v8", v8)):
        if not t.is_cuda or t.dtype != torch.uint8 or t.dim() != 4 or not t.is_contiguous() or t.shape != q8.shape:
            raise ValueError(f"{name} must be contiguous CUDA uint8 (E4M3 codes) shaped like q8")
    B, H, N, d = q8.shape
    need = mxfp8_scale_bytes(B, H, N, d)
    for name, t in (("q_sf", q_sf), ("k_sf", k_sf), ("v_sf", v_sf)):
        if not t.is_cuda or t.dtype != torch.uint8 or t.numel() < need:
            raise ValueError(f"{name} must be a CUDA uint8 scale array of >= {need} bytes")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    h = _stream_handle(stream)
    ptrs = [_ptr(t) for t in (q8, q_sf, k8, k_sf, v8, v_sf, o, lse)]
    if unroll_kv and (tau != 0.0 or exp2_emu16 != 0 or p_scaling != P_SCALE_BLOCK_AMAX):
        raise ValueError("the unroll-KV schedule runs with tau = 0, exp2_emu16 = 0 and p_scaling = 0")
    with torch.cuda.device(q8.device):
        if unroll_kv:
            st = lib().attn_fwd_mxfp8_unroll_kv(*ptrs, B, H, N, d, int(bool(causal)), float(scale), h)
        elif tau == 0.0 and exp2_emu16 == 0 and p_scaling == P_SCALE_BLOCK_AMAX:
            st = lib().attn_fwd_mxfp8(*ptrs, B, H, N, d, int(bool(causal)), float(scale), h)
        else:
            st = lib().attn_fwd_mxfp8_ex(*ptrs, B, H, N, d, int(bool(causal)), float(scale), float(tau),
                                         int(exp2_emu16), int(p_scaling), h)
    _check(st, "attn_fwd_mxfp8")
    return o, lse


def exp2_emulated(x: torch.Tensor, stream=None) -> torch.Tensor:
    """The kernels' software exp2 applied elementwise (float32 CUDA tensor)."""
    if not x.is_cuda or x.dtype != torch.float32 or not x.is_contiguous():
        raise ValueError("x must be a contiguous CUDA float32 tensor")
    y = torch.empty_like(x)
    with torch.cuda.device(x.device):
        _check(lib().attn_exp2_emulated(_ptr(x), _ptr(y), x.numel(), _stream_handle(stream)),
               "attn_exp2_emulated")
    return y


def device_status(stream=None) -> Status:
    """Synchronise and read (and clear) the device error word."""
    return Status(lib().attn_get_device_status(_stream_handle(stream)))


def status_string(status: int) -> str:
    return lib().attn_status_string(int(status)).decode()


def version() -> int:
    return lib().attn_version()
