"""ctypes binding of the C ABI in include/attn.h.

Argument marshalling only: PyTorch supplies device memory and the current
stream, every step of the computation runs in the CUDA library.  There is no
fallback: if libattn.so is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn.so")

ATTN_OK = 0
STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_CUDA",
          4: "ATTN_ERR_TIMEOUT", 5: "ATTN_ERR_NO_DEVICE", 6: "ATTN_ERR_SCRATCH_LIMIT", 7: "ATTN_ERR_BAD_INDEX"}
ATTN_ERR_TIMEOUT, ATTN_ERR_BAD_INDEX = 4, 7  # device-side errors that get_error() reports

# Every symbol the header declares, with (restype, argtypes).
_P, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_fwd_host_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "attn_fwd_host": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _SZ, _P]),
    "attn_decode_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "attn_bwd_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _SZ, _P]),
    "attn_decode": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _SZ, _P]),
    "attn_decode_multi_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "attn_decode_multi": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _SZ, _P]),
    "attn_decode_paged": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _SZ, _P]),
    "attn_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "attn_fwd_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_rotate_quantize_fp8": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "attn_rotate_quantize_fp8_many": (_I, [_P, _I, _P, _I, _P]),
    "attn_get_error": (_I, [_P]),
    "attn_debug_stall_role_waits": (None, [_I]),
    "attn_debug_skew_roles": (None, [_I]),
    "attn_status_str": (ctypes.c_char_p, [_I]),
    "attn_version": (ctypes.c_char_p, []),
}

_lib = None
_lock = threading.Lock()


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


def lib() -> ctypes.CDLL:
    """Load libattn.so once (after torch's CUDA runtime, so both share it)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"CUDA library {LIB_PATH} is not built; run "
                        "`python -m exact_tiled_attention_15_gb300.build` (nvcc, sm_103a)")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(status: int, what: str):
    if status != ATTN_OK:
        raise AttnError(status, what)


def _need(t, name, dtype, dims):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dimensions, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _need_like(t, name, dtype, shape, device):
    """A caller-supplied input or output: right dtype, exact shape, contiguous,
    on the same device as the query -- the library writes through its raw
    pointer and trusts these."""
    _need(t, name, dtype, len(shape))
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


def _need_workspace(t, name, nbytes, device):
    """Caller-supplied scratch: a contiguous CUDA tensor on `device` of at least
    `nbytes` bytes (the library also checks the byte count it is given)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be a CUDA tensor on {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name} holds {t.numel() * t.element_size()} bytes, {nbytes} needed")


def _out(t, name, dtype, shape, device):
    """The given output tensor after checking it, or a new one."""
    if t is None:
        return torch.empty(shape, device=device, dtype=dtype)
    _need_like(t, name, dtype, shape, device)
    return t


def fwd(q, k, v, causal=False, scale=None, return_lse=True, out=None, lse_out=None):
    """bf16 prefill forward.  q [B,Hq,Sq,D], k/v [B,Hkv,Sk,D] -> (o, lse)."""
    _need(q, "q", torch.bfloat16, 4)
    _need(k, "k", torch.bfloat16, 4)
    _need(v, "v", torch.bfloat16, 4)
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    if tuple(v.shape) != tuple(k.shape) or k.shape[0] != B or k.shape[3] != D:
        raise ValueError("k and v must be [B, Hkv, Sk, D] matching q")
    _need_like(k, "k", torch.bfloat16, k.shape, q.device)
    _need_like(v, "v", torch.bfloat16, k.shape, q.device)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    o = _out(out, "out", torch.bfloat16, q.shape, q.device)
    lse = _out(lse_out, "lse_out", torch.float32, (B, Hq, Sq), q.device) if return_lse else None
    st = lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Sk, D,
                        1 if causal else 0, scale, _stream(q.device))
    _check(st, "attn_fwd")
    return o, lse


def _need_host(t, name, dtype, dims):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dimensions, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def fwd_host_workspace_bytes(B, Hq, Hkv, Sq, Sk, D) -> int:
    return int(lib().attn_fwd_host_workspace_bytes(B, Hq, Hkv, Sq, Sk, D))


def fwd_host(q, k, v, causal=False, scale=None, out=None, lse_out=None, workspace=None, device=None):
    """fwd on host (CPU, ideally pinned) tensors; copies and kernels overlap in
    chunks.  Returns (o, lse) as host tensors, valid once the current CUDA
    stream of ``device`` has been synchronised."""
    _need_host(q, "q", torch.bfloat16, 4)
    _need_host(k, "k", torch.bfloat16, 4)
    _need_host(v, "v", torch.bfloat16, 4)
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    if tuple(v.shape) != tuple(k.shape) or k.shape[0] != B or k.shape[3] != D:
        raise ValueError("k and v must be [B, Hkv, Sk, D] matching q")
    dev = torch.device("cuda") if device is None else torch.device(device)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    o = out if out is not None else torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    lse = lse_out if lse_out is not None else torch.empty(B, Hq, Sq, dtype=torch.float32, pin_memory=True)
    _need_host(o, "out", torch.bfloat16, 4)
    _need_host(lse, "lse_out", torch.float32, 3)
    if tuple(o.shape) != tuple(q.shape) or tuple(lse.shape) != (B, Hq, Sq):
        raise ValueError("out must be shaped like q and lse_out [B, Hq, Sq]")
    nbytes = fwd_host_workspace_bytes(B, Hq, Hkv, Sq, Sk, D)
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    _need_workspace(workspace, "workspace", nbytes, dev)
    st = lib().attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, Hq, Hkv,
                             Sq, Sk, D, 1 if causal else 0, scale, _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(dev))
    _check(st, "attn_fwd_host")
    return o, lse


def bwd(q, k, v, o, lse, dout, causal=False, scale=None, workspace=None):
    """Gradients of fwd: (dq, dk, dv) for the given dout, from q, k, v, o and the forward's lse."""
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _need(t, name, torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    if tuple(v.shape) != tuple(k.shape) or k.shape[0] != B or k.shape[3] != D:
        raise ValueError("k and v must be [B, Hkv, Sk, D] matching q")
    for name, t in (("k", k), ("v", v)):
        _need_like(t, name, torch.bfloat16, k.shape, q.device)
    for name, t in (("o", o), ("dout", dout)):
        _need_like(t, name, torch.bfloat16, q.shape, q.device)
    _need_like(lse, "lse", torch.float32, (B, Hq, Sq), q.device)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    nbytes = int(lib().attn_bwd_workspace_bytes(B, Hq, Sq, D))
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), device=q.device, dtype=torch.uint8)
    _need_workspace(workspace, "workspace", nbytes, q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv),
                        B, Hq, Hkv, Sq, Sk, D, 1 if causal else 0, scale, _ptr(workspace),
                        workspace.numel() * workspace.element_size(), _stream(q.device))
    _check(st, "attn_bwd")
    return dq, dk, dv


def decode_workspace_bytes(B, Hq, Hkv, Lmax, D) -> int:
    return int(lib().attn_decode_workspace_bytes(B, Hq, Hkv, Lmax, D))


def decode(q, kcache, vcache, seqlens, scale=None, workspace=None, return_lse=True, out=None, lse_out=None):
    """Decode: q [B,Hq,D] against cache [B,Hkv,Lmax,D] with seqlens [B] int32 -> (o, lse)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(kcache, "kcache", torch.bfloat16, 4)
    _need(vcache, "vcache", torch.bfloat16, 4)
    _need(seqlens, "seqlens", torch.int32, 1)
    B, Hq, D = q.shape
    Hkv, Lmax = kcache.shape[1], kcache.shape[2]
    if tuple(vcache.shape) != tuple(kcache.shape) or kcache.shape[0] != B or kcache.shape[3] != D:
        raise ValueError("kcache and vcache must be [B, Hkv, Lmax, D] matching q")
    if seqlens.shape[0] != B:
        raise ValueError("seqlens must have B entries")
    for name, t in (("kcache", kcache), ("vcache", vcache)):
        _need_like(t, name, torch.bfloat16, kcache.shape, q.device)
    _need_like(seqlens, "seqlens", torch.int32, (B,), q.device)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    nbytes = decode_workspace_bytes(B, Hq, Hkv, Lmax, D)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), device=q.device, dtype=torch.uint8)
    _need_workspace(workspace, "workspace", nbytes, q.device)
    o = _out(out, "out", torch.bfloat16, q.shape, q.device)
    lse = _out(lse_out, "lse_out", torch.float32, (B, Hq), q.device) if return_lse else None
    st = lib().attn_decode(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(seqlens), _ptr(o), _ptr(lse),
                           B, Hq, Hkv, Lmax, D, scale, _ptr(workspace), workspace.numel() * workspace.element_size(),
                           _stream(q.device))
    _check(st, "attn_decode")
    return o, lse


def decode_multi(q, kcache, vcache, seqlens, causal=True, scale=None, workspace=None, return_lse=True, out=None,
                 lse_out=None):
    """T query tokens per sequence: q [B,Hq,T,D] against cache [B,Hkv,Lmax,D] -> (o [B,Hq,T,D], lse [B,Hq,T])."""
    _need(q, "q", torch.bfloat16, 4)
    _need(kcache, "kcache", torch.bfloat16, 4)
    _need(vcache, "vcache", torch.bfloat16, 4)
    _need(seqlens, "seqlens", torch.int32, 1)
    B, Hq, T, D = q.shape
    Hkv, Lmax = kcache.shape[1], kcache.shape[2]
    if tuple(vcache.shape) != tuple(kcache.shape) or kcache.shape[0] != B or kcache.shape[3] != D:
        raise ValueError("kcache and vcache must be [B, Hkv, Lmax, D] matching q")
    if seqlens.shape[0] != B:
        raise ValueError("seqlens must have B entries")
    for name, t in (("kcache", kcache), ("vcache", vcache)):
        _need_like(t, name, torch.bfloat16, kcache.shape, q.device)
    _need_like(seqlens, "seqlens", torch.int32, (B,), q.device)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    nbytes = int(lib().attn_decode_multi_workspace_bytes(B, Hq, Hkv, T, Lmax, D))
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), device=q.device, dtype=torch.uint8)
    _need_workspace(workspace, "workspace", nbytes, q.device)
    o = _out(out, "out", torch.bfloat16, q.shape, q.device)
    lse = _out(lse_out, "lse_out", torch.float32, (B, Hq, T), q.device) if return_lse else None
    st = lib().attn_decode_multi(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(seqlens), _ptr(o), _ptr(lse), B, Hq, Hkv,
                                 T, Lmax, D, 1 if causal else 0, scale, _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(q.device))
    _check(st, "attn_decode_multi")
    return o, lse


def decode_paged(q, k_pages, v_pages, block_table, seqlens, scale=None, workspace=None, return_lse=True,
                 out=None, lse_out=None):
    """Decode against a paged cache: pools [num_pages, Hkv, page_size, D] bf16,
    block_table [B, max_blocks] int32 -> (o, lse)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seqlens, "seqlens", torch.int32, 1)
    B, Hq, D = q.shape
    num_pages, Hkv, page_size = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    max_blocks = block_table.shape[1]
    if tuple(v_pages.shape) != tuple(k_pages.shape) or k_pages.shape[3] != D:
        raise ValueError("k_pages and v_pages must be [num_pages, Hkv, page_size, D] matching q")
    if block_table.shape[0] != B or seqlens.shape[0] != B:
        raise ValueError("block_table and seqlens must have B rows")
    for name, t in (("k_pages", k_pages), ("v_pages", v_pages)):
        _need_like(t, name, torch.bfloat16, k_pages.shape, q.device)
    _need_like(block_table, "block_table", torch.int32, (B, max_blocks), q.device)
    _need_like(seqlens, "seqlens", torch.int32, (B,), q.device)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    nbytes = decode_workspace_bytes(B, Hq, Hkv, max_blocks * page_size, D)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), device=q.device, dtype=torch.uint8)
    _need_workspace(workspace, "workspace", nbytes, q.device)
    o = _out(out, "out", torch.bfloat16, q.shape, q.device)
    lse = _out(lse_out, "lse_out", torch.float32, (B, Hq), q.device) if return_lse else None
    st = lib().attn_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seqlens), _ptr(o),
                                 _ptr(lse), B, Hq, Hkv, page_size, max_blocks, num_pages, D, scale, _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(q.device))
    _check(st, "attn_decode_paged")
    return o, lse


def decode_noalloc(q, kcache, vcache, seqlens, scale=None, return_lse=True, out=None, lse_out=None):
    """decode() for callers that cannot allocate device scratch: uses the
    library's fixed 16 MiB static scratch (see attn_decode_noalloc in attn.h);
    concurrent calls on one device must be serialised."""
    _need(q, "q", torch.bfloat16, 3)
    _need(kcache, "kcache", torch.bfloat16, 4)
    _need(vcache, "vcache", torch.bfloat16, 4)
    _need(seqlens, "seqlens", torch.int32, 1)
    B, Hq, D = q.shape
    Hkv, Lmax = kcache.shape[1], kcache.shape[2]
    if tuple(vcache.shape) != tuple(kcache.shape) or kcache.shape[0] != B or kcache.shape[3] != D:
        raise ValueError("kcache and vcache must be [B, Hkv, Lmax, D] matching q")
    if seqlens.shape[0] != B:
        raise ValueError("seqlens must have B entries")
    for name, t in (("kcache", kcache), ("vcache", vcache)):
        _need_like(t, name, torch.bfloat16, kcache.shape, q.device)
    _need_like(seqlens, "seqlens", torch.int32, (B,), q.device)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    o = _out(out, "out", torch.bfloat16, q.shape, q.device)
    lse = _out(lse_out, "lse_out", torch.float32, (B, Hq), q.device) if return_lse else None
    st = lib().attn_decode_noalloc(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(seqlens), _ptr(o), _ptr(lse),
                                   B, Hq, Hkv, Lmax, D, scale, _stream(q.device))
    _check(st, "attn_decode_noalloc")
    return o, lse


def fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal=False, scale=None, return_lse=True, out=None,
            lse_out=None):
    """FP8 e4m3 prefill: codes (uint8) plus one fp32 scale per 128x128 tile -> (o bf16, lse)."""
    for name, t in (("q8", q8), ("k8", k8), ("v8", v8)):
        _need(t, name, torch.uint8, 4)
    for name, t in (("q_scale", q_scale), ("k_scale", k_scale), ("v_scale", v_scale)):
        _need(t, name, torch.float32, 4)
    B, Hq, Sq, D = q8.shape
    Hkv, Sk = k8.shape[1], k8.shape[2]
    if tuple(v8.shape) != tuple(k8.shape):
        raise ValueError("k8 and v8 must have the same shape")
    nt = lambda s: -(-s // 128)  # noqa: E731
    if tuple(q_scale.shape) != (B, Hq, nt(Sq), nt(D)) or tuple(k_scale.shape) != (B, Hkv, nt(Sk), nt(D)) \
            or tuple(v_scale.shape) != (B, Hkv, nt(Sk), nt(D)):
        raise ValueError("scales must be [B, H, ceil(S/128), ceil(D/128)]")
    for name, t in (("k8", k8), ("v8", v8)):
        _need_like(t, name, torch.uint8, k8.shape, q8.device)
    for name, t in (("q_scale", q_scale), ("k_scale", k_scale), ("v_scale", v_scale)):
        _need_like(t, name, torch.float32, t.shape, q8.device)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    o = _out(out, "out", torch.bfloat16, (B, Hq, Sq, D), q8.device)
    lse = _out(lse_out, "lse_out", torch.float32, (B, Hq, Sq), q8.device) if return_lse else None
    st = lib().attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
                            _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Sk, D, 1 if causal else 0, scale,
                            _stream(q8.device))
    _check(st, "attn_fwd_fp8")
    return o, lse


def rotate_quantize_fp8(x, signs=None, codes=None, scales=None):
    """bf16 x [B,H,S,D] -> (e4m3 codes uint8 [B,H,S,D], scales fp32 [B,H,ceil(S/128),1]), D = 64 or 128.
    With signs ([D] float32 of +-1) the rows are first multiplied by H_D diag(signs) / sqrt(D)."""
    _need(x, "x", torch.bfloat16, 4)
    B, H, S, D = x.shape
    if signs is not None:
        _need(signs, "signs", torch.float32, 1)
        if signs.shape[0] != D:
            raise ValueError("signs must have D entries")
        _need_like(signs, "signs", torch.float32, (D,), x.device)
    codes = _out(codes, "codes", torch.uint8, (B, H, S, D), x.device)
    scales = _out(scales, "scales", torch.float32, (B, H, -(-S // 128), 1), x.device)
    st = lib().attn_rotate_quantize_fp8(_ptr(x), _ptr(codes), _ptr(scales), _ptr(signs), B, H, S, D,
                                        _stream(x.device))
    _check(st, "attn_rotate_quantize_fp8")
    return codes, scales


class QuantTensor(ctypes.Structure):
    """attn_quant_tensor of include/attn.h."""
    _fields_ = [("x", _P), ("codes", _P), ("scales", _P), ("B", _I), ("H", _I), ("S", _I), ("rotate", _I)]


QUANT_MAX_TENSORS = 4


def rotate_quantize_fp8_many(xs, signs=None, rotate=None, outs=None):
    """rotate_quantize_fp8 of several bf16 [B,H,S,D] tensors (one D, 64 or 128) in one launch.
    rotate[i] (default: every tensor when signs is given) says whether xs[i] is
    rotated with signs; outs[i] is a preallocated (codes, scales) pair or None.
    Returns [(codes, scales), ...] in the order of xs."""
    n = len(xs)
    if not 1 <= n <= QUANT_MAX_TENSORS:
        raise ValueError(f"between 1 and {QUANT_MAX_TENSORS} tensors")
    rotate = [signs is not None] * n if rotate is None else [bool(r) for r in rotate]
    if len(rotate) != n or (outs is not None and len(outs) != n):
        raise ValueError("rotate and outs need one entry per tensor")
    if any(rotate) and signs is None:
        raise ValueError("a rotated tensor needs signs")
    for i, x in enumerate(xs):
        _need(x, f"xs[{i}]", torch.bfloat16, 4)
        if x.device != xs[0].device:
            raise ValueError(f"xs[{i}] must be on {xs[0].device}")
        if x.shape[3] != xs[0].shape[3]:
            raise ValueError(f"xs[{i}] must have the head dimension of xs[0]")
    dev = xs[0].device
    D = int(xs[0].shape[3])
    if signs is not None:
        _need_like(signs, "signs", torch.float32, (D,), dev)
    descs = (QuantTensor * n)()
    results = []
    for i, x in enumerate(xs):
        B, H, S, D = x.shape
        c, sc = (None, None) if outs is None or outs[i] is None else outs[i]
        c = _out(c, f"codes[{i}]", torch.uint8, (B, H, S, D), dev)
        sc = _out(sc, f"scales[{i}]", torch.float32, (B, H, -(-S // 128), 1), dev)
        descs[i] = QuantTensor(x.data_ptr(), c.data_ptr(), sc.data_ptr(), B, H, S, int(rotate[i]))
        results.append((c, sc))
    st = lib().attn_rotate_quantize_fp8_many(ctypes.cast(descs, _P), n, _ptr(signs if any(rotate) else None), D,
                                             _stream(dev))
    _check(st, "attn_rotate_quantize_fp8_many")
    return results


def get_error(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device error word."""
    return int(lib().attn_get_error(_stream(device)))


def debug_stall_role_waits(enable: bool) -> None:
    """Test hook: later forward/backward calls wait for a signal nothing gives
    (bounded at 1 ms) and report ATTN_ERR_TIMEOUT; False restores them."""
    lib().attn_debug_stall_role_waits(1 if enable else 0)


def debug_skew_roles(enable: bool) -> None:
    """Test hook: later FP8 forward calls run with fixed delays in two warp
    roles, so the others run ahead of them; False restores them."""
    lib().attn_debug_skew_roles(1 if enable else 0)


def version() -> str:
    return lib().attn_version().decode()
