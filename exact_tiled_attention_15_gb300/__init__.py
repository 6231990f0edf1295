"""Exact tiled attention for GB300 (sm_103a).

    from exact_tiled_attention_15_gb300 import fwd, decode, fwd_fp8

``fwd``      bf16 prefill (causal or not, MHA/GQA/MQA) -> (O, LSE)
``fwd_host`` the same on host tensors, copies overlapped with the kernels
``bwd``      its gradients (dQ, dK, dV), recomputing P from LSE
``decode``   one query token per sequence against a KV cache -> (O, LSE)
``decode_paged``  the same against a paged KV cache (block table) -> (O, LSE)
``decode_multi``  T <= 16 query tokens per sequence (speculative verification) -> (O, LSE)
``fwd_fp8``  FP8 e4m3 prefill with one scale per 128x128 tile -> (O, LSE)
``rotate_quantize_fp8``  Hadamard rotation + per-tile e4m3 quantisation of its inputs
``rotate_quantize_fp8_many``  the same for up to four tensors (Q, K, V) in one launch
``get_error``  synchronise and read (and clear) the device error word

All of them call the C ABI of libattn.so (include/attn.h) on the current CUDA
stream; the library is loaded on first use and a missing library raises.
"""
from ._lib import ATTN_ERR_BAD_INDEX, ATTN_ERR_TIMEOUT, STATUS, AttnError, bwd, debug_skew_roles, debug_stall_role_waits, decode, decode_multi, decode_noalloc, decode_paged, decode_workspace_bytes, fwd, fwd_fp8, fwd_host, fwd_host_workspace_bytes, get_error, lib, rotate_quantize_fp8, rotate_quantize_fp8_many, version  # noqa: F401
