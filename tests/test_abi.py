"""The C ABI on the CPU: the library loads, exports every declared symbol, and
rejects bad arguments on the host before any CUDA work."""
import ctypes
import os
import re

import pytest

import exact_tiled_attention_15_gb300 as eta
from exact_tiled_attention_15_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")

INVALID, UNSUPPORTED = 1, 2
A = 0x10000  # a 16-byte aligned fake device address: never dereferenced by these calls


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z_0-9]*\s*\*?\s*(attn_[a-z_0-9]+)\s*\(", text, flags=re.M)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        from exact_tiled_attention_15_gb300.build import build
        build()
    return eta.lib()


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    assert {"attn_fwd", "attn_decode", "attn_decode_workspace_bytes", "attn_fwd_fp8", "attn_get_error",
            "attn_status_str", "attn_version"} <= names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(_lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), name
    assert set(declared_functions()) <= set(_lib.SIGNATURES)


def test_status_strings(lib):
    for code, name in _lib.STATUS.items():
        assert lib.attn_status_str(code).decode() == name
    assert lib.attn_version().decode().count(".") == 2


def test_status_table_matches_header_enum():
    """The binding's status table is the header's attn_status enum, value for value."""
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    enum = text[text.index("typedef enum"):text.index("} attn_status;")]
    declared = {int(v): n for n, v in re.findall(r"(ATTN_\w+)\s*=\s*(\d+)", enum)}
    assert declared == _lib.STATUS
    assert (_lib.ATTN_ERR_TIMEOUT, _lib.ATTN_ERR_BAD_INDEX) == (4, 7)


def p(x):
    return ctypes.c_void_p(x)


def fwd(lib, q=A, k=A, v=A, o=A, lse=None, B=1, Hq=2, Hkv=2, Sq=128, Sk=128, D=128, causal=0, scale=0.1):
    return lib.attn_fwd(p(q), p(k), p(v), p(o), p(lse), B, Hq, Hkv, Sq, Sk, D, causal, scale, None)


def test_fwd_rejects_bad_arguments_on_host(lib):
    assert fwd(lib, q=0) == INVALID
    assert fwd(lib, o=0) == INVALID
    assert fwd(lib, Hq=3, Hkv=2) == INVALID
    assert fwd(lib, B=0) == INVALID
    assert fwd(lib, Sq=0) == INVALID
    assert fwd(lib, Sk=-1) == INVALID
    assert fwd(lib, scale=0.0) == INVALID
    assert fwd(lib, scale=float("nan")) == INVALID
    assert fwd(lib, scale=float("inf")) == INVALID
    assert fwd(lib, k=A + 8) == INVALID          # misaligned for TMA
    assert fwd(lib, lse=A + 2) == INVALID
    assert fwd(lib, D=96) == UNSUPPORTED
    assert fwd(lib, D=256) == UNSUPPORTED


def fp8(lib, D=128, qs=A, Hq=2, Hkv=2):
    return lib.attn_fwd_fp8(p(A), p(A), p(A), p(qs), p(A), p(A), p(A), None, 1, Hq, Hkv, 256, 256, D, 0, 0.1, None)


def test_fp8_rejects_bad_arguments_on_host(lib):
    assert fp8(lib, qs=0) == INVALID
    assert fp8(lib, qs=A + 2) == INVALID
    assert fp8(lib, Hq=4, Hkv=3) == INVALID
    assert fp8(lib, D=96) == UNSUPPORTED  # D in {64, 128}
    assert fp8(lib, D=256) == UNSUPPORTED


def test_decode_workspace_and_validation(lib):
    n = lib.attn_decode_workspace_bytes(64, 32, 8, 8192, 128)
    assert n > 0 and n % 4 == 0
    assert lib.attn_decode_workspace_bytes(0, 32, 8, 8192, 128) == 0
    assert lib.attn_decode_workspace_bytes(2, 6, 4, 100, 128) == 0  # Hq % Hkv != 0
    # workspace grows with Lmax and with the number of query heads
    assert lib.attn_decode_workspace_bytes(64, 32, 8, 16384, 128) >= n
    assert lib.attn_decode_workspace_bytes(64, 64, 8, 8192, 128) > n

    def dec(ws=A, wsb=n, seq=A, D=128, Hq=32, Hkv=8, scale=0.1):
        return lib.attn_decode(p(A), p(A), p(A), p(seq), p(A), None, 64, Hq, Hkv, 8192, D, scale, p(ws), wsb, None)

    assert dec(ws=0) == INVALID
    assert dec(wsb=n - 1) == INVALID
    assert dec(ws=A + 16) == INVALID       # workspace must be 256-byte aligned
    assert dec(seq=0) == INVALID
    assert dec(seq=A + 1) == INVALID
    assert dec(Hq=30) == INVALID
    assert dec(scale=-1.0) == INVALID
    m = lib.attn_decode_workspace_bytes(64, 32, 8, 8192, 80)
    assert lib.attn_decode(p(A), p(A), p(A), p(A), p(A), None, 64, 32, 8, 8192, 80, 0.1, p(A), m, None) == UNSUPPORTED


def test_python_binding_rejects_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        eta.fwd(q, q, q)
    with pytest.raises((TypeError, ValueError)):
        eta.fwd(q.float(), q, q)
    with pytest.raises(TypeError):
        eta.fwd("q", q, q)


def test_decode_paged_validation(lib):
    n = lib.attn_decode_workspace_bytes(4, 8, 2, 16 * 64, 128)

    def dec(ps=64, table=A, mb=16, npages=40, wsb=n, D=128):
        return lib.attn_decode_paged(p(A), p(A), p(A), p(table), p(A), p(A), None, 4, 8, 2, ps, mb, npages, D, 0.1,
                                     p(A), wsb, None)

    assert dec(table=0) == INVALID
    assert dec(table=A + 2) == INVALID
    assert dec(npages=0) == INVALID
    assert dec(wsb=n - 1) == INVALID
    assert dec(ps=48, mb=20, wsb=lib.attn_decode_workspace_bytes(4, 8, 2, 48 * 20, 128)) == UNSUPPORTED
    assert dec(D=80, wsb=lib.attn_decode_workspace_bytes(4, 8, 2, 1024, 80)) == UNSUPPORTED


def test_bwd_validation(lib):
    n = lib.attn_bwd_workspace_bytes(1, 2, 128, 128)
    assert n > 0 and lib.attn_bwd_workspace_bytes(0, 2, 128, 128) == 0

    def bwd(lse=A, ws=A, wsb=n, D=128, Hkv=2):
        return lib.attn_bwd(p(A), p(A), p(A), p(A), p(lse), p(A), p(A), p(A), p(A), 1, 2, Hkv, 128, 128, D, 1, 0.1,
                            p(ws), wsb, None)

    assert bwd(lse=0) == INVALID
    assert bwd(ws=A + 64) == INVALID
    assert bwd(wsb=n - 1) == INVALID
    assert bwd(Hkv=3) == INVALID
    assert bwd(D=96, wsb=lib.attn_bwd_workspace_bytes(1, 2, 128, 96)) == UNSUPPORTED  # D in {64, 128}


def test_fwd_host_validation(lib):
    """The host-buffer forward checks its arguments before any CUDA call; its
    workspace holds three chunk buffers of whole (batch, KV head) units."""
    n = lib.attn_fwd_host_workspace_bytes(2, 32, 32, 4096, 4096, 128)
    assert n > 0 and lib.attn_fwd_host_workspace_bytes(2, 32, 3, 4096, 4096, 128) == 0
    assert lib.attn_fwd_host_workspace_bytes(0, 32, 32, 4096, 4096, 128) == 0
    # more units never need less scratch, and a unit is at least the bytes of its Q, K, V, O, LSE
    assert lib.attn_fwd_host_workspace_bytes(4, 32, 32, 4096, 4096, 128) >= n
    unit = 4096 * 128 * 2 * 4 + 4096 * 4
    assert n >= 3 * unit

    def host(q=A, ws=A, wsb=n, Hkv=32, D=128):
        return lib.attn_fwd_host(p(q), p(A), p(A), p(A), p(A), 2, 32, Hkv, 4096, 4096, D, 1, 0.1, p(ws), wsb, None)

    assert host(q=0) == INVALID
    assert host(ws=0) == INVALID
    assert host(ws=A + 16) == INVALID
    assert host(wsb=n - 1) == INVALID
    assert host(Hkv=3) == INVALID
    assert host(D=96, wsb=lib.attn_fwd_host_workspace_bytes(2, 32, 32, 4096, 4096, 96)) == UNSUPPORTED


def test_rotate_quantize_many_validation(lib):
    """The multi-tensor quantise call checks every descriptor on the host."""
    T = _lib.QuantTensor

    def many(items, n=None, signs=A, D=128):
        arr = (T * max(1, len(items)))(*items)
        return lib.attn_rotate_quantize_fp8_many(ctypes.cast(arr, ctypes.c_void_p), len(items) if n is None else n,
                                                 p(signs), D, None)

    good = T(A, A, A, 2, 4, 300, 1)
    assert many([good], n=0) == INVALID
    assert lib.attn_rotate_quantize_fp8_many(None, 1, p(A), 128, None) == INVALID
    assert many([good] * 5) == UNSUPPORTED                    # more than ATTN_QUANT_MAX_TENSORS
    assert many([good, T(0, A, A, 2, 4, 300, 0)]) == INVALID  # NULL input
    assert many([good, T(A, A + 8, A, 2, 4, 300, 0)]) == INVALID  # codes not 16-byte aligned
    assert many([good, T(A, A, A + 2, 2, 4, 300, 0)]) == INVALID  # scales not 4-byte aligned
    assert many([good, T(A, A, A, 2, 0, 300, 0)]) == INVALID   # H < 1
    assert many([good], signs=0) == INVALID                      # a rotated tensor needs signs
    assert many([good], signs=A + 2) == INVALID
    assert many([good], D=96) == UNSUPPORTED  # D in {64, 128}
    assert many([T(A, A, A, 1 << 16, 1 << 15, 128, 0)], signs=0) == UNSUPPORTED  # B * H > 2^30
